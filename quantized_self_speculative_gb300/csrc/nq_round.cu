// nq_round.cu -- round bookkeeping of speculative decoding: the tokens a pass
// consumes become its input rows, the draft's greedy choice becomes the next
// drafted token, and the tokens a round emits extend the sequence.
//
// "How Speculative Decoding Speeds Up Inference", "Drafting and checking
// tokens": the draft proposes k tokens one at a time (each from the previous
// one), the target checks all of them in one pass over k+1 positions, the
// matching prefix is kept and the target's token replaces the first
// mismatch; that token starts the next round.  BitNest, Fig. 4 / "KV cache
// nesting": the entries the verify pass computed for the rejected suffix are
// discarded, so the cache keeps the first out_cnt of the k+1 positions.
//
// All of it is device-side so that a whole round (k draft passes, one verify
// pass, acceptance and commit) can be queued, or captured in a CUDA graph,
// with no host round trip.
#include "nq_internal.cuh"

namespace nq {
namespace {

constexpr int kEmbedThreads = 128;

// One CTA per output row: 16-byte copies of the table row (d % 8 == 0).
__global__ void __launch_bounds__(kEmbedThreads)
embed_kernel(const uint16_t *__restrict__ table, int V, int d, const int32_t *__restrict__ ids, int ids_stride,
             const int32_t *__restrict__ x0, int k, uint16_t *__restrict__ out, unsigned int *status)
{
    const int m = blockIdx.x;
    int id;
    if (x0) {   // round layout: row m = b (k+1) + j takes x0[b] at j = 0, ids[b k + j - 1] after
        const int b = m / (k + 1), j = m % (k + 1);
        id = j == 0 ? x0[b] : ids[static_cast<size_t>(b) * k + (j - 1)];
    } else {
        id = ids[static_cast<size_t>(m) * ids_stride];
    }
    const bool ok = id >= 0 && id < V;
    if (!ok && threadIdx.x == 0) set_status(status, NQ_DEV_BAD_TOKEN);
    const uint4 *src = reinterpret_cast<const uint4 *>(table + static_cast<size_t>(ok ? id : 0) * d);
    uint4 *dst = reinterpret_cast<uint4 *>(out + static_cast<size_t>(m) * d);
    for (int i = threadIdx.x; i < d / 8; i += kEmbedThreads) dst[i] = ok ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
}

// One thread per row: append the emitted tokens, advance the length, set the
// next round's first input token.
__global__ void commit_kernel(const int32_t *__restrict__ out_tok, const int32_t *__restrict__ out_cnt, int B, int k,
                              int32_t *__restrict__ seq, int32_t *__restrict__ seq_len, int max_len,
                              int32_t *__restrict__ x0, unsigned int *status)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int c = out_cnt[b];
    if (c < 1 || c > k + 1) {          // not the output of an acceptance call: nothing is appended
        set_status(status, NQ_DEV_BAD_TOKEN);
        return;
    }
    const int L = seq_len[b];
    const int room = max_len - L > 0 ? max_len - L : 0;
    const int n = c < room ? c : room;
    if (n < c) set_status(status, NQ_DEV_SEQ_FULL);
    for (int i = 0; i < n; ++i)
        seq[static_cast<size_t>(b) * max_len + L + i] = out_tok[static_cast<size_t>(b) * (k + 1) + i];
    seq_len[b] = L + n;
    x0[b] = out_tok[static_cast<size_t>(b) * (k + 1) + c - 1];
}

inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace nq

extern "C" nq_status nq_embed_rows(const uint16_t *table, int V, int d, const int32_t *ids, int ids_stride, int M,
                                   uint16_t *out, cudaStream_t stream)
{
    if (!table || !ids || !out || V < 1 || d < 8 || d % 8 != 0 || M < 1 || M > (1 << 24) || ids_stride < 1)
        return NQ_ERR_ARG;
    if (!nq::aligned16(table) || !nq::aligned16(out) || !nq::aligned4(ids)) return NQ_ERR_ALIGN;
    unsigned int *status = nq::device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    nq::embed_kernel<<<M, nq::kEmbedThreads, 0, stream>>>(table, V, d, ids, ids_stride, nullptr, 0, out, status);
    return nq::cuda_status(cudaGetLastError());
}

extern "C" nq_status nq_embed_round(const uint16_t *table, int V, int d, const int32_t *x0, const int32_t *draft,
                                    int B, int k, uint16_t *out, cudaStream_t stream)
{
    if (!table || !x0 || !out || V < 1 || d < 8 || d % 8 != 0 || B < 1 || k < 0 || k > 16 || (k > 0 && !draft) ||
        static_cast<long long>(B) * (k + 1) > (1 << 24))
        return NQ_ERR_ARG;
    if (!nq::aligned16(table) || !nq::aligned16(out) || !nq::aligned4(x0) || (draft && !nq::aligned4(draft)))
        return NQ_ERR_ALIGN;
    unsigned int *status = nq::device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    nq::embed_kernel<<<B * (k + 1), nq::kEmbedThreads, 0, stream>>>(table, V, d, draft, 1, x0, k, out, status);
    return nq::cuda_status(cudaGetLastError());
}

extern "C" nq_status spec_round_commit(const int32_t *out_tok, const int32_t *out_cnt, int B, int k, int32_t *seq,
                                       int32_t *seq_len, int max_len, int32_t *x0, cudaStream_t stream)
{
    if (!out_tok || !out_cnt || !seq || !seq_len || !x0 || B < 1 || B > 65535 || k < 0 || k > 16 || max_len < 1)
        return NQ_ERR_ARG;
    if (!nq::aligned4(out_tok) || !nq::aligned4(out_cnt) || !nq::aligned4(seq) || !nq::aligned4(seq_len) ||
        !nq::aligned4(x0))
        return NQ_ERR_ALIGN;
    unsigned int *status = nq::device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    nq::commit_kernel<<<(B + 255) / 256, 256, 0, stream>>>(out_tok, out_cnt, B, k, seq, seq_len, max_len, x0, status);
    return nq::cuda_status(cudaGetLastError());
}
