// nq_kv.cu -- the nested KV cache: appending quantised K/V rows, and decode
// attention that reads the 4-bit base view (draft) or the full 8-bit view
// (verify) of the same cache.
//
// BitNest, Fig. 4 ("KV nesting during speculative decoding"): the draft stage
// reads only the low-bit base view of the cache, verification reads the full
// b_kv + r_kv-bit view, accepted entries stay and the rejected suffix is
// discarded; Fig. 5 and Tables 9-11: reading the KV4 base while drafting is
// what pays at long context.  Each K or V row of head_dim values is quantised
// exactly like a NESTED44 weight row (groups of `group` values along the head
// dimension, s = fp16(absmax / 7), base q4 and refinement r), so the draft
// value of an element is s q4 and the target value (s / 16)(16 q4 + r).
//
// Attention (one launch + a combine): the cache rows of a (sequence, kv head)
// are cut into 256-row splits; a CTA of four warps takes one split and up to
// eight query vectors (query heads sharing the kv head, times query rows).
// Scores: lane t of a warp owns cache row t of a 32-row block and dots its
// decoded K row with the query vectors (held in shared memory); online
// softmax per query vector across the blocks; values: the two half-warps take
// alternate rows of the block, each lane 8 consecutive dimensions of the
// decoded V row.  The splits' (max, sum, output) partials are merged by a
// second kernel.  The cache rows are streamed once per CTA group (query-vector
// groups of one split run side by side and share them in L2).
#include "nq_internal.cuh"

namespace nq {
namespace {

constexpr int kKvWarps = 4;
constexpr int kSplit = 256;                 // cache rows per CTA
constexpr int kQvCap = 8;                   // query vectors per CTA at most
constexpr int kAppendWarps = 8;

struct Cache {
    int B, H, d, G, L;
    const uint8_t *kb, *kr, *vb, *vr;
    const __half *ks, *vs;
};

// Quantise row (b, h, i) of the new K or V rows (one warp per (row, group)).
template <int G>
__global__ void __launch_bounds__(kAppendWarps * 32)
kv_append_kernel(const float *__restrict__ src, int B, int H, int n_new, int d, int L, const int32_t *__restrict__ pos,
                 uint8_t *__restrict__ base, uint8_t *__restrict__ resid, __half *__restrict__ scales,
                 unsigned int *status)
{
    constexpr int E = G / 32;
    const int gpr = d / G;
    const long long job = static_cast<long long>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
    if (job >= static_cast<long long>(B) * H * n_new * gpr) return;
    const int lane = threadIdx.x & 31;
    const int grp = static_cast<int>(job % gpr);
    const long long rowi = job / gpr;                     // (b, h, i)
    const int i = static_cast<int>(rowi % n_new);
    const int h = static_cast<int>((rowi / n_new) % H);
    const int b = static_cast<int>(rowi / (static_cast<long long>(n_new) * H));
    const int t = pos[b] + i;
    if (t < 0 || t >= L) {
        if (lane == 0) set_status(status, NQ_DEV_SEQ_FULL);
        return;
    }
    const float *w = src + rowi * d + static_cast<size_t>(grp) * G + lane * E;
    float v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = w[e];
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const __half sh = __float2half_rn(__fdiv_rn(amax, 7.0f));
    const float s = __half2float(sh);
    uint32_t bb = 0, rr = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        int q4, r;
        nested_quantise(v[e], s, q4, r);
        bb |= static_cast<uint32_t>(q4 & 15) << (4 * e);
        rr |= static_cast<uint32_t>(r & 15) << (4 * e);
    }
    const size_t row = (static_cast<size_t>(b) * H + h) * L + t;
    const size_t off = row * (d / 2) + static_cast<size_t>(grp) * (G / 2) + lane * (E / 2);
    if (E == 4) {
        *reinterpret_cast<uint16_t *>(base + off) = static_cast<uint16_t>(bb);
        *reinterpret_cast<uint16_t *>(resid + off) = static_cast<uint16_t>(rr);
    } else {
        base[off] = static_cast<uint8_t>(bb);
        resid[off] = static_cast<uint8_t>(rr);
    }
    if (lane == 0) scales[row * gpr + grp] = sh;
}

// Element values of one 32-bit word per plane (8 consecutive elements, element
// 2j in the low nibble of byte j): s q4 (PLANES == 1) or (s / 16)(16 q4 + r).
template <int PLANES>
__device__ __forceinline__ void decode8(uint32_t bw, uint32_t rw, float s, float (&o)[8])
{
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int q4 = static_cast<int>(bw << (28 - 4 * e)) >> 28;
        if constexpr (PLANES == 2) {
            const int r = static_cast<int>(rw << (28 - 4 * e)) >> 28;
            o[e] = __fmul_rn(__fmul_rn(s, 0.0625f), static_cast<float>(16 * q4 + r));
        } else {
            o[e] = __fmul_rn(s, static_cast<float>(q4));
        }
    }
}

// Partial attention of one split of cache rows for up to kQvMax query vectors.
// Query vector v (0..nqv-1 of this CTA's group) = (query row m, query head hq)
// with hq = kvh * g + (v' % g), m = v' / g for v' = qv0 + v.
template <int PLANES, int D, int QV>
__global__ void __launch_bounds__(kKvWarps * 32)
attn_split_kernel(Cache C, const float *__restrict__ q, int M, int Hq, const int32_t *__restrict__ len, float scale,
                  float *__restrict__ part, int nsplit)
{
    static_assert(D == 128 || D == 64, "head_dim 64 or 128");
    constexpr int kQvMax = QV;                // query vectors per CTA (1, 2, 4 or 8)
    constexpr int DW = D / 8;                 // 32-bit words per plane per row
    const int g = Hq / C.H, nq_all = M * g, qgroups = (nq_all + QV - 1) / QV;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z / qgroups, qg = blockIdx.z % qgroups;
    const int qv0 = qg * kQvMax, nqv = min(kQvMax, nq_all - qv0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ __align__(16) float qs[kQvMax][D];
    __shared__ float red_m[kKvWarps][kQvMax], red_l[kKvWarps][kQvMax];
    __shared__ __align__(16) float red_o[kKvWarps][kQvMax][D];
    const int Lb = min(len[b], C.L);
    int lim[kQvMax];                          // rows < lim[v] are visible to query vector v
#pragma unroll
    for (int v = 0; v < kQvMax; ++v) {
        const int vv = qv0 + (v < nqv ? v : 0);
        const int m = vv / g;
        lim[v] = v < nqv ? Lb - (M - 1 - m) : 0;
    }
    for (int i = threadIdx.x; i < kQvMax * D; i += kKvWarps * 32) {
        const int v = i / D, j = i % D;
        float x = 0.0f;
        if (v < nqv) {
            const int vv = qv0 + v, m = vv / g, hq = kvh * g + vv % g;
            x = __fmul_rn(q[((static_cast<size_t>(b) * M + m) * Hq + hq) * D + j], scale);
        }
        qs[v][j] = x;
    }
    __syncthreads();

    const size_t rowbase = (static_cast<size_t>(b) * C.H + kvh) * C.L;
    const int gpr = D / C.G;
    float mrun[kQvMax], lrun[kQvMax], acc[kQvMax][8];
#pragma unroll
    for (int v = 0; v < kQvMax; ++v) {
        mrun[v] = -INFINITY;
        lrun[v] = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[v][e] = 0.0f;
    }
    const int t_begin = split * kSplit, t_end = min(t_begin + kSplit, Lb);
    constexpr int LPR = D / 8, RPS = 32 / LPR;           // values: lanes per row, rows per step
    const int half = lane / LPR, dl = lane % LPR;        // row offset within a step, dims 8 dl .. 8 dl + 7
    for (int tb = t_begin + 32 * warp; tb < t_end; tb += 32 * kKvWarps) {
        // ---- scores: lane = cache row tb + lane
        const int t = tb + lane;
        float sc[kQvMax];
#pragma unroll
        for (int v = 0; v < kQvMax; ++v) sc[v] = 0.0f;
        if (t < t_end) {
            const uint4 *kb4 = reinterpret_cast<const uint4 *>(C.kb + (rowbase + t) * (D / 2));
            const uint4 *kr4 = reinterpret_cast<const uint4 *>(C.kr + (rowbase + t) * (D / 2));
#pragma unroll
            for (int c4 = 0; c4 < DW / 4; ++c4) {
                const uint4 bw = __ldg(kb4 + c4);
                const uint4 rw = PLANES == 2 ? __ldg(kr4 + c4) : make_uint4(0, 0, 0, 0);
                const uint32_t bws[4] = {bw.x, bw.y, bw.z, bw.w}, rws[4] = {rw.x, rw.y, rw.z, rw.w};
#pragma unroll
                for (int w4 = 0; w4 < 4; ++w4) {
                    const int e0 = 8 * (4 * c4 + w4);
                    const float s = __half2float(C.ks[(rowbase + t) * gpr + e0 / C.G]);
                    float kv[8];
                    decode8<PLANES>(bws[w4], rws[w4], s, kv);
#pragma unroll
                    for (int v = 0; v < kQvMax; ++v) {
                        const float4 qa = *reinterpret_cast<const float4 *>(&qs[v][e0]);
                        const float4 qb = *reinterpret_cast<const float4 *>(&qs[v][e0 + 4]);
                        float a = sc[v];
                        a = fmaf(qa.x, kv[0], a); a = fmaf(qa.y, kv[1], a); a = fmaf(qa.z, kv[2], a);
                        a = fmaf(qa.w, kv[3], a); a = fmaf(qb.x, kv[4], a); a = fmaf(qb.y, kv[5], a);
                        a = fmaf(qb.z, kv[6], a); a = fmaf(qb.w, kv[7], a);
                        sc[v] = a;
                    }
                }
            }
        }
        // ---- online softmax per query vector (rows beyond a vector's limit: -inf)
        float p[kQvMax];
#pragma unroll
        for (int v = 0; v < kQvMax; ++v) {
            const float s = (t < t_end && t < lim[v]) ? sc[v] : -INFINITY;
            float mb = s;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
            const float mn = fmaxf(mrun[v], mb);
            const float alpha = mn == -INFINITY ? 1.0f : __expf(mrun[v] - mn);
            p[v] = mn == -INFINITY ? 0.0f : __expf(s - mn);
            float ps = p[v];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            lrun[v] = fmaf(lrun[v], alpha, ps);
            mrun[v] = mn;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[v][e] *= alpha;
        }
        // ---- values: row tb + RPS i + half, dims 8 dl .. 8 dl + 7
        const int nrow = min(32, t_end - tb);
        for (int i = 0; RPS * i < nrow; ++i) {
            const int r = RPS * i + half;
            const int tt = tb + r;
            float vv[8];
            if (r < nrow) {
                const size_t row = rowbase + tt;
                const uint32_t bw = __ldg(reinterpret_cast<const uint32_t *>(C.vb + row * (D / 2)) + dl);
                const uint32_t rw = PLANES == 2 ? __ldg(reinterpret_cast<const uint32_t *>(C.vr + row * (D / 2)) + dl) : 0u;
                decode8<PLANES>(bw, rw, __half2float(C.vs[row * gpr + (8 * dl) / C.G]), vv);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) vv[e] = 0.0f;
            }
#pragma unroll
            for (int v = 0; v < kQvMax; ++v) {
                const float pr = __shfl_sync(0xffffffffu, p[v], r < 32 ? r : 0);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[v][e] = fmaf(pr, vv[e], acc[v][e]);
            }
        }
    }
    // ---- merge the row groups of the warp, then the warps of the CTA
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
        for (int v = 0; v < kQvMax; ++v)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[v][e] += __shfl_xor_sync(0xffffffffu, acc[v][e], o);
    if (lane == 0)
        for (int v = 0; v < kQvMax; ++v) { red_m[warp][v] = mrun[v]; red_l[warp][v] = lrun[v]; }
    if (half == 0)
        for (int v = 0; v < kQvMax; ++v)
#pragma unroll
            for (int e = 0; e < 8; ++e) red_o[warp][v][8 * dl + e] = acc[v][e];
    __syncthreads();
    for (int i = threadIdx.x; i < nqv * (D + 2); i += kKvWarps * 32) {
        const int v = i / (D + 2), j = i % (D + 2);
        float M2 = -INFINITY;
        for (int w = 0; w < kKvWarps; ++w) M2 = fmaxf(M2, red_m[w][v]);
        float val = 0.0f;
        if (j == D) {
            val = M2;
        } else {
            for (int w = 0; w < kKvWarps; ++w) {
                const float f = red_m[w][v] == -INFINITY ? 0.0f : __expf(red_m[w][v] - M2);
                val += f * (j == D + 1 ? red_l[w][v] : red_o[w][v][j]);
            }
        }
        const int vv = qv0 + v, m = vv / g, hq = kvh * g + vv % g;
        part[((((static_cast<size_t>(b) * M + m) * Hq + hq) * nsplit) + split) * (D + 2) + j] = val;
    }
}

// out[b][m][hq][:] = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s over the splits.
template <int D>
__global__ void __launch_bounds__(D)
attn_combine_kernel(const float *__restrict__ part, int nsplit, float *__restrict__ out)
{
    const size_t vec = blockIdx.x;            // (b, m, hq)
    const float *p = part + vec * nsplit * (D + 2);
    float M2 = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M2 = fmaxf(M2, p[static_cast<size_t>(s) * (D + 2) + D]);
    float num = 0.0f, den = 0.0f;
    for (int s = 0; s < nsplit; ++s) {
        const float ms = p[static_cast<size_t>(s) * (D + 2) + D];
        if (ms == -INFINITY) continue;
        const float f = __expf(ms - M2);
        num = fmaf(f, p[static_cast<size_t>(s) * (D + 2) + threadIdx.x], num);
        den = fmaf(f, p[static_cast<size_t>(s) * (D + 2) + D + 1], den);
    }
    out[vec * D + threadIdx.x] = den > 0.0f ? num / den : 0.0f;
}

template <int PLANES, int D>
void launch_attn_qv(int qv, dim3 grid, cudaStream_t s, Cache C, const float *q, int M, int Hq, const int32_t *len,
                    float scale, float *part, int nsplit)
{
    switch (qv) {
    case 1: attn_split_kernel<PLANES, D, 1><<<grid, kKvWarps * 32, 0, s>>>(C, q, M, Hq, len, scale, part, nsplit); break;
    case 2: attn_split_kernel<PLANES, D, 2><<<grid, kKvWarps * 32, 0, s>>>(C, q, M, Hq, len, scale, part, nsplit); break;
    case 4: attn_split_kernel<PLANES, D, 4><<<grid, kKvWarps * 32, 0, s>>>(C, q, M, Hq, len, scale, part, nsplit); break;
    default: attn_split_kernel<PLANES, D, kQvCap><<<grid, kKvWarps * 32, 0, s>>>(C, q, M, Hq, len, scale, part, nsplit); break;
    }
}
void launch_attn(int planes, int d, int qv, dim3 grid, cudaStream_t s, Cache C, const float *q, int M, int Hq,
                 const int32_t *len, float scale, float *part, int nsplit)
{
    if (d == 128) {
        if (planes == 1) launch_attn_qv<1, 128>(qv, grid, s, C, q, M, Hq, len, scale, part, nsplit);
        else launch_attn_qv<2, 128>(qv, grid, s, C, q, M, Hq, len, scale, part, nsplit);
    } else {
        if (planes == 1) launch_attn_qv<1, 64>(qv, grid, s, C, q, M, Hq, len, scale, part, nsplit);
        else launch_attn_qv<2, 64>(qv, grid, s, C, q, M, Hq, len, scale, part, nsplit);
    }
}

nq_status check_cache(const nq_kv_cache *c)
{
    if (!c || c->batch < 1 || c->heads_kv < 1 || c->max_len < 1) return NQ_ERR_ARG;
    if (!(c->head_dim == 64 || c->head_dim == 128) || !(c->group == 64 || c->group == 128) || c->group > c->head_dim)
        return NQ_ERR_SHAPE;
    if (!c->k_base || !c->k_resid || !c->k_scales || !c->v_base || !c->v_resid || !c->v_scales) return NQ_ERR_ARG;
    if (!aligned16(c->k_base) || !aligned16(c->k_resid) || !aligned16(c->k_scales) || !aligned16(c->v_base) ||
        !aligned16(c->v_resid) || !aligned16(c->v_scales))
        return NQ_ERR_ALIGN;
    return NQ_OK;
}

int n_splits(int max_len) { return (max_len + kSplit - 1) / kSplit; }

}  // namespace
}  // namespace nq

extern "C" nq_status nq_kv_cache_bytes(int batch, int heads_kv, int head_dim, int group, int max_len,
                                       size_t *plane_bytes, size_t *scale_bytes)
{
    if (batch < 1 || heads_kv < 1 || max_len < 1) return NQ_ERR_ARG;
    if (!(head_dim == 64 || head_dim == 128) || !(group == 64 || group == 128) || group > head_dim) return NQ_ERR_SHAPE;
    const size_t rows = static_cast<size_t>(batch) * heads_kv * max_len;
    if (plane_bytes) *plane_bytes = rows * (head_dim / 2);
    if (scale_bytes) *scale_bytes = rows * (head_dim / group) * 2;
    return NQ_OK;
}

extern "C" nq_status nq_kv_append(const nq_kv_cache *cache, const float *k_new, const float *v_new, int n_new,
                                  const int32_t *pos, cudaStream_t stream)
{
    nq_status st = nq::check_cache(cache);
    if (st != NQ_OK) return st;
    if (!k_new || !v_new || !pos || n_new < 1 || n_new > cache->max_len) return NQ_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(k_new) & 15u) || (reinterpret_cast<uintptr_t>(v_new) & 15u) ||
        (reinterpret_cast<uintptr_t>(pos) & 3u))
        return NQ_ERR_ALIGN;
    unsigned int *status = nq::device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    const nq_kv_cache &c = *cache;
    const long long jobs = static_cast<long long>(c.batch) * c.heads_kv * n_new * (c.head_dim / c.group);
    const int grid = static_cast<int>((jobs + nq::kAppendWarps - 1) / nq::kAppendWarps);
    for (int which = 0; which < 2; ++which) {
        const float *src = which ? v_new : k_new;
        auto *base = static_cast<uint8_t *>(which ? c.v_base : c.k_base);
        auto *resid = static_cast<uint8_t *>(which ? c.v_resid : c.k_resid);
        auto *sc = static_cast<__half *>(which ? c.v_scales : c.k_scales);
        if (c.group == 128)
            nq::kv_append_kernel<128><<<grid, nq::kAppendWarps * 32, 0, stream>>>(
                src, c.batch, c.heads_kv, n_new, c.head_dim, c.max_len, pos, base, resid, sc, status);
        else
            nq::kv_append_kernel<64><<<grid, nq::kAppendWarps * 32, 0, stream>>>(
                src, c.batch, c.heads_kv, n_new, c.head_dim, c.max_len, pos, base, resid, sc, status);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return NQ_ERR_CUDA;
    }
    return NQ_OK;
}

extern "C" size_t nq_attn_workspace_bytes(int batch, int M, int heads_q, int head_dim, int max_len)
{
    if (batch < 1 || M < 1 || heads_q < 1 || max_len < 1 || !(head_dim == 64 || head_dim == 128)) return 0;
    return static_cast<size_t>(batch) * M * heads_q * nq::n_splits(max_len) * (head_dim + 2) * sizeof(float);
}

extern "C" nq_status nq_attn_decode(const nq_kv_cache *cache, const float *q, int M, int heads_q, const int32_t *len,
                                    int planes, float scale, float *out, void *ws, size_t ws_bytes,
                                    cudaStream_t stream)
{
    nq_status st = nq::check_cache(cache);
    if (st != NQ_OK) return st;
    const nq_kv_cache &c = *cache;
    if (!q || !len || !out || M < 1 || M > c.max_len || heads_q < c.heads_kv || heads_q % c.heads_kv != 0 ||
        (planes != 1 && planes != 2) || !(scale > 0.0f))
        return NQ_ERR_ARG;
    if (!nq::aligned16(q) || !nq::aligned16(out) || (reinterpret_cast<uintptr_t>(len) & 3u)) return NQ_ERR_ALIGN;
    if (!ws || ws_bytes < nq_attn_workspace_bytes(c.batch, M, heads_q, c.head_dim, c.max_len)) return NQ_ERR_WORKSPACE;
    if (!nq::aligned16(ws)) return NQ_ERR_ALIGN;
    const int nsplit = nq::n_splits(c.max_len);
    const int g = heads_q / c.heads_kv, nq_all = M * g;
    const int qv = nq_all <= 1 ? 1 : (nq_all <= 2 ? 2 : (nq_all <= 4 ? 4 : nq::kQvCap));
    const int qgroups = (nq_all + qv - 1) / qv;
    if (static_cast<long long>(c.batch) * qgroups > 65535) return NQ_ERR_SHAPE;
    nq::Cache C{c.batch, c.heads_kv, c.head_dim, c.group, c.max_len,
                static_cast<const uint8_t *>(c.k_base), static_cast<const uint8_t *>(c.k_resid),
                static_cast<const uint8_t *>(c.v_base), static_cast<const uint8_t *>(c.v_resid),
                static_cast<const __half *>(c.k_scales), static_cast<const __half *>(c.v_scales)};
    float *part = static_cast<float *>(ws);
    dim3 grid(nsplit, c.heads_kv, c.batch * qgroups);
    nq::launch_attn(planes, c.head_dim, qv, grid, stream, C, q, M, heads_q, len, scale, part, nsplit);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return NQ_ERR_CUDA;
    const int nvec = c.batch * M * heads_q;
    if (c.head_dim == 128) nq::attn_combine_kernel<128><<<nvec, 128, 0, stream>>>(part, nsplit, out);
    else nq::attn_combine_kernel<64><<<nvec, 64, 0, stream>>>(part, nsplit, out);
    return nq::cuda_status(cudaGetLastError());
}
