// nq_accept.cu -- the verification step of a speculative round: which
// drafted tokens to keep.
//
// "How Speculative Decoding Speeds Up Inference": draft k tokens, check all k
// positions in one target pass, keep the matching prefix, the target's token
// replaces the first mismatch, 1..k+1 tokens per pass (Table 1); with
// sampling, accept each draft token with probability min(1, p/q) and after a
// rejection resample from normalise(max(0, p - q)) (Leviathan et al.; Chen et
// al.), which follows the target distribution exactly.
//
// Design: one pass over the logits.  The grid is (chunk of 4096 entries,
// vector, row); every CTA reduces its chunk and writes a partial to the
// workspace; the last CTA of a row (atomic ticket, no spin-waits) combines the
// partials, decides, and -- for sampling -- draws the replacement / bonus
// token from the two vectors of the chosen position, which are still warm in
// L2.  All fp32 arithmetic of the sampled path follows the fixed recipe
// documented in nq.h so that decisions are reproducible bit for bit.
#include <algorithm>
#include <mutex>

#include "nq_internal.cuh"

namespace nq {
namespace {

constexpr int kThreads = 256;
constexpr int kLeaf = 16;
constexpr int kChunk = kThreads * kLeaf;     // vocabulary entries per workspace partial slot
constexpr int kGreedyChunk = 4 * kChunk;     // vocabulary entries per greedy CTA
constexpr int kMaxChunks = 128;              // V <= 524288
constexpr int kBlock = 4 * kChunk;           // vocabulary entries per sampling CTA (1024 leaves)
constexpr int kMaxBlocks = kMaxChunks / 4;   // 32
constexpr int kMaxK = 16;
constexpr float kLog2e = 1.44269504088896340736f;

inline int n_chunks(int V) { return (V + kChunk - 1) / kChunk; }
inline int n_greedy_chunks(int V) { return (V + kGreedyChunk - 1) / kGreedyChunk; }
inline int n_blocks(int V) { return (V + kBlock - 1) / kBlock; }
inline size_t counters_bytes(int B) { return (static_cast<size_t>(B) * 4 + 255) / 256 * 256; }

// ------------------------------------------------------------------ greedy

struct ValIdx { float v; int i; };

__device__ __forceinline__ ValIdx better(ValIdx a, ValIdx b)
{
    // larger value wins, lowest index on ties
    return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

__device__ __forceinline__ ValIdx warp_best(ValIdx a)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ValIdx b{__shfl_xor_sync(0xffffffffu, a.v, o), __shfl_xor_sync(0xffffffffu, a.i, o)};
        a = better(a, b);
    }
    return a;
}

__global__ void __launch_bounds__(kThreads)
greedy_kernel(const int32_t *__restrict__ draft, const float *__restrict__ tgt, int k, int V,
              int32_t *__restrict__ out_tok, int32_t *__restrict__ out_cnt,
              unsigned int *__restrict__ counters, float2 *__restrict__ part, unsigned int *status)
{
    __shared__ ValIdx red[kThreads / 32];
    __shared__ bool last;
    __shared__ int tj[kMaxK + 1];
    const int C = gridDim.x, c = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *vec = tgt + (static_cast<size_t>(b) * (k + 1) + j) * V;

    ValIdx best{-INFINITY, 0x7fffffff};
    float finite = 0.0f;   // becomes NaN if any entry is not finite
    const int x0 = c * kGreedyChunk;
    if ((V & 3) == 0) {
        // two batches of eight 16-byte loads per thread (eight in flight)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float4 v[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int x = x0 + (8 * h + r) * (kThreads * 4) + threadIdx.x * 4;
                v[r] = x < V ? __ldcs(reinterpret_cast<const float4 *>(vec + x)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int x = x0 + (8 * h + r) * (kThreads * 4) + threadIdx.x * 4;
                if (x < V) {
                    finite = __fmaf_rn(0.0f, v[r].x, finite); finite = __fmaf_rn(0.0f, v[r].y, finite);
                    finite = __fmaf_rn(0.0f, v[r].z, finite); finite = __fmaf_rn(0.0f, v[r].w, finite);
                    best = better(best, ValIdx{v[r].x, x});
                    best = better(best, ValIdx{v[r].y, x + 1});
                    best = better(best, ValIdx{v[r].z, x + 2});
                    best = better(best, ValIdx{v[r].w, x + 3});
                }
            }
        }
    } else {
        for (int e = threadIdx.x; e < kGreedyChunk; e += kThreads) {
            const int x = x0 + e;
            if (x < V) {
                const float v = vec[x];
                finite = __fmaf_rn(0.0f, v, finite);
                best = better(best, ValIdx{v, x});
            }
        }
    }
    if (finite != 0.0f) set_status(status, NQ_DEV_NONFINITE);
    best = warp_best(best);
    if (lane == 0) red[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        ValIdx r = red[0];
        for (int w = 1; w < kThreads / 32; ++w) r = better(r, red[w]);
        part[(static_cast<size_t>(b) * (k + 1) + j) * C + c] = make_float2(r.v, __int_as_float(r.i));
        __threadfence();
        const unsigned int prev = atomicAdd(&counters[b], 1u);
        last = prev == static_cast<unsigned int>((k + 1) * C - 1);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();

    // last CTA of row b: t_j = best over the chunk partials of position j
    for (int jj = warp; jj <= k; jj += kThreads / 32) {
        ValIdx r{-INFINITY, 0x7fffffff};
        for (int cc = lane; cc < C; cc += 32) {
            const float2 p = __ldcg(part + (static_cast<size_t>(b) * (k + 1) + jj) * C + cc);
            r = better(r, ValIdx{p.x, __float_as_int(p.y)});
        }
        r = warp_best(r);
        if (lane == 0) tj[jj] = r.i;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int n = k;
        for (int jj = 0; jj < k; ++jj) {
            const int d = draft[static_cast<size_t>(b) * k + jj];
            if (d < 0 || d >= V) set_status(status, NQ_DEV_BAD_TOKEN);
            if (d != tj[jj] && n == k) n = jj;
        }
        for (int jj = 0; jj <= k; ++jj)
            out_tok[static_cast<size_t>(b) * (k + 1) + jj] = jj < n ? draft[static_cast<size_t>(b) * k + jj] : (jj == n ? tj[n] : -1);
        out_cnt[b] = n + 1;
        counters[b] = 0;   // ready for the next call
    }
}

// ------------------------------------------------------------------ sampled
//
// Leaves of the recipe: the vocabulary is cut into blocks of 16384 entries of
// 1024 leaves; leaf 4T + q (T = 0..255, q = 0..3) of block b holds the entries
// b*16384 + 4096*q + 1024*r + 4*T + j (r, j = 0..3), in (r, j) order, and has
// global index 1024*b + 4T + q.  Thread T of a 256-thread CTA owns the four
// consecutive leaves 4T..4T+3 of a block and reads them with sixteen coalesced
// 16-byte loads.  Absent entries (>= V) are read as -inf: they cannot raise a
// maximum and contribute an exact zero to every sum.

struct SampleRec {      // per-row decision, written by pass A, read by pass B
    int js;             // first rejected position, or k if all accepted
    int resid;          // 1: draw from max(0, p_js - q_js); 0: draw from p_js
    float u;            // the draw's uniform
    float Mp, invSp, Mq, invSq;
    int pad;
};

// Workspace layout shared by the greedy and sampled calls.
struct WsLayout {
    size_t counters_a, counters_b, part, rec, qsum, lsum, total;
};

inline size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// Every section starts on a 256-byte boundary (the kernels use 16-byte
// vector accesses on some of them).
inline WsLayout ws_layout(int B, int k, int V)
{
    const size_t C = static_cast<size_t>(n_chunks(V));   // greedy partials per vector (>= blocks)
    const size_t NB = static_cast<size_t>(n_blocks(V));
    WsLayout L;
    L.counters_a = 0;
    L.counters_b = align256(static_cast<size_t>(B) * 4);
    L.part = L.counters_b + align256(static_cast<size_t>(B) * 4);
    L.rec = L.part + align256(static_cast<size_t>(B) * (2 * k + 1) * C * sizeof(float2));
    L.qsum = L.rec + align256(static_cast<size_t>(B) * sizeof(SampleRec));   // 4 quarter nodes per block
    L.lsum = L.qsum + align256(static_cast<size_t>(B) * NB * 4 * sizeof(float));
    L.total = L.lsum + static_cast<size_t>(B) * NB * 4 * kThreads * sizeof(float);
    return L;
}

__device__ __forceinline__ int leaf_entry(int blk, int T, int q, int e)
{
    return blk * kBlock + 4096 * q + 1024 * (e >> 2) + 4 * T + (e & 3);
}

// Leaf (blk, 4T + q); `full` means the whole block lies inside [0, V).
__device__ __forceinline__ void load_leaf(const float *vec, int V, bool full, int blk, int T, int q, float (&l)[kLeaf])
{
    const int base = leaf_entry(blk, T, q, 0);
    if (full) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(vec + base + 1024 * r));
            l[4 * r] = v.x; l[4 * r + 1] = v.y; l[4 * r + 2] = v.z; l[4 * r + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < kLeaf; ++e) {
            const int x = base + 1024 * (e >> 2) + (e & 3);
            l[e] = x < V ? __ldcg(vec + x) : -INFINITY;
        }
    }
}

__device__ __forceinline__ bool block_full(int V, int blk) { return (V & 3) == 0 && (blk + 1) * kBlock <= V; }

// (mz, s) of a leaf with at least one present entry.
__device__ __forceinline__ MaxSum leaf_ms(const float (&l)[kLeaf], float c)
{
    float mx = l[0];
#pragma unroll
    for (int e = 1; e < kLeaf; ++e) mx = fmaxf(mx, l[e]);
    const float mz = __fmul_rn(mx, c);
    const unsigned long long c2 = f2_pack(c, c), nmz2 = f2_pack(-mz, -mz);
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < kLeaf; e += 2) {
        const float2 x = exp2_canon_x2(f2_fma(f2_pack(l[e], l[e + 1]), c2, nmz2));
        s = __fadd_rn(__fadd_rn(s, x.x), x.y);
    }
    return MaxSum{mz, s};
}

// Pairwise tree over 32 lanes (lane i holds node i of the level below).
__device__ __forceinline__ MaxSum warp_tree_ms(MaxSum a, int lane, int levels)
{
    for (int lv = 0; lv < levels; ++lv) {
        const int o = 1 << lv;
        MaxSum b{__shfl_xor_sync(0xffffffffu, a.m, o), __shfl_xor_sync(0xffffffffu, a.s, o)};
        a = (lane & o) ? ms_merge(b, a) : ms_merge(a, b);   // left operand = lower index
    }
    return a;
}

__device__ __forceinline__ float warp_tree_sum(float a, int levels)
{
    for (int lv = 0; lv < levels; ++lv) a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 1 << lv));
    return a;
}

struct RowRoots { float M, inv_s; };

__device__ __forceinline__ float leaf_factor(float mz_leaf, float M, float inv_s)
{
    return __fmul_rn(exp2_canon(__fsub_rn(mz_leaf, M)), inv_s);
}

// ---- pass A: one block of one vector; the last CTA of a row decides.
__global__ void __launch_bounds__(kThreads, 6)
sample_a_kernel(const int32_t *__restrict__ draft, const float *__restrict__ dlog, const float *__restrict__ tlog,
                int k, int V, float c, const uint64_t *__restrict__ seeds, uint64_t round,
                unsigned int *__restrict__ counters, float2 *__restrict__ part, SampleRec *__restrict__ rec,
                unsigned int *status)
{
    // the resample pass may be scheduled now; it waits (griddepcontrol.wait) for
    // this grid to complete before reading anything this grid writes
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ MaxSum red[kThreads / 32];
    __shared__ RowRoots roots[2 * kMaxK + 1];
    __shared__ bool last;
    const int NBK = gridDim.x, blk = blockIdx.x, v = blockIdx.y, b = blockIdx.z;
    const int NV = 2 * k + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, T = threadIdx.x;
    // vectors 0..k: target positions 0..k; k+1..2k: draft positions 0..k-1
    const float *vec = v <= k ? tlog + (static_cast<size_t>(b) * (k + 1) + v) * V
                              : dlog + (static_cast<size_t>(b) * k + (v - k - 1)) * V;
    {
        const bool full = block_full(V, blk);
        float finite = 0.0f;   // becomes NaN if a present entry is not finite
        MaxSum ms[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float l[kLeaf];
            load_leaf(vec, V, full, blk, T, q, l);
            if (full) {
#pragma unroll
                for (int e = 0; e < kLeaf; ++e) finite = __fmaf_rn(0.0f, l[e], finite);
                ms[q] = leaf_ms(l, c);
            } else if (leaf_entry(blk, T, q, 0) < V) {
#pragma unroll
                for (int e = 0; e < kLeaf; ++e)
                    if (leaf_entry(blk, T, q, e) < V) finite = __fmaf_rn(0.0f, l[e], finite);
                ms[q] = leaf_ms(l, c);
            } else {
                ms[q] = MaxSum{-INFINITY, 0.0f};
            }
            finite = __fmaf_rn(0.0f, ms[q].m == -INFINITY ? 0.0f : ms[q].m, finite);
        }
        if (finite != 0.0f) set_status(status, NQ_DEV_NONFINITE);
        MaxSum a = ms_merge(ms_merge(ms[0], ms[1]), ms_merge(ms[2], ms[3]));
        a = warp_tree_ms(a, lane, 5);
        if (lane == 0) red[warp] = a;
        __syncthreads();
        if (warp == 0) {
            MaxSum w8 = lane < kThreads / 32 ? red[lane] : MaxSum{-INFINITY, 0.0f};
            w8 = warp_tree_ms(w8, lane, 3);
            if (lane == 0) {
                part[(static_cast<size_t>(b) * NV + v) * NBK + blk] = make_float2(w8.m, w8.s);
                __threadfence();
                const unsigned int prev = atomicAdd(&counters[b], 1u);
                last = prev == static_cast<unsigned int>(NV * NBK - 1);
            }
        }
        __syncthreads();
        if (!last) return;
        __threadfence();
    }

    // ---- last CTA of row b: roots (M, 1/S) of the 2k+1 vectors (lane = block)
    for (int vv = warp; vv < NV; vv += kThreads / 32) {
        MaxSum a{-INFINITY, 0.0f};
        if (lane < NBK) {
            const float2 p = __ldcg(part + (static_cast<size_t>(b) * NV + vv) * NBK + lane);
            a = MaxSum{p.x, p.y};
        }
        a = warp_tree_ms(a, lane, 5);
        if (lane == 0) roots[vv] = RowRoots{a.m, __frcp_rn(a.s)};
    }
    __syncthreads();

    // ---- decisions: accept d_j iff u_j < p_j(d_j) / q_j(d_j); first rejection j*
    if (warp == 0) {
        const uint64_t seed = seeds[b];
        bool reject = false;
        if (lane < k) {
            const int j = lane;
            const int d = draft[static_cast<size_t>(b) * k + j];
            if (d < 0 || d >= V) {
                set_status(status, NQ_DEV_BAD_TOKEN);
                reject = true;
            } else {
                const float *pv = tlog + (static_cast<size_t>(b) * (k + 1) + j) * V;
                const float *qv = dlog + (static_cast<size_t>(b) * k + j) * V;
                const int bd = d / kBlock, o = d - bd * kBlock;
                const int qd = o >> 12, o2 = o & 4095;
                const int Td = (o2 & 1023) >> 2, ed = 4 * (o2 >> 10) + (o2 & 3);
                const bool fd = block_full(V, bd);
                float lp[kLeaf], lq[kLeaf];
                load_leaf(pv, V, fd, bd, Td, qd, lp);
                load_leaf(qv, V, fd, bd, Td, qd, lq);
                float mp = lp[0], mq = lq[0];
#pragma unroll
                for (int e = 1; e < kLeaf; ++e) { mp = fmaxf(mp, lp[e]); mq = fmaxf(mq, lq[e]); }
                const float mzp = __fmul_rn(mp, c), mzq = __fmul_rn(mq, c);
                float ld_p = lp[0], ld_q = lq[0];
#pragma unroll
                for (int e = 1; e < kLeaf; ++e) if (e == ed) { ld_p = lp[e]; ld_q = lq[e]; }
                const float p = __fmul_rn(exp2_canon(__fmaf_rn(ld_p, c, -mzp)), leaf_factor(mzp, roots[j].M, roots[j].inv_s));
                const float q = __fmul_rn(exp2_canon(__fmaf_rn(ld_q, c, -mzq)),
                                          leaf_factor(mzq, roots[k + 1 + j].M, roots[k + 1 + j].inv_s));
                const float ratio = __fdiv_rn(p, q);
                const float u = philox_uniform(seed, static_cast<uint32_t>(j), 0u, round);
                reject = !(u < ratio);
            }
        }
        const unsigned int rej = __ballot_sync(0xffffffffu, reject);
        if (lane == 0) {
            const int js = rej ? __ffs(rej) - 1 : k;
            SampleRec r;
            r.js = js;
            r.resid = js < k;
            r.u = philox_uniform(seed, static_cast<uint32_t>(js), js < k ? 1u : 2u, round);
            r.Mp = roots[js].M;
            r.invSp = roots[js].inv_s;
            r.Mq = js < k ? roots[k + 1 + js].M : 0.0f;
            r.invSq = js < k ? roots[k + 1 + js].inv_s : 0.0f;
            r.pad = 0;
            rec[b] = r;
            counters[b] = 0;   // ready for the next call
        }
    }
}

// Sampling weights of leaf (blk, 4T + q) of row b's chosen position and their
// serial sum: max(0, p - q) (resid) or p.  The logits are loaded separately
// (load_pq) so that the next leaf's loads can overlap this leaf's arithmetic.
__device__ __forceinline__ void load_pq(const float *pv, const float *qv, bool resid, int V, int blk, int T, int q,
                                        float (&lp)[kLeaf], float (&lq)[kLeaf])
{
    if (leaf_entry(blk, T, q, 0) >= V) return;
    const bool full = block_full(V, blk);
    load_leaf(pv, V, full, blk, T, q, lp);
    if (resid) load_leaf(qv, V, full, blk, T, q, lq);
}

template <bool KEEP>
__device__ __forceinline__ float leaf_weights(const float (&lp)[kLeaf], const float (&lq)[kLeaf], bool resid, int V,
                                              int blk, int T, int q, float c, const SampleRec &R, float (&w)[kLeaf])
{
    if (leaf_entry(blk, T, q, 0) >= V) {
        if (KEEP) {
#pragma unroll
            for (int e = 0; e < kLeaf; ++e) w[e] = 0.0f;
        }
        return 0.0f;
    }
    float mp = lp[0];
#pragma unroll
    for (int e = 1; e < kLeaf; ++e) mp = fmaxf(mp, lp[e]);
    const float mzp = __fmul_rn(mp, c);
    const float Fp = leaf_factor(mzp, R.Mp, R.invSp);
    float s = 0.0f;
    if (resid) {
        float mq = lq[0];
#pragma unroll
        for (int e = 1; e < kLeaf; ++e) mq = fmaxf(mq, lq[e]);
        const float mzq = __fmul_rn(mq, c);
        const float Fq = leaf_factor(mzq, R.Mq, R.invSq);
        const unsigned long long c2 = f2_pack(c, c), nmzp = f2_pack(-mzp, -mzp), nmzq = f2_pack(-mzq, -mzq);
#pragma unroll
        for (int e = 0; e < kLeaf; e += 2) {
            const float2 ep = exp2_canon_x2(f2_fma(f2_pack(lp[e], lp[e + 1]), c2, nmzp));
            const float2 eq = exp2_canon_x2(f2_fma(f2_pack(lq[e], lq[e + 1]), c2, nmzq));
            const float d0 = __fsub_rn(__fmul_rn(ep.x, Fp), __fmul_rn(eq.x, Fq));
            const float d1 = __fsub_rn(__fmul_rn(ep.y, Fp), __fmul_rn(eq.y, Fq));
            const float w0 = d0 > 0.0f ? d0 : 0.0f, w1 = d1 > 0.0f ? d1 : 0.0f;
            s = __fadd_rn(__fadd_rn(s, w0), w1);
            if (KEEP) { w[e] = w0; w[e + 1] = w1; }
        }
    } else {
        const unsigned long long c2 = f2_pack(c, c), nmzp = f2_pack(-mzp, -mzp);
#pragma unroll
        for (int e = 0; e < kLeaf; e += 2) {
            const float2 ep = exp2_canon_x2(f2_fma(f2_pack(lp[e], lp[e + 1]), c2, nmzp));
            const float w0 = __fmul_rn(ep.x, Fp), w1 = __fmul_rn(ep.y, Fp);
            s = __fadd_rn(__fadd_rn(s, w0), w1);
            if (KEEP) { w[e] = w0; w[e + 1] = w1; }
        }
    }
    return s;
}

// Sum over the 1024 leaves of block blk by the fixed pairwise tree (valid in
// thread 0); optionally stores the 1024 leaf sums (index 4T + q) at lsum.
__device__ float block_sum(float *warp_sum, float *lsum, const float *pv, const float *qv, bool resid, int V,
                           int blk, float c, const SampleRec &R)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, T = threadIdx.x;
    float w[kLeaf];
    float lp[2][kLeaf], lq[2][kLeaf];
    float ls[4];
    load_pq(pv, qv, resid, V, blk, T, 0, lp[0], lq[0]);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (q + 1 < 4) load_pq(pv, qv, resid, V, blk, T, q + 1, lp[(q + 1) & 1], lq[(q + 1) & 1]);
        ls[q] = leaf_weights<false>(lp[q & 1], lq[q & 1], resid, V, blk, T, q, c, R, w);
    }
    if (lsum) *reinterpret_cast<float4 *>(lsum + 4 * T) = make_float4(ls[0], ls[1], ls[2], ls[3]);
    float s = __fadd_rn(__fadd_rn(ls[0], ls[1]), __fadd_rn(ls[2], ls[3]));
    s = warp_tree_sum(s, 5);
    if (lane == 0) warp_sum[warp] = s;
    __syncthreads();
    float tot = 0.0f;
    if (warp == 0) tot = warp_tree_sum(lane < kThreads / 32 ? warp_sum[lane] : 0.0f, 3);
    __syncthreads();
    return tot;
}

// Descend the pairwise sum tree over 32 leaves held one per lane (index =
// lane; pads are zeros).  Level sums are formed as left + right by xor
// shuffles (fp addition commutes exactly); at each level go left if t < left
// or the right sum is not positive, else t -= left.  Returns the chosen lane;
// every lane computes the same result and t.
__device__ __forceinline__ int warp_descend32(float v, float &t)
{
    float s[6];
    s[0] = v;
#pragma unroll
    for (int l = 0; l < 5; ++l) s[l + 1] = __fadd_rn(s[l], __shfl_xor_sync(0xffffffffu, s[l], 1 << l));
    int base = 0;
#pragma unroll
    for (int l = 4; l >= 0; --l) {
        const float left = __shfl_sync(0xffffffffu, s[l], base);
        const float right = __shfl_sync(0xffffffffu, s[l], base + (1 << l));
        if (!(t < left || !(right > 0.0f))) {
            t = __fsub_rn(t, left);
            base += 1 << l;
        }
    }
    return base;
}

// ---- pass B: one block of the chosen position of one row; the last CTA of
// the row descends the sum tree and writes the row's tokens.
__global__ void __launch_bounds__(kThreads, 4)
sample_b_kernel(const int32_t *__restrict__ draft, const float *__restrict__ dlog, const float *__restrict__ tlog,
                int k, int V, float c, int32_t *__restrict__ out_tok, int32_t *__restrict__ out_cnt,
                unsigned int *__restrict__ counters, const SampleRec *__restrict__ rec, float *__restrict__ qsum,
                float *__restrict__ lsum)
{
    // launched as a programmatic dependent of the decision pass: wait for that
    // grid to complete (its records and partials visible) before anything else
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float warp_sum[kThreads / 32];
    __shared__ __align__(16) float btree[2 * kMaxBlocks];
    __shared__ bool last;
    __shared__ int pick;
    const int NBK = gridDim.x >> 2, blk = blockIdx.x >> 2, q = blockIdx.x & 3, b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const SampleRec R = rec[b];
    const float *pv = tlog + (static_cast<size_t>(b) * (k + 1) + R.js) * V;
    const float *qv = R.js < k ? dlog + (static_cast<size_t>(b) * k + R.js) * V : pv;
    bool resid = R.resid != 0;

    // one leaf per thread: leaf 256 q + T of block blk, so the CTA holds 256
    // consecutive leaves and forms their node of the block's pairwise sum tree
    // (lanes, then warps); its leaf sum goes to lsum, the node to qsum
    float *blk_lsum = lsum + (static_cast<size_t>(b) * NBK + blk) * (4 * kThreads);
    const int leaf = kThreads * q + threadIdx.x, Tl = leaf >> 2, ql = leaf & 3;   // leaf = 4 Tl + ql
    float ls;
    {
        float lp[kLeaf], lq[kLeaf], w[kLeaf];
        load_pq(pv, qv, resid, V, blk, Tl, ql, lp, lq);
        ls = leaf_weights<false>(lp, lq, resid, V, blk, Tl, ql, c, R, w);
        blk_lsum[leaf] = ls;
    }
    ls = warp_tree_sum(ls, 5);
    if (lane == 0) warp_sum[warp] = ls;
    __syncthreads();
    if (warp == 0) {
        const float node = warp_tree_sum(lane < kThreads / 32 ? warp_sum[lane] : 0.0f, 3);
        if (lane == 0) {
            qsum[(static_cast<size_t>(b) * NBK + blk) * 4 + q] = node;
            __threadfence();
            const unsigned int prev = atomicAdd(&counters[b], 1u);
            last = prev == static_cast<unsigned int>(4 * NBK - 1);
        }
    }
    __syncthreads();
    if (!last) return;
    __threadfence();

    // block totals: the top two levels of each block's tree over its four
    // quarter nodes, (q0 + q1) + (q2 + q3)
    for (int bb = threadIdx.x; bb < NBK; bb += kThreads) {
        const float4 n4 = __ldcg(reinterpret_cast<const float4 *>(qsum + (static_cast<size_t>(b) * NBK + bb) * 4));
        btree[bb] = __fadd_rn(__fadd_rn(n4.x, n4.y), __fadd_rn(n4.z, n4.w));
    }
    __syncthreads();
    // all-zero residual (rounding): draw from p_js instead (all threads rebuild the leaf sums)
    if (resid) {
        float r = warp == 0 ? (lane < NBK ? btree[lane] : 0.0f) : 0.0f;
        if (warp == 0) r = warp_tree_sum(r, 5);
        if (threadIdx.x == 0) pick = r > 0.0f ? 1 : 0;
        __syncthreads();
        if (pick == 0) {
            resid = false;
            for (int bb = 0; bb < NBK; ++bb) {
                const float sb = block_sum(warp_sum, lsum + (static_cast<size_t>(b) * NBK + bb) * (4 * kThreads), pv, qv,
                                           false, V, bb, c, R);
                if (threadIdx.x == 0) btree[bb] = sb;
            }
        }
        __syncthreads();
    }
    if (warp != 0) return;

    // warp 0: block tree (32 lanes, zero pads), then the chosen block's leaf tree
    const float bval = lane < NBK ? btree[lane] : 0.0f;
    const float root = warp_tree_sum(bval, 5);
    float t = __fmul_rn(R.u, root);
    const int bstar = warp_descend32(bval, t);
    float v[32];
    {
        const float4 *src = reinterpret_cast<const float4 *>(lsum + (static_cast<size_t>(b) * NBK + bstar) * (4 * kThreads)) + 8 * lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 x = __ldcg(src + i);
            v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
        }
    }
    float lsum32[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) lsum32[i] = v[i];
#pragma unroll
    for (int w = 1; w < 32; w <<= 1)
#pragma unroll
        for (int i = 0; i < 32; i += 2 * w) v[i] = __fadd_rn(v[i], v[i + w]);
    const int lane_star = warp_descend32(v[0], t);
    float mine = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float x = __shfl_sync(0xffffffffu, lsum32[i], lane_star);
        if (lane == i) mine = x;
    }
    const int lstar = 32 * lane_star + warp_descend32(mine, t);

    // the chosen leaf: 16 lanes reload one entry each, the weights are formed
    // exactly as in the leaf sums, lane 0 scans them in entry order
    const int Ts = lstar >> 2, qs = lstar & 3;
    const int e = lane & 15;
    const int x = leaf_entry(bstar, Ts, qs, e);
    const bool present = x < V;
    const float lp = present ? __ldcg(pv + x) : -INFINITY;
    const float lq = present && resid ? __ldcg(qv + x) : -INFINITY;
    float mp = lp, mq = lq;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
        mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, o));
        mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
    }
    const float mzp = __fmul_rn(mp, c);
    float we = __fmul_rn(exp2_canon(__fmaf_rn(lp, c, -mzp)), leaf_factor(mzp, R.Mp, R.invSp));
    if (resid) {
        const float mzq = __fmul_rn(mq, c);
        const float qe = __fmul_rn(exp2_canon(__fmaf_rn(lq, c, -mzq)), leaf_factor(mzq, R.Mq, R.invSq));
        const float d = __fsub_rn(we, qe);
        we = d > 0.0f ? d : 0.0f;
    }
    if (!present) we = 0.0f;
    int pk = -1;
    float run = 0.0f;
#pragma unroll
    for (int i = 0; i < kLeaf; ++i) {
        const float wi = __shfl_sync(0xffffffffu, we, i);
        const int xi = leaf_entry(bstar, Ts, qs, i);
        if (xi < V && pk < 0) {
            run = __fadd_rn(run, wi);
            if (t < run) pk = xi;
        }
    }
    // fallback: the last entry of the leaf with a positive weight
#pragma unroll
    for (int i = kLeaf - 1; i >= 0; --i) {
        const float wi = __shfl_sync(0xffffffffu, we, i);
        const int xi = leaf_entry(bstar, Ts, qs, i);
        if (pk < 0 && xi < V && wi > 0.0f) pk = xi;
    }
    if (lane == 0) {
        const int js = R.js;
        for (int jj = 0; jj <= k; ++jj)
            out_tok[static_cast<size_t>(b) * (k + 1) + jj] = jj < js ? draft[static_cast<size_t>(b) * k + jj] : (jj == js ? pk : -1);
        out_cnt[b] = js + 1;
        counters[b] = 0;
    }
}

nq_status check_accept(int B, int k, int V, const void *ws, size_t ws_bytes)
{
    if (B < 1 || B > 65535 || k < 1 || k > kMaxK || V < 1 || V > kMaxChunks * kChunk) return NQ_ERR_ARG;
    if (!ws) return NQ_ERR_ARG;
    if (!aligned16(ws)) return NQ_ERR_ALIGN;
    if (ws_bytes < ws_layout(B, k, V).total) return NQ_ERR_WORKSPACE;
    return NQ_OK;
}

}  // namespace
}  // namespace nq

extern "C" size_t spec_accept_workspace_bytes(int B, int k, int V)
{
    if (B < 1 || B > 65535 || k < 1 || k > nq::kMaxK || V < 1 || V > nq::kMaxChunks * nq::kChunk) return 0;
    return nq::ws_layout(B, k, V).total;
}

extern "C" nq_status spec_accept_greedy(const int32_t *draft, const float *tgt_logits, int B, int k, int V,
                                        int32_t *out_tok, int32_t *out_cnt, void *ws, size_t ws_bytes,
                                        cudaStream_t stream)
{
    nq_status st = nq::check_accept(B, k, V, ws, ws_bytes);
    if (st != NQ_OK) return st;
    if (!draft || !tgt_logits || !out_tok || !out_cnt) return NQ_ERR_ARG;
    if (!nq::aligned16(draft) || !nq::aligned16(tgt_logits) || !nq::aligned16(out_tok) || !nq::aligned16(out_cnt))
        return NQ_ERR_ALIGN;
    unsigned int *status = nq::device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    const nq::WsLayout L = nq::ws_layout(B, k, V);
    char *w = static_cast<char *>(ws);
    dim3 grid(nq::n_greedy_chunks(V), k + 1, B);
    nq::greedy_kernel<<<grid, nq::kThreads, 0, stream>>>(draft, tgt_logits, k, V, out_tok, out_cnt,
                                                         reinterpret_cast<unsigned int *>(w + L.counters_a),
                                                         reinterpret_cast<float2 *>(w + L.part), status);
    return nq::cuda_status(cudaGetLastError());
}

extern "C" nq_status spec_accept_sample(const int32_t *draft, const float *draft_logits, const float *tgt_logits,
                                        int B, int k, int V, float temperature, const uint64_t *seeds,
                                        uint64_t round, int32_t *out_tok, int32_t *out_cnt, void *ws,
                                        size_t ws_bytes, cudaStream_t stream)
{
    nq_status st = nq::check_accept(B, k, V, ws, ws_bytes);
    if (st != NQ_OK) return st;
    if (!(temperature > 0.0f) || !(temperature < INFINITY)) return NQ_ERR_ARG;
    if (!draft || !draft_logits || !tgt_logits || !seeds || !out_tok || !out_cnt) return NQ_ERR_ARG;
    if (!nq::aligned16(draft) || !nq::aligned16(draft_logits) || !nq::aligned16(tgt_logits) ||
        !nq::aligned16(seeds) || !nq::aligned16(out_tok) || !nq::aligned16(out_cnt))
        return NQ_ERR_ALIGN;
    unsigned int *status = nq::device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    const float c = nq::kLog2e / temperature;   // IEEE division on the host (round to nearest)
    const nq::WsLayout L = nq::ws_layout(B, k, V);
    char *w = static_cast<char *>(ws);
    auto *rec = reinterpret_cast<nq::SampleRec *>(w + L.rec);
    dim3 grid_a(nq::n_blocks(V), 2 * k + 1, B);
    nq::sample_a_kernel<<<grid_a, nq::kThreads, 0, stream>>>(draft, draft_logits, tgt_logits, k, V, c, seeds, round,
                                                             reinterpret_cast<unsigned int *>(w + L.counters_a),
                                                             reinterpret_cast<float2 *>(w + L.part), rec, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return NQ_ERR_CUDA;
    // pass B as a programmatic dependent launch when pass A fills the GPU: its
    // CTAs are scheduled while pass A drains and block in griddepcontrol.wait
    // until pass A completes.  Below one wave of pass-A CTAs (B = 1 rounds)
    // a plain launch measured faster inside a decode round (32 vs 37 us with
    // the dependent launch); griddepcontrol.wait returns at once then.
    const bool dependent = static_cast<long long>(grid_a.x) * grid_a.y * grid_a.z >= nq::sm_count();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4 * nq::n_blocks(V), B);   // one CTA per (block, leaf quarter q)
    cfg.blockDim = dim3(nq::kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, nq::sample_b_kernel, draft, draft_logits, tgt_logits, k, V, c, out_tok, out_cnt,
                           reinterpret_cast<unsigned int *>(w + L.counters_b), static_cast<const nq::SampleRec *>(rec),
                           reinterpret_cast<float *>(w + L.qsum), reinterpret_cast<float *>(w + L.lsum));
    return nq::cuda_status(e);
}

// ------------------------------------------------------------------ allocation-free greedy acceptance
//
// For callers that cannot allocate device memory at the call site (their
// device memory is owned by another component -- e.g. a serving runtime whose
// allocator holds a fixed budget -- or they must not risk a failing or
// blocking allocation in the decode loop): the workspace of the greedy
// acceptance lives in a fixed array compiled into this file.  Every GPU that
// loads the library holds it until the process exits.  All calls share it.

namespace nq {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;   // 1 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64];

// Device address of the scratch array on the current device, looked up once
// per device with that device current (host code may not use the symbol).
void *noalloc_scratch()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace
}  // namespace nq

extern "C" nq_status spec_accept_greedy_noalloc(const int32_t *draft, const float *tgt_logits, int B, int k, int V,
                                                int32_t *out_tok, int32_t *out_cnt, cudaStream_t stream)
{
    if (B < 1 || B > 65535 || k < 1 || k > nq::kMaxK || V < 1 || V > nq::kMaxChunks * nq::kChunk) return NQ_ERR_ARG;
    if (!draft || !tgt_logits || !out_tok || !out_cnt) return NQ_ERR_ARG;
    if (!nq::aligned16(draft) || !nq::aligned16(tgt_logits) || !nq::aligned16(out_tok) || !nq::aligned16(out_cnt))
        return NQ_ERR_ALIGN;
    const size_t counters = nq::counters_bytes(B);
    const size_t need = counters + static_cast<size_t>(B) * (k + 1) * nq::n_chunks(V) * sizeof(float2);
    if (need > nq::kNoAllocScratchBytes) return NQ_ERR_WORKSPACE;
    unsigned char *scratch = static_cast<unsigned char *>(nq::noalloc_scratch());
    unsigned int *status = nq::device_status_ptr();
    if (!scratch || !status) return NQ_ERR_CUDA;
    // the per-row tickets must start at zero; the partials are overwritten
    if (cudaMemsetAsync(scratch, 0, counters, stream) != cudaSuccess) return NQ_ERR_CUDA;
    dim3 grid(nq::n_greedy_chunks(V), k + 1, B);
    nq::greedy_kernel<<<grid, nq::kThreads, 0, stream>>>(draft, tgt_logits, k, V, out_tok, out_cnt,
                                                         reinterpret_cast<unsigned int *>(scratch),
                                                         reinterpret_cast<float2 *>(scratch + counters), status);
    return nq::cuda_status(cudaGetLastError());
}
