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
constexpr int kChunk = kThreads * kLeaf;     // vocabulary entries per CTA
constexpr int kMaxChunks = 128;              // V <= 524288
constexpr int kMaxK = 16;
constexpr float kLog2e = 1.44269504088896340736f;

inline int n_chunks(int V) { return (V + kChunk - 1) / kChunk; }
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
    const int x0 = c * kChunk;
    if ((V & 3) == 0) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int x = x0 + r * (kThreads * 4) + threadIdx.x * 4;
            if (x < V) {
                const float4 v = __ldcs(reinterpret_cast<const float4 *>(vec + x));
                finite = __fmaf_rn(0.0f, v.x, finite); finite = __fmaf_rn(0.0f, v.y, finite);
                finite = __fmaf_rn(0.0f, v.z, finite); finite = __fmaf_rn(0.0f, v.w, finite);
                best = better(best, ValIdx{v.x, x});
                best = better(best, ValIdx{v.y, x + 1});
                best = better(best, ValIdx{v.z, x + 2});
                best = better(best, ValIdx{v.w, x + 3});
            }
        }
    } else {
        for (int e = threadIdx.x; e < kChunk; e += kThreads) {
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

// Load the (up to) 16 logits of leaf L of a vector; entries past V are -inf.
__device__ __forceinline__ void load_leaf(const float *vec, int V, int L, float (&l)[kLeaf])
{
    const int x0 = L * kLeaf;
    if ((V & 3) == 0 && x0 + kLeaf <= V) {
        const float4 *p = reinterpret_cast<const float4 *>(vec + x0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 v = __ldcg(p + q);
            l[4 * q] = v.x; l[4 * q + 1] = v.y; l[4 * q + 2] = v.z; l[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < kLeaf; ++e) l[e] = x0 + e < V ? __ldcg(vec + x0 + e) : -INFINITY;
    }
}

// Leaf statistics of the recipe: raw max -> mz = RN(max * c); s = serial sum
// of exp2(fma(l, c, -mz)).  Returns (-inf, 0) for a leaf wholly past V.
__device__ __forceinline__ MaxSum leaf_stats(const float (&l)[kLeaf], int n_valid, float c, float &finite)
{
    if (n_valid <= 0) return MaxSum{-INFINITY, 0.0f};
    float mx = l[0];
#pragma unroll
    for (int e = 0; e < kLeaf; ++e) {
        if (e < n_valid) {
            mx = fmaxf(mx, l[e]);
            finite = __fmaf_rn(0.0f, l[e], finite);
        }
    }
    const float mz = __fmul_rn(mx, c);
    finite = __fmaf_rn(0.0f, mz, finite);
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < kLeaf; ++e)
        if (e < n_valid) s = __fadd_rn(s, exp2_canon(__fmaf_rn(l[e], c, -mz)));
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

// Probability of entry x (leaf max mz recomputed from the leaf's logits).
__device__ __forceinline__ float prob_of(float lx, float mz_leaf, float c, RowRoots r)
{
    const float F = __fmul_rn(exp2_canon(__fsub_rn(mz_leaf, r.M)), r.inv_s);
    return __fmul_rn(exp2_canon(__fmaf_rn(lx, c, -mz_leaf)), F);
}

// Weights of the sampling distribution for one leaf: the residual
// max(0, p - q) (resid == true) or the target probabilities p.
__device__ __forceinline__ void leaf_weights(const float *pv, const float *qv, bool resid, int V, int L, float c,
                                             RowRoots rp, RowRoots rq, float (&w)[kLeaf], int &n_valid)
{
    n_valid = min(kLeaf, V - L * kLeaf);
    if (n_valid <= 0) {
#pragma unroll
        for (int e = 0; e < kLeaf; ++e) w[e] = 0.0f;
        return;
    }
    float lp[kLeaf];
    load_leaf(pv, V, L, lp);
    float mx = lp[0];
#pragma unroll
    for (int e = 0; e < kLeaf; ++e) if (e < n_valid) mx = fmaxf(mx, lp[e]);
    const float mzp = __fmul_rn(mx, c);
#pragma unroll
    for (int e = 0; e < kLeaf; ++e) w[e] = e < n_valid ? prob_of(lp[e], mzp, c, rp) : 0.0f;
    if (resid) {
        float lq[kLeaf];
        load_leaf(qv, V, L, lq);
        float mq = lq[0];
#pragma unroll
        for (int e = 0; e < kLeaf; ++e) if (e < n_valid) mq = fmaxf(mq, lq[e]);
        const float mzq = __fmul_rn(mq, c);
#pragma unroll
        for (int e = 0; e < kLeaf; ++e) {
            if (e < n_valid) {
                const float d = __fsub_rn(w[e], prob_of(lq[e], mzq, c, rq));
                w[e] = d > 0.0f ? d : 0.0f;
            }
        }
    }
}

struct SampleSmem {
    MaxSum red[kThreads / 32];
    RowRoots roots[2 * kMaxK + 1];
    float chunk_sum[2 * kMaxChunks];     // chunk-level tree (levels stacked)
    float leaf_sum[2 * kThreads];        // leaf-level tree of one chunk (levels stacked)
    float warp_sum[kThreads / 32];
    int jstar;
    int pick;
    bool last;
};

// Sum of the sampling weights of every leaf of chunk cc, reduced to the chunk
// total by a fixed pairwise tree; optionally keeps the leaf-level tree.
__device__ float chunk_weight_sum(SampleSmem &sm, const float *pv, const float *qv, bool resid, int V, int cc,
                                  float c, RowRoots rp, RowRoots rq, bool keep_levels)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float w[kLeaf];
    int nv;
    leaf_weights(pv, qv, resid, V, cc * kThreads + threadIdx.x, c, rp, rq, w, nv);
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < kLeaf; ++e) if (e < nv) s = __fadd_rn(s, w[e]);
    if (keep_levels) sm.leaf_sum[threadIdx.x] = s;
    s = warp_tree_sum(s, 5);
    if (lane == 0) sm.warp_sum[warp] = s;
    __syncthreads();
    float tot = 0.0f;
    if (threadIdx.x < 32) {
        float v = lane < kThreads / 32 ? sm.warp_sum[lane] : 0.0f;
        v = warp_tree_sum(v, 3);
        tot = v;
    }
    if (keep_levels) {
        // levels 1..8 of the 256-leaf tree, stacked after level 0
        int in = 0, width = kThreads;
        while (width > 1) {
            const int out = in + width;
            for (int i = threadIdx.x; i < width / 2; i += kThreads)
                sm.leaf_sum[out + i] = __fadd_rn(sm.leaf_sum[in + 2 * i], sm.leaf_sum[in + 2 * i + 1]);
            __syncthreads();
            in = out;
            width >>= 1;
        }
    }
    __syncthreads();
    return tot;   // valid in thread 0 (warp 0)
}

__global__ void __launch_bounds__(kThreads)
sample_kernel(const int32_t *__restrict__ draft, const float *__restrict__ dlog, const float *__restrict__ tlog,
              int k, int V, float c, const uint64_t *__restrict__ seeds, uint64_t round,
              int32_t *__restrict__ out_tok, int32_t *__restrict__ out_cnt,
              unsigned int *__restrict__ counters, float2 *__restrict__ part, unsigned int *status)
{
    __shared__ SampleSmem sm;
    const int C = gridDim.x, cidx = blockIdx.x, v = blockIdx.y, b = blockIdx.z;
    const int NV = 2 * k + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // vectors 0..k: target positions 0..k; k+1..2k: draft positions 0..k-1
    const float *vec = v <= k ? tlog + (static_cast<size_t>(b) * (k + 1) + v) * V
                              : dlog + (static_cast<size_t>(b) * k + (v - k - 1)) * V;

    // ---- pass A: (max, sum) of this chunk's 256 leaves
    {
        const int L = cidx * kThreads + threadIdx.x;
        float l[kLeaf];
        const int nv = min(kLeaf, V - L * kLeaf);
        float finite = 0.0f;
        MaxSum ms{-INFINITY, 0.0f};
        if (nv > 0) {
            const int x0 = L * kLeaf;
            if ((V & 3) == 0 && nv == kLeaf) {
                const float4 *p = reinterpret_cast<const float4 *>(vec + x0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 t4 = __ldcg(p + q);
                    l[4 * q] = t4.x; l[4 * q + 1] = t4.y; l[4 * q + 2] = t4.z; l[4 * q + 3] = t4.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < kLeaf; ++e) l[e] = e < nv ? vec[x0 + e] : 0.0f;
            }
            ms = leaf_stats(l, nv, c, finite);
        }
        if (finite != 0.0f) set_status(status, NQ_DEV_NONFINITE);
        ms = warp_tree_ms(ms, lane, 5);
        if (lane == 0) sm.red[warp] = ms;
        __syncthreads();
        if (warp == 0) {
            MaxSum a = lane < kThreads / 32 ? sm.red[lane] : MaxSum{-INFINITY, 0.0f};
            a = warp_tree_ms(a, lane, 3);
            if (lane == 0) {
                part[(static_cast<size_t>(b) * NV + v) * C + cidx] = make_float2(a.m, a.s);
                __threadfence();
                const unsigned int prev = atomicAdd(&counters[b], 1u);
                sm.last = prev == static_cast<unsigned int>(NV * C - 1);
            }
        }
        __syncthreads();
        if (!sm.last) return;
        __threadfence();
    }

    // ---- last CTA of row b: roots (M, 1/S) of all 2k+1 vectors
    for (int vv = warp; vv < NV; vv += kThreads / 32) {
        // lane holds chunks 4*lane .. 4*lane+3 (levels 9, 10 locally, then 11.. across lanes)
        MaxSum n4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int cc = 4 * lane + q;
            if (cc < C) {
                const float2 p = __ldcg(part + (static_cast<size_t>(b) * NV + vv) * C + cc);
                n4[q] = MaxSum{p.x, p.y};
            } else {
                n4[q] = MaxSum{-INFINITY, 0.0f};
            }
        }
        MaxSum a = ms_merge(ms_merge(n4[0], n4[1]), ms_merge(n4[2], n4[3]));
        a = warp_tree_ms(a, lane, 5);
        if (lane == 0) sm.roots[vv] = RowRoots{a.m, __frcp_rn(a.s)};
    }
    __syncthreads();

    // ---- decisions: accept d_j iff u_j < p_j(d_j) / q_j(d_j), first rejection j*
    const uint64_t seed = seeds[b];
    if (warp == 0) {
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
                const int L = d / kLeaf;
                float lp[kLeaf], lq[kLeaf];
                load_leaf(pv, V, L, lp);
                load_leaf(qv, V, L, lq);
                const int nv = min(kLeaf, V - L * kLeaf);
                float mp = lp[0], mq = lq[0];
#pragma unroll
                for (int e = 0; e < kLeaf; ++e) if (e < nv) { mp = fmaxf(mp, lp[e]); mq = fmaxf(mq, lq[e]); }
                const float p = prob_of(lp[d - L * kLeaf], __fmul_rn(mp, c), c, sm.roots[j]);
                const float q = prob_of(lq[d - L * kLeaf], __fmul_rn(mq, c), c, sm.roots[k + 1 + j]);
                const float ratio = __fdiv_rn(p, q);
                const float u = philox_uniform(seed, static_cast<uint32_t>(j), 0u, round);
                reject = !(u < ratio);
            }
        }
        const unsigned int rej = __ballot_sync(0xffffffffu, reject);
        if (lane == 0) sm.jstar = rej ? __ffs(rej) - 1 : k;
    }
    __syncthreads();
    const int js = sm.jstar;

    // ---- draw the replacement (residual at j*) or the bonus token (p_k)
    const float *pv = tlog + (static_cast<size_t>(b) * (k + 1) + js) * V;
    const float *qv = js < k ? dlog + (static_cast<size_t>(b) * k + js) * V : pv;
    const RowRoots rp = sm.roots[js];
    const RowRoots rq = js < k ? sm.roots[k + 1 + js] : sm.roots[js];
    bool resid = js < k;
    const float u = philox_uniform(seed, static_cast<uint32_t>(js), resid ? 1u : 2u, round);
    int Cp = 1;
    while (Cp < C) Cp <<= 1;
    for (int attempt = 0; attempt < 2; ++attempt) {
        for (int cc = 0; cc < Cp; ++cc) {
            const float s = cc < C ? chunk_weight_sum(sm, pv, qv, resid, V, cc, c, rp, rq, false) : 0.0f;
            if (threadIdx.x == 0) sm.chunk_sum[cc] = s;
        }
        __syncthreads();
        // chunk-level levels stacked: level 0 at [0, Cp), level l after
        {
            int in = 0, width = Cp;
            while (width > 1) {
                const int out = in + width;
                for (int i = threadIdx.x; i < width / 2; i += kThreads)
                    sm.chunk_sum[out + i] = __fadd_rn(sm.chunk_sum[in + 2 * i], sm.chunk_sum[in + 2 * i + 1]);
                __syncthreads();
                in = out;
                width >>= 1;
            }
        }
        const float R = sm.chunk_sum[2 * Cp - 2];
        if (R > 0.0f || !resid) break;
        resid = false;   // all-zero residual: draw from p_j* instead
        __syncthreads();
    }
    const float R = sm.chunk_sum[2 * Cp - 2];
    // descend the chunk-level tree (every thread follows the same path)
    float t = __fmul_rn(u, R);
    int node = 0;
    {
        // level offsets: level l (width Cp >> l) starts at Cp*(2 - 2^(1-l)) = sum of wider levels
        int levels = 0;
        while ((1 << levels) < Cp) ++levels;
        for (int lv = levels; lv >= 1; --lv) {
            int off_child = 0;
            for (int q = 0; q < lv - 1; ++q) off_child += Cp >> q;
            const float left = sm.chunk_sum[off_child + 2 * node], right = sm.chunk_sum[off_child + 2 * node + 1];
            if (t < left || !(right > 0.0f)) node = 2 * node;
            else { t = __fsub_rn(t, left); node = 2 * node + 1; }
        }
    }
    __syncthreads();
    const int cstar = node;
    chunk_weight_sum(sm, pv, qv, resid, V, cstar, c, rp, rq, true);
    // descend the 256-leaf tree of chunk c*
    {
        int leaf = 0;
        for (int lv = 8; lv >= 1; --lv) {
            int off_child = 0;
            for (int q = 0; q < lv - 1; ++q) off_child += kThreads >> q;
            const float left = sm.leaf_sum[off_child + 2 * leaf], right = sm.leaf_sum[off_child + 2 * leaf + 1];
            if (t < left || !(right > 0.0f)) leaf = 2 * leaf;
            else { t = __fsub_rn(t, left); leaf = 2 * leaf + 1; }
        }
        if (threadIdx.x == 0) {
            const int L = cstar * kThreads + leaf;
            float w[kLeaf];
            int nv;
            leaf_weights(pv, qv, resid, V, L, c, rp, rq, w, nv);
            int pick = -1;
            float run = 0.0f;
            for (int e = 0; e < nv && pick < 0; ++e) {
                run = __fadd_rn(run, w[e]);
                if (t < run) pick = e;
            }
            for (int e = nv - 1; e >= 0 && pick < 0; --e)
                if (w[e] > 0.0f) pick = e;
            sm.pick = pick < 0 ? -1 : L * kLeaf + pick;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int tok = sm.pick;
        for (int jj = 0; jj <= k; ++jj)
            out_tok[static_cast<size_t>(b) * (k + 1) + jj] = jj < js ? draft[static_cast<size_t>(b) * k + jj] : (jj == js ? tok : -1);
        out_cnt[b] = js + 1;
        counters[b] = 0;
    }
}

nq_status check_accept(int B, int k, int V, const void *ws, size_t ws_bytes)
{
    if (B < 1 || B > 65535 || k < 1 || k > kMaxK || V < 1 || V > kMaxChunks * kChunk) return NQ_ERR_ARG;
    if (!ws) return NQ_ERR_ARG;
    if (!aligned16(ws)) return NQ_ERR_ALIGN;
    if (ws_bytes < spec_accept_workspace_bytes(B, k, V)) return NQ_ERR_WORKSPACE;
    return NQ_OK;
}

}  // namespace
}  // namespace nq

extern "C" size_t spec_accept_workspace_bytes(int B, int k, int V)
{
    if (B < 1 || B > 65535 || k < 1 || k > nq::kMaxK || V < 1 || V > nq::kMaxChunks * nq::kChunk) return 0;
    return nq::counters_bytes(B) + static_cast<size_t>(B) * (2 * k + 1) * nq::n_chunks(V) * sizeof(float2);
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
    unsigned int *counters = static_cast<unsigned int *>(ws);
    float2 *part = reinterpret_cast<float2 *>(static_cast<char *>(ws) + nq::counters_bytes(B));
    dim3 grid(nq::n_chunks(V), k + 1, B);
    nq::greedy_kernel<<<grid, nq::kThreads, 0, stream>>>(draft, tgt_logits, k, V, out_tok, out_cnt, counters, part, status);
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
    unsigned int *counters = static_cast<unsigned int *>(ws);
    float2 *part = reinterpret_cast<float2 *>(static_cast<char *>(ws) + nq::counters_bytes(B));
    dim3 grid(nq::n_chunks(V), 2 * k + 1, B);
    nq::sample_kernel<<<grid, nq::kThreads, 0, stream>>>(draft, draft_logits, tgt_logits, k, V, c, seeds, round,
                                                         out_tok, out_cnt, counters, part, status);
    return nq::cuda_status(cudaGetLastError());
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
    dim3 grid(nq::n_chunks(V), k + 1, B);
    nq::greedy_kernel<<<grid, nq::kThreads, 0, stream>>>(draft, tgt_logits, k, V, out_tok, out_cnt,
                                                         reinterpret_cast<unsigned int *>(scratch),
                                                         reinterpret_cast<float2 *>(scratch + counters), status);
    return nq::cuda_status(cudaGetLastError());
}
