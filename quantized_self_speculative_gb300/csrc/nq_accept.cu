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
// Leaves of the recipe: 16 consecutive vocabulary entries in index order
// (leaf i holds entries 16 i .. 16 i + 15); a block of 1024 leaves (16384
// entries) is the unit of one pass-A CTA.  Four lanes share a leaf: lane
// 4 g + qq of a warp holds entries 4 qq .. 4 qq + 3 of its group's leaf (one
// 16-byte load, so a warp's load instruction reads eight 64-byte leaves in
// full sectors).  The leaf's maximum and sum are formed across the four lanes
// with xor shuffles: the maximum, and (Q0 + Q1) + (Q2 + Q3) of the serial
// quarter sums Q -- the same bits on all four lanes, since fp32 max and
// addition commute.  Absent entries (>= V) are read as -inf: they cannot
// raise a maximum and contribute an exact zero to every sum; a leaf with no
// present entry is a pad, (-inf, 0) or 0.

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

// The four entries x .. x + 3 (x a multiple of 4) of one vector; `full` means
// they are all present and 16-byte aligned.
__device__ __forceinline__ float4 load_quarter(const float *vec, int V, bool full, int x)
{
    if (full) return __ldcg(reinterpret_cast<const float4 *>(vec + x));
    if ((V & 3) == 0)
        return x < V ? __ldcg(reinterpret_cast<const float4 *>(vec + x))
                     : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    return make_float4(x < V ? __ldcg(vec + x) : -INFINITY, x + 1 < V ? __ldcg(vec + x + 1) : -INFINITY,
                       x + 2 < V ? __ldcg(vec + x + 2) : -INFINITY, x + 3 < V ? __ldcg(vec + x + 3) : -INFINITY);
}

__device__ __forceinline__ bool block_full(int V, int blk) { return (V & 3) == 0 && (blk + 1) * kBlock <= V; }

// Leaf maximum and leaf sum across the four lanes sharing a leaf.
__device__ __forceinline__ float leaf_max4(float m)
{
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    return fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
}
__device__ __forceinline__ float leaf_sum4(float s)
{
    s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 1));   // Q0 + Q1 | Q2 + Q3
    return __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 2)); // (Q0 + Q1) + (Q2 + Q3)
}
__device__ __forceinline__ float quad_max(float4 v) { return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)); }

// Canonical base-2 exponents t(x) = fma(l(x), c, -mz) of a quarter, exponentiated.
__device__ __forceinline__ void quad_exp2(float4 v, float c, float mz, float2 &e01, float2 &e23)
{
    const unsigned long long c2 = f2_pack(c, c), nmz = f2_pack(-mz, -mz);
    e01 = exp2_canon_x2(f2_fma(f2_pack(v.x, v.y), c2, nmz));
    e23 = exp2_canon_x2(f2_fma(f2_pack(v.z, v.w), c2, nmz));
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

// p(x) of entry x of one vector (recipe: RN(e2(t(x)) F_leaf), with the
// maximum of the 16-entry leaf that holds x).
__device__ __forceinline__ float prob_at(const float *vec, int V, int x, float c, RowRoots root)
{
    const int leaf = x >> 4, r_x = (x & 15) >> 2, j_x = x & 3;
    float mx = -INFINITY, lx = -INFINITY;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const float4 v = load_quarter(vec, V, false, kLeaf * leaf + 4 * r);
        mx = fmaxf(mx, quad_max(v));
        if (r == r_x) lx = j_x == 0 ? v.x : (j_x == 1 ? v.y : (j_x == 2 ? v.z : v.w));
    }
    const float mz = __fmul_rn(mx, c);
    return __fmul_rn(exp2_canon(__fmaf_rn(lx, c, -mz)), leaf_factor(mz, root.M, root.inv_s));
}

// ---- pass A: one block of one vector; the last CTA of a row decides.
// Warp w covers leaves 128 w .. 128 w + 127 of the block; lane group g (four
// lanes) covers 16 of them, 16 g + n, in four batches b (n = 4 i + b,
// i = 0..3, one load each).  After batch b, lane qq keeps leaf 4 qq + b, so
// each lane ends with four consecutive leaves, 4 qq .. 4 qq + 3 of its group:
// lane index = position of its 4-leaf node, and the warp tree over lanes is
// the pairwise tree over the warp's 128 leaves.
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
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, qq = lane & 3;
    // vectors 0..k: target positions 0..k; k+1..2k: draft positions 0..k-1
    const float *vec = v <= k ? tlog + (static_cast<size_t>(b) * (k + 1) + v) * V
                              : dlog + (static_cast<size_t>(b) * k + (v - k - 1)) * V;
    {
        const bool full = block_full(V, blk);
        const int gleaf = blk * (kBlock / kLeaf) + 128 * warp + 16 * (lane >> 2);   // the group's first leaf
        float finite = 0.0f;   // becomes NaN if a present entry or leaf maximum is not finite
        MaxSum mine[4];
#pragma unroll
        for (int bt = 0; bt < 4; ++bt) {
            float4 x4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) x4[i] = load_quarter(vec, V, full, kLeaf * (gleaf + 4 * i + bt) + 4 * qq);
            MaxSum keep{-INFINITY, 0.0f};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int leaf = gleaf + 4 * i + bt, x = kLeaf * leaf + 4 * qq;
                const bool present = full || kLeaf * leaf < V;
                const float4 q = x4[i];
                if (full) {
                    finite = __fmaf_rn(0.0f, q.x, finite); finite = __fmaf_rn(0.0f, q.y, finite);
                    finite = __fmaf_rn(0.0f, q.z, finite); finite = __fmaf_rn(0.0f, q.w, finite);
                } else {
                    if (x < V) finite = __fmaf_rn(0.0f, q.x, finite);
                    if (x + 1 < V) finite = __fmaf_rn(0.0f, q.y, finite);
                    if (x + 2 < V) finite = __fmaf_rn(0.0f, q.z, finite);
                    if (x + 3 < V) finite = __fmaf_rn(0.0f, q.w, finite);
                }
                const float mz = __fmul_rn(leaf_max4(quad_max(q)), c);
                float2 e01, e23;
                quad_exp2(q, c, mz, e01, e23);
                const float s = leaf_sum4(__fadd_rn(__fadd_rn(__fadd_rn(e01.x, e01.y), e23.x), e23.y));
                if (present) finite = __fmaf_rn(0.0f, mz, finite);
                if (i == qq) keep = present ? MaxSum{mz, s} : MaxSum{-INFINITY, 0.0f};
            }
            mine[bt] = keep;
        }
        if (finite != 0.0f) set_status(status, NQ_DEV_NONFINITE);
        MaxSum a = ms_merge(ms_merge(mine[0], mine[1]), ms_merge(mine[2], mine[3]));
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
                const float p = prob_at(tlog + (static_cast<size_t>(b) * (k + 1) + j) * V, V, d, c, roots[j]);
                const float q = prob_at(dlog + (static_cast<size_t>(b) * k + j) * V, V, d, c, roots[k + 1 + j]);
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

// Sampling weights of one quarter of a leaf of row b's chosen position and
// their serial sum: max(0, RN(p - q)) (resid) or p, with p = RN(e2(t_p) Fp).
// Called by all four lanes of the leaf (the leaf maxima are shuffled).
__device__ __forceinline__ float quarter_weights(float4 lp, float4 lq, bool resid, float c, const SampleRec &R,
                                                 float (&w)[4])
{
    const float mzp = __fmul_rn(leaf_max4(quad_max(lp)), c);
    const float Fp = leaf_factor(mzp, R.Mp, R.invSp);
    float2 p01, p23;
    quad_exp2(lp, c, mzp, p01, p23);
    w[0] = __fmul_rn(p01.x, Fp); w[1] = __fmul_rn(p01.y, Fp);
    w[2] = __fmul_rn(p23.x, Fp); w[3] = __fmul_rn(p23.y, Fp);
    if (resid) {
        const float mzq = __fmul_rn(leaf_max4(quad_max(lq)), c);
        const float Fq = leaf_factor(mzq, R.Mq, R.invSq);
        float2 q01, q23;
        quad_exp2(lq, c, mzq, q01, q23);
        const float d0 = __fsub_rn(w[0], __fmul_rn(q01.x, Fq)), d1 = __fsub_rn(w[1], __fmul_rn(q01.y, Fq));
        const float d2 = __fsub_rn(w[2], __fmul_rn(q23.x, Fq)), d3 = __fsub_rn(w[3], __fmul_rn(q23.y, Fq));
        w[0] = d0 > 0.0f ? d0 : 0.0f; w[1] = d1 > 0.0f ? d1 : 0.0f;
        w[2] = d2 > 0.0f ? d2 : 0.0f; w[3] = d3 > 0.0f ? d3 : 0.0f;
    }
    return __fadd_rn(__fadd_rn(__fadd_rn(w[0], w[1]), w[2]), w[3]);
}

// Leaf sums of the 256 consecutive leaves leaf0 .. leaf0 + 255 of row b's
// chosen position (all threads of the CTA take part): they are stored at
// out[0..255] and the node of the pairwise sum tree over them is returned
// (valid in warp 0).  Warp w covers leaves 32 w .. 32 w + 31; its lane group
// g the four leaves 4 g + i (one load per lane each), of which lane qq keeps
// leaf 4 g + qq, so lane index = leaf index within the warp.
__device__ float quarter_block(float *warp_sum, float *out, const float *pv, const float *qv, bool resid, int V,
                               int leaf0, float c, const SampleRec &R)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, qq = lane & 3;
    const int gl = leaf0 + 32 * warp + 4 * (lane >> 2);
    const bool full = (V & 3) == 0 && kLeaf * (leaf0 + kThreads) <= V;
    float4 lp[4], lq[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        lp[i] = load_quarter(pv, V, full, kLeaf * (gl + i) + 4 * qq);
        lq[i] = resid ? load_quarter(qv, V, full, kLeaf * (gl + i) + 4 * qq) : lp[i];
    }
    float keep = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float w[4];
        const float s = leaf_sum4(quarter_weights(lp[i], lq[i], resid, c, R, w));
        const bool present = full || kLeaf * (gl + i) < V;
        if (i == qq) keep = present ? s : 0.0f;
    }
    out[32 * warp + lane] = keep;
    const float node = warp_tree_sum(keep, 5);
    if (lane == 0) warp_sum[warp] = node;
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

// ---- pass B: one quarter (256 leaves) of one block of the chosen position
// of one row; the last CTA of the row descends the sum tree and writes the
// row's tokens.
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
    constexpr int kBlockLeaves = kBlock / kLeaf;   // 1024
    const int NBK = gridDim.x >> 2, blk = blockIdx.x >> 2, q = blockIdx.x & 3, b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const SampleRec R = rec[b];
    const float *pv = tlog + (static_cast<size_t>(b) * (k + 1) + R.js) * V;
    const float *qv = R.js < k ? dlog + (static_cast<size_t>(b) * k + R.js) * V : pv;
    bool resid = R.resid != 0;

    // this CTA's node of the block's pairwise sum tree (leaf sums go to lsum,
    // the node to qsum)
    {
        const float node = quarter_block(warp_sum, lsum + (static_cast<size_t>(b) * NBK + blk) * kBlockLeaves + kThreads * q,
                                         pv, qv, resid, V, blk * kBlockLeaves + kThreads * q, c, R);
        if (threadIdx.x == 0) {
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
                float n4[4];
                for (int qb = 0; qb < 4; ++qb)
                    n4[qb] = quarter_block(warp_sum,
                                           lsum + (static_cast<size_t>(b) * NBK + bb) * kBlockLeaves + kThreads * qb,
                                           pv, qv, false, V, bb * kBlockLeaves + kThreads * qb, c, R);
                if (threadIdx.x == 0) btree[bb] = __fadd_rn(__fadd_rn(n4[0], n4[1]), __fadd_rn(n4[2], n4[3]));
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
        const float4 *src = reinterpret_cast<const float4 *>(lsum + (static_cast<size_t>(b) * NBK + bstar) * kBlockLeaves) + 8 * lane;
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
    const int lstar = bstar * kBlockLeaves + 32 * lane_star + warp_descend32(mine, t);   // global leaf index

    // the chosen leaf: lanes e and e + 16 reload entry e, the weights are
    // formed exactly as in the leaf sums, lane 0 scans them in entry order
    const int e = lane & 15;
    const int x = kLeaf * lstar + e;
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
        const int xi = kLeaf * lstar + i;
        if (xi < V && pk < 0) {
            run = __fadd_rn(run, wi);
            if (t < run) pk = xi;
        }
    }
    // fallback: the last entry of the leaf with a positive weight
#pragma unroll
    for (int i = kLeaf - 1; i >= 0; --i) {
        const float wi = __shfl_sync(0xffffffffu, we, i);
        const int xi = kLeaf * lstar + i;
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
    // one (value, index) partial per (row, position, greedy CTA of 16384 entries)
    const size_t need = counters + static_cast<size_t>(B) * (k + 1) * nq::n_greedy_chunks(V) * sizeof(float2);
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
