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
// Design.  Greedy: one pass over the logits; the grid is (chunk of 16384
// entries, vector, row), every CTA reduces its chunk and writes a partial to
// the workspace, the last CTA of a row (atomic ticket, no spin-waits) combines
// the partials and decides.  Sampled: three launches -- pass A reduces every
// segment of every vector to its (max, sum) with no hand-off between warps, a
// decision kernel (one CTA per row) forms the roots, decides and draws the
// bonus token, pass B resamples the rows with a rejection.  All fp32
// arithmetic of the sampled path follows the fixed recipe documented in nq.h
// so that decisions are reproducible bit for bit.
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
              int32_t *__restrict__ out_tok, int tok_stride, int32_t *__restrict__ out_cnt,
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
            out_tok[static_cast<size_t>(b) * tok_stride + jj] = jj < n ? draft[static_cast<size_t>(b) * k + jj] : (jj == n ? tj[n] : -1);
        if (out_cnt) out_cnt[b] = n + 1;
        counters[b] = 0;   // ready for the next call
    }
}

// ------------------------------------------------------------------ sampled
//
// Arithmetic of the recipe (spec_accept_sample in nq.h): segments of 1024
// consecutive vocabulary entries carry the maximum every base-2 exponent is
// taken against; a leaf of 16 consecutive entries is summed as two serial
// chains, over its even and over its odd entries, E + O; a segment's sum is
// the pairwise tree over its 64 leaves; segments merge pairwise as (max, sum)
// nodes.
//
// Work unit: one warp, one segment at a time.  Lane l computes entries
// 32 l .. 32 l + 31 (leaves 2 l and 2 l + 1).  The warp stages its segments in
// its own slice of shared memory with cp.async: copy instruction t of lane l
// reads the 16 bytes at entry 128 t + 4 l (512 contiguous bytes per
// instruction) and stores them as chunk c = l % 8 of row r = 4 t + l / 8,
// at position c ^ (r % 8) of that 128-byte row, so that the lane that owns
// row r later reads its eight chunks with no bank conflict.  Loads in flight
// cost no registers, and the warps of pass A are independent: each writes its
// own partial and leaves (no ticket, no fence, no CTA-wide barrier); in pass
// B each warp takes a ticket and the last warp of a row finishes the row.
//
// The chains of a leaf run on the packed fp32 adds, the even and the odd
// chain in the two halves of one register pair; products that feed an add
// are formed with scalar __fmul_rn, since a packed multiply followed by a
// packed add may be fused into one fma by the code generator.  Absent
// entries (>= V) are read as -inf: they cannot raise a maximum and contribute
// an exact zero to every sum.

constexpr int kSeg = 1024;                       // entries per segment
constexpr int kSegPerBlock = kBlock / kSeg;      // 16 per pass-A CTA (two per warp)
constexpr int kLeavesPerSeg = kSeg / kLeaf;      // 64
#ifndef NQ_SAMPLE_WARPS
#define NQ_SAMPLE_WARPS 2
#endif
#ifndef NQ_SAMPLE_CTAS
#define NQ_SAMPLE_CTAS 14
#endif
constexpr int kWarpsS = NQ_SAMPLE_WARPS;         // warps per sampling CTA
constexpr int kThreadsS = 32 * kWarpsS;
constexpr int kSmemS = kWarpsS * 2 * kSeg * 4;   // two 4 KB segment buffers per warp
constexpr int kSampleCtas = NQ_SAMPLE_CTAS;      // resident CTAs per SM (launch bounds)

inline int n_segments_padded(int V) { return n_blocks(V) * kSegPerBlock; }

struct SampleRec {      // per-row decision, written by the decision kernel, read by pass B
    int js;             // first rejected position, or k if all accepted
    int resid;          // 1: draw from max(0, p_js - q_js); 0: draw from p_js
    float u;            // the draw's uniform
    float Mp, invSp, Mq, invSq;
    int done;           // 1: the decision kernel drew the token (bonus draw from p_k)
};

// Workspace layout shared by the greedy and sampled calls.
struct WsLayout {
    size_t counters_a, counters_b, part, rec, segmax, segsum, ssum, lsum, partu, total;
};

inline size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// Every section starts on a 256-byte boundary (the kernels use 8- and 16-byte
// vector accesses on some of them).
inline WsLayout ws_layout(int B, int k, int V)
{
    const size_t C = static_cast<size_t>(n_chunks(V));   // greedy partials per vector
    const size_t NSP = static_cast<size_t>(n_segments_padded(V));
    const size_t NV = static_cast<size_t>(2 * k + 1);
    WsLayout L;
    L.counters_a = 0;
    L.counters_b = align256(static_cast<size_t>(B) * 4);
    L.part = L.counters_b + align256(static_cast<size_t>(B) * 4);
    // greedy: one (value, index) per 4096-entry chunk; sampled: one (max, sum)
    // per segment pair (warp of pass A), NSP / 2 of them
    const size_t P = C > NSP / 2 ? C : NSP / 2;
    L.rec = L.part + align256(static_cast<size_t>(B) * NV * P * sizeof(float2));
    L.segmax = L.rec + align256(static_cast<size_t>(B) * sizeof(SampleRec));        // per (row, vector, segment)
    L.segsum = L.segmax + align256(static_cast<size_t>(B) * NV * NSP * sizeof(float));   // per (row, vector, segment)
    L.ssum = L.segsum + align256(static_cast<size_t>(B) * NV * NSP * sizeof(float));
    L.lsum = L.ssum + align256(static_cast<size_t>(B) * NSP * sizeof(float));         // per (row, segment)
    L.partu = L.lsum + align256(static_cast<size_t>(B) * NSP * kLeavesPerSeg * sizeof(float));  // features: u per partial
    L.total = L.partu + static_cast<size_t>(B) * NV * P * sizeof(float);
    return L;
}

// Stage the 1024 entries x0 .. x0 + 1023 of one vector in `buf` (4 KB of the
// warp's shared memory) in the swizzled row layout; absent entries are zero.
// al >= 1 (V % 4 == 0, 16-byte aligned vectors): cp.async, completed by the
// caller's wait; al == 0: synchronous loads.
__device__ __forceinline__ void stage_segment(float *buf, const float *vec, int V, int x0, int al)
{
    const int lane = threadIdx.x & 31;
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(buf));
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const int x = x0 + 128 * t + 4 * lane;
        const int r = 4 * t + (lane >> 3), cch = lane & 7;
        const uint32_t dst = sbase + static_cast<uint32_t>(r * 128 + ((cch ^ (r & 7)) << 4));
        if (al >= 1) {
            const int bytes = x < V ? 16 : 0;
            const float *src = x < V ? vec + x : vec;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(bytes) : "memory");
        } else {
            float4 q;
            q.x = x < V ? __ldcg(vec + x) : 0.0f;
            q.y = x + 1 < V ? __ldcg(vec + x + 1) : 0.0f;
            q.z = x + 2 < V ? __ldcg(vec + x + 2) : 0.0f;
            q.w = x + 3 < V ? __ldcg(vec + x + 3) : 0.0f;
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" :: "r"(dst), "f"(q.x), "f"(q.y), "f"(q.z), "f"(q.w) : "memory");
        }
    }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// This lane's 32 entries of a staged segment (np of them present; the rest -inf).
__device__ __forceinline__ void read_lane(const float *buf, int np, float (&v)[32])
{
    const int lane = threadIdx.x & 31;
    const uint32_t row = static_cast<uint32_t>(__cvta_generic_to_shared(buf)) + static_cast<uint32_t>(lane * 128);
#pragma unroll
    for (int cch = 0; cch < 8; ++cch) {
        float4 q;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(q.x), "=f"(q.y), "=f"(q.z), "=f"(q.w) : "r"(row + static_cast<uint32_t>((cch ^ (lane & 7)) << 4)));
        v[4 * cch] = q.x; v[4 * cch + 1] = q.y; v[4 * cch + 2] = q.z; v[4 * cch + 3] = q.w;
    }
    if (np < 32) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = i < np ? v[i] : -INFINITY;
    }
}

__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Smallest of three, NaN if any operand is NaN.
__device__ __forceinline__ float min3_nan(float a, float b, float c)
{
    float d;
    asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float pair_sum(unsigned long long eo)
{
    const float2 v = f2_unpack(eo);
    return __fadd_rn(v.x, v.y);
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

__device__ __forceinline__ float warp_max(float m)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    return m;
}

// (mz, s) of one segment; every lane of the warp calls it with its 32 entries,
// np of which are present.  `finite` becomes NaN if a present entry's
// exponent t is not finite (a non-finite logit or segment maximum).
//
// With FEAT it also returns u = sum of e2(t) t over the segment (t relative to
// the segment maximum), from which the distribution's entropy follows; any
// order of summation (a float feature, not a decision).
template <bool FEAT = false>
__device__ __forceinline__ MaxSum segment_ms(const float (&v)[32], int np, float c, float &finite, float *u_out = nullptr)
{
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; i += 2) mx = max3(mx, v[i], v[i + 1]);
    const float mz = __fmul_rn(warp_max(mx), c);
    const unsigned long long c2 = f2_pack(c, c), nmz = f2_pack(-mz, -mz), z2 = f2_pack(0.0f, 0.0f);
    unsigned long long fin = z2, eo[2], uu = z2;
    // A lane whose 32 entries are all present and whose smallest exponent
    // t = l c - mz is at least -125 (t grows with l, so that one t bounds the
    // rest; NaN fails the test) needs neither the underflow select nor the
    // per-entry finiteness check: every t lies in [-125, 0.5].
    bool fast = false;
    if (np == 32) {
        float mn = v[0];
#pragma unroll
        for (int i = 1; i < 31; i += 2) mn = min3_nan(mn, v[i], v[i + 1]);
        mn = min3_nan(mn, v[31], v[31]);
        fast = __fmaf_rn(mn, c, -mz) >= -125.0f;
    }
    if (fast) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const unsigned long long t = f2_fma(f2_pack(v[16 * h + 2 * p], v[16 * h + 2 * p + 1]), c2, nmz);
                const float2 e = exp2_canon_x2_inrange(t);
                eo[h] = p == 0 ? f2_pack(e.x, e.y) : f2_add(eo[h], f2_pack(e.x, e.y));
                if constexpr (FEAT) uu = f2_fma(f2_pack(e.x, e.y), t, uu);
            }
        }
    } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const unsigned long long t = f2_fma(f2_pack(v[16 * h + 2 * p], v[16 * h + 2 * p + 1]), c2, nmz);
                fin = f2_fma(z2, t, fin);
                const float2 e = exp2_canon_x2(t);
                eo[h] = p == 0 ? f2_pack(e.x, e.y) : f2_add(eo[h], f2_pack(e.x, e.y));
                if constexpr (FEAT) {
                    // absent entries: t = -inf, e = 0; count their product as 0
                    const float2 tv = f2_unpack(t);
                    uu = f2_fma(f2_pack(e.x, e.y), f2_pack(e.x > 0.0f ? tv.x : 0.0f, e.y > 0.0f ? tv.y : 0.0f), uu);
                }
            }
        }
        if (np == 32) {
            const float2 f = f2_unpack(fin);
            finite = __fadd_rn(finite, __fadd_rn(f.x, f.y));
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < np) finite = __fmaf_rn(0.0f, __fmaf_rn(v[i], c, -mz), finite);
        }
    }
    // warp-wide from here (every lane, whichever branch it took)
    if constexpr (FEAT) *u_out = warp_tree_sum(pair_sum(uu), 5);
    const float s = warp_tree_sum(__fadd_rn(pair_sum(eo[0]), pair_sum(eo[1])), 5);
    return MaxSum{mz, s};
}

struct RowRoots { float M, inv_s; };

// (max, sum, u) merge for the entropy feature: the larger max survives, the
// smaller node's sum and u are rescaled by f = e2(d), d = m_small - m_large,
// and u also gains d s_small (its exponents move by d).  Pads: (-inf, 0, 0).
struct MSU { float m, s, u; };
__device__ __forceinline__ MSU msu_merge(MSU a, MSU b)
{
    const bool a_big = a.m >= b.m || b.m != b.m;
    const MSU big = a_big ? a : b, sm = a_big ? b : a;
    if (sm.m == -INFINITY) return big;
    const float d = __fsub_rn(sm.m, big.m), f = exp2_canon(d);
    return MSU{big.m, __fmaf_rn(sm.s, f, big.s), __fmaf_rn(__fmaf_rn(d, sm.s, sm.u), f, big.u)};
}

__device__ __forceinline__ float seg_factor(float mz_seg, float M, float inv_s)
{
    return __fmul_rn(exp2_canon(__fsub_rn(mz_seg, M)), inv_s);
}

// p(x) of entry x of one vector (recipe: RN(e2(t(x)) F_seg)).
__device__ __forceinline__ float prob_from(float lx, float mz, float c, RowRoots root)
{
    return __fmul_rn(exp2_canon(__fmaf_rn(lx, c, -mz)), seg_factor(mz, root.M, root.inv_s));
}

// Sampling weights of a lane's 32 entries of row b's chosen position,
// max(0, RN(p - q)) (resid) or p, with p = RN(e2(t_p) Fp); returns the two
// leaf sums (entries 0..15 and 16..31).
__device__ __forceinline__ float2 lane_leaf_sums(const float (&lp)[32], const float (&lq)[32], bool resid,
                                                 float c, float mzp, float Fp, float mzq, float Fq)
{
    const unsigned long long c2 = f2_pack(c, c), nmzp = f2_pack(-mzp, -mzp), nmzq = f2_pack(-mzq, -mzq);
    unsigned long long eo[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int i = 16 * h + 2 * p;
            const float2 ep = exp2_canon_x2(f2_fma(f2_pack(lp[i], lp[i + 1]), c2, nmzp));
            float w0 = __fmul_rn(ep.x, Fp), w1 = __fmul_rn(ep.y, Fp);
            if (resid) {
                const float2 eq = exp2_canon_x2(f2_fma(f2_pack(lq[i], lq[i + 1]), c2, nmzq));
                const float d0 = __fsub_rn(w0, __fmul_rn(eq.x, Fq)), d1 = __fsub_rn(w1, __fmul_rn(eq.y, Fq));
                w0 = d0 > 0.0f ? d0 : 0.0f;
                w1 = d1 > 0.0f ? d1 : 0.0f;
            }
            eo[h] = p == 0 ? f2_pack(w0, w1) : f2_add(eo[h], f2_pack(w0, w1));
        }
    }
    return make_float2(pair_sum(eo[0]), pair_sum(eo[1]));
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

// The row's emitted tokens: draft[b][0..js-1], then tok, then -1 pads.
__device__ __forceinline__ void write_row(int32_t *out_tok, int32_t *out_cnt, const int32_t *draft, int b, int k,
                                          int js, int tok)
{
    for (int jj = 0; jj <= k; ++jj)
        out_tok[static_cast<size_t>(b) * (k + 1) + jj] = jj < js ? draft[static_cast<size_t>(b) * k + jj] : (jj == js ? tok : -1);
    out_cnt[b] = js + 1;
}

// Scan leaf `leaf` of the chosen position with the remaining t (one warp):
// lanes e and e + 16 form entry e's weight exactly as in the leaf sums, the
// entries are scanned in order; the first whose running sum exceeds t is the
// token (fallback: the last entry of the leaf with a positive weight).
__device__ int scan_leaf(const float *pv, const float *qv, bool resid, int V, int leaf, float c, float mzp, float Fp,
                         float mzq, float Fq, float t)
{
    const int lane = threadIdx.x & 31;
    const int x = kLeaf * leaf + (lane & 15);
    const bool present = x < V;
    const float lp = present ? __ldcg(pv + x) : -INFINITY;
    float we = __fmul_rn(exp2_canon(__fmaf_rn(lp, c, -mzp)), Fp);
    if (resid) {
        const float lq = present ? __ldcg(qv + x) : -INFINITY;
        const float d = __fsub_rn(we, __fmul_rn(exp2_canon(__fmaf_rn(lq, c, -mzq)), Fq));
        we = d > 0.0f ? d : 0.0f;
    }
    if (!present) we = 0.0f;
    int pk = -1;
    float run = 0.0f;
#pragma unroll
    for (int i = 0; i < kLeaf; ++i) {
        const float wi = __shfl_sync(0xffffffffu, we, i);
        const int xi = kLeaf * leaf + i;
        if (xi < V && pk < 0) {
            run = __fadd_rn(run, wi);
            if (t < run) pk = xi;
        }
    }
#pragma unroll
    for (int i = kLeaf - 1; i >= 0; --i) {
        const float wi = __shfl_sync(0xffffffffu, we, i);
        const int xi = kLeaf * leaf + i;
        if (pk < 0 && xi < V && wi > 0.0f) pk = xi;
    }
    return pk;
}

// Choose one of the 64 leaves of segment sg from this lane's pair of leaf
// sums (leaves 2 l and 2 l + 1): the pairwise tree over the lanes' pairs,
// then the pair; returns the global leaf index and updates t.
__device__ __forceinline__ int descend_segment(float2 lpair, int sg, float &t)
{
    const int pstar = warp_descend32(__fadd_rn(lpair.x, lpair.y), t);
    const float left = __shfl_sync(0xffffffffu, lpair.x, pstar), right = __shfl_sync(0xffffffffu, lpair.y, pstar);
    int leaf = kLeavesPerSeg * sg + 2 * pstar;
    if (!(t < left || !(right > 0.0f))) {
        t = __fsub_rn(t, left);
        leaf += 1;
    }
    return leaf;
}

// A draw from p of one target vector by the recipe's two-level rule (one warp;
// every lane returns the token): segment weights W = RN(s_seg F_seg) from the
// segment maxima and sums of the (max, sum) pass, the pairwise tree over the
// (up to 512) segments with 16 consecutive segments per lane, t = RN(u R);
// then the chosen segment's 64 leaf sums of p, its leaf tree and the scan of
// the chosen leaf.
__device__ int sample_p_warp(const float *pv, int V, const float *smz, const float *ssum, int NSP, float c, float M,
                             float invS, float u)
{
    const int lane = threadIdx.x & 31;
    float w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int sg = 16 * lane + i;
        w[i] = 0.0f;
        if (sg < NSP && sg * kSeg < V) w[i] = __fmul_rn(__ldcg(ssum + sg), seg_factor(__ldcg(smz + sg), M, invS));
    }
    float n[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) n[i] = w[i];
#pragma unroll
    for (int wd = 1; wd < 16; wd <<= 1)
#pragma unroll
        for (int i = 0; i < 16; i += 2 * wd) n[i] = __fadd_rn(n[i], n[i + wd]);
    const float root = warp_tree_sum(n[0], 5);
    float t = __fmul_rn(u, root);
    const int lstar = warp_descend32(n[0], t);
    float mine = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float x = __shfl_sync(0xffffffffu, w[i], lstar);
        if (lane == i) mine = x;
    }
    const int sg = 16 * lstar + warp_descend32(mine, t);   // lanes 16..31 hold zeros
    const float mz = __ldcg(smz + sg);
    const float F = seg_factor(mz, M, invS);
    const int x0 = sg * kSeg + 32 * lane;
    float l[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) l[i] = x0 + i < V ? __ldcg(pv + x0 + i) : -INFINITY;
    const float2 lpair = lane_leaf_sums(l, l, false, c, mz, F, 0.0f, 0.0f);
    const int leaf = descend_segment(lpair, sg, t);
    return scan_leaf(pv, pv, false, V, leaf, c, mz, F, 0.0f, 0.0f, t);
}

// ---- pass A: warp w of CTA (x, v, b) reduces segments 2 g and 2 g + 1
// (g = kWarpsS x + w) of vector v of row b, staged in buf (the caller has
// committed one cp.async group per segment): their (max, sum) go to segmax /
// segsum and their merge to part (with u to partu when FEAT and v is a draft
// vector).  No warp waits for another: the roots and the decisions are taken
// by the decision kernel after the pass, which costs one launch (overlapped
// as a dependent launch) and takes a fence and an atomic ticket off every
// warp's path (84 against 89 us at B = 64, k = 4, V = 152064).
template <bool FEAT>
__device__ __forceinline__ void reduce_pair(int k, int V, float c, float2 *__restrict__ part, float *__restrict__ segmax,
                                       float *__restrict__ segsum, float *__restrict__ partu, unsigned int *status,
                                       int NW, int b, int v, int g, const float *buf)
{
    const int NV = 2 * k + 1, NSP = 2 * NW;
    const int lane = threadIdx.x & 31;
    float *segm = segmax + (static_cast<size_t>(b) * NV + v) * NSP;
    float *segs = segsum + (static_cast<size_t>(b) * NV + v) * NSP;
    float finite = 0.0f;
    MaxSum seg[2];
    float su[2] = {0.0f, 0.0f};
    const bool want_u = FEAT && v > k;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        if (i == 0) cp_async_wait<1>(); else cp_async_wait<0>();   // segment 1 still in flight for i = 0
        __syncwarp();
        const int sg = 2 * g + i;
        seg[i] = MaxSum{-INFINITY, 0.0f};
        if (sg * kSeg < V) {                          // warp-uniform
            const int np = min(max(V - (sg * kSeg + 32 * lane), 0), 32);
            float l[32];
            read_lane(buf + i * kSeg, np, l);
            if (want_u) seg[i] = segment_ms<true>(l, np, c, finite, &su[i]);
            else seg[i] = segment_ms(l, np, c, finite);
            if (lane == 0) {
                segm[sg] = seg[i].m;
                segs[sg] = seg[i].s;
            }
        }
    }
    if (finite != 0.0f) set_status(status, NQ_DEV_NONFINITE);
    const MaxSum a = ms_merge(seg[0], seg[1]);
    if (want_u && lane == 0)
        partu[(static_cast<size_t>(b) * NV + v) * NW + g] =
            msu_merge(MSU{seg[0].m, seg[0].s, su[0]}, MSU{seg[1].m, seg[1].s, su[1]}).u;
    if (lane == 0) part[(static_cast<size_t>(b) * NV + v) * NW + g] = make_float2(a.m, a.s);
}

template <bool FEAT>
__global__ void __launch_bounds__(kThreadsS, kSampleCtas)
sample_a_kernel(const float *__restrict__ dlog, const float *__restrict__ tlog, int k, int V, float c, int al,
                float2 *__restrict__ part, float *__restrict__ segmax, float *__restrict__ segsum,
                float *__restrict__ partu, unsigned int *status)
{
    // the decision kernel may be scheduled now; it waits (griddepcontrol.wait)
    // for this grid to complete before reading anything this grid writes
    asm volatile("griddepcontrol.launch_dependents;");
    extern __shared__ __align__(128) float smem_s[];
    const int warp = threadIdx.x >> 5;
    const int v = blockIdx.y, b = blockIdx.z, g = blockIdx.x * kWarpsS + warp, NW = gridDim.x * kWarpsS;
    float *buf = smem_s + warp * 2 * kSeg;
    // vectors 0..k: target positions 0..k; k+1..2k: draft positions 0..k-1
    const float *vec = v <= k ? tlog + (static_cast<size_t>(b) * (k + 1) + v) * V
                              : dlog + (static_cast<size_t>(b) * k + (v - k - 1)) * V;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        if ((2 * g + i) * kSeg < V) stage_segment(buf + i * kSeg, vec, V, (2 * g + i) * kSeg, al);
        cp_async_commit();
    }
    reduce_pair<FEAT>(k, V, c, part, segmax, segsum, partu, status, NW, b, v, g, buf);
}

// ---- decision kernel: CTA b takes row b.  Warp w forms the roots (M, 1/S) of
// vectors w, w + kDecWarps, ... from pass A's partials (warp 0 first loads the
// logits at the drafted ids); then warp 0 takes the row's decisions while
// warp 1 draws the bonus token from p_k, and warp 0 writes the record the
// resample pass reads (and the row's tokens when every draft is accepted).
constexpr int kDecWarps = 16;

template <bool FEAT>
__global__ void __launch_bounds__(kDecWarps * 32)
decide_kernel(const int32_t *__restrict__ draft, const float *__restrict__ dlog, const float *__restrict__ tlog,
              int k, int V, float c, const uint64_t *__restrict__ seeds, uint64_t round,
              const float2 *__restrict__ part, const float *__restrict__ segmax, const float *__restrict__ segsum,
              const float *__restrict__ partu, SampleRec *__restrict__ rec, int32_t *__restrict__ out_tok,
              int32_t *__restrict__ out_cnt, float *__restrict__ feat, unsigned int *status, int NW)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ float2 sroot[2 * kMaxK + 1];
    __shared__ float sent[2 * kMaxK + 1];
    __shared__ int sbonus;
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NV = 2 * k + 1, NSP = 2 * NW;
    const float *segrow = segmax + static_cast<size_t>(b) * NV * NSP;
    // warp 0, lane j < k: the logits and segment maxima at the drafted id d_j,
    // loaded while the roots are formed
    int dj = 0;
    float lxp = 0.0f, mzp = 0.0f, lxq = 0.0f, mzq = 0.0f;
    if (warp == 0 && lane < k) {
        dj = draft[static_cast<size_t>(b) * k + lane];
        if (dj >= 0 && dj < V) {
            lxp = __ldcg(tlog + (static_cast<size_t>(b) * (k + 1) + lane) * V + dj);
            mzp = __ldcg(segrow + static_cast<size_t>(lane) * NSP + (dj >> 10));
            lxq = __ldcg(dlog + (static_cast<size_t>(b) * k + lane) * V + dj);
            mzq = __ldcg(segrow + static_cast<size_t>(k + 1 + lane) * NSP + (dj >> 10));
        }
    }
    for (int v = warp; v < NV; v += kDecWarps) {
        MaxSum n[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int gi = 8 * lane + i;
            n[i] = MaxSum{-INFINITY, 0.0f};
            if (gi < NW) {
                const float2 p = __ldcg(part + (static_cast<size_t>(b) * NV + v) * NW + gi);
                n[i] = MaxSum{p.x, p.y};
            }
        }
        MaxSum a = ms_merge(ms_merge(ms_merge(n[0], n[1]), ms_merge(n[2], n[3])),
                            ms_merge(ms_merge(n[4], n[5]), ms_merge(n[6], n[7])));
        a = warp_tree_ms(a, lane, 5);
        if (FEAT && v > k) {
            // entropy of the draft distribution in nats: H = ln 2 (log2 S - U / S),
            // U = sum of 2^(l c - M) (l c - M) over the vector
            MSU nu[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int gi = 8 * lane + i;
                nu[i] = MSU{n[i].m, n[i].s, gi < NW ? __ldcg(partu + (static_cast<size_t>(b) * NV + v) * NW + gi) : 0.0f};
            }
            MSU r = msu_merge(msu_merge(msu_merge(nu[0], nu[1]), msu_merge(nu[2], nu[3])),
                              msu_merge(msu_merge(nu[4], nu[5]), msu_merge(nu[6], nu[7])));
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const MSU other{__shfl_xor_sync(0xffffffffu, r.m, o), __shfl_xor_sync(0xffffffffu, r.s, o),
                                __shfl_xor_sync(0xffffffffu, r.u, o)};
                r = msu_merge(r, other);
            }
            if (lane == 0) sent[v] = 0.69314718f * (log2f(r.s) - r.u / r.s);
        }
        if (lane == 0) sroot[v] = make_float2(a.m, __frcp_rn(a.s));
    }
    __syncthreads();
    if (warp > 1) return;
    auto root_of = [&](int vv) { const float2 r = sroot[vv]; return RowRoots{r.x, r.y}; };
    const uint64_t seed = seeds[b];
    if (warp == 1) {
        // the bonus token from p_k by the two-level rule (segment weights from
        // pass A), drawn while warp 0 decides; used if every draft is accepted
        const RowRoots rk = root_of(k);
        const int pk = sample_p_warp(tlog + (static_cast<size_t>(b) * (k + 1) + k) * V, V,
                                     segrow + static_cast<size_t>(k) * NSP,
                                     segsum + (static_cast<size_t>(b) * NV + k) * NSP, NSP, c, rk.M, rk.inv_s,
                                     philox_uniform(seed, static_cast<uint32_t>(k), 2u, round));
        if (lane == 0) sbonus = pk;
        asm volatile("bar.sync 1, 64;" ::: "memory");   // warps 0 and 1: sbonus is written
        return;
    }

    // ---- warp 0.  Decisions: accept d_j iff u_j < p_j(d_j) / q_j(d_j); first
    // rejection j*
    bool reject = false;
    float conf = 0.0f;
    if (lane < k) {
        const int j = lane;
        if (dj < 0 || dj >= V) {
            set_status(status, NQ_DEV_BAD_TOKEN);
            reject = true;
        } else {
            const float p = prob_from(lxp, mzp, c, root_of(j));
            const float q = prob_from(lxq, mzq, c, root_of(k + 1 + j));
            conf = q;
            const float ratio = __fdiv_rn(p, q);
            const float u = philox_uniform(seed, static_cast<uint32_t>(j), 0u, round);
            reject = !(u < ratio);
        }
    }
    if constexpr (FEAT) {
        // the step's features over the k drafted positions (lanes 0..k-1)
        const float h = lane < k ? sent[k + 1 + lane] : 0.0f;
        float sh = h, sc = conf, mh = lane < k ? h : -INFINITY, mc = lane < k ? conf : INFINITY;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            sh += __shfl_xor_sync(0xffffffffu, sh, o);
            sc += __shfl_xor_sync(0xffffffffu, sc, o);
            mh = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, o));
            mc = fminf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
        }
        if (lane == 0) {
            float *f = feat + static_cast<size_t>(b) * 4;
            f[0] = sh / k; f[1] = sc / k; f[2] = mh; f[3] = mc;
        }
    }
    const unsigned int rej = __ballot_sync(0xffffffffu, reject);
    const int js = rej ? __ffs(rej) - 1 : k;
    // every draft accepted: the bonus token (warp 1's draw), and the resample
    // pass skips the row
    asm volatile("bar.sync 1, 64;" ::: "memory");       // warps 0 and 1: sbonus is written
    if (js == k && lane == 0) write_row(out_tok, out_cnt, draft, b, k, k, sbonus);
    if (lane == 0) {
        const RowRoots rp = root_of(js);
        SampleRec r;
        r.js = js;
        r.resid = js < k;
        r.u = philox_uniform(seed, static_cast<uint32_t>(js), js < k ? 1u : 2u, round);
        r.Mp = rp.M;
        r.invSp = rp.inv_s;
        if (js < k) {
            const RowRoots rq = root_of(k + 1 + js);
            r.Mq = rq.M;
            r.invSq = rq.inv_s;
        } else {
            r.Mq = 0.0f;
            r.invSq = 0.0f;
        }
        r.done = js == k;
        rec[b] = r;
    }
}

// Leaf sums of segment sg of row b's chosen position from its staged entries
// (pbuf, and qbuf for the residual), stored at lrow[64 sg + ...]; returns the
// segment's sum (every lane).
__device__ __forceinline__ float segment_leaf_sums(const float *pbuf, const float *qbuf, bool resid, int V, int sg,
                                                   float c, const SampleRec &R, const float *smp, const float *smq,
                                                   float *lrow)
{
    const int lane = threadIdx.x & 31;
    const int np = min(max(V - (sg * kSeg + 32 * lane), 0), 32);
    const float mzp = __ldcg(smp + sg);
    const float Fp = seg_factor(mzp, R.Mp, R.invSp);
    float lp[32], lq[32];
    read_lane(pbuf, np, lp);
    float2 ls;
    if (resid) {
        const float mzq = __ldcg(smq + sg);
        const float Fq = seg_factor(mzq, R.Mq, R.invSq);
        read_lane(qbuf, np, lq);
        ls = lane_leaf_sums(lp, lq, true, c, mzp, Fp, mzq, Fq);
    } else {
        ls = lane_leaf_sums(lp, lp, false, c, mzp, Fp, 0.0f, 0.0f);
    }
    *reinterpret_cast<float2 *>(lrow + kLeavesPerSeg * sg + 2 * lane) = ls;
    return warp_tree_sum(__fadd_rn(ls.x, ls.y), 5);
}

// ---- pass B: warp w of CTA (x, b) forms the leaf sums of segment kWarpsS x + w of
// row b's chosen position; the last warp of the row descends the sum tree
// and writes the row's tokens.
__global__ void __launch_bounds__(kThreadsS, kSampleCtas)
sample_b_kernel(const int32_t *__restrict__ draft, const float *__restrict__ dlog, const float *__restrict__ tlog,
                int k, int V, float c, int al, int32_t *__restrict__ out_tok, int32_t *__restrict__ out_cnt,
                unsigned int *__restrict__ counters, const SampleRec *__restrict__ rec,
                const float *__restrict__ segmax, const float *__restrict__ segsum, float *__restrict__ ssum,
                float *__restrict__ lsum)
{
    // launched as a programmatic dependent of the decision pass: wait for that
    // grid to complete (its records and partials visible) before anything else
    asm volatile("griddepcontrol.wait;" ::: "memory");
    extern __shared__ __align__(128) float smem_s[];
    const int NSP = gridDim.x * kWarpsS, NV = 2 * k + 1, NBK = NSP / kSegPerBlock, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sg = blockIdx.x * kWarpsS + warp;
    float *pbuf = smem_s + warp * 2 * kSeg, *qbuf = pbuf + kSeg;
    const SampleRec R = rec[b];
    if (R.done) return;                                  // the decision kernel drew the bonus token
    const float *pv = tlog + (static_cast<size_t>(b) * (k + 1) + R.js) * V;
    const float *qv = R.js < k ? dlog + (static_cast<size_t>(b) * k + R.js) * V : pv;
    const float *smp = segmax + (static_cast<size_t>(b) * NV + R.js) * NSP;
    const float *smq = segmax + (static_cast<size_t>(b) * NV + (R.js < k ? k + 1 + R.js : R.js)) * NSP;
    float *lrow = lsum + static_cast<size_t>(b) * NSP * kLeavesPerSeg;
    float *srow = ssum + static_cast<size_t>(b) * NSP;
    bool resid = R.resid != 0;

    bool last;
    {
        float s = 0.0f;
        if (sg * kSeg < V) {                              // warp-uniform
            stage_segment(pbuf, pv, V, sg * kSeg, al);
            if (resid) stage_segment(qbuf, qv, V, sg * kSeg, al);
            cp_async_commit();
            cp_async_wait<0>();
            __syncwarp();
            s = segment_leaf_sums(pbuf, qbuf, resid, V, sg, c, R, smp, smq, lrow);
        } else {
            *reinterpret_cast<float2 *>(lrow + kLeavesPerSeg * sg + 2 * lane) = make_float2(0.0f, 0.0f);
        }
        unsigned int prev = 0;
        __syncwarp();   // every lane's leaf sums are ordered before lane 0's fence
        if (lane == 0) {
            srow[sg] = s;
            __threadfence();
            prev = atomicAdd(&counters[b], 1u);
        }
        last = __shfl_sync(0xffffffffu, prev, 0) == static_cast<unsigned int>(NSP - 1);
    }
    if (!last) return;
    __threadfence();

    // ---- last warp of row b.  Block totals (lane = block): pairwise over the
    // block's 16 segment sums.
    auto block_total = [&](int bb) {
        float n[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) n[i] = __ldcg(srow + kSegPerBlock * bb + i);
#pragma unroll
        for (int w = 1; w < 16; w <<= 1)
#pragma unroll
            for (int i = 0; i < 16; i += 2 * w) n[i] = __fadd_rn(n[i], n[i + w]);
        return n[0];
    };
    float bval = lane < NBK ? block_total(lane) : 0.0f;
    // all-zero residual (rounding): draw from p_js instead, by the two-level rule
    const float root = warp_tree_sum(bval, 5);
    if (resid && !(root > 0.0f)) {
        const int pk = sample_p_warp(pv, V, smp, segsum + (static_cast<size_t>(b) * NV + R.js) * NSP, NSP, c, R.Mp,
                                     R.invSp, R.u);
        if (lane == 0) {
            write_row(out_tok, out_cnt, draft, b, k, R.js, pk);
            counters[b] = 0;
        }
        return;
    }

    // descent: blocks (32 lanes, zero pads), the chosen block's 16 segments,
    // the chosen segment's 64 leaves (pairs per lane, then the pair)
    float t = __fmul_rn(R.u, root);
    const int bstar = warp_descend32(bval, t);
    const float sval = lane < kSegPerBlock ? __ldcg(srow + kSegPerBlock * bstar + lane) : 0.0f;
    const int sstar = kSegPerBlock * bstar + warp_descend32(sval, t);
    const float2 lpair = __ldcg(reinterpret_cast<const float2 *>(lrow + kLeavesPerSeg * sstar) + lane);
    const int lstar = descend_segment(lpair, sstar, t);
    const float mzp = __ldcg(smp + sstar);
    const float Fp = seg_factor(mzp, R.Mp, R.invSp);
    float mzq = 0.0f, Fq = 0.0f;
    if (resid) {
        mzq = __ldcg(smq + sstar);
        Fq = seg_factor(mzq, R.Mq, R.invSq);
    }
    const int pk = scan_leaf(pv, qv, resid, V, lstar, c, mzp, Fp, mzq, Fq, t);
    if (lane == 0) {
        write_row(out_tok, out_cnt, draft, b, k, R.js, pk);
        counters[b] = 0;
    }
}

// Opt the two sampling kernels into their 64 KB of dynamic shared memory,
// once per device.
cudaError_t allow_sampling_smem()
{
    static std::mutex mu;
    static bool done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(sample_a_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemS);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(sample_a_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemS);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(sample_b_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemS);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

// k = 0 only for the draft argmax (no drafts, one position per row).
nq_status check_accept(int B, int k, int V, const void *ws, size_t ws_bytes)
{
    if (B < 1 || B > 65535 || k < 0 || k > kMaxK || V < 1 || V > kMaxChunks * kChunk) return NQ_ERR_ARG;
    if (!ws) return NQ_ERR_ARG;
    if (!aligned16(ws)) return NQ_ERR_ALIGN;
    if (ws_bytes < ws_layout(B, k, V).total) return NQ_ERR_WORKSPACE;
    return NQ_OK;
}

}  // namespace
}  // namespace nq

extern "C" size_t spec_accept_workspace_bytes(int B, int k, int V)
{
    if (B < 1 || B > 65535 || k < 0 || k > nq::kMaxK || V < 1 || V > nq::kMaxChunks * nq::kChunk) return 0;
    return nq::ws_layout(B, k, V).total;
}

extern "C" nq_status spec_accept_greedy(const int32_t *draft, const float *tgt_logits, int B, int k, int V,
                                        int32_t *out_tok, int32_t *out_cnt, void *ws, size_t ws_bytes,
                                        cudaStream_t stream)
{
    if (k < 1) return NQ_ERR_ARG;
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
    nq::greedy_kernel<<<grid, nq::kThreads, 0, stream>>>(draft, tgt_logits, k, V, out_tok, k + 1, out_cnt,
                                                         reinterpret_cast<unsigned int *>(w + L.counters_a),
                                                         reinterpret_cast<float2 *>(w + L.part), status);
    return nq::cuda_status(cudaGetLastError());
}

extern "C" nq_status spec_draft_argmax(const float *logits, int M, int V, int32_t *tok, int tok_stride, void *ws,
                                       size_t ws_bytes, cudaStream_t stream)
{
    // the greedy kernel with no drafts: t_0 = argmax of each row, emitted alone
    nq_status st = nq::check_accept(M, 0, V, ws, ws_bytes);
    if (st != NQ_OK) return st;
    if (!logits || !tok || tok_stride < 1) return NQ_ERR_ARG;
    if (!nq::aligned16(logits) || (reinterpret_cast<uintptr_t>(tok) & 3u) != 0) return NQ_ERR_ALIGN;
    unsigned int *status = nq::device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    const nq::WsLayout L = nq::ws_layout(M, 0, V);
    char *w = static_cast<char *>(ws);
    dim3 grid(nq::n_greedy_chunks(V), 1, M);
    nq::greedy_kernel<<<grid, nq::kThreads, 0, stream>>>(nullptr, logits, 0, V, tok, tok_stride, nullptr,
                                                         reinterpret_cast<unsigned int *>(w + L.counters_a),
                                                         reinterpret_cast<float2 *>(w + L.part), status);
    return nq::cuda_status(cudaGetLastError());
}

namespace nq {
namespace {
nq_status launch_sample(const int32_t *draft, const float *draft_logits, const float *tgt_logits, int B, int k,
                        int V, float temperature, const uint64_t *seeds, uint64_t round, int32_t *out_tok,
                        int32_t *out_cnt, void *ws, size_t ws_bytes, float *features, cudaStream_t stream)
{
    if (k < 1) return NQ_ERR_ARG;
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
    auto *segmax = reinterpret_cast<float *>(w + L.segmax);
    // staging: cp.async of 16-byte pieces when every vector starts on a
    // 16-byte boundary (V % 4 == 0; the pointers are 16-byte aligned)
    const int al = (V % 4) == 0 ? 1 : 0;
    if (nq::allow_sampling_smem() != cudaSuccess) return NQ_ERR_CUDA;
    const int nsp = nq::n_segments_padded(V);
    dim3 grid_a(nsp / (2 * nq::kWarpsS), 2 * k + 1, B);   // one warp per segment pair
    auto ka = features ? nq::sample_a_kernel<true> : nq::sample_a_kernel<false>;
    ka<<<grid_a, nq::kThreadsS, nq::kSmemS, stream>>>(draft_logits, tgt_logits, k, V, c, al,
                                                      reinterpret_cast<float2 *>(w + L.part), segmax,
                                                      reinterpret_cast<float *>(w + L.segsum),
                                                      reinterpret_cast<float *>(w + L.partu), status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return NQ_ERR_CUDA;
    // the decision kernel and pass B as programmatic dependent launches when
    // pass A fills the GPU: their CTAs are scheduled while the grid before
    // drains and block in griddepcontrol.wait until it completes.  Below one
    // wave of pass-A CTAs (B = 1 rounds) plain launches measured faster inside
    // a decode round (32 vs 37 us with dependent launches); griddepcontrol.wait
    // returns at once then.
    const bool dependent = static_cast<long long>(grid_a.x) * grid_a.y * grid_a.z >= nq::sm_count();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(nq::kDecWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, features ? nq::decide_kernel<true> : nq::decide_kernel<false>, draft, draft_logits,
                           tgt_logits, k, V, c, seeds, round, static_cast<const float2 *>(reinterpret_cast<float2 *>(w + L.part)),
                           static_cast<const float *>(segmax), static_cast<const float *>(reinterpret_cast<float *>(w + L.segsum)),
                           static_cast<const float *>(reinterpret_cast<float *>(w + L.partu)), rec, out_tok, out_cnt,
                           features, status, nsp / 2);
    if (e != cudaSuccess) return NQ_ERR_CUDA;
    cfg.gridDim = dim3(nsp / nq::kWarpsS, B);   // one warp per segment
    cfg.blockDim = dim3(nq::kThreadsS);
    cfg.dynamicSmemBytes = nq::kSmemS;
    e = cudaLaunchKernelEx(&cfg, nq::sample_b_kernel, draft, draft_logits, tgt_logits, k, V, c, al, out_tok, out_cnt,
                           reinterpret_cast<unsigned int *>(w + L.counters_b), static_cast<const nq::SampleRec *>(rec),
                           static_cast<const float *>(segmax), static_cast<const float *>(reinterpret_cast<float *>(w + L.segsum)),
                           reinterpret_cast<float *>(w + L.ssum), reinterpret_cast<float *>(w + L.lsum));
    return nq::cuda_status(e);
}
}  // namespace
}  // namespace nq


extern "C" nq_status spec_accept_sample(const int32_t *draft, const float *draft_logits, const float *tgt_logits,
                                        int B, int k, int V, float temperature, const uint64_t *seeds,
                                        uint64_t round, int32_t *out_tok, int32_t *out_cnt, void *ws,
                                        size_t ws_bytes, cudaStream_t stream)
{
    return nq::launch_sample(draft, draft_logits, tgt_logits, B, k, V, temperature, seeds, round, out_tok, out_cnt,
                             ws, ws_bytes, nullptr, stream);
}

extern "C" nq_status spec_accept_sample_features(const int32_t *draft, const float *draft_logits,
                                                 const float *tgt_logits, int B, int k, int V, float temperature,
                                                 const uint64_t *seeds, uint64_t round, int32_t *out_tok,
                                                 int32_t *out_cnt, float *features, void *ws, size_t ws_bytes,
                                                 cudaStream_t stream)
{
    if (!features) return NQ_ERR_ARG;
    if (!nq::aligned16(features)) return NQ_ERR_ALIGN;
    return nq::launch_sample(draft, draft_logits, tgt_logits, B, k, V, temperature, seeds, round, out_tok, out_cnt,
                             ws, ws_bytes, features, stream);
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
    nq::greedy_kernel<<<grid, nq::kThreads, 0, stream>>>(draft, tgt_logits, k, V, out_tok, k + 1, out_cnt,
                                                         reinterpret_cast<unsigned int *>(scratch),
                                                         reinterpret_cast<float2 *>(scratch + counters), status);
    return nq::cuda_status(cudaGetLastError());
}
