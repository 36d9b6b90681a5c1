// nq_linear.cu -- weight-streaming linears of quantized self-speculative
// decoding: the draft GEMV (base plane only) and the verify GEMM (both planes
// = the 8-bit target), plus the FP8 and FP16 verify tiers.
//
// BitNest, Fig. 2 / Fig. 3: drafting reads only the 4-bit base plane;
// verification reads both 4-bit planes and rebuilds the 8-bit target
// 16*q4 + r at step s/16.  SpecQuant Sec. III.A: Q8 (FP8) and Q16 (FP16)
// parents of the same base.
//
// Design (GB300, HBM-bound at M <= 16):
//  * One persistent launch streams every linear of a batch (e.g. a whole
//    model pass): each CTA takes a contiguous, cost-balanced range of 16-row
//    units, and each warp walks the flat (unit, group) sequence of its rows
//    with 128-bit non-allocating loads several quantisation groups ahead in a
//    register ring that continues across unit boundaries (no drain, no copies;
//    a step costs one compare for unit and segment bookkeeping).
//  * Dequantisation costs 5 integer ops per 8 weights: a nibble pair masked to
//    bits 0-3 (or 4-7) of each half and XOR-ed with 8 is, read as an fp16x2,
//    exactly (code + 8) * 2^-24 (or 16x that) -- fp16 subnormals.  The x16
//    pairs meet activations staged as x/16, the +8 offset is removed by
//    starting the group's accumulator at -8 * 2^-24 * sum(x), and the factor
//    2^24 is folded into the group scale.
//  * The contraction runs on the warp MMA (m16n8k16, fp16 in, fp32
//    accumulate) with the 16 weight rows as the A operand and the M <= 16
//    activation rows as one or two 8-column B tiles.  Each group uses two
//    short accumulator chains per plane; the scale is applied once per group.
//  * The K order inside every group is fixed, so an output element is
//    computed by the same operations whatever M is (batch invariance).
//  * Activations are staged in shared memory only when the problem (or the
//    staged K segment) changes, converted to fp16, permuted into operand
//    order and interleaved so that B-fragment loads are conflict-free.
#include <algorithm>
#include <atomic>

#include "nq_internal.cuh"

namespace nq {
// Tensor-memory path for M >= 16 (nq_tc.cu).
bool tc_route(int count, const nq_weights *w, int M, bool verify);
size_t tc_workspace_bytes(int count, const nq_weights *w, int M);
nq_status tc_run(int count, const nq_weights *w, const uint16_t *const *x, int M, float *const *y, bool verify,
                 void *ws, cudaStream_t stream);
}  // namespace nq

namespace nq {
namespace {

constexpr int kRowPad = 64;           // activation row stride = 64 (mod 128) bytes -> conflict-free B loads
constexpr int kMaxM = 16;             // activation rows per launch (two 8-column MMA tiles)
constexpr int kXsMax = 112 * 1024;    // dynamic shared memory cap per CTA (two CTAs fit one SM)
// Activation staging cap: whole activation rows up to K = 11008 at M <= 5
// with 16-warp units (one CTA per SM), segments beyond.  Shared memory is
// carved out of L1, so the cap trades restaging against L1: whole rows
// measured best on whole-model passes (LLaMA-2-7B verify at M = 5: 0.779 of
// the HBM roof at 112 KB against 0.736 at 56 KB, Qwen2.5-7B FP8 verify at
// M = 9: 0.770 against 0.745; the draft unchanged); with two 8-warp CTAs per
// SM anything above 40 KB was slower.
constexpr int kXsStageWide = 112 * 1024;  // 16-warp units (one CTA per SM)
constexpr int kXsStage = 40 * 1024;       // 8- and 4-warp units

enum Kind { kNib = 0, kFp8 = 1, kFp16 = 2 };

struct Prob {
    const uint8_t *base;
    const uint8_t *resid;
    const void *scales;
    const void *x;          // bf16 [M][k], or int8 codes [M][k] when the batch is a8
    const float *sx;        // a8: the activation rows' scales [M]
    float *y;
    long long cost_begin;   // sum over earlier problems of units * k (load balancing)
    int n, k, unit_begin, pad;
};

template <int MAXP>
struct Batch {
    long long total_cost;
    int count, total_units, M, xs_bytes;
    int a8, pad;            // a8: int8 activation codes (exact in fp16), y scaled by sx
    Prob p[MAXP];
};

constexpr int kSmallBatch = 4;
constexpr int kLargeBatch = 256;

__device__ __forceinline__ uint4 lds128(const unsigned char *p) { return *reinterpret_cast<const uint4 *>(p); }

template <int MAXP>
__device__ __forceinline__ int find_problem(const Batch<MAXP> &B, int u)
{
    int lo = 0, hi = B.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (B.p[mid].unit_begin <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// D = C + A * B with fp16 inputs and fp32 accumulators.
__device__ __forceinline__ void mma_f16_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// fp16x2 operand pairs of one 32-bit word of nibbles (elements k0..k7 of 8):
// lo1 = (k0, k4) and hi1 = (k2, k6) as (code + 8) * 2^-24;
// lo16 = (k1, k5) and hi16 = (k3, k7) as 16 (code + 8) * 2^-24.
struct NibPairs { uint32_t lo1, hi1, lo16, hi16; };

// One XOR turns the eight signed nibbles into offset binary (code + 8); each
// pair is then a single AND with one immediate.
__device__ __forceinline__ NibPairs nib_pairs(uint32_t w)
{
    const uint32_t u = w ^ 0x88888888u;
    const uint32_t u8 = u >> 8;
    NibPairs r;
    r.lo1 = u & 0x000F000Fu;
    r.lo16 = u & 0x00F000F0u;
    r.hi1 = u8 & 0x000F000Fu;
    r.hi16 = u8 & 0x00F000F0u;
    return r;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(lo))) |
           (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(hi))) << 16);
}

__device__ __forceinline__ float h_lo(uint32_t v) { return __half2float(__ushort_as_half(static_cast<unsigned short>(v))); }
__device__ __forceinline__ float h_hi(uint32_t v) { return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16))); }

// ------------------------------------------------------------------ streaming kernel

// Geometry of one chunk of K (the unit of the prefetch ring) per weight kind:
// nibbles use one quantisation group per chunk; E4M3 and fp16 rows give each
// lane 16 contiguous bytes per row per chunk.
template <int KIND, int G>
struct Geo {
    static constexpr int CH = KIND == kNib ? G : (KIND == kFp8 ? 64 : 32);   // inputs per chunk
    static constexpr int VB = KIND == kNib ? G / 8 : 16;                     // bytes per lane per row per plane
    static constexpr int WORDS = VB / 4;
    static constexpr int IPL = CH / 4;                                       // inputs per lane per chunk
    static constexpr int CHB = 2 * CH;                                       // staged fp16 bytes per chunk per row
    static constexpr int PIECES = CHB / 64;                                  // 16-byte activation pieces per lane
    __host__ __device__ static constexpr size_t row_bytes(int k)
    {
        return KIND == kNib ? static_cast<size_t>(k) / 2 : (KIND == kFp8 ? static_cast<size_t>(k) : 2 * static_cast<size_t>(k));
    }
};

template <int KIND, int PLANES, int G>
struct Slot {
    uint32_t w[PLANES][2][Geo<KIND, G>::WORDS];   // [plane][row g / g+8][word]
    unsigned short s[2];                           // nibbles: fp16 group scales of rows g, g+8
};

// First unit whose cost-prefix is >= target (units of one problem cost K each).
template <int MAXP>
__device__ __forceinline__ int unit_at_cost(const Batch<MAXP> &B, long long target)
{
    if (target >= B.total_cost) return B.total_units;
    int lo = 0, hi = B.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (B.p[mid].cost_begin <= target) lo = mid; else hi = mid - 1;
    }
    const Prob &P = B.p[lo];
    const long long off = target - P.cost_begin;
    return P.unit_begin + static_cast<int>((off + P.k - 1) / P.k);
}

template <int MAXP>
__device__ __forceinline__ int units_of(const Batch<MAXP> &B, int pi)
{
    return (pi + 1 < B.count ? B.p[pi + 1].unit_begin : B.total_units) - B.p[pi].unit_begin;
}

// Each CTA streams a contiguous, cost-balanced range of row units; every warp
// walks the flat (unit, chunk) sequence of its 16 rows with a prefetch ring
// that continues across unit boundaries.  Activations are restaged only when
// the problem (or the staged K segment) changes.
template <int KIND, int PLANES, int G, int NT, int WARPS, int MAXP>
__global__ void __launch_bounds__(WARPS * 32)
stream_kernel(const __grid_constant__ Batch<MAXP> B, unsigned int *status)
{
    using Gm = Geo<KIND, G>;
    constexpr int THREADS = WARPS * 32;
    constexpr int CH = Gm::CH, VB = Gm::VB, WORDS = Gm::WORDS, CHB = Gm::CHB, IPL = Gm::IPL;
    constexpr int MT = 8 * NT;
    constexpr int CORR = KIND == kNib ? MT * 4 : 0;   // offset-correction bytes per chunk
    constexpr int LANE_BYTES = 2 * PLANES * VB;
    // ring slots (R - 1 chunks in flight), measured per kind on whole-model
    // passes: nibbles 3 (both planes) / 5 (one plane, 128-input groups); E4M3
    // and fp16 rows 7 with one 8-column tile and 6 with two (4% faster than 5
    // for E4M3 at M = 3..7).  Nibbles with two tiles (M = 9..16) keep one slot
    // less, so that 16-warp units fit 128 registers a thread.
    constexpr int R = KIND == kNib ? (LANE_BYTES >= 64 ? (NT == 2 ? 2 : 3) : (LANE_BYTES >= 32 ? (NT == 2 ? 4 : 5) : 8))
                                   : (NT == 1 ? 7 : 6);
    constexpr int ROWS = 16 * WARPS;
    constexpr float kNeg8Ulp = -4.76837158203125e-07f;   // -8 * 2^-24

    extern __shared__ __align__(16) unsigned char smem[];
    const int M = B.M;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;

    const int ub = unit_at_cost(B, B.total_cost * blockIdx.x / gridDim.x);
    const int ue = unit_at_cost(B, B.total_cost * (blockIdx.x + 1) / gridDim.x);
    if (ub >= ue) return;

    // total steps (chunks) of this CTA's range
    const int first_pi = find_problem(B, ub);
    long long steps_ll = 0;
    for (int pi = first_pi; pi < B.count && B.p[pi].unit_begin < ue; ++pi) {
        const int a = max(ub, B.p[pi].unit_begin), b = min(ue, B.p[pi].unit_begin + units_of(B, pi));
        steps_ll += static_cast<long long>(b - a) * (B.p[pi].k / CH);
    }
    const int steps = static_cast<int>(steps_ll);

    // ---- load cursor (runs R-1 steps ahead of the compute cursor)
    int l_u = ub, l_pi = first_pi, l_c = 0, l_ng = 0;
    const uint8_t *lw[PLANES][2];
    const unsigned short *ls[2] = {nullptr, nullptr};
    auto l_setup = [&]() {
        const Prob &P = B.p[l_pi];
        const int N = P.n;
        l_ng = P.k / CH;
        const size_t rowb = Gm::row_bytes(P.k);
        const int rg = (l_u - P.unit_begin) * ROWS + warp * 16 + g;
        const int r0 = rg < N ? rg : 0, r1 = rg + 8 < N ? rg + 8 : 0;
        lw[0][0] = P.base + static_cast<size_t>(r0) * rowb + VB * t;
        lw[0][1] = P.base + static_cast<size_t>(r1) * rowb + VB * t;
        if constexpr (PLANES == 2) {
            lw[1][0] = P.resid + static_cast<size_t>(r0) * rowb + VB * t;
            lw[1][1] = P.resid + static_cast<size_t>(r1) * rowb + VB * t;
        }
        if constexpr (KIND == kNib) {
            ls[0] = static_cast<const unsigned short *>(P.scales) + static_cast<size_t>(r0) * l_ng;
            ls[1] = static_cast<const unsigned short *>(P.scales) + static_cast<size_t>(r1) * l_ng;
        }
    };
    auto issue = [&](Slot<KIND, PLANES, G> &S) {
        const size_t off = static_cast<size_t>(l_c) * (4 * VB);
#pragma unroll
        for (int p = 0; p < PLANES; ++p)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if constexpr (VB == 16) {
                    const uint4 v = ld_stream_v4(lw[p][r] + off);
                    S.w[p][r][0] = v.x; S.w[p][r][1] = v.y; S.w[p][r][2] = v.z; S.w[p][r][3] = v.w;
                } else {
                    const uint2 v = ld_stream_v2(lw[p][r] + off);
                    S.w[p][r][0] = v.x; S.w[p][r][1] = v.y;
                }
            }
        if constexpr (KIND == kNib) {
            S.s[0] = ld_nc_u16(ls[0] + l_c);
            S.s[1] = ld_nc_u16(ls[1] + l_c);
        }
        if (++l_c == l_ng) {
            l_c = 0;
            if (++l_u < ue) {
                if (l_pi + 1 < B.count && l_u >= B.p[l_pi + 1].unit_begin) ++l_pi;
                l_setup();
            }
        }
    };

    // ---- compute cursor: the next chunk to compute is (c_u, c_grp); an
    // "event" (unit end / unit start / new activation segment) happens when
    // c_grp reaches seg_end, so a step costs one compare.
    int c_u = ub, c_pi = first_pi, c_grp = 0, seg_end = 0;
    int c_N = 0, c_ng = 0, c_K = 0, c_rg = 0;
    bool in_unit = false;
    int staged_pi = -1, staged_begin = -1, cps = 1, RS = 0;
    const void *c_x = nullptr;
    const float *c_sx = nullptr;
    float *c_y = nullptr;
    const float *c_rs = nullptr;   // FP8 row scales
    unsigned char *xs = smem;
    float *corr = reinterpret_cast<float *>(smem);

    // Stage activations of chunks [c_begin, c_begin + nch) of the compute
    // cursor's problem in fp16.  Nibbles: operand order (x0,x4)(x2,x6)
    // (x1/16,x5/16)(x3/16,x7/16) per 8 inputs plus the offset correction
    // -8 * 2^-24 * sum(x) per (chunk, row); E4M3 / fp16: natural order.
    auto stage = [&](int c_begin, int nch) {
        const int items_row = nch * (CH / 8);
        const int total = M * items_row;
        const int total_pad = (total + THREADS - 1) / THREADS * THREADS;
        bool range = false;
        for (int i = threadIdx.x; i < total_pad; i += THREADS) {
            const bool valid = i < total;
            const int m = valid ? i / items_row : 0, it = valid ? i % items_row : 0;
            const size_t xoff = static_cast<size_t>(m) * c_K + static_cast<size_t>(c_begin) * CH + it * 8;
            float x0, x1, x2, x3, x4, x5, x6, x7;
            if (B.a8) {
                // eight int8 codes (|code| <= 127: exact in fp16, and so is code / 16)
                uint2 v = make_uint2(0u, 0u);
                if (valid) v = *reinterpret_cast<const uint2 *>(static_cast<const int8_t *>(c_x) + xoff);
                x0 = static_cast<float>(static_cast<int8_t>(v.x)); x1 = static_cast<float>(static_cast<int8_t>(v.x >> 8));
                x2 = static_cast<float>(static_cast<int8_t>(v.x >> 16)); x3 = static_cast<float>(static_cast<int8_t>(v.x >> 24));
                x4 = static_cast<float>(static_cast<int8_t>(v.y)); x5 = static_cast<float>(static_cast<int8_t>(v.y >> 8));
                x6 = static_cast<float>(static_cast<int8_t>(v.y >> 16)); x7 = static_cast<float>(static_cast<int8_t>(v.y >> 24));
            } else {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (valid) v = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(c_x) + xoff);
                x0 = __uint_as_float(v.x << 16); x1 = __uint_as_float(v.x & 0xFFFF0000u);
                x2 = __uint_as_float(v.y << 16); x3 = __uint_as_float(v.y & 0xFFFF0000u);
                x4 = __uint_as_float(v.z << 16); x5 = __uint_as_float(v.z & 0xFFFF0000u);
                x6 = __uint_as_float(v.w << 16); x7 = __uint_as_float(v.w & 0xFFFF0000u);
            }
            const float amax = fmaxf(fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3))),
                                     fmaxf(fmaxf(fabsf(x4), fabsf(x5)), fmaxf(fabsf(x6), fabsf(x7))));
            range |= amax > 65504.0f;
            const int cl = it / (CH / 8), kk = (it % (CH / 8)) * 8;
            if constexpr (KIND == kNib) {
                uint4 o;
                o.x = pack_h2(x0, x4);
                o.y = pack_h2(x2, x6);
                o.z = pack_h2(__fmul_rn(x1, 0.0625f), __fmul_rn(x5, 0.0625f));
                o.w = pack_h2(__fmul_rn(x3, 0.0625f), __fmul_rn(x7, 0.0625f));
                const int tl = kk / IPL, wd = (kk % IPL) / 8;
                if (valid) *reinterpret_cast<uint4 *>(xs + m * RS + cl * CHB + (4 * wd + tl) * 16) = o;
                // sum of the staged values as the MMA sees them: x~ at even k, 16 * (x/16)~ at odd k
                const float se = __fadd_rn(__fadd_rn(h_lo(o.x), h_hi(o.x)), __fadd_rn(h_lo(o.y), h_hi(o.y)));
                const float so = __fadd_rn(__fadd_rn(h_lo(o.z), h_hi(o.z)), __fadd_rn(h_lo(o.w), h_hi(o.w)));
                float sum = __fmaf_rn(16.0f, so, se);
#pragma unroll
                for (int o2 = 1; o2 < CH / 8; o2 <<= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, o2));
                if (valid && kk == 0) corr[cl * MT + m] = __fmul_rn(kNeg8Ulp, sum);
            } else {
                const uint4 o = make_uint4(pack_h2(x0, x1), pack_h2(x2, x3), pack_h2(x4, x5), pack_h2(x6, x7));
                // lane kk / IPL reads its IPL inputs as PIECES 16-byte pieces, interleaved across lanes
                const int tl = kk / IPL, pc = (kk % IPL) / 8;
                if (valid) *reinterpret_cast<uint4 *>(xs + m * RS + cl * CHB + (4 * pc + tl) * 16) = o;
            }
        }
        if constexpr (KIND == kNib)
            for (int i = threadIdx.x; i < nch * (MT - M); i += THREADS)
                corr[(i / (MT - M)) * MT + M + i % (MT - M)] = 0.0f;
        if (range) set_status(status, NQ_DEV_ACT_RANGE);
    };

    const unsigned char *xrow[NT];   // row base of each 8-column tile in the staged segment
    int xstep[NT];
    const unsigned char *xp[NT];     // current chunk
    const float *cp = corr;          // current chunk's offset corrections (nibbles)
    float y[NT][4], y2[NT][4];

    auto store_unit = [&]() {
        float rs0 = 1.0f, rs1 = 1.0f;
        if constexpr (KIND == kFp8) {
            rs0 = c_rg < c_N ? c_rs[c_rg] : 0.0f;
            rs1 = c_rg + 8 < c_N ? c_rs[c_rg + 8] : 0.0f;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = nt * 8 + 2 * t + (e & 1);
                const int row = e < 2 ? c_rg : c_rg + 8;
                float val = y[nt][e];
                if constexpr (KIND != kNib) val = __fadd_rn(val, y2[nt][e]);
                if constexpr (KIND == kFp8) val = __fmul_rn(e < 2 ? rs0 : rs1, val);
                if (m < M && row < c_N) {
                    if (B.a8) val = __fmul_rn(c_sx[m], val);
                    c_y[static_cast<size_t>(m) * c_N + row] = val;
                }
            }
        }
    };

    auto event = [&]() {
        if (in_unit && c_grp == c_ng) {
            store_unit();
            in_unit = false;
            ++c_u;
            if (c_pi + 1 < B.count && c_u >= B.p[c_pi + 1].unit_begin) ++c_pi;
        }
        if (!in_unit) {
            const Prob &P = B.p[c_pi];
            c_N = P.n; c_K = P.k; c_ng = c_K / CH; c_x = P.x; c_sx = P.sx; c_y = P.y;
            c_rs = static_cast<const float *>(P.scales);
            c_rg = (c_u - P.unit_begin) * ROWS + warp * 16 + g;
            c_grp = 0;
            in_unit = true;
            if (staged_pi != c_pi) {
                cps = (B.xs_bytes - M * kRowPad) / (M * CHB + CORR);
                cps = cps >= c_ng ? c_ng : max(1, cps);
                RS = cps * CHB + kRowPad;
                corr = reinterpret_cast<float *>(smem + M * RS);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int m = nt * 8 + g;
                    xrow[nt] = xs + (m < M ? m : 0) * RS + t * 16;
                    xstep[nt] = m < M ? CHB : 0;
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) { y[nt][e] = 0.0f; y2[nt][e] = 0.0f; }
        }
        seg_end = min(c_ng, c_grp + cps);
        if (staged_pi != c_pi || staged_begin != c_grp) {
            __syncthreads();
            stage(c_grp, seg_end - c_grp);
            __syncthreads();
            staged_pi = c_pi;
            staged_begin = c_grp;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) xp[nt] = xrow[nt];
        cp = corr + 2 * t;
    };

    // E4M3 / fp16 chunk: lane t holds IPL consecutive inputs of rows g, g+8;
    // each 16-byte activation piece covers words 2 pc and 2 pc + 1
    auto fp_chunk = [&](const Slot<KIND, PLANES, G> &S, float (&acc)[NT][4]) {
#pragma unroll
        for (int pc = 0; pc < Gm::PIECES; ++pc) {
            uint4 bq[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) bq[nt] = lds128(xp[nt] + pc * 64);
            // this piece covers words 2 pc and 2 pc + 1 of each row (4 inputs per word)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t a0, a1, a2, a3;
                if constexpr (KIND == kFp8) {
                    e4m3x4_to_f16x2x2(S.w[0][0][2 * pc + h], a0, a2);
                    e4m3x4_to_f16x2x2(S.w[0][1][2 * pc + h], a1, a3);
                } else {
                    a0 = S.w[0][0][2 * h]; a2 = S.w[0][0][2 * h + 1];
                    a1 = S.w[0][1][2 * h]; a3 = S.w[0][1][2 * h + 1];
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_f16(acc[nt], a0, a1, a2, a3, h ? bq[nt].z : bq[nt].x, h ? bq[nt].w : bq[nt].y);
            }
        }
    };

    // one chunk of this warp's 16 rows; the E4M3 / fp16 kinds alternate two
    // accumulator sets (two independent chains, summed at the unit end) by the
    // chunk's index in its row range, so the summation order of a row never
    // depends on where its unit falls in a CTA's range (batch invariance)
    auto compute = [&](const Slot<KIND, PLANES, G> &S) {
        if (c_grp == seg_end) event();
        if constexpr (KIND == kNib) {
            float accA[NT][PLANES][4], accB[NT][PLANES][4];
#pragma unroll
            for (int wd = 0; wd < WORDS; ++wd) {
                uint4 bq[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) bq[nt] = lds128(xp[nt] + wd * 64);
#pragma unroll
                for (int p = 0; p < PLANES; ++p) {
                    const NibPairs a = nib_pairs(S.w[p][0][wd]), b = nib_pairs(S.w[p][1][wd]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (wd == 0) {
                            const float2 cc = *reinterpret_cast<const float2 *>(cp + nt * 8);
                            mma_f16_c(accA[nt][p], a.lo1, b.lo1, a.hi1, b.hi1, bq[nt].x, bq[nt].y, cc.x, cc.y, cc.x, cc.y);
                            mma_f16_c(accB[nt][p], a.lo16, b.lo16, a.hi16, b.hi16, bq[nt].z, bq[nt].w, 0.f, 0.f, 0.f, 0.f);
                        } else {
                            mma_f16(accA[nt][p], a.lo1, b.lo1, a.hi1, b.hi1, bq[nt].x, bq[nt].y);
                            mma_f16(accB[nt][p], a.lo16, b.lo16, a.hi16, b.hi16, bq[nt].z, bq[nt].w);
                        }
                    }
                }
            }
            // group scale x 2^24 (undoes the subnormal encoding); refinement plane at s/16
            const float s0f = __fmul_rn(__half2float(__ushort_as_half(S.s[0])), 16777216.0f);
            const float s1f = __fmul_rn(__half2float(__ushort_as_half(S.s[1])), 16777216.0f);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float sc = e < 2 ? s0f : s1f;
                    y[nt][e] = __fmaf_rn(sc, __fadd_rn(accA[nt][0][e], accB[nt][0][e]), y[nt][e]);
                    if constexpr (PLANES == 2)
                        y[nt][e] = __fmaf_rn(__fmul_rn(sc, 0.0625f), __fadd_rn(accA[nt][1][e], accB[nt][1][e]), y[nt][e]);
                }
            }
            cp += MT;
        } else {
            if (c_grp & 1) fp_chunk(S, y2); else fp_chunk(S, y);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) xp[nt] += xstep[nt];
        ++c_grp;
    };

    Slot<KIND, PLANES, G> ring[R];
    l_setup();
#pragma unroll
    for (int i = 0; i < R - 1; ++i)
        if (i < steps) issue(ring[i]);

    int s0 = 0;
    for (; s0 + 2 * R - 2 < steps; s0 += R) {     // every load of the block is in range
#pragma unroll
        for (int i = 0; i < R; ++i) {
            issue(ring[(i + R - 1) % R]);
            compute(ring[i]);
        }
    }
    for (; s0 < steps; s0 += R) {                  // tail
#pragma unroll
        for (int i = 0; i < R; ++i) {
            if (s0 + i < steps) {
                if (s0 + i + R - 1 < steps) issue(ring[(i + R - 1) % R]);
                compute(ring[i]);
            }
        }
    }
    if (in_unit) store_unit();
}

// ------------------------------------------------------------------ host side

template <typename F>
int occupancy_of(F kernel, int threads, int smem)
{
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, threads, smem) != cudaSuccess || o < 1) o = 1;
    return o;
}

// Units, shared memory and launch for one kernel instantiation.
// Resident CTAs per SM for a kernel at a given dynamic shared memory size,
// cached per 1 KiB bucket (the launch configuration is a pure function of it).
template <typename F>
int cached_occupancy(F kernel, int threads, int smem, std::atomic<int> (&cache)[kXsMax / 1024 + 1])
{
    const int bucket = (smem + 1023) / 1024;
    int o = cache[bucket].load(std::memory_order_relaxed);
    if (o == 0) {
        o = occupancy_of(kernel, threads, bucket * 1024);
        cache[bucket].store(o, std::memory_order_relaxed);
    }
    return o;
}

// Opt a kernel into the large dynamic shared memory size, once per process.
template <typename F>
cudaError_t allow_large_smem(F kernel, std::atomic<int> &done)
{
    if (done.load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kXsMax);
    if (e == cudaSuccess) done.store(1, std::memory_order_release);
    return e;
}

template <int KIND, int PLANES, int G, int NT, int WARPS, int MAXP>
cudaError_t launch_stream(Batch<MAXP> &b, cudaStream_t s, unsigned int *status)
{
    auto k = stream_kernel<KIND, PLANES, G, NT, WARPS, MAXP>;
    static std::atomic<int> attr{0};
    static std::atomic<int> occ[kXsMax / 1024 + 1];
    const cudaError_t e = allow_large_smem(k, attr);
    if (e != cudaSuccess) return e;
    const int grid = std::max(1, std::min(b.total_units, sm_count() * cached_occupancy(k, WARPS * 32, b.xs_bytes, occ)));
    k<<<grid, WARPS * 32, b.xs_bytes, s>>>(b, status);
    return cudaGetLastError();
}

// 16-warp (256-row) units: one CTA per SM at 128 registers, so each SM holds
// one staged copy of the activations instead of two (less shared memory, a
// larger L1; measured 3-13% faster on whole-model passes at M = 1..9).  The
// nibble kernels with two 8-column tiles need more than 128 registers and keep
// 8-warp units.
template <int KIND, int PLANES, int G, int NT, int MAXP>
cudaError_t dispatch_w(Batch<MAXP> &b, int warps, cudaStream_t s, unsigned int *st)
{
    if constexpr (MAXP == kSmallBatch) {
        return launch_stream<KIND, PLANES, G, NT, 4, MAXP>(b, s, st);
    } else {
        if (warps == 16) return launch_stream<KIND, PLANES, G, NT, 16, MAXP>(b, s, st);
        return warps == 8 ? launch_stream<KIND, PLANES, G, NT, 8, MAXP>(b, s, st)
                          : launch_stream<KIND, PLANES, G, NT, 4, MAXP>(b, s, st);
    }
}

template <int MAXP>
cudaError_t launch_kind(int kind, int planes, int group, int nt, int warps, Batch<MAXP> &b, cudaStream_t s,
                        unsigned int *st)
{
    if (kind == kNib) {
        if (planes == 1) {
            if (group == 128) return nt == 1 ? dispatch_w<kNib, 1, 128, 1>(b, warps, s, st) : dispatch_w<kNib, 1, 128, 2>(b, warps, s, st);
            return nt == 1 ? dispatch_w<kNib, 1, 64, 1>(b, warps, s, st) : dispatch_w<kNib, 1, 64, 2>(b, warps, s, st);
        }
        if (group == 128) return nt == 1 ? dispatch_w<kNib, 2, 128, 1>(b, warps, s, st) : dispatch_w<kNib, 2, 128, 2>(b, warps, s, st);
        return nt == 1 ? dispatch_w<kNib, 2, 64, 1>(b, warps, s, st) : dispatch_w<kNib, 2, 64, 2>(b, warps, s, st);
    }
    if (kind == kFp8) return nt == 1 ? dispatch_w<kFp8, 1, 0, 1>(b, warps, s, st) : dispatch_w<kFp8, 1, 0, 2>(b, warps, s, st);
    return nt == 1 ? dispatch_w<kFp16, 1, 0, 1>(b, warps, s, st) : dispatch_w<kFp16, 1, 0, 2>(b, warps, s, st);
}

// Validate one layer for the given pass; returns the kernel family.
nq_status check_layer(const nq_weights &w, bool verify, int &kind, int &planes)
{
    size_t bb, rb, sb;
    nq_status st = nq_packed_bytes(w.n_out, w.k_in, w.group, w.format, &bb, &rb, &sb);
    if (st != NQ_OK) return st;
    switch (w.format) {
    case NQ_FMT_NESTED44: kind = kNib; planes = verify ? 2 : 1; break;
    case NQ_FMT_INT4: if (verify) return NQ_ERR_ARG; kind = kNib; planes = 1; break;
    case NQ_FMT_FP8E4M3_ROW: if (!verify) return NQ_ERR_ARG; kind = kFp8; planes = 1; break;
    case NQ_FMT_FP16: if (!verify) return NQ_ERR_ARG; kind = kFp16; planes = 1; break;
    default: return NQ_ERR_ARG;
    }
    if (!w.base || (planes == 2 && !w.resid) || ((kind == kNib || kind == kFp8) && !w.scales)) return NQ_ERR_ARG;
    if (!aligned16(w.base) || (planes == 2 && !aligned16(w.resid)) || ((kind == kNib || kind == kFp8) && !aligned16(w.scales)))
        return NQ_ERR_ALIGN;
    if (w.n_out > (1 << 28)) return NQ_ERR_SHAPE;
    return NQ_OK;
}

// Dynamic shared memory for a launch: all activation rows of the widest layer
// (in fp16, padded rows, plus offset corrections), capped by the unit width.
int xs_bytes_for(int kind, int M, int kmax, int group, int warps)
{
    const int ch = kind == kNib ? group : (kind == kFp8 ? 64 : 32);
    const int chunks = kmax / ch;
    const int mt = M > 8 ? 16 : 8;
    const long long need = static_cast<long long>(M) * (chunks * 2 * ch + kRowPad) +
                           (kind == kNib ? static_cast<long long>(chunks) * mt * 4 : 0);
    return static_cast<int>(std::min<long long>(need, warps == 16 ? kXsStageWide : kXsStage));
}

template <int MAXP>
nq_status run_batch(int count, const nq_weights *w, const void *const *x, int M, float *const *y,
                    int kind, int planes, int group, cudaStream_t stream, const float *const *sx = nullptr)
{
    unsigned int *status = device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    Batch<MAXP> b{};
    for (int m0 = 0; m0 < M; m0 += kMaxM) {
        const int Mc = std::min(kMaxM, M - m0);
        for (int i0 = 0; i0 < count; i0 += MAXP) {
            const int cnt = std::min(MAXP, count - i0);
            int kmax = 0;
            long long rows16 = 0;
            for (int i = 0; i < cnt; ++i) {
                kmax = std::max(kmax, w[i0 + i].k_in);
                rows16 += (w[i0 + i].n_out + 15) / 16;
            }
            // the widest units (16, 8 or 4 warps of 16 rows) that still fill the GPU twice
            const int nt = Mc > 8 ? 2 : 1;
            int warps = 4;
            if (MAXP == kLargeBatch) {
                // (nibbles with two tiles used 8-warp units at 150 registers, one
                // CTA per SM, until their ring lost a slot and 16-warp units fit:
                // M = 16 draft 0.21 -> 0.42 and M = 9 0.29 -> 0.52 of the copy
                // bandwidth on the LLaMA-3-8B pass)
                if (rows16 / 16 >= 2LL * sm_count()) warps = 16;
                else if (rows16 / 8 >= 2LL * sm_count()) warps = 8;
            }
            const int rows_per_unit = 16 * warps;
            long long units = 0, cost = 0;
            for (int i = 0; i < cnt; ++i) {
                const nq_weights &L = w[i0 + i];
                Prob &p = b.p[i];
                p.base = static_cast<const uint8_t *>(L.base);
                p.resid = static_cast<const uint8_t *>(L.resid);
                p.scales = L.scales;
                // bf16 rows (2 bytes an input) or, with sx, int8 codes (1 byte)
                p.x = static_cast<const char *>(x[i0 + i]) + static_cast<size_t>(m0) * L.k_in * (sx ? 1 : 2);
                p.sx = sx ? sx[i0 + i] + m0 : nullptr;
                p.y = y[i0 + i] + static_cast<size_t>(m0) * L.n_out;
                p.n = L.n_out;
                p.k = L.k_in;
                p.unit_begin = static_cast<int>(units);
                p.cost_begin = cost;
                p.pad = 0;
                const long long nu = (L.n_out + rows_per_unit - 1) / rows_per_unit;
                units += nu;
                cost += nu * L.k_in;
            }
            if (units > 0x7fffffffLL) return NQ_ERR_SHAPE;
            b.total_cost = cost;
            b.count = cnt;
            b.total_units = static_cast<int>(units);
            b.M = Mc;
            b.a8 = sx ? 1 : 0;
            b.xs_bytes = xs_bytes_for(kind, Mc, kmax, group, warps);
            const cudaError_t e = launch_kind<MAXP>(kind, planes, group, nt, warps, b, stream, status);
            if (e != cudaSuccess) return NQ_ERR_CUDA;
        }
    }
    return NQ_OK;
}

nq_status linear_entry(int count, const nq_weights *w, const uint16_t *const *x, int M, float *const *y,
                       bool verify, cudaStream_t stream, bool with_ws = false, void *ws = nullptr,
                       size_t ws_bytes = 0)
{
    if (count < 1 || !w || !x || !y) return NQ_ERR_ARG;
    if (M < 1 || M > 4096) return NQ_ERR_ARG;
    int kind = -1, planes = 0, group = 0;
    for (int i = 0; i < count; ++i) {
        int k2, p2;
        nq_status st = check_layer(w[i], verify, k2, p2);
        if (st != NQ_OK) return st;
        const int g2 = k2 == kNib ? w[i].group : 0;
        if (i == 0) { kind = k2; planes = p2; group = g2; }
        else if (k2 != kind || p2 != planes || g2 != group) return NQ_ERR_ARG;   // one kernel family per call
        if (!x[i] || !y[i]) return NQ_ERR_ARG;
        if (!aligned16(x[i]) || !aligned16(y[i])) return NQ_ERR_ALIGN;
    }
    if (with_ws && tc_route(count, w, M, verify)) {
        if (!ws || ws_bytes < tc_workspace_bytes(count, w, M)) return NQ_ERR_WORKSPACE;
        if (!aligned16(ws)) return NQ_ERR_ALIGN;
        return tc_run(count, w, x, M, y, verify, ws, stream);
    }
    const void *const *xv = reinterpret_cast<const void *const *>(x);
    return count <= kSmallBatch ? run_batch<kSmallBatch>(count, w, xv, M, y, kind, planes, group, stream)
                                : run_batch<kLargeBatch>(count, w, xv, M, y, kind, planes, group, stream);
}

}  // namespace

// Int8-activation linears (nested planes: NESTED44 both planes or one, INT4
// base plane) on the streaming kernel: the codes are staged like bf16
// activations (exactly, as fp16), every per-group dot of codes is exact in the
// fp32 accumulators, y = s_x sum_g s_g dot_g.  Arguments checked by the caller.
nq_status linear_a8_entry(int count, const nq_weights *w, const int8_t *const *xq, const float *const *sx, int M,
                          bool verify, float *const *y, cudaStream_t stream)
{
    const int group = w[0].group;
    const void *const *xv = reinterpret_cast<const void *const *>(xq);
    return count <= kSmallBatch
               ? run_batch<kSmallBatch>(count, w, xv, M, y, kNib, verify ? 2 : 1, group, stream, sx)
               : run_batch<kLargeBatch>(count, w, xv, M, y, kNib, verify ? 2 : 1, group, stream, sx);
}

}  // namespace nq

extern "C" nq_status nq_draft_gemv(const nq_weights *w, const uint16_t *x, int M, float *y, cudaStream_t stream)
{
    if (!w) return NQ_ERR_ARG;
    return nq::linear_entry(1, w, &x, M, &y, false, stream);
}

extern "C" nq_status nq_verify_gemm(const nq_weights *w, const uint16_t *x, int M, float *y, cudaStream_t stream)
{
    if (!w) return NQ_ERR_ARG;
    return nq::linear_entry(1, w, &x, M, &y, true, stream);
}

extern "C" nq_status nq_draft_gemv_batch(int count, const nq_weights *w, const uint16_t *const *x, int M,
                                         float *const *y, cudaStream_t stream)
{
    return nq::linear_entry(count, w, x, M, y, false, stream);
}

extern "C" nq_status nq_verify_gemm_batch(int count, const nq_weights *w, const uint16_t *const *x, int M,
                                          float *const *y, cudaStream_t stream)
{
    return nq::linear_entry(count, w, x, M, y, true, stream);
}

extern "C" size_t nq_linear_workspace_bytes(int count, const nq_weights *w, int M, int verify)
{
    if (count < 1 || !w || M < 1 || M > 4096) return 0;
    for (int i = 0; i < count; ++i) {
        int k2, p2;
        if (nq::check_layer(w[i], verify != 0, k2, p2) != NQ_OK) return 0;
    }
    return nq::tc_route(count, w, M, verify != 0) ? nq::tc_workspace_bytes(count, w, M) : 0;
}

extern "C" nq_status nq_draft_gemv_batch_ws(int count, const nq_weights *w, const uint16_t *const *x, int M,
                                            float *const *y, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    return nq::linear_entry(count, w, x, M, y, false, stream, true, ws, ws_bytes);
}

extern "C" nq_status nq_verify_gemm_batch_ws(int count, const nq_weights *w, const uint16_t *const *x, int M,
                                             float *const *y, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    return nq::linear_entry(count, w, x, M, y, true, stream, true, ws, ws_bytes);
}
