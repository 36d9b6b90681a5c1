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
//  * Persistent CTAs walk a flat list of 64-row units over all linears of a
//    batch (one launch streams a whole model pass: no inter-kernel gaps).
//  * Each warp owns 16 output rows and streams them with 128-bit
//    non-allocating loads, prefetched D quantisation groups ahead in registers.
//  * Nibbles become bf16 with one LOP3 per pair (magic-number 128 + (nib^8)),
//    the contraction runs on the warp MMA (m16n8k16, fp32 accumulate) with the
//    weight rows as the 16-row A operand and the M <= 16 activation rows as
//    one or two 8-column B tiles.  The +136 bias of the codes is removed by
//    starting each group's accumulator at -136 * sum(x over the group).
//  * Per-group scales are applied once per group in fp32.  The K order of
//    every group is fixed, so each output element is computed by the same
//    operations whatever M is (batch invariance).
//  * Activations are staged once per unit in shared memory, permuted to the
//    operand order and interleaved so that B-fragment loads are conflict-free.
#include <algorithm>
#include <mutex>

#include "nq_internal.cuh"

namespace nq {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerUnit = 16 * kWarps;
constexpr int kXsBytes = 40 * 1024;   // dynamic shared memory: staged activations + bias terms
constexpr int kRowPad = 64;           // x row stride = 64 (mod 128) bytes -> conflict-free B loads
constexpr int kMaxM = 16;             // activation rows per launch (two 8-column MMA tiles)

enum Kind { kNib = 0, kFp8 = 1, kFp16 = 2 };

struct Prob {
    const uint8_t *base;
    const uint8_t *resid;
    const void *scales;
    const uint16_t *x;
    float *y;
    int n, k, unit_begin, pad;
};

template <int MAXP>
struct Batch {
    int count, total_units, M, pad;
    Prob p[MAXP];
};

constexpr int kSmallBatch = 4;
constexpr int kLargeBatch = 256;

template <int KIND, int G>
struct Geom {
    static constexpr int CH = G;                              // inputs per chunk (= quantisation group for nibbles)
    static constexpr int VB = KIND == kNib ? G / 8 : 16;      // bytes per lane per row per plane per chunk
    static constexpr int WORDS = VB / 4;
    static constexpr int CHB = CH * 2;                        // staged activation bytes per chunk per row
    static constexpr int ROWB_NUM = KIND == kNib ? 1 : (KIND == kFp8 ? 2 : 4);  // row bytes = k * ROWB_NUM / 2
};

template <int KIND, int PLANES, int G>
struct Slot {
    uint32_t w[PLANES][2][Geom<KIND, G>::WORDS];
    unsigned short s[2];
};

template <int KIND, int PLANES, int G>
__device__ __forceinline__ void load_slot(Slot<KIND, PLANES, G> &S, const uint8_t *const (&plane_g)[2],
                                          const uint8_t *const (&plane_g8)[2], int c,
                                          const unsigned short *sc_g, const unsigned short *sc_g8)
{
    using Gm = Geom<KIND, G>;
    const size_t off = static_cast<size_t>(c) * (4 * Gm::VB);
#pragma unroll
    for (int p = 0; p < PLANES; ++p) {
        if constexpr (Gm::VB == 16) {
            uint4 a = ld_stream_v4(plane_g[p] + off), b = ld_stream_v4(plane_g8[p] + off);
            S.w[p][0][0] = a.x; S.w[p][0][1] = a.y; S.w[p][0][2] = a.z; S.w[p][0][3] = a.w;
            S.w[p][1][0] = b.x; S.w[p][1][1] = b.y; S.w[p][1][2] = b.z; S.w[p][1][3] = b.w;
        } else {
            uint2 a = ld_stream_v2(plane_g[p] + off), b = ld_stream_v2(plane_g8[p] + off);
            S.w[p][0][0] = a.x; S.w[p][0][1] = a.y;
            S.w[p][1][0] = b.x; S.w[p][1][1] = b.y;
        }
    }
    if constexpr (KIND == kNib) {
        S.s[0] = ld_nc_u16(sc_g + c);
        S.s[1] = ld_nc_u16(sc_g8 + c);
    }
}

__device__ __forceinline__ uint4 lds128(const unsigned char *p) { return *reinterpret_cast<const uint4 *>(p); }

template <int KIND, int PLANES, int G, int NT, int MAXP>
__global__ void __launch_bounds__(kThreads)
linear_kernel(const __grid_constant__ Batch<MAXP> B)
{
    using Gm = Geom<KIND, G>;
    constexpr int CH = Gm::CH, VB = Gm::VB, WORDS = Gm::WORDS, CHB = Gm::CHB;
    constexpr int MT = 8 * NT;
    constexpr int LANE_BYTES = 2 * PLANES * VB;                   // per chunk
    constexpr int D = LANE_BYTES >= 128 ? 1 : 128 / LANE_BYTES;   // prefetch depth (chunks)
    constexpr int CORR = KIND == kNib ? MT * 4 : 0;               // bias-term bytes per chunk

    extern __shared__ __align__(16) unsigned char smem[];
    const int M = B.M;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;

    for (int u = blockIdx.x; u < B.total_units; u += gridDim.x) {
        int lo = 0, hi = B.count - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (B.p[mid].unit_begin <= u) lo = mid; else hi = mid - 1;
        }
        const Prob &P = B.p[lo];
        const int N = P.n, K = P.k, NCH = K / CH;
        const int rg = (u - P.unit_begin) * kRowsPerUnit + warp * 16 + g, rg8 = rg + 8;
        const bool vg = rg < N, vg8 = rg8 < N;
        const size_t rowb = static_cast<size_t>(K) * Gm::ROWB_NUM / 2;
        const uint8_t *pg[2], *pg8[2];
        pg[0] = P.base + static_cast<size_t>(vg ? rg : 0) * rowb + VB * t;
        pg8[0] = P.base + static_cast<size_t>(vg8 ? rg8 : 0) * rowb + VB * t;
        pg[1] = PLANES == 2 ? P.resid + static_cast<size_t>(vg ? rg : 0) * rowb + VB * t : pg[0];
        pg8[1] = PLANES == 2 ? P.resid + static_cast<size_t>(vg8 ? rg8 : 0) * rowb + VB * t : pg8[0];
        const unsigned short *scg = static_cast<const unsigned short *>(P.scales) + static_cast<size_t>(vg ? rg : 0) * NCH;
        const unsigned short *scg8 = static_cast<const unsigned short *>(P.scales) + static_cast<size_t>(vg8 ? rg8 : 0) * NCH;

        // chunks per staged segment of activations
        int cps = (kXsBytes - M * kRowPad) / (M * CHB + CORR);
        if (cps > NCH) cps = NCH;
        const int RS = cps * CHB + kRowPad;
        unsigned char *xs = smem;
        float *corr = reinterpret_cast<float *>(smem + M * RS);

        Slot<KIND, PLANES, G> ring[D];
#pragma unroll
        for (int i = 0; i < D; ++i)
            if (i < NCH) load_slot(ring[i], pg, pg8, i, scg, scg8);

        // stage activations of chunks [c_begin, c_begin + cps) into shared memory
        auto stage = [&](int c_begin) {
            const int nch = min(cps, NCH - c_begin);
            const int items_row = nch * (CH / 8);
            const int total = M * items_row;
            const int total_pad = (total + kThreads - 1) / kThreads * kThreads;
            for (int i = threadIdx.x; i < total_pad; i += kThreads) {
                const bool valid = i < total;
                const int m = valid ? i / items_row : 0, it = valid ? i % items_row : 0;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (valid)
                    v = *reinterpret_cast<const uint4 *>(P.x + static_cast<size_t>(m) * K +
                                                         static_cast<size_t>(c_begin) * CH + it * 8);
                const int cl = it / (CH / 8), kk = (it % (CH / 8)) * 8;
                if constexpr (KIND == kNib) {
                    // operand order within 8 inputs: 0,4,1,5,2,6,3,7 (matches nib_pair_bf16)
                    uint4 o;
                    o.x = __byte_perm(v.x, v.z, 0x5410);
                    o.y = __byte_perm(v.x, v.z, 0x7632);
                    o.z = __byte_perm(v.y, v.w, 0x5410);
                    o.w = __byte_perm(v.y, v.w, 0x7632);
                    const int tl = kk / (2 * VB), wd = (kk % (2 * VB)) / 8;
                    if (valid) *reinterpret_cast<uint4 *>(xs + m * RS + cl * CHB + (4 * wd + tl) * 16) = o;
                    const float x0 = __uint_as_float(v.x << 16), x1 = __uint_as_float(v.x & 0xFFFF0000u);
                    const float x2 = __uint_as_float(v.y << 16), x3 = __uint_as_float(v.y & 0xFFFF0000u);
                    const float x4 = __uint_as_float(v.z << 16), x5 = __uint_as_float(v.z & 0xFFFF0000u);
                    const float x6 = __uint_as_float(v.w << 16), x7 = __uint_as_float(v.w & 0xFFFF0000u);
                    float s = __fadd_rn(__fadd_rn(__fadd_rn(x0, x1), __fadd_rn(x2, x3)),
                                        __fadd_rn(__fadd_rn(x4, x5), __fadd_rn(x6, x7)));
#pragma unroll
                    for (int o2 = 1; o2 < CH / 8; o2 <<= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o2));
                    if (valid && kk == 0) corr[cl * MT + m] = __fmul_rn(-136.0f, s);
                } else {
                    // bf16 -> fp16 (round to nearest), natural order
                    uint32_t h[4];
                    const uint32_t src[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const __half lo16 = __float2half_rn(__uint_as_float(src[q] << 16));
                        const __half hi16 = __float2half_rn(__uint_as_float(src[q] & 0xFFFF0000u));
                        h[q] = static_cast<uint32_t>(__half_as_ushort(lo16)) |
                               (static_cast<uint32_t>(__half_as_ushort(hi16)) << 16);
                    }
                    int pos;
                    if constexpr (KIND == kFp8) pos = 4 * ((kk % 16) / 8) + kk / 16;   // lane kk/16, piece (kk%16)/8
                    else pos = kk / 8;
                    if (valid) *reinterpret_cast<uint4 *>(xs + m * RS + cl * CHB + pos * 16) = make_uint4(h[0], h[1], h[2], h[3]);
                }
            }
            if constexpr (KIND == kNib)
                for (int i = threadIdx.x; i < nch * (MT - M); i += kThreads)
                    corr[(i / (MT - M)) * MT + M + i % (MT - M)] = 0.0f;
        };

        __syncthreads();   // the previous unit is done with shared memory
        stage(0);
        __syncthreads();

        int mrow[NT];
        bool mvalid[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mrow[nt] = nt * 8 + g;
            mvalid[nt] = mrow[nt] < M;
        }

        float yacc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) yacc[nt][i] = 0.0f;

        int seg_begin = 0;
        for (int c0 = 0; c0 < NCH; c0 += D) {
#pragma unroll
            for (int i = 0; i < D; ++i) {
                const int c = c0 + i;
                if (c < NCH) {
                    if (c - seg_begin >= cps) {
                        seg_begin = c;
                        __syncthreads();
                        stage(seg_begin);
                        __syncthreads();
                    }
                    const Slot<KIND, PLANES, G> cur = ring[i];
                    if (c + D < NCH) load_slot(ring[i], pg, pg8, c + D, scg, scg8);
                    const int cl = c - seg_begin;
                    const unsigned char *xc[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) xc[nt] = xs + (mvalid[nt] ? mrow[nt] : 0) * RS + cl * CHB;

                    if constexpr (KIND == kNib) {
                        float acc[NT][PLANES][4];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const float2 cc = *reinterpret_cast<const float2 *>(corr + cl * MT + nt * 8 + 2 * t);
#pragma unroll
                            for (int p = 0; p < PLANES; ++p) {
                                acc[nt][p][0] = cc.x; acc[nt][p][1] = cc.y;
                                acc[nt][p][2] = cc.x; acc[nt][p][3] = cc.y;
                            }
                        }
#pragma unroll
                        for (int wd = 0; wd < WORDS; ++wd) {
                            uint4 bq[NT];
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                bq[nt] = mvalid[nt] ? lds128(xc[nt] + (4 * wd + t) * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
                            for (int p = 0; p < PLANES; ++p) {
                                const uint32_t Wg = cur.w[p][0][wd], W8 = cur.w[p][1][wd];
                                {
                                    const uint32_t a0 = nib_pair_bf16<0>(Wg), a2 = nib_pair_bf16<1>(Wg);
                                    const uint32_t a1 = nib_pair_bf16<0>(W8), a3 = nib_pair_bf16<1>(W8);
#pragma unroll
                                    for (int nt = 0; nt < NT; ++nt) mma_bf16(acc[nt][p], a0, a1, a2, a3, bq[nt].x, bq[nt].y);
                                }
                                {
                                    const uint32_t a0 = nib_pair_bf16<2>(Wg), a2 = nib_pair_bf16<3>(Wg);
                                    const uint32_t a1 = nib_pair_bf16<2>(W8), a3 = nib_pair_bf16<3>(W8);
#pragma unroll
                                    for (int nt = 0; nt < NT; ++nt) mma_bf16(acc[nt][p], a0, a1, a2, a3, bq[nt].z, bq[nt].w);
                                }
                            }
                        }
                        const float sg = __half2float(__ushort_as_half(cur.s[0]));
                        const float sg8 = __half2float(__ushort_as_half(cur.s[1]));
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            yacc[nt][0] = __fmaf_rn(sg, acc[nt][0][0], yacc[nt][0]);
                            yacc[nt][1] = __fmaf_rn(sg, acc[nt][0][1], yacc[nt][1]);
                            yacc[nt][2] = __fmaf_rn(sg8, acc[nt][0][2], yacc[nt][2]);
                            yacc[nt][3] = __fmaf_rn(sg8, acc[nt][0][3], yacc[nt][3]);
                            if constexpr (PLANES == 2) {
                                const float rg16 = __fmul_rn(sg, 0.0625f), rg816 = __fmul_rn(sg8, 0.0625f);
                                yacc[nt][0] = __fmaf_rn(rg16, acc[nt][1][0], yacc[nt][0]);
                                yacc[nt][1] = __fmaf_rn(rg16, acc[nt][1][1], yacc[nt][1]);
                                yacc[nt][2] = __fmaf_rn(rg816, acc[nt][1][2], yacc[nt][2]);
                                yacc[nt][3] = __fmaf_rn(rg816, acc[nt][1][3], yacc[nt][3]);
                            }
                        }
                    } else if constexpr (KIND == kFp8) {
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            uint4 bq[NT];
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                bq[nt] = mvalid[nt] ? lds128(xc[nt] + (4 * q + t) * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int s = 2 * q + h;
                                uint32_t a0, a2, a1, a3;
                                e4m3x4_to_f16x2x2(cur.w[0][0][s], a0, a2);
                                e4m3x4_to_f16x2x2(cur.w[0][1][s], a1, a3);
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
                                    mma_f16(yacc[nt], a0, a1, a2, a3, h ? bq[nt].z : bq[nt].x, h ? bq[nt].w : bq[nt].y);
                            }
                        }
                    } else {
                        uint4 bq[NT];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            bq[nt] = mvalid[nt] ? lds128(xc[nt] + t * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma_f16(yacc[nt], cur.w[0][0][0], cur.w[0][1][0], cur.w[0][0][1], cur.w[0][1][1], bq[nt].x, bq[nt].y);
                            mma_f16(yacc[nt], cur.w[0][0][2], cur.w[0][1][2], cur.w[0][0][3], cur.w[0][1][3], bq[nt].z, bq[nt].w);
                        }
                    }
                }
            }
        }

        float rs_g = 1.0f, rs_g8 = 1.0f;
        if constexpr (KIND == kFp8) {
            const float *rsc = static_cast<const float *>(P.scales);
            rs_g = vg ? rsc[rg] : 0.0f;
            rs_g8 = vg8 ? rsc[rg8] : 0.0f;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = nt * 8 + 2 * t + (i & 1);
                const bool top = i < 2;
                const int row = top ? rg : rg8;
                if (m < M && (top ? vg : vg8)) {
                    float v = yacc[nt][i];
                    if constexpr (KIND == kFp8) v = __fmul_rn(top ? rs_g : rs_g8, v);
                    P.y[static_cast<size_t>(m) * N + row] = v;
                }
            }
        }
    }
}

// ------------------------------------------------------------------ host side

template <int KIND, int PLANES, int G, int NT, int MAXP>
int occupancy()
{
    static std::once_flag once;
    static int occ = 1;
    std::call_once(once, [] {
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, linear_kernel<KIND, PLANES, G, NT, MAXP>, kThreads, kXsBytes) ==
                cudaSuccess && o > 0)
            occ = o;
    });
    return occ;
}

template <int KIND, int PLANES, int G, int NT, int MAXP>
cudaError_t launch_t(const Batch<MAXP> &b, cudaStream_t stream)
{
    const int grid = std::min(b.total_units, sm_count() * occupancy<KIND, PLANES, G, NT, MAXP>());
    linear_kernel<KIND, PLANES, G, NT, MAXP><<<grid, kThreads, kXsBytes, stream>>>(b);
    return cudaGetLastError();
}

template <int MAXP>
cudaError_t launch_kind(int kind, int planes, int group, int nt, const Batch<MAXP> &b, cudaStream_t s)
{
    if (kind == kNib) {
        if (planes == 1) {
            if (group == 128) return nt == 1 ? launch_t<kNib, 1, 128, 1>(b, s) : launch_t<kNib, 1, 128, 2>(b, s);
            return nt == 1 ? launch_t<kNib, 1, 64, 1>(b, s) : launch_t<kNib, 1, 64, 2>(b, s);
        }
        if (group == 128) return nt == 1 ? launch_t<kNib, 2, 128, 1>(b, s) : launch_t<kNib, 2, 128, 2>(b, s);
        return nt == 1 ? launch_t<kNib, 2, 64, 1>(b, s) : launch_t<kNib, 2, 64, 2>(b, s);
    }
    if (kind == kFp8) return nt == 1 ? launch_t<kFp8, 1, 64, 1>(b, s) : launch_t<kFp8, 1, 64, 2>(b, s);
    return nt == 1 ? launch_t<kFp16, 1, 32, 1>(b, s) : launch_t<kFp16, 1, 32, 2>(b, s);
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
    const long long units = (static_cast<long long>(w.n_out) + kRowsPerUnit - 1) / kRowsPerUnit;
    if (units > (1LL << 30)) return NQ_ERR_SHAPE;
    return NQ_OK;
}

template <int MAXP>
nq_status run_batch(int count, const nq_weights *w, const uint16_t *const *x, int M, float *const *y,
                    int kind, int planes, int group, cudaStream_t stream)
{
    Batch<MAXP> b{};
    for (int m0 = 0; m0 < M; m0 += kMaxM) {
        const int Mc = std::min(kMaxM, M - m0);
        for (int i0 = 0; i0 < count; i0 += MAXP) {
            const int cnt = std::min(MAXP, count - i0);
            long long units = 0;
            for (int i = 0; i < cnt; ++i) {
                const nq_weights &L = w[i0 + i];
                Prob &p = b.p[i];
                p.base = static_cast<const uint8_t *>(L.base);
                p.resid = static_cast<const uint8_t *>(L.resid);
                p.scales = L.scales;
                p.x = x[i0 + i] + static_cast<size_t>(m0) * L.k_in;
                p.y = y[i0 + i] + static_cast<size_t>(m0) * L.n_out;
                p.n = L.n_out;
                p.k = L.k_in;
                p.unit_begin = static_cast<int>(units);
                p.pad = 0;
                units += (L.n_out + kRowsPerUnit - 1) / kRowsPerUnit;
            }
            if (units > 0x7fffffffLL) return NQ_ERR_SHAPE;
            b.count = cnt;
            b.total_units = static_cast<int>(units);
            b.M = Mc;
            const cudaError_t e = launch_kind<MAXP>(kind, planes, group, Mc > 8 ? 2 : 1, b, stream);
            if (e != cudaSuccess) return NQ_ERR_CUDA;
        }
    }
    return NQ_OK;
}

nq_status linear_entry(int count, const nq_weights *w, const uint16_t *const *x, int M, float *const *y,
                       bool verify, cudaStream_t stream)
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
    return count <= kSmallBatch ? run_batch<kSmallBatch>(count, w, x, M, y, kind, planes, group, stream)
                                : run_batch<kLargeBatch>(count, w, x, M, y, kind, planes, group, stream);
}

}  // namespace
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
