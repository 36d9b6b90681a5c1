// nq_a8.cu -- int8-activation linears over the nested planes ("W4A8 -> W8A8").
//
// BitNest, Table 1 (draft -> target "W4A8 -> W8A8") and Table 12: the draft
// multiplies the 4-bit base codes, the target the 8-bit codes, both against
// 8-bit activations.  Activations are quantised per row, s_x = fp32(absmax /
// 127), code = clamp(rint(x / s_x), -127, 127); per weight group the dot
// product of codes is an exact integer, scaled by the group scale (s for the
// base codes, s / 16 for the 8-bit codes) and by s_x.
//
// The integer dots run on the CUDA cores (dp4a: four 8-bit products and an
// add per instruction): GB300's int8 tensor rate is far below its fp16 rate
// and at decode batch sizes the pass is bound by the weight stream anyway.
// The nibbles become offset-binary bytes (q4 + 8, or q8 + 136 = 16 (q4 + 8) +
// (r + 8), which needs no borrow), an unsigned-by-signed dp4a takes them
// against the activation codes, and the offset comes out once per 32 inputs:
// dot(q, x) = dot(q + off, x) - off sum(x).
//
// Work: one warp takes 4 rows of a linear (a unit) and streams their K in
// steps of 1024 inputs, lane l holding inputs 32 l .. 32 l + 31 of each step
// (one 16-byte load per plane and row), so the activation codes a lane loads
// serve four rows.  Units of all linears of a call form one flat list that
// persistent warps take in turn.
#include "nq_internal.cuh"

#include <algorithm>

namespace nq {
namespace {

constexpr int kA8Rows = 4;                  // rows per warp unit
constexpr int kA8Warps = 8;
constexpr int kA8MaxP = 256;                // linears per launch
constexpr int kA8MaxM = 8;                  // activation rows per launch

struct A8Prob {
    const uint8_t *base, *resid;
    const uint16_t *scales;
    const int8_t *xq;                       // [M][k]
    const float *sx;                        // [M]
    float *y;                               // [M][n]
    int n, k, unit_begin, pad;
};
struct A8Batch {
    int count, total_units, M, pad;
    A8Prob p[kA8MaxP];
};

__device__ __forceinline__ uint32_t dp4a_us(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The codes of one 32-bit word per plane (8 consecutive inputs) as two words
// of offset-binary bytes in input order: inputs 0..3 and 4..7.
template <int PLANES>
__device__ __forceinline__ void codes8(uint32_t b, uint32_t r, uint32_t &lo, uint32_t &hi)
{
    const uint32_t bx = b ^ 0x88888888u;
    uint32_t ev, od;                         // bytes of the even inputs (0, 2, 4, 6) and of the odd ones
    if constexpr (PLANES == 2) {
        const uint32_t rx = r ^ 0x88888888u;
        ev = ((bx << 4) & 0xF0F0F0F0u) | (rx & 0x0F0F0F0Fu);
        od = (bx & 0xF0F0F0F0u) | ((rx >> 4) & 0x0F0F0F0Fu);
    } else {
        (void)r;
        ev = bx & 0x0F0F0F0Fu;
        od = (bx >> 4) & 0x0F0F0F0Fu;
    }
    lo = __byte_perm(ev, od, 0x5140);        // inputs 0, 1, 2, 3
    hi = __byte_perm(ev, od, 0x7362);        // inputs 4, 5, 6, 7
}

template <int PLANES, int G, int MM>
__global__ void __launch_bounds__(kA8Warps * 32, 2)
a8_kernel(const __grid_constant__ A8Batch B)
{
    constexpr int kOff = PLANES == 2 ? 136 : 8;
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kA8Warps + (threadIdx.x >> 5), nw = gridDim.x * kA8Warps;
    const int M = B.M;
    for (int u = gw; u < B.total_units; u += nw) {
        int pi = 0;
        {
            int lo = 0, hi = B.count - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (B.p[mid].unit_begin <= u) lo = mid; else hi = mid - 1;
            }
            pi = lo;
        }
        const A8Prob &P = B.p[pi];
        const int r0 = (u - P.unit_begin) * kA8Rows;
        const int gpr = P.k / G;
        float acc[kA8Rows][MM];
#pragma unroll
        for (int i = 0; i < kA8Rows; ++i)
#pragma unroll
            for (int m = 0; m < MM; ++m) acc[i][m] = 0.0f;
        for (int k0 = 32 * lane; k0 < P.k; k0 += 1024) {
            // activation codes of inputs k0 .. k0 + 31 and their sums
            uint4 xw[MM][2];
            int xs[MM];
#pragma unroll
            for (int m = 0; m < MM; ++m) {
                if (m < M) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(P.xq + static_cast<size_t>(m) * P.k + k0);
                    xw[m][0] = __ldg(src);
                    xw[m][1] = __ldg(src + 1);
                } else {
                    xw[m][0] = make_uint4(0, 0, 0, 0);
                    xw[m][1] = make_uint4(0, 0, 0, 0);
                }
                int s = 0;
                s = dp4a_ss(0x01010101u, xw[m][0].x, s); s = dp4a_ss(0x01010101u, xw[m][0].y, s);
                s = dp4a_ss(0x01010101u, xw[m][0].z, s); s = dp4a_ss(0x01010101u, xw[m][0].w, s);
                s = dp4a_ss(0x01010101u, xw[m][1].x, s); s = dp4a_ss(0x01010101u, xw[m][1].y, s);
                s = dp4a_ss(0x01010101u, xw[m][1].z, s); s = dp4a_ss(0x01010101u, xw[m][1].w, s);
                xs[m] = s;
            }
#pragma unroll
            for (int i = 0; i < kA8Rows; ++i) {
                const int row = r0 + i;
                if (row >= P.n) break;
                const size_t off = static_cast<size_t>(row) * (P.k / 2) + k0 / 2;
                const uint4 bw = ld_stream_v4(P.base + off);
                const uint4 rw = PLANES == 2 ? ld_stream_v4(P.resid + off) : make_uint4(0, 0, 0, 0);
                const float sw = __half2float(__ushort_as_half(ld_nc_u16(P.scales + static_cast<size_t>(row) * gpr + k0 / G)));
                const float S = PLANES == 2 ? __fmul_rn(sw, 0.0625f) : sw;
                uint32_t c[8];
                codes8<PLANES>(bw.x, rw.x, c[0], c[1]);
                codes8<PLANES>(bw.y, rw.y, c[2], c[3]);
                codes8<PLANES>(bw.z, rw.z, c[4], c[5]);
                codes8<PLANES>(bw.w, rw.w, c[6], c[7]);
#pragma unroll
                for (int m = 0; m < MM; ++m) {
                    uint32_t d = 0;
                    d = dp4a_us(c[0], xw[m][0].x, d); d = dp4a_us(c[1], xw[m][0].y, d);
                    d = dp4a_us(c[2], xw[m][0].z, d); d = dp4a_us(c[3], xw[m][0].w, d);
                    d = dp4a_us(c[4], xw[m][1].x, d); d = dp4a_us(c[5], xw[m][1].y, d);
                    d = dp4a_us(c[6], xw[m][1].z, d); d = dp4a_us(c[7], xw[m][1].w, d);
                    const int dot = static_cast<int>(d) - kOff * xs[m];
                    acc[i][m] = fmaf(S, static_cast<float>(dot), acc[i][m]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kA8Rows; ++i)
#pragma unroll
            for (int m = 0; m < MM; ++m) {
                float v = acc[i][m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[i][m] = v;
            }
        if (lane < kA8Rows * MM) {
            const int i = lane / MM, m = lane % MM, row = r0 + i;
            float v = 0.0f;
#pragma unroll
            for (int ii = 0; ii < kA8Rows; ++ii)
#pragma unroll
                for (int mm = 0; mm < MM; ++mm)
                    if (ii == i && mm == m) v = acc[ii][mm];
            if (m < M && row < P.n) P.y[static_cast<size_t>(m) * P.n + row] = __fmul_rn(P.sx[m], v);
        }
    }
}

constexpr int kQThreads = 256;

// One CTA per activation row: absmax, then the codes.
__global__ void __launch_bounds__(kQThreads)
quant_act_kernel(const uint16_t *__restrict__ x, int K, int8_t *__restrict__ xq, float *__restrict__ sx,
                 unsigned int *status)
{
    __shared__ float red[kQThreads / 32];
    const uint16_t *src = x + static_cast<size_t>(blockIdx.x) * K;
    float amax = 0.0f;
    for (int i = threadIdx.x; i < K; i += kQThreads) amax = fmaxf(amax, fabsf(__uint_as_float(static_cast<uint32_t>(src[i]) << 16)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < kQThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    if (!(amax <= 3.0e38f)) {
        if (threadIdx.x == 0) set_status(status, NQ_DEV_NONFINITE);
        amax = 0.0f;
    }
    const float s = __fdiv_rn(amax, 127.0f);
    if (threadIdx.x == 0) sx[blockIdx.x] = s;
    int8_t *dst = xq + static_cast<size_t>(blockIdx.x) * K;
    for (int i = threadIdx.x; i < K; i += kQThreads) {
        int q = 0;
        if (s > 0.0f) {
            const float r = rintf(__fdiv_rn(__uint_as_float(static_cast<uint32_t>(src[i]) << 16), s));
            q = r < -127.0f ? -127 : (r > 127.0f ? 127 : static_cast<int>(r));
        }
        dst[i] = static_cast<int8_t>(q);
    }
}

template <int PLANES, int G>
cudaError_t launch_a8(const A8Batch &b, int mm, cudaStream_t s)
{
    const int grid = std::max(1, std::min((b.total_units + kA8Warps - 1) / kA8Warps, sm_count() * 8));
    switch (mm) {
    case 1: a8_kernel<PLANES, G, 1><<<grid, kA8Warps * 32, 0, s>>>(b); break;
    case 2: a8_kernel<PLANES, G, 2><<<grid, kA8Warps * 32, 0, s>>>(b); break;
    case 3: a8_kernel<PLANES, G, 3><<<grid, kA8Warps * 32, 0, s>>>(b); break;
    case 4: a8_kernel<PLANES, G, 4><<<grid, kA8Warps * 32, 0, s>>>(b); break;
    case 5: a8_kernel<PLANES, G, 5><<<grid, kA8Warps * 32, 0, s>>>(b); break;
    case 6: a8_kernel<PLANES, G, 6><<<grid, kA8Warps * 32, 0, s>>>(b); break;
    case 7: a8_kernel<PLANES, G, 7><<<grid, kA8Warps * 32, 0, s>>>(b); break;
    default: a8_kernel<PLANES, G, 8><<<grid, kA8Warps * 32, 0, s>>>(b); break;
    }
    return cudaGetLastError();
}

}  // namespace
}  // namespace nq

extern "C" nq_status nq_quantize_act_int8(const uint16_t *x, int M, int K, int8_t *xq, float *sx, cudaStream_t stream)
{
    if (!x || !xq || !sx || M < 1 || M > 65535 || K < 1) return NQ_ERR_ARG;
    if (!nq::aligned16(x) || !nq::aligned16(xq) || !nq::aligned16(sx)) return NQ_ERR_ALIGN;
    unsigned int *status = nq::device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    nq::quant_act_kernel<<<M, nq::kQThreads, 0, stream>>>(x, K, xq, sx, status);
    return nq::cuda_status(cudaGetLastError());
}

extern "C" nq_status nq_linear_a8_batch(int count, const nq_weights *w, const int8_t *const *xq,
                                        const float *const *sx, int M, int verify, float *const *y,
                                        cudaStream_t stream)
{
    if (count < 1 || !w || !xq || !sx || !y || M < 1 || M > 4096) return NQ_ERR_ARG;
    const int planes = verify ? 2 : 1;
    int group = 0;
    for (int i = 0; i < count; ++i) {
        const nq_weights &L = w[i];
        size_t bb, rb, sb;
        const nq_status st = nq_packed_bytes(L.n_out, L.k_in, L.group, L.format, &bb, &rb, &sb);
        if (st != NQ_OK) return st;
        if (!(L.format == NQ_FMT_NESTED44 || (L.format == NQ_FMT_INT4 && !verify))) return NQ_ERR_ARG;
        if (i == 0) group = L.group;
        else if (L.group != group) return NQ_ERR_ARG;
        if (!L.base || !L.scales || (verify && !L.resid) || !xq[i] || !sx[i] || !y[i]) return NQ_ERR_ARG;
        if (!nq::aligned16(L.base) || !nq::aligned16(L.scales) || (verify && !nq::aligned16(L.resid)) ||
            !nq::aligned16(xq[i]) || !nq::aligned16(y[i]) || (reinterpret_cast<uintptr_t>(sx[i]) & 3u))
            return NQ_ERR_ALIGN;
    }
    nq::A8Batch b{};
    for (int m0 = 0; m0 < M; m0 += nq::kA8MaxM) {
        const int Mc = std::min(nq::kA8MaxM, M - m0);
        const int mm = Mc;   // an exact instantiation for every M up to 8
        for (int i0 = 0; i0 < count; i0 += nq::kA8MaxP) {
            const int cnt = std::min(nq::kA8MaxP, count - i0);
            long long units = 0;
            for (int i = 0; i < cnt; ++i) {
                const nq_weights &L = w[i0 + i];
                nq::A8Prob &p = b.p[i];
                p.base = static_cast<const uint8_t *>(L.base);
                p.resid = static_cast<const uint8_t *>(L.resid);
                p.scales = static_cast<const uint16_t *>(L.scales);
                p.xq = xq[i0 + i] + static_cast<size_t>(m0) * L.k_in;
                p.sx = sx[i0 + i] + m0;
                p.y = y[i0 + i] + static_cast<size_t>(m0) * L.n_out;
                p.n = L.n_out;
                p.k = L.k_in;
                p.unit_begin = static_cast<int>(units);
                p.pad = 0;
                units += (L.n_out + nq::kA8Rows - 1) / nq::kA8Rows;
            }
            if (units > 0x7fffffffLL) return NQ_ERR_SHAPE;
            b.count = cnt;
            b.total_units = static_cast<int>(units);
            b.M = Mc;
            cudaError_t e;
            if (planes == 2) e = group == 128 ? nq::launch_a8<2, 128>(b, mm, stream) : nq::launch_a8<2, 64>(b, mm, stream);
            else e = group == 128 ? nq::launch_a8<1, 128>(b, mm, stream) : nq::launch_a8<1, 64>(b, mm, stream);
            if (e != cudaSuccess) return NQ_ERR_CUDA;
        }
    }
    return NQ_OK;
}
