// nq_a8.cu -- int8-activation linears over the nested planes ("W4A8 -> W8A8").
//
// BitNest, Table 1 (draft -> target "W4A8 -> W8A8") and Table 12: the draft
// multiplies the 4-bit base codes, the target the 8-bit codes, both against
// 8-bit activations.  Activations are quantised per row, s_x = fp32(absmax /
// 127), code = clamp(rint(x / s_x), -127, 127); per weight group the dot
// product of codes is an exact integer, scaled by the group scale (s for the
// base codes, s / 16 for the 8-bit codes) and by s_x.
//
// The linears run on the streaming weight kernel of nq_linear.cu (warp MMA,
// one weight stream): an int8 code and code / 16 are exact in fp16, the
// offset-binary weight codes enter as fp16 subnormals, and every per-group
// partial sum is an integer multiple of 2^-24 below 2^-4, so the group dots
// come out of the fp32 accumulators exactly; only the scaling rounds.  This
// file holds the activation quantiser and the entry point.

#include "nq_internal.cuh"

namespace nq {
namespace {

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
    return nq::linear_a8_entry(count, w, xq, sx, M, verify != 0, y, stream);
}
