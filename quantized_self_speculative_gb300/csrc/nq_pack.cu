// nq_pack.cu -- offline weight preparation (not part of a decoding round).
//
// NESTED44 / INT4 (BitNest, Fig. 2 and Fig. 3): per (row, group of G inputs)
// s = fp16(absmax / 7); base q4 = clamp(rint(w/s), -8, 7); refinement
// r = clamp(rint(16 (w/s - q4)), -8, 7); two's-complement nibbles, element 2j
// in the low nibble of byte j.  FP8E4M3_ROW / FP16: SpecQuant Sec. III.A tiers.
// One warp quantises one (row, group); every intermediate is an IEEE fp32
// operation with round-to-nearest so the codes are reproducible bit for bit.
#include "nq_internal.cuh"

namespace nq {
namespace {

constexpr int kPackWarps = 8;

// Each lane owns E = G/32 consecutive weights of the group.
template <int G>
__global__ void __launch_bounds__(kPackWarps * 32)
pack_nested_kernel(const float *__restrict__ w, int n, int k, uint8_t *__restrict__ base,
                   uint8_t *__restrict__ resid, __half *__restrict__ scales)
{
    constexpr int E = G / 32;
    const int groups_per_row = k / G;
    const long long job = static_cast<long long>(blockIdx.x) * kPackWarps + (threadIdx.x >> 5);
    if (job >= static_cast<long long>(n) * groups_per_row) return;
    const int lane = threadIdx.x & 31;
    const int row = static_cast<int>(job / groups_per_row), grp = static_cast<int>(job % groups_per_row);
    const float *src = w + static_cast<size_t>(row) * k + static_cast<size_t>(grp) * G + lane * E;
    float v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = src[e];
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
    const size_t off = static_cast<size_t>(row) * (k / 2) + static_cast<size_t>(grp) * (G / 2) + lane * (E / 2);
    if (E == 4) {
        *reinterpret_cast<uint16_t *>(base + off) = static_cast<uint16_t>(bb);
        if (resid) *reinterpret_cast<uint16_t *>(resid + off) = static_cast<uint16_t>(rr);
    } else {
        base[off] = static_cast<uint8_t>(bb);
        if (resid) resid[off] = static_cast<uint8_t>(rr);
    }
    if (lane == 0) scales[static_cast<size_t>(row) * groups_per_row + grp] = sh;
}

constexpr int kRowThreads = 256;

// One CTA per row: absmax over the row, then per-weight E4M3 encoding.
__global__ void __launch_bounds__(kRowThreads)
pack_fp8_kernel(const float *__restrict__ w, int k, uint8_t *__restrict__ codes, float *__restrict__ row_scale)
{
    __shared__ float red[kRowThreads / 32];
    const float *src = w + static_cast<size_t>(blockIdx.x) * k;
    float amax = 0.0f;
    for (int i = threadIdx.x; i < k; i += kRowThreads) amax = fmaxf(amax, fabsf(src[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < kRowThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    const float s = __fdiv_rn(amax, 448.0f);
    if (threadIdx.x == 0) row_scale[blockIdx.x] = s;
    uint8_t *dst = codes + static_cast<size_t>(blockIdx.x) * k;
    for (int i = threadIdx.x; i < k; i += kRowThreads)
        dst[i] = s == 0.0f ? 0 : static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(src[i], s), __NV_SATFINITE, __NV_E4M3));
}

__global__ void pack_fp16_kernel(const float *__restrict__ w, size_t count, __half *__restrict__ out)
{
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        out[i] = __float2half_rn(w[i]);
}

}  // namespace
}  // namespace nq

extern "C" nq_status nq_packed_bytes(int n_out, int k_in, int group, int format,
                                     size_t *base_bytes, size_t *resid_bytes, size_t *scale_bytes)
{
    if (n_out < 1 || k_in < 64) return NQ_ERR_SHAPE;
    if (k_in % 64 != 0) return NQ_ERR_SHAPE;
    const size_t nk = static_cast<size_t>(n_out) * static_cast<size_t>(k_in);
    size_t b = 0, r = 0, s = 0;
    switch (format) {
    case NQ_FMT_NESTED44:
    case NQ_FMT_INT4:
        if (group != 64 && group != 128) return NQ_ERR_SHAPE;
        if (k_in % group != 0) return NQ_ERR_SHAPE;
        b = nk / 2;
        r = format == NQ_FMT_NESTED44 ? nk / 2 : 0;
        s = static_cast<size_t>(n_out) * (k_in / group) * sizeof(uint16_t);
        break;
    case NQ_FMT_FP8E4M3_ROW: b = nk; s = static_cast<size_t>(n_out) * sizeof(float); break;
    case NQ_FMT_FP16: b = nk * 2; break;
    default: return NQ_ERR_ARG;
    }
    if (base_bytes) *base_bytes = b;
    if (resid_bytes) *resid_bytes = r;
    if (scale_bytes) *scale_bytes = s;
    return NQ_OK;
}

extern "C" nq_status nq_pack_weights(const float *w, const nq_weights *out, cudaStream_t stream)
{
    if (!w || !out) return NQ_ERR_ARG;
    size_t bb, rb, sb;
    nq_status st = nq_packed_bytes(out->n_out, out->k_in, out->group, out->format, &bb, &rb, &sb);
    if (st != NQ_OK) return st;
    if (!out->base || (rb && !out->resid) || (sb && !out->scales)) return NQ_ERR_ARG;
    if (!nq::aligned16(w) || !nq::aligned16(out->base) || (rb && !nq::aligned16(out->resid)) ||
        (sb && !nq::aligned16(out->scales)))
        return NQ_ERR_ALIGN;
    const int n = out->n_out, k = out->k_in;
    switch (out->format) {
    case NQ_FMT_NESTED44:
    case NQ_FMT_INT4: {
        uint8_t *resid = out->format == NQ_FMT_NESTED44 ? static_cast<uint8_t *>(out->resid) : nullptr;
        const long long jobs = static_cast<long long>(n) * (k / out->group);
        const long long blocks = (jobs + nq::kPackWarps - 1) / nq::kPackWarps;
        if (blocks > 0x7fffffffLL) return NQ_ERR_SHAPE;
        if (out->group == 128)
            nq::pack_nested_kernel<128><<<static_cast<unsigned>(blocks), nq::kPackWarps * 32, 0, stream>>>(
                w, n, k, static_cast<uint8_t *>(out->base), resid, static_cast<__half *>(out->scales));
        else
            nq::pack_nested_kernel<64><<<static_cast<unsigned>(blocks), nq::kPackWarps * 32, 0, stream>>>(
                w, n, k, static_cast<uint8_t *>(out->base), resid, static_cast<__half *>(out->scales));
        break;
    }
    case NQ_FMT_FP8E4M3_ROW:
        nq::pack_fp8_kernel<<<n, nq::kRowThreads, 0, stream>>>(w, k, static_cast<uint8_t *>(out->base),
                                                             static_cast<float *>(out->scales));
        break;
    case NQ_FMT_FP16:
        nq::pack_fp16_kernel<<<nq::sm_count() * 8, 256, 0, stream>>>(w, static_cast<size_t>(n) * k,
                                                                    static_cast<__half *>(out->base));
        break;
    default: return NQ_ERR_ARG;
    }
    return nq::cuda_status(cudaGetLastError());
}
