// nq_internal.cuh -- device helpers and host plumbing shared by the libnq
// translation units.  Product code only (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/nq.h"

namespace nq {

// ---------------------------------------------------------------- host side
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the sticky status word of the current device (set up once
// per device with cudaGetSymbolAddress); nullptr if that failed.
unsigned int *device_status_ptr();

// Multiprocessor count of the current device (cached).
int sm_count();

inline nq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NQ_OK : NQ_ERR_CUDA; }

// Int8-activation linears on the streaming weight kernel (nq_linear.cu);
// arguments already checked.
nq_status linear_a8_entry(int count, const nq_weights *w, const int8_t *const *xq, const float *const *sx, int M,
                          bool verify, float *const *y, cudaStream_t stream);

// ---------------------------------------------------------------- device side
__device__ __forceinline__ void set_status(unsigned int *status, unsigned int bits)
{
    if (status) atomicOr(status, bits);
}

// Streamed 16/8/4-byte global loads that bypass L1 allocation (read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void *p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ unsigned short ld_nc_u16(const void *p)
{
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// D += A(16x16) * B(16x8), fp16 inputs, fp32 accumulators (warp MMA).
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four E4M3 codes (bytes 0..3 of w) -> two f16x2 (bytes 0,1 and 2,3), exact.
// Byte 2i goes to the low half of the result, byte 2i+1 to the high half.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; cvt.rn.f16x2.e4m3x2 %0, l; cvt.rn.f16x2.e4m3x2 %1, h; }"
        : "=r"(lo), "=r"(hi) : "r"(w));
}

// ---------------------------------------------------------------- nested quantiser
// BitNest Fig. 2 reading: with the group scale s = fp16(absmax / 7), base
// q4 = clamp(rint(w / s), -8, 7) and refinement r = clamp(rint(16 (w / s - q4)),
// -8, 7); s == 0 gives zeros.  IEEE fp32 with round to nearest throughout, so
// the codes are reproducible bit for bit (weights and KV rows alike).
__device__ __forceinline__ int nested_clamp(float v)
{
    int i = static_cast<int>(v);
    return i < -8 ? -8 : (i > 7 ? 7 : i);
}
__device__ __forceinline__ void nested_quantise(float w, float s, int &q4, int &r)
{
    if (s == 0.0f) { q4 = 0; r = 0; return; }
    float x = __fdiv_rn(w, s);
    q4 = nested_clamp(rintf(x));
    float err = __fmul_rn(__fsub_rn(x, static_cast<float>(q4)), 16.0f);
    r = nested_clamp(rintf(err));
}

// ---------------------------------------------------------------- canonical
// fp32 recipe of the sampled acceptance (see spec_accept_sample in nq.h):
// base-2 exponential of t <= 0.5: 0 below -125, else P(f) 2^n with n =
// rint(t), f = t - n (exact) and P the degree-6 Taylor polynomial of 2^f,
// coefficients ln2^i / i! rounded to fp32, Horner with fused multiply-add.
// rint is taken by adding 1.5 * 2^23 (round to nearest even; the integer
// lands in the low mantissa bits of the sum) and 2^n is applied by adding n
// to the exponent field, so no conversion instructions are needed.
__device__ __forceinline__ float exp2_canon(float t)
{
    const float c0 = 1.0f, c1 = 0.693147180559945309417f, c2 = 0.240226506959100712333f,
                c3 = 0.0555041086648215799531f, c4 = 0.00961812910762847716197f,
                c5 = 0.00133335581464284434234f, c6 = 0.000154035303933816099545f;
    const float tc = fmaxf(t, -125.0f);
    const float big = __fadd_rn(tc, 12582912.0f);
    const float n = __fsub_rn(big, 12582912.0f);
    const float f = __fsub_rn(tc, n);
    float p = __fmaf_rn(c6, f, c5);
    p = __fmaf_rn(p, f, c4);
    p = __fmaf_rn(p, f, c3);
    p = __fmaf_rn(p, f, c2);
    p = __fmaf_rn(p, f, c1);
    p = __fmaf_rn(p, f, c0);
    const float r = __int_as_float(__float_as_int(p) + (__float_as_int(big) << 23));
    return t < -125.0f ? 0.0f : r;
}

// Two canonical exp2 evaluations at once with the packed fp32 instructions
// (add/sub/fma .rn.f32x2 perform two independent IEEE operations, so each
// lane rounds exactly as exp2_canon does).  The clamp at -125 is not needed:
// t < -125 returns 0 by the final select, and t >= -125 is unchanged.
__device__ __forceinline__ unsigned long long f2_pack(float a, float b)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long r)
{
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c)
{
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float2 exp2_canon_x2(unsigned long long t)
{
    const unsigned long long mag = f2_pack(12582912.0f, 12582912.0f);
    const unsigned long long big = f2_add(t, mag);
    const unsigned long long f = f2_sub(t, f2_sub(big, mag));
    unsigned long long p = f2_fma(f2_pack(0.000154035303933816099545f, 0.000154035303933816099545f), f,
                                  f2_pack(0.00133335581464284434234f, 0.00133335581464284434234f));
    p = f2_fma(p, f, f2_pack(0.00961812910762847716197f, 0.00961812910762847716197f));
    p = f2_fma(p, f, f2_pack(0.0555041086648215799531f, 0.0555041086648215799531f));
    p = f2_fma(p, f, f2_pack(0.240226506959100712333f, 0.240226506959100712333f));
    p = f2_fma(p, f, f2_pack(0.693147180559945309417f, 0.693147180559945309417f));
    p = f2_fma(p, f, f2_pack(1.0f, 1.0f));
    const float2 pv = f2_unpack(p), bv = f2_unpack(big), tv = f2_unpack(t);
    const float ra = __int_as_float(__float_as_int(pv.x) + (__float_as_int(bv.x) << 23));
    const float rb = __int_as_float(__float_as_int(pv.y) + (__float_as_int(bv.y) << 23));
    return make_float2(tv.x < -125.0f ? 0.0f : ra, tv.y < -125.0f ? 0.0f : rb);
}

// exp2_canon_x2 for exponents known to lie in [-125, 0.5] (no underflow
// select; same results as exp2_canon_x2 there).
__device__ __forceinline__ float2 exp2_canon_x2_inrange(unsigned long long t)
{
    const unsigned long long mag = f2_pack(12582912.0f, 12582912.0f);
    const unsigned long long big = f2_add(t, mag);
    const unsigned long long f = f2_sub(t, f2_sub(big, mag));
    unsigned long long p = f2_fma(f2_pack(0.000154035303933816099545f, 0.000154035303933816099545f), f,
                                  f2_pack(0.00133335581464284434234f, 0.00133335581464284434234f));
    p = f2_fma(p, f, f2_pack(0.00961812910762847716197f, 0.00961812910762847716197f));
    p = f2_fma(p, f, f2_pack(0.0555041086648215799531f, 0.0555041086648215799531f));
    p = f2_fma(p, f, f2_pack(0.240226506959100712333f, 0.240226506959100712333f));
    p = f2_fma(p, f, f2_pack(0.693147180559945309417f, 0.693147180559945309417f));
    p = f2_fma(p, f, f2_pack(1.0f, 1.0f));
    const float2 pv = f2_unpack(p), bv = f2_unpack(big);
    return make_float2(__int_as_float(__float_as_int(pv.x) + (__float_as_int(bv.x) << 23)),
                       __int_as_float(__float_as_int(pv.y) + (__float_as_int(bv.y) << 23)));
}

struct MaxSum { float m, s; };

// Merge two (max, sum) nodes; the larger max survives, the other sum is
// rescaled by 2^(m_small - m_large) with one fma; ties keep `a` as the larger.
// Branch-free (lanes of a warp merging different pairs never diverge).  A
// (-inf, 0) pad is the identity: its rescale factor is exp2(-inf) = 0 and
// fma(0, 0, s) = s; two pads give a pad.
__device__ __forceinline__ MaxSum ms_merge(MaxSum a, MaxSum b)
{
    const bool a_big = a.m >= b.m || b.m != b.m;
    const float big_m = a_big ? a.m : b.m, small_m = a_big ? b.m : a.m;
    const float big_s = a_big ? a.s : b.s, small_s = a_big ? b.s : a.s;
    const float d = small_m == -INFINITY ? -INFINITY : __fsub_rn(small_m, big_m);
    return MaxSum{big_m, __fmaf_rn(small_s, exp2_canon(d), big_s)};
}

// Philox4x32-10 (Salmon et al., SC'11).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

// Uniform in [0,1) for (row seed, position, purpose, round): word 0's top 24 bits.
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint32_t j, uint32_t purpose, uint64_t round)
{
    uint4 o = philox4x32_10(make_uint4(j, purpose, static_cast<uint32_t>(round), static_cast<uint32_t>(round >> 32)),
                            make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)));
    return __fmul_rn(__uint2float_rn(o.x >> 8), 5.9604644775390625e-08f);
}

}  // namespace nq
