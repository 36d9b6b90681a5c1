// nq_tc.cu -- nested-nibble linears at M >= 16 activation rows on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// The draft and verify linears of a batched speculative round (BitNest Fig. 2:
// drafting reads the base plane, verification rebuilds the 8-bit target from
// both planes; Fig. 3: two 4-bit planes of N/2 bytes each) become dense
// contractions once M reaches a few tens of rows: at M = 144 the verify pass
// does 288 FLOP per weight byte, beyond any warp-MMA path.  Here each CTA owns
// a tile of 128 weight rows and streams its K:
//
//   * warp 22 loads the packed nibble planes of the tile's next k-blocks
//     into shared-memory stages with TMA (one 128-row x 64-byte box per
//     plane, 64-byte swizzle), several k-blocks ahead;
//   * warps 0-15 (one thread per weight row = one tensor-memory lane; two
//     groups of eight take alternate k-blocks, two warps per row quarter
//     each taking half of the k-block) decode the
//     weights to fp16(q * s), exactly rounded, into a tensor-memory A stage
//     (64 columns per 128 inputs) with tcgen05.st;
//   * warp 20 copies the activations of the k-block (already fp16, in the
//     MMA's 128-byte-swizzled K-major layout, written once per call by
//     tc_stage_kernel into the caller's workspace) into a shared-memory B
//     stage with one bulk copy;
//   * warp 21 issues tcgen05.mma (M = 128, N = padded M, K = 16; A from tensor
//     memory, B from shared memory, fp32 accumulators in tensor memory) and
//     tcgen05.commit to release the stages;
//   * warps 16-19 read the finished accumulators (tcgen05.ld) and store y.
//
// Decoding: offset-binary codes land in fp16 subnormals (code * 2^-24) with
// integer masks only; one fma per pair, fma(code * 2^-24, s * 2^20, -8 s) with
// code = q8 + 128 (verify; the byte holds q8 + 136 and an exact subnormal
// subtract removes the 8) or 16 (q4 + 8) (draft), yields fp16(q8 * s / 16) or
// fp16(q4 * s) with one rounding.  Groups with s * 2^20 beyond the fp16 range (s > 0.0625) take an
// equivalent exact path (1024-biased fp16 integer, subtract, multiply) with
// the same result.  Stage hand-offs: a weight stage is read through the
// generic proxy and refilled by TMA through the async proxy, so the readers
// fence (fence.proxy.async) before releasing it; every tcgen05.commit is
// issued by the thread whose MMAs it must track.  Every wait on an mbarrier
// is bounded by a timer; on a timeout the CTA sets NQ_DEV_TIMEOUT, drains its
// copies and MMAs, frees its tensor memory (kept if the MMA drain itself gave
// up, since MMAs might still write it) and returns.
#include "nq_internal.cuh"

#include <cuda.h>           // CUtensorMap (types only; the encoder is fetched through the runtime)
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

namespace nq {
namespace {

constexpr int kTcMinM = 16;            // smallest M routed here
constexpr int kTcMaxN = 256;           // activation rows per launch (MMA N)
constexpr int kTcTile = 128;           // weight rows per tile (MMA M)
constexpr int kTcKB = 128;             // inputs per k-block at wide N (8 MMAs of K = 16)
constexpr int kTcKBWide = 256;         // inputs per k-block when the padded M is at most 64
constexpr int kTcMaxP = 64;            // linears per launch (two 128-byte tensor maps each)
constexpr int kTcThreads = 736;        // warps 0-15 decode, 16-19 epilogue, 20 B copy, 21 MMA, 22 weight loads
constexpr int kTmemCols = 512;
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s per wait

struct TcProb {
    const uint8_t *base;
    const uint8_t *resid;
    const uint16_t *scales;
    const uint16_t *x;     // bf16 [M][k] (rows of this M chunk)
    uint16_t *xs;          // staged fp16 activations in the workspace
    float *y;              // fp32 [M][n] (rows of this M chunk)
    int n, k, tile_begin, pad;
};

struct TcBatch {
    CUtensorMap maps[kTcMaxP][2];   // base / refinement plane: uint8 [n][k/2], box 64 B x 128 rows, 64-byte swizzle
    int count, total_tiles, M, Npad, group, sb, sa, nd, ws;
    TcProb p[kTcMaxP];
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// try_wait with a suspend-time hint: a waiting warp sleeps (up to 10 ms) until
// the phase completes instead of spinning and taking issue slots from the
// warps that do the work.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(bar), "r"(parity), "r"(10000000u) : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Wait for the phase of `bar` with the given parity.  Gives up after
// limit_ns (sets the CTA's abort flag and NQ_DEV_TIMEOUT) or when another
// role of the CTA has given up; returns false then.
__device__ __noinline__ bool mbar_wait_until(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             unsigned int *status, unsigned long long limit_ns)
{
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            set_status(status, NQ_DEV_TIMEOUT);
            return false;
        }
    }
}
__device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                               unsigned int *status)
{
    return mbar_wait_until(bar, parity, abort_flag, status, kWaitNs);
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned int *status)
{
    return mbar_test(bar, parity) || mbar_wait_slow(bar, parity, abort_flag, status);
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// One lane of a converged warp (the warp's loop state stays warp-uniform, so
// descriptors and addresses live in uniform registers for tcgen05 issue).
__device__ __forceinline__ bool elect_one()
{
    uint32_t e;
    asm volatile("{ .reg .b32 r; .reg .pred p; elect.sync r|p, 0xffffffff; selp.u32 %0, 1, 0, p; }" : "=r"(e));
    return e != 0;
}
// The same, also returning the elected lane's id (the same value on every lane).
__device__ __forceinline__ bool elect_one(uint32_t &leader)
{
    uint32_t e, l;
    asm volatile("{ .reg .pred p; elect.sync %1|p, 0xffffffff; selp.u32 %0, 1, 0, p; }" : "=r"(e), "=r"(l));
    leader = l;
    return e != 0;
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// D[128 x N] (+)= A[128 x 16] (tensor memory, fp16) * B[16 x N] (shared, fp16)
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                 "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
                 "r"(v[15]) : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                   "=r"(v[15])
                 : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row core
// groups 1024 bytes apart (stride byte offset), leading byte offset unused
// for this layout (encoded as 1), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulators, fp16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t f16_idesc(int m, int n)
{
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t dup_h(unsigned short h) { return static_cast<uint32_t>(h) * 0x10001u; }
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// Per-group decoding constants: fast = fma(code * 2^-24, F, C) with F = s 2^20,
// C = -8 s (both exact in fp16 when s <= 0x2BFF); slow = (1024 + code) - bias,
// times S (s/16 for the verify codes, s for the draft codes).  For a normal s
// the constants are exponent shifts of its bits (F: +20, C: +3 and negate,
// s/16: -4); s = 0 gives zeros; subnormal s (below 2^-14) goes through fp32.
struct GroupK {
    uint32_t F, C, S;
    bool fast;
};
template <int PLANES>
__device__ __forceinline__ GroupK group_consts(unsigned short s_bits)
{
    GroupK g;
    const uint32_t sb = s_bits & 0x7FFFu;
    g.fast = sb <= 0x2BFFu;
    if (sb >= 0x0400u || sb == 0u) {
        const uint32_t sign = s_bits & 0x8000u;
        const uint32_t f = sb ? (sb + (20u << 10)) | sign : 0u;
        const uint32_t c = sb ? ((sb + (3u << 10)) | 0x8000u) ^ sign : 0u;
        const uint32_t sv = (PLANES == 2 ? (sb >= (5u << 10) ? sb - (4u << 10) : 0u) : sb) | sign;
        g.F = f * 0x10001u;
        g.C = c * 0x10001u;
        g.S = sv * 0x10001u;
        if (PLANES == 2 && sb != 0 && sb < (5u << 10)) {   // s/16 subnormal (s < 2^-10): exact via fp32
            g.S = dup_h(__half_as_ushort(__float2half_rn(__fmul_rn(__half2float(__ushort_as_half(s_bits)), 0.0625f))));
        }
    } else {
        const float s = __half2float(__ushort_as_half(s_bits));
        g.F = dup_h(__half_as_ushort(__float2half_rn(__fmul_rn(s, 1048576.0f))));
        g.C = dup_h(__half_as_ushort(__float2half_rn(__fmul_rn(s, -8.0f))));
        g.S = dup_h(__half_as_ushort(__float2half_rn(PLANES == 2 ? __fmul_rn(s, 0.0625f) : s)));
    }
    return g;
}

// Decode one 32-bit word per plane (8 consecutive inputs) into 4 fp16x2
// registers in the MMA order (0,4)(1,5)(2,6)(3,7).  FAST: one fma per pair;
// otherwise the biased-integer path (any s).
template <int PLANES, bool FAST>
__device__ __forceinline__ void decode_word(uint32_t b, uint32_t r, const GroupK &g, uint32_t *o)
{
    uint32_t c[4];   // codes as fp16 subnormals: (q8 + 136) or 16 (q4 + 8), times 2^-24
    const uint32_t bx = b ^ 0x88888888u;
    if constexpr (PLANES == 2) {
        const uint32_t rx = r ^ 0x88888888u;
        // byte c of L: inputs 2c (base nibble high, refinement nibble low); H: inputs
        // 2c+1.  Each byte is 16 (q4 + 8) + (r + 8) = q8 + 136 in [0, 255]: q8 spans
        // [-136, 119], so no byte-wide offset of 128 exists and the remaining -8 is
        // taken per half below, where the sign fits.
        const uint32_t L = ((bx << 4) & 0xF0F0F0F0u) | (rx & 0x0F0F0F0Fu);
        const uint32_t H = (bx & 0xF0F0F0F0u) | ((rx >> 4) & 0x0F0F0F0Fu);
        c[0] = L & 0x00FF00FFu;
        c[1] = H & 0x00FF00FFu;
        c[2] = __byte_perm(L, 0u, 0x4341);   // bytes 1 and 3 of L into the low byte of each half
        c[3] = __byte_perm(H, 0u, 0x4341);
    } else {
        (void)r;
        c[0] = (bx << 4) & 0x00F000F0u;
        c[1] = bx & 0x00F000F0u;
        c[2] = (bx >> 4) & 0x00F000F0u;
        c[3] = (bx >> 8) & 0x00F000F0u;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // verify: (q8 + 136) 2^-24 - 8 2^-24 is exact on the subnormal grid (sign
        // included), leaving (q8 + 128) 2^-24 for the fma
        const uint32_t cf = PLANES == 2 ? hsub2_u(c[i], 0x00080008u) : c[i];
        if constexpr (FAST) {
            o[i] = hfma2_u(cf, g.F, g.C);
        } else {
            const uint32_t slow = PLANES == 2 ? hmul2_u(hsub2_u(c[i] | 0x64006400u, 0x64886488u), g.S)    // 1160
                                              : hmul2_u(hsub2_u((c[i] >> 4) | 0x64006400u, 0x64086408u), g.S);  // 1032
            o[i] = g.fast ? hfma2_u(cf, g.F, g.C) : slow;
        }
    }
}

__device__ __forceinline__ int tile_problem(const TcBatch &B, int tile)
{
    int lo = 0, hi = B.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (B.p[mid].tile_begin <= tile) lo = mid; else hi = mid - 1;
    }
    return lo;
}
// ---------------------------------------------------------------- activation pre-pass
// x (bf16, [M][k]) -> fp16 in the workspace, per k-block of 64 inputs a
// [Npad][128 B] block: row m, 16-byte chunk c (inputs 8c..8c+7 in the order
// 0,4,1,5,2,6,3,7) stored at chunk position c ^ (m & 7) -- the 128-byte
// swizzle the tensor cores apply to a 1024-byte aligned shared-memory tile.
// Rows M..Npad-1 are zero.
__global__ void __launch_bounds__(256) tc_stage_kernel(const __grid_constant__ TcBatch B, unsigned int *status)
{
    const TcProb &P = B.p[blockIdx.y];
    const int Npad = B.Npad, M = B.M, K = P.k;
    const long long total = static_cast<long long>(K / 8) * Npad;
    bool range = false;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i & 7);
        const long long am = i >> 3;
        const int m = static_cast<int>(am % Npad), a = static_cast<int>(am / Npad);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (m < M) v = *reinterpret_cast<const uint4 *>(P.x + static_cast<size_t>(m) * K + a * 64 + c * 8);
        const float x0 = __uint_as_float(v.x << 16), x1 = __uint_as_float(v.x & 0xFFFF0000u);
        const float x2 = __uint_as_float(v.y << 16), x3 = __uint_as_float(v.y & 0xFFFF0000u);
        const float x4 = __uint_as_float(v.z << 16), x5 = __uint_as_float(v.z & 0xFFFF0000u);
        const float x6 = __uint_as_float(v.w << 16), x7 = __uint_as_float(v.w & 0xFFFF0000u);
        const float amax = fmaxf(fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3))),
                                 fmaxf(fmaxf(fabsf(x4), fabsf(x5)), fmaxf(fabsf(x6), fabsf(x7))));
        range |= amax > 65504.0f;
        uint4 o;
        o.x = h2_bits(__floats2half2_rn(x0, x4));
        o.y = h2_bits(__floats2half2_rn(x1, x5));
        o.z = h2_bits(__floats2half2_rn(x2, x6));
        o.w = h2_bits(__floats2half2_rn(x3, x7));
        *reinterpret_cast<uint4 *>(P.xs + (static_cast<size_t>(a) * Npad + m) * 64 + ((c ^ (m & 7)) * 8)) = o;
    }
    if (range) set_status(status, NQ_DEV_ACT_RANGE);
}

// Slot and phase parity of a ring of n mbarrier-guarded stages, advanced
// incrementally (integer division by a runtime n is an emulated sequence).
struct Ring {
    int slot, phase, n;
    __device__ explicit Ring(int n_, int start = 0) : slot(start % n_), phase((start / n_) & 1), n(n_) {}
    __device__ void step(int by = 1)
    {
        slot += by;
        if (slot >= n) { slot -= n; phase ^= 1; }
    }
};

// ---------------------------------------------------------------- main kernel
// Tiles are dealt round-robin (CTA c takes tiles c, c + grid, ...), so the
// CTAs running at any moment work on neighbouring tiles of one or two linears
// and share their staged activations in L2.
template <int KB>
struct TileSeq {
    int tile, pi, kb, nkb;
    __device__ void init(const TcBatch &B)
    {
        tile = blockIdx.x;
        kb = 0;
        if (tile < B.total_tiles) { pi = tile_problem(B, tile); nkb = B.p[pi].k / KB; }
        else { pi = 0; nkb = 1; }
    }
    __device__ void next(const TcBatch &B)
    {
        if (++kb == nkb) {
            kb = 0;
            tile += gridDim.x;
            if (tile < B.total_tiles) { pi = tile_problem(B, tile); nkb = B.p[pi].k / KB; }
        }
    }
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// Weight stage: per plane 128 rows of KB/2 bytes as TMA writes them with the
// 64-byte (KB = 128) or 128-byte (KB = 256) swizzle of a 1024-byte aligned
// stage: the 16-byte piece p of row r sits at p ^ ((r >> 1) & 3) or p ^ (r & 7),
// so the 8 rows read by a quarter warp (same logical piece) fall in 8
// different bank groups.
template <int KB>
__host__ __device__ constexpr uint32_t wpos(int row, int piece)
{
    return KB == 128 ? static_cast<uint32_t>(row * 64 + ((piece ^ ((row >> 1) & 3)) << 4))
                     : static_cast<uint32_t>(row * 128 + ((piece ^ (row & 7)) << 4));
}

template <int PLANES, int G, int KB>
__global__ void __launch_bounds__(kTcThreads, 1) tc_kernel(const __grid_constant__ TcBatch B, unsigned int *status)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (sbase - raw);
    const int Npad = B.Npad, SB = B.sb, SA = B.sa, ND = B.nd, WS = B.ws;
    const uint32_t stage_bytes = 2u * KB * static_cast<uint32_t>(Npad);   // KB/64 swizzle atoms of Npad x 128 B
    constexpr uint32_t kPlaneBytes = kTcTile * (KB / 2);
    constexpr int kACols = KB / 2;                                         // tensor-memory columns per A stage
    constexpr uint32_t kWStage = PLANES * kPlaneBytes;          // 1024-byte multiple (TMA swizzle atoms)
    const uint32_t wbase = sbase + static_cast<uint32_t>(SB) * stage_bytes;
    // barriers: a_full[4] a_empty[4] b_full[8] b_empty[8] d_full[2] d_empty[2] done w_full[12] w_empty[12]
    // done_all
    const uint32_t bars = wbase + static_cast<uint32_t>(WS) * kWStage;
    auto A_FULL = [&](int i) { return bars + 8u * i; };
    auto A_EMPTY = [&](int i) { return bars + 8u * (4 + i); };
    auto B_FULL = [&](int i) { return bars + 8u * (8 + i); };
    auto B_EMPTY = [&](int i) { return bars + 8u * (16 + i); };
    auto D_FULL = [&](int i) { return bars + 8u * (24 + i); };
    auto D_EMPTY = [&](int i) { return bars + 8u * (26 + i); };
    // 32 arrivals: the MMA warp's final commits (lanes that issued MMAs) and
    // plain arrivals (lanes that issued none)
    const uint32_t DONE_ALL = bars + 8u * 53;
    auto W_FULL = [&](int i) { return bars + 8u * (29 + i); };
    auto W_EMPTY = [&](int i) { return bars + 8u * (41 + i); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + (bars - sbase) + 8 * 56);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *keep_tmem = reinterpret_cast<volatile int *>(tmem_slot + 2);   // set if the MMA drain gave up

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) { mbar_init(A_FULL(i), 8); mbar_init(A_EMPTY(i), 1); }
        for (int i = 0; i < 8; ++i) { mbar_init(B_FULL(i), 1); mbar_init(B_EMPTY(i), 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(D_FULL(i), 1); mbar_init(D_EMPTY(i), 4); }
        mbar_init(DONE_ALL, 32);
        for (int i = 0; i < 12; ++i) { mbar_init(W_FULL(i), 1); mbar_init(W_EMPTY(i), 8); }
        *abort_flag = 0;
        *keep_tmem = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 20) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    int steps = 0;
    for (int t = blockIdx.x; t < B.total_tiles; t += gridDim.x) steps += B.p[tile_problem(B, t)].k / KB;
    const uint32_t dcol0 = static_cast<uint32_t>(SA) * kACols;

    if (warp == 22 && steps > 0) {
        // ------------------------------------------------ weight loader: one elected lane issues
        // the TMA boxes of each k-block into the next free stage
        if (elect_one()) {
            TileSeq<KB> q;
            q.init(B);
            int last_phase[12];
            for (int i = 0; i < 12; ++i) last_phase[i] = -1;
            Ring w(WS);
            for (int it = 0; it < steps; ++it, w.step()) {
                const int st = w.slot;
                if (!mbar_wait(W_EMPTY(st), w.phase ^ 1, abort_flag, status)) break;
                const TcProb &P = B.p[q.pi];
                const int r0 = (q.tile - P.tile_begin) * kTcTile;
                const uint32_t dst = wbase + static_cast<uint32_t>(st) * kWStage;
                // one arrival with the byte count; rows beyond n are zero-filled by TMA
                mbar_expect_tx(W_FULL(st), PLANES * kPlaneBytes);
#pragma unroll
                for (int p = 0; p < PLANES; ++p)
                    tma_load_2d(dst + static_cast<uint32_t>(p) * kPlaneBytes, &B.maps[q.pi][p], q.kb * (KB / 2), r0, W_FULL(st));
                last_phase[st] = w.phase;
                q.next(B);
            }
            // every TMA box issued has landed before the CTA may exit
            for (int i = 0; i < WS && i < 12; ++i)
                if (last_phase[i] >= 0) {
                    volatile int never = 0;
                    mbar_wait(W_FULL(i), static_cast<uint32_t>(last_phase[i]), &never, status);
                }
        }
        __syncwarp();
    } else if (warp < 16 && steps > 0) {
        // ------------------------------------------------ decode warps: two groups of eight take
        // alternate k-blocks; in a group, warp w decodes rows 32 (w % 4) .. + 31 (its
        // tensor-memory lane quarter) and half h = (w / 4) % 2 of the k-block (inputs
        // h KB/2 .. + KB/2 - 1, A-stage columns h KB/4 .. + KB/4 - 1), in chunks of 64
        // inputs (8 words per plane, 32 columns)
        constexpr int kChunks = KB / 128;   // 64-input chunks per half k-block
        const int grp = warp >> 3, half = (warp >> 2) & 1, row = 32 * (warp & 3) + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + static_cast<uint32_t>(half * (KB / 4));
        TileSeq<KB> q;
        q.init(B);
        if (grp == 1) q.next(B);
        // this row's group scales for the chunks of its half, loaded from global one
        // k-block of this group ahead
        auto scales_of = [&](const TileSeq<KB> &c, unsigned short (&out)[kChunks]) {
            const TcProb &P = B.p[c.pi];
            const int n0 = (c.tile - P.tile_begin) * kTcTile + row;
            const size_t base = static_cast<size_t>(n0 < P.n ? n0 : 0) * (P.k / G);
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch)
                out[ch] = ld_nc_u16(P.scales + base + (static_cast<size_t>(c.kb) * KB + half * (KB / 2) + 64 * ch) / G);
        };
        unsigned short s_next[kChunks];
        scales_of(q, s_next);
        Ring w(WS, grp), a(SA, grp);
        for (int it = grp; it < steps; it += 2, w.step(2), a.step(2)) {
            unsigned short sbits[kChunks];
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch) sbits[ch] = s_next[ch];
            TileSeq<KB> q2 = q;
            q2.next(B);
            q2.next(B);
            if (it + 2 < steps) scales_of(q2, s_next);
            const int st = w.slot, sa = a.slot;
            bool ok = mbar_wait(W_FULL(st), w.phase, abort_flag, status);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint32_t src = wbase + static_cast<uint32_t>(st) * kWStage;
            uint32_t bw[8 * kChunks], rw[8 * kChunks];
#pragma unroll
            for (int j = 0; j < 2 * kChunks; ++j) {
                const uint32_t at = src + wpos<KB>(row, 2 * kChunks * half + j);
                const uint4 v = lds128(at);
                bw[4 * j] = v.x; bw[4 * j + 1] = v.y; bw[4 * j + 2] = v.z; bw[4 * j + 3] = v.w;
                const uint4 r = PLANES == 2 ? lds128(at + kPlaneBytes) : make_uint4(0, 0, 0, 0);
                rw[4 * j] = r.x; rw[4 * j + 1] = r.y; rw[4 * j + 2] = r.z; rw[4 * j + 3] = r.w;
            }
            // the stage is refilled by TMA (async proxy) once every decode warp has
            // arrived: order this thread's shared-memory reads (generic proxy)
            // before that write.  Without the fence a refill could land before a
            // lane's read and feed that row the next k-block's codes (seen as rare
            // run-to-run differences in single rows at M = 144).
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(W_EMPTY(st));
            GroupK g[kChunks];
            bool all_fast = true;
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch) {
                g[ch] = group_consts<PLANES>(sbits[ch]);
                all_fast = all_fast && g[ch].fast;
            }
            all_fast = __all_sync(0xffffffffu, all_fast);
            ok = mbar_wait(A_EMPTY(sa), a.phase ^ 1, abort_flag, status);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch) {
                uint32_t v[32];
                if (all_fast) {
#pragma unroll
                    for (int w8 = 0; w8 < 8; ++w8)
                        decode_word<PLANES, true>(bw[8 * ch + w8], rw[8 * ch + w8], g[ch], &v[4 * w8]);
                } else {
#pragma unroll
                    for (int w8 = 0; w8 < 8; ++w8)
                        decode_word<PLANES, false>(bw[8 * ch + w8], rw[8 * ch + w8], g[ch], &v[4 * w8]);
                }
                const uint32_t col = lane_addr + static_cast<uint32_t>(kACols * sa + 32 * ch);
                tc_st16(col, *reinterpret_cast<const uint32_t(*)[16]>(&v[0]));
                tc_st16(col + 16, *reinterpret_cast<const uint32_t(*)[16]>(&v[16]));
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(A_FULL(sa));
            q = q2;
        }
    } else if (warp < 20 && steps > 0) {
        // ------------------------------------------------ epilogue warps
        const int qd = warp - 16;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        Ring d(ND);
        for (int tile = blockIdx.x; tile < B.total_tiles; tile += gridDim.x, d.step()) {
            const int db = d.slot;
            bool w_ok = mbar_wait(D_FULL(db), d.phase, abort_flag, status);
            if (!__all_sync(0xffffffffu, w_ok)) break;
            tc_fence_after();
            const TcProb &P = B.p[tile_problem(B, tile)];
            const int n = (tile - P.tile_begin) * kTcTile + 32 * qd + lane;
            const bool valid = n < P.n;
            for (int c0 = 0; c0 < Npad; c0 += 16) {
                uint32_t v[16];
                tc_ld16(lane_addr + dcol0 + static_cast<uint32_t>(db * Npad + c0), v);
                tc_wait_ld();
                if (valid) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < B.M) P.y[static_cast<size_t>(c0 + j) * P.n + n] = __uint_as_float(v[j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(D_EMPTY(db));
        }
    } else if (warp == 20 && lane == 0 && steps > 0) {
        // ------------------------------------------------ activation copies
        TileSeq<KB> q;
        q.init(B);
        int last_phase[8];
        for (int i = 0; i < 8; ++i) last_phase[i] = -1;
        Ring r(SB);
        for (int it = 0; it < steps; ++it, r.step()) {
            const int sb = r.slot;
            if (!mbar_wait(B_EMPTY(sb), r.phase ^ 1, abort_flag, status)) break;
            const TcProb &P = B.p[q.pi];
            mbar_expect_tx(B_FULL(sb), stage_bytes);
            bulk_g2s(sbase + static_cast<uint32_t>(sb) * stage_bytes,
                     P.xs + static_cast<size_t>(q.kb) * (stage_bytes / 2), stage_bytes, B_FULL(sb));
            last_phase[sb] = r.phase;
            q.next(B);
        }
        // every copy issued has landed before the CTA may exit
        for (int i = 0; i < SB && i < 8; ++i)
            if (last_phase[i] >= 0) {
                volatile int never = 0;
                mbar_wait(B_FULL(i), static_cast<uint32_t>(last_phase[i]), &never, status);
            }
    } else if (warp == 21 && steps > 0) {
        // ------------------------------------------------ MMA issue (the whole warp runs the
        // loop and waits; one elected lane issues the MMAs and commits)
        const uint32_t idesc = f16_idesc(kTcTile, Npad);
        Ring a(SA), r(SB), d(ND);
        bool ok = true;
        uint32_t issued_by = 0;   // lanes that have issued MMAs (the same mask on every lane)
        for (int tile = blockIdx.x; ok && tile < B.total_tiles; tile += gridDim.x, d.step()) {
            const int nkb = B.p[tile_problem(B, tile)].k / KB;
            const int db = d.slot;
            if (!__all_sync(0xffffffffu, mbar_wait(D_EMPTY(db), d.phase ^ 1, abort_flag, status))) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + dcol0 + static_cast<uint32_t>(db * Npad);
            const bool last_tile = tile + static_cast<int>(gridDim.x) >= B.total_tiles;
            for (int kb = 0; kb < nkb; ++kb, a.step(), r.step()) {
                const int sa = a.slot, sb = r.slot;
                bool w_ok = mbar_wait(A_FULL(sa), a.phase, abort_flag, status) &&
                            mbar_wait(B_FULL(sb), r.phase, abort_flag, status);
                if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
                tc_fence_after();
                const uint32_t b0 = sbase + static_cast<uint32_t>(sb) * stage_bytes;
                // every commit comes from the thread that issued the MMAs it must
                // track (a commit covers the issuing thread's own prior MMAs)
                uint32_t leader;
                if (elect_one(leader)) {
#pragma unroll
                    for (int t = 0; t < KB / 16; ++t) {
                        const uint32_t a_tmem = tmem + static_cast<uint32_t>(kACols * sa + 8 * t);
                        const uint64_t bd = sw128_desc(b0 + static_cast<uint32_t>((t >> 2) * Npad * 128 + (t & 3) * 32));
                        tc_mma(d_tmem, a_tmem, bd, idesc, (kb | t) != 0 ? 1u : 0u);
                    }
                    tc_commit(A_EMPTY(sa));
                    tc_commit(B_EMPTY(sb));
                    if (kb == nkb - 1) tc_commit(D_FULL(db));
                }
                __syncwarp();
                issued_by |= 1u << leader;
            }
            if (!ok) break;
        }
        // every MMA of this CTA has completed before tensor memory is freed, on
        // the normal path and after a wait gave up mid-tile alike: a lane that
        // issued MMAs commits to DONE_ALL (the commit tracks that lane's own
        // earlier MMAs), every other lane arrives on it without a commit, so no
        // commit is ever issued by a thread with no MMA behind it
        if (issued_by) {
            if ((issued_by >> lane) & 1u) tc_commit(DONE_ALL);
            else mbar_arrive(DONE_ALL);
            __syncwarp();
            volatile int never = 0;
            const bool drained = mbar_wait(DONE_ALL, 0, &never, status);
            // the drain itself gave up (sets NQ_DEV_TIMEOUT): MMAs may still
            // write tensor memory, so it is not freed
            if (!__all_sync(0xffffffffu, drained) && lane == 0) *keep_tmem = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 20 && *keep_tmem == 0) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------- bounded-wait self-test
// One warp waits, through the library's bounded wait, on an mbarrier that no
// thread or copy ever completes: the wait gives up after limit_ns, sets
// NQ_DEV_TIMEOUT and the kernel returns.  Nothing is in flight, so the
// context stays usable.
__global__ void __launch_bounds__(32) wait_selftest_kernel(unsigned long long limit_ns, unsigned int *status)
{
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const bool ok = mbar_test(b, 0) || mbar_wait_until(b, 0, &abort_flag, status, limit_ns);
    (void)__all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------- host side
int npad_of(int M) { return (std::min(M, kTcMaxN) + 15) / 16 * 16; }

size_t stage_region_bytes(int k, int npad) { return (static_cast<size_t>(2) * npad * k + 1023) / 1024 * 1024; }

bool tc_routable(int count, const nq_weights *w, int M, bool verify)
{
    if (M < kTcMinM) return false;
    for (int i = 0; i < count; ++i) {
        const int f = w[i].format;
        if (!(f == NQ_FMT_NESTED44 || (f == NQ_FMT_INT4 && !verify))) return false;
        if (w[i].k_in % kTcKB != 0 || (w[i].group != 64 && w[i].group != 128)) return false;
    }
    return true;
}

size_t tc_workspace(int count, const nq_weights *w, int M)
{
    const int npad = npad_of(M);
    size_t best = 0;
    for (int i0 = 0; i0 < count; i0 += kTcMaxP) {
        size_t sum = 0;
        for (int i = i0; i < std::min(count, i0 + kTcMaxP); ++i) sum += stage_region_bytes(w[i].k_in, npad);
        best = std::max(best, sum);
    }
    return best;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D map of one nibble plane: uint8 [n][k/2], box kb/2 bytes x 128 rows with
// the swizzle of the same width (64 or 128 bytes).
bool encode_plane(CUtensorMap *map, const void *plane, int n, int k, int kb)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k / 2), static_cast<cuuint64_t>(n)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k / 2)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kb / 2), static_cast<cuuint32_t>(kTcTile)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(plane), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, kb == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename F>
cudaError_t set_smem(F kernel, int bytes, std::atomic<int> &done)
{
    if (done.load() >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.store(bytes);
    return e;
}

template <int PLANES, int G, int KB>
cudaError_t launch_tc(TcBatch &b, int smem, cudaStream_t s, unsigned int *status)
{
    auto k = tc_kernel<PLANES, G, KB>;
    static std::atomic<int> attr{0};
    const cudaError_t e = set_smem(k, smem, attr);
    if (e != cudaSuccess) return e;
    const int grid = std::max(1, std::min(b.total_tiles, sm_count()));
    k<<<grid, kTcThreads, smem, s>>>(b, status);
    return cudaGetLastError();
}

}  // namespace

// Runs the batch on the tensor-memory path.  Preconditions (checked by the
// caller): tc_routable(), layers validated, ws of tc_workspace() bytes.
nq_status tc_run(int count, const nq_weights *w, const uint16_t *const *x, int M, float *const *y, bool verify,
                 void *ws, cudaStream_t stream)
{
    unsigned int *status = device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    const int planes = verify ? 2 : 1, group = w[0].group;
    bool k256 = true;   // every layer splits into 256-input k-blocks
    for (int i = 0; i < count; ++i) k256 = k256 && (w[i].k_in % kTcKBWide == 0);
    TcBatch b{};
    for (int m0 = 0; m0 < M; m0 += kTcMaxN) {
        const int Mc = std::min(kTcMaxN, M - m0);
        const int npad = npad_of(Mc);
        // 256-input k-blocks halve the per-k-block hand-offs per weight byte; they
        // fit tensor memory (3 x 128 A columns + 2 x Npad accumulator columns)
        // when Npad <= 64
        const int KB = (k256 && npad <= 64) ? kTcKBWide : kTcKB;
        const int acols = KB / 2;
        const uint32_t stage_bytes = 2u * KB * npad;
        const uint32_t wstage = planes * kTcTile * (KB / 2);
        // shared memory: up to 96 KB of weight stages in flight per SM (at least 3
        // stages), the rest for activation stages (2 to 8)
        const uint32_t avail = 222u * 1024u - 2048u;
        const int wsn = std::max(3, std::min(planes == 2 ? 4 : 8, static_cast<int>((avail - 4 * stage_bytes) / wstage)));
        const int sb = std::max(2, std::min(8, static_cast<int>((avail - wsn * wstage) / stage_bytes)));
        const int sa = (4 * acols + 2 * npad <= kTmemCols) ? 4 : 3;
        const int nd = (sa * acols + 2 * npad <= kTmemCols) ? 2 : 1;
        // 1 CTA per SM: the kernel allocates all 512 tensor-memory columns
        const int smem = std::max<int>(static_cast<int>(sb * stage_bytes + wsn * wstage) + 8 * 56 + 64 + 1024,
                                       120 * 1024);
        for (int i0 = 0; i0 < count; i0 += kTcMaxP) {
            const int cnt = std::min(kTcMaxP, count - i0);
            long long tiles = 0;
            size_t off = 0;
            int kmax = 0;
            for (int i = 0; i < cnt; ++i) {
                const nq_weights &L = w[i0 + i];
                TcProb &p = b.p[i];
                p.base = static_cast<const uint8_t *>(L.base);
                p.resid = static_cast<const uint8_t *>(L.resid);
                p.scales = static_cast<const uint16_t *>(L.scales);
                p.x = x[i0 + i] + static_cast<size_t>(m0) * L.k_in;
                p.y = y[i0 + i] + static_cast<size_t>(m0) * L.n_out;
                p.xs = reinterpret_cast<uint16_t *>(static_cast<unsigned char *>(ws) + off);
                p.n = L.n_out;
                p.k = L.k_in;
                p.tile_begin = static_cast<int>(tiles);
                p.pad = 0;
                if (!encode_plane(&b.maps[i][0], L.base, L.n_out, L.k_in, KB) ||
                    (planes == 2 && !encode_plane(&b.maps[i][1], L.resid, L.n_out, L.k_in, KB)))
                    return NQ_ERR_CUDA;
                const long long nt = (L.n_out + kTcTile - 1) / kTcTile;
                tiles += nt;
                off += stage_region_bytes(L.k_in, npad);
                kmax = std::max(kmax, L.k_in);
            }
            if (tiles > 0x7fffffffLL) return NQ_ERR_SHAPE;
            b.count = cnt;
            b.total_tiles = static_cast<int>(tiles);
            b.M = Mc;
            b.Npad = npad;
            b.group = group;
            b.sb = sb;
            b.sa = sa;
            b.nd = nd;
            b.ws = wsn;
            const long long chunks = static_cast<long long>(kmax / 8) * npad;
            const int gx = static_cast<int>(std::min<long long>((chunks + 255) / 256, 4096));
            tc_stage_kernel<<<dim3(gx, cnt), 256, 0, stream>>>(b, status);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return NQ_ERR_CUDA;
            if (KB == kTcKB) {
                if (planes == 2) e = group == 128 ? launch_tc<2, 128, 128>(b, smem, stream, status) : launch_tc<2, 64, 128>(b, smem, stream, status);
                else e = group == 128 ? launch_tc<1, 128, 128>(b, smem, stream, status) : launch_tc<1, 64, 128>(b, smem, stream, status);
            } else {
                if (planes == 2) e = group == 128 ? launch_tc<2, 128, 256>(b, smem, stream, status) : launch_tc<2, 64, 256>(b, smem, stream, status);
                else e = group == 128 ? launch_tc<1, 128, 256>(b, smem, stream, status) : launch_tc<1, 64, 256>(b, smem, stream, status);
            }
            if (e != cudaSuccess) return NQ_ERR_CUDA;
        }
    }
    return NQ_OK;
}

bool tc_route(int count, const nq_weights *w, int M, bool verify) { return tc_routable(count, w, M, verify); }
size_t tc_workspace_bytes(int count, const nq_weights *w, int M) { return tc_workspace(count, w, M); }

}  // namespace nq

extern "C" nq_status nq_selftest_bounded_wait(uint32_t limit_us, cudaStream_t stream)
{
    if (limit_us < 1 || limit_us > 1000000) return NQ_ERR_ARG;
    unsigned int *status = nq::device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    nq::wait_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<unsigned long long>(limit_us) * 1000ull, status);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}
