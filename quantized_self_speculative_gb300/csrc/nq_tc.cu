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
//   * warps 0-3 (one thread per weight row = one tensor-memory lane) load the
//     packed nibbles and the group scale straight from HBM into a register
//     ring and write the decoded weights, fp16(q * s) exactly rounded, into a
//     tensor-memory A stage (64 columns per 128 inputs) with tcgen05.st;
//   * warp 8 copies the activations of the k-block (already fp16, in the
//     MMA's 128-byte-swizzled K-major layout, written once per call by
//     tc_stage_kernel into the caller's workspace) into a shared-memory B
//     stage with one bulk copy;
//   * warp 9 issues tcgen05.mma (M = 128, N = padded M, K = 16; A from tensor
//     memory, B from shared memory, fp32 accumulators in tensor memory) and
//     tcgen05.commit to release the stages;
//   * warps 4-7 read the finished accumulators (tcgen05.ld) and store y.
//
// Decoding: offset-binary codes land in fp16 subnormals (code * 2^-24) with
// integer masks only; one fma per pair, fma(code * 2^-24, s * 2^20, -8 s),
// yields fp16(q8 * s / 16) (verify) or fp16(q4 * s) (draft) with one
// rounding.  Groups with s * 2^20 beyond the fp16 range (s > 0.0625) take an
// equivalent exact path (1024-biased fp16 integer, subtract, multiply) with
// the same result.  Every wait on an mbarrier is bounded by a timer; on a
// timeout the CTA sets NQ_DEV_TIMEOUT, drains its copies and MMAs, frees its
// tensor memory and returns.
#include "nq_internal.cuh"

#include <algorithm>
#include <atomic>

namespace nq {
namespace {

constexpr int kTcMinM = 16;            // smallest M routed here
constexpr int kTcMaxN = 256;           // activation rows per launch (MMA N)
constexpr int kTcTile = 128;           // weight rows per tile (MMA M)
constexpr int kTcKB = 128;             // inputs per k-block (8 MMAs of K = 16)
constexpr int kTcMaxP = 128;           // linears per launch
constexpr int kTcThreads = 320;        // warps 0-3 decode, 4-7 epilogue, 8 copy, 9 MMA
constexpr int kTmemCols = 512;
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s per wait

struct TcProb {
    const uint8_t *base;
    const uint8_t *resid;
    const uint16_t *scales;
    const uint16_t *x;     // bf16 [M][k] (rows of this M chunk)
    uint16_t *xs;          // staged fp16 activations in the workspace
    float *y;              // fp32 [M][n] (rows of this M chunk)
    long long cost_begin;  // prefix of tiles * k over the batch
    int n, k, tile_begin, pad;
};

struct TcBatch {
    long long total_cost;
    int count, total_tiles, M, Npad, group, sb, sa, nd;
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
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `bar` with the given parity.  Gives up after kWaitNs
// (sets the CTA's abort flag and NQ_DEV_TIMEOUT) or when another role of the
// CTA has given up; returns false then.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                       unsigned int *status)
{
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (unsigned int i = 1;; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > kWaitNs) {
                *abort_flag = 1;
                set_status(status, NQ_DEV_TIMEOUT);
                return false;
            }
        }
    }
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
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
// 16-byte read-only load kept in L1: the 32 lanes of a warp read 32 rows, and
// the second half of each 32-byte sector is used by the next load.
__device__ __forceinline__ uint4 ld_nc_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// Per-group decoding constants: fast = fma(code * 2^-24, F, C) with F = s 2^20,
// C = -8 s (both exact in fp16 when s <= 0x2BFF); slow = (1024 + code) - bias,
// times s16 (s/16 for the verify codes, s for the draft codes).
struct GroupK {
    uint32_t F, C, S;
    bool fast;
};
template <int PLANES>
__device__ __forceinline__ GroupK group_consts(unsigned short s_bits)
{
    GroupK g;
    const float s = __half2float(__ushort_as_half(s_bits));
    g.fast = (s_bits & 0x7FFFu) <= 0x2BFFu;
    g.F = dup_h(__half_as_ushort(__float2half_rn(__fmul_rn(s, 1048576.0f))));
    g.C = dup_h(__half_as_ushort(__float2half_rn(__fmul_rn(s, -8.0f))));
    g.S = dup_h(__half_as_ushort(__float2half_rn(PLANES == 2 ? __fmul_rn(s, 0.0625f) : s)));
    return g;
}

// Decode one 32-bit word per plane (8 consecutive inputs) into 4 fp16x2
// registers in the MMA order (0,4)(1,5)(2,6)(3,7).
template <int PLANES>
__device__ __forceinline__ void decode_word(uint32_t b, uint32_t r, const GroupK &g, uint32_t *o)
{
    uint32_t c0, c1, c2, c3;   // codes as fp16 subnormals: (q8 + 128) or 16 (q4 + 8), times 2^-24
    const uint32_t bx = b ^ 0x88888888u;
    if constexpr (PLANES == 2) {
        const uint32_t rx = r ^ 0x88888888u;
        // byte c of L: inputs 2c (base nibble high, refinement nibble low); H: inputs 2c+1
        const uint32_t L = (((bx << 4) & 0xF0F0F0F0u) | (rx & 0x0F0F0F0Fu)) - 0x08080808u;
        const uint32_t H = ((bx & 0xF0F0F0F0u) | ((rx >> 4) & 0x0F0F0F0Fu)) - 0x08080808u;
        c0 = L & 0x00FF00FFu;
        c1 = H & 0x00FF00FFu;
        c2 = (L >> 8) & 0x00FF00FFu;
        c3 = (H >> 8) & 0x00FF00FFu;
        if (g.fast) {
            o[0] = hfma2_u(c0, g.F, g.C);
            o[1] = hfma2_u(c1, g.F, g.C);
            o[2] = hfma2_u(c2, g.F, g.C);
            o[3] = hfma2_u(c3, g.F, g.C);
        } else {
            const uint32_t bias = 0x64806480u;   // fp16 1152 = 1024 + 128
            o[0] = hmul2_u(hsub2_u(c0 | 0x64006400u, bias), g.S);
            o[1] = hmul2_u(hsub2_u(c1 | 0x64006400u, bias), g.S);
            o[2] = hmul2_u(hsub2_u(c2 | 0x64006400u, bias), g.S);
            o[3] = hmul2_u(hsub2_u(c3 | 0x64006400u, bias), g.S);
        }
    } else {
        (void)r;
        c0 = (bx << 4) & 0x00F000F0u;
        c1 = bx & 0x00F000F0u;
        c2 = (bx >> 4) & 0x00F000F0u;
        c3 = (bx >> 8) & 0x00F000F0u;
        if (g.fast) {
            o[0] = hfma2_u(c0, g.F, g.C);
            o[1] = hfma2_u(c1, g.F, g.C);
            o[2] = hfma2_u(c2, g.F, g.C);
            o[3] = hfma2_u(c3, g.F, g.C);
        } else {
            const uint32_t bias = 0x64086408u;   // fp16 1032 = 1024 + 8
            o[0] = hmul2_u(hsub2_u((c0 >> 4) | 0x64006400u, bias), g.S);
            o[1] = hmul2_u(hsub2_u((c1 >> 4) | 0x64006400u, bias), g.S);
            o[2] = hmul2_u(hsub2_u((c2 >> 4) | 0x64006400u, bias), g.S);
            o[3] = hmul2_u(hsub2_u((c3 >> 4) | 0x64006400u, bias), g.S);
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
// First tile whose cost prefix is >= target.
__device__ __forceinline__ int tile_at_cost(const TcBatch &B, long long target)
{
    if (target >= B.total_cost) return B.total_tiles;
    int lo = 0, hi = B.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (B.p[mid].cost_begin <= target) lo = mid; else hi = mid - 1;
    }
    const TcProb &P = B.p[lo];
    return P.tile_begin + static_cast<int>((target - P.cost_begin + P.k - 1) / P.k);
}

// Walks the (tile, k-block) sequence of a CTA's tile range.
struct Cursor {
    int tile, pi, kb, nkb;
    __device__ void init(const TcBatch &B, int t)
    {
        tile = t;
        pi = tile_problem(B, t);
        kb = 0;
        nkb = B.p[pi].k / kTcKB;
    }
    __device__ void next(const TcBatch &B)
    {
        if (++kb == nkb) {
            kb = 0;
            ++tile;
            while (pi + 1 < B.count && tile >= B.p[pi + 1].tile_begin) ++pi;
            nkb = B.p[pi].k / kTcKB;
        }
    }
};

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

// ---------------------------------------------------------------- main kernel
template <int PLANES>
struct DqSlot {
    uint32_t b[16];
    uint32_t r[PLANES == 2 ? 16 : 1];
    unsigned short s[2];
};

template <int PLANES, int G>
__global__ void __launch_bounds__(kTcThreads, 1) tc_kernel(const __grid_constant__ TcBatch B, unsigned int *status)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (sbase - raw);
    const int Npad = B.Npad, SB = B.sb, SA = B.sa, ND = B.nd;
    const uint32_t stage_bytes = 256u * static_cast<uint32_t>(Npad);
    // barriers: a_full[4] a_empty[4] b_full[8] b_empty[8] d_full[2] d_empty[2] done
    const uint32_t bars = sbase + static_cast<uint32_t>(SB) * stage_bytes;
    auto A_FULL = [&](int i) { return bars + 8u * i; };
    auto A_EMPTY = [&](int i) { return bars + 8u * (4 + i); };
    auto B_FULL = [&](int i) { return bars + 8u * (8 + i); };
    auto B_EMPTY = [&](int i) { return bars + 8u * (16 + i); };
    auto D_FULL = [&](int i) { return bars + 8u * (24 + i); };
    auto D_EMPTY = [&](int i) { return bars + 8u * (26 + i); };
    const uint32_t DONE = bars + 8u * 28;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + static_cast<size_t>(SB) * stage_bytes + 8 * 32);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) { mbar_init(A_FULL(i), 4); mbar_init(A_EMPTY(i), 1); }
        for (int i = 0; i < 8; ++i) { mbar_init(B_FULL(i), 1); mbar_init(B_EMPTY(i), 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(D_FULL(i), 1); mbar_init(D_EMPTY(i), 4); }
        mbar_init(DONE, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 8) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int tb = tile_at_cost(B, B.total_cost * blockIdx.x / gridDim.x);
    const int te = tile_at_cost(B, B.total_cost * (blockIdx.x + 1) / gridDim.x);
    int steps = 0;
    if (tb < te) {
        Cursor c;
        c.init(B, tb);
        for (int pi = c.pi; pi < B.count && B.p[pi].tile_begin < te; ++pi) {
            const int t_end = pi + 1 < B.count ? B.p[pi + 1].tile_begin : B.total_tiles;
            const int a = max(tb, B.p[pi].tile_begin), b = min(te, t_end);
            steps += (b - a) * (B.p[pi].k / kTcKB);
        }
    }
    const uint32_t dcol0 = static_cast<uint32_t>(SA) * 64u;

    if (warp < 4 && steps > 0) {
        // ------------------------------------------------ decode warps
        constexpr int R = PLANES == 2 ? 3 : 4;
        const int row = threadIdx.x;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
        Cursor lc, cc;
        lc.init(B, tb);
        cc.init(B, tb);
        DqSlot<PLANES> ring[R];
        auto issue = [&](DqSlot<PLANES> &S) {
            const TcProb &P = B.p[lc.pi];
            const int n = (lc.tile - P.tile_begin) * kTcTile + row;
            const size_t nn = static_cast<size_t>(n < P.n ? n : 0);
            const size_t rowb = static_cast<size_t>(P.k) / 2;
            const uint8_t *pb = P.base + nn * rowb + static_cast<size_t>(lc.kb) * 64;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 v = ld_nc_v4(pb + 16 * q);
                S.b[4 * q] = v.x; S.b[4 * q + 1] = v.y; S.b[4 * q + 2] = v.z; S.b[4 * q + 3] = v.w;
            }
            if constexpr (PLANES == 2) {
                const uint8_t *pr = P.resid + nn * rowb + static_cast<size_t>(lc.kb) * 64;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v = ld_nc_v4(pr + 16 * q);
                    S.r[4 * q] = v.x; S.r[4 * q + 1] = v.y; S.r[4 * q + 2] = v.z; S.r[4 * q + 3] = v.w;
                }
            }
            const int ng = P.k / G;
            const uint16_t *ps = P.scales + nn * ng + static_cast<size_t>(lc.kb) * (kTcKB / G);
            S.s[0] = ld_nc_u16(ps);
            S.s[1] = G == 64 ? ld_nc_u16(ps + 1) : S.s[0];
            lc.next(B);
        };
        int a_iter = 0;
        bool ok = true;
        auto compute = [&](const DqSlot<PLANES> &S) {
            const int sa = a_iter % SA;
            const uint32_t par = ((a_iter / SA) & 1) ^ 1;
            bool w_ok = mbar_wait(A_EMPTY(sa), par, abort_flag, status);
            w_ok = __all_sync(0xffffffffu, w_ok);
            if (!w_ok) { ok = false; return; }
            tc_fence_after();
            const GroupK g0 = group_consts<PLANES>(S.s[0]);
            const GroupK g1 = G == 64 ? group_consts<PLANES>(S.s[1]) : g0;
#pragma unroll
            for (int part = 0; part < 4; ++part) {
                uint32_t v[16];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int wd = 4 * part + w;
                    decode_word<PLANES>(S.b[wd], S.r[PLANES == 2 ? wd : 0], wd < 8 ? g0 : g1, &v[4 * w]);
                }
                tc_st16(lane_addr + static_cast<uint32_t>(64 * sa + 16 * part), v);
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(A_FULL(sa));
            ++a_iter;
            cc.next(B);
        };
#pragma unroll
        for (int i = 0; i < R - 1; ++i)
            if (i < steps) issue(ring[i]);
        int s0 = 0;
        for (; ok && s0 + 2 * R - 2 < steps; s0 += R) {
#pragma unroll
            for (int i = 0; i < R; ++i) {
                issue(ring[(i + R - 1) % R]);
                if (ok) compute(ring[i]);
            }
        }
        for (; ok && s0 < steps; s0 += R) {
#pragma unroll
            for (int i = 0; i < R; ++i) {
                if (s0 + i < steps && ok) {
                    if (s0 + i + R - 1 < steps) issue(ring[(i + R - 1) % R]);
                    compute(ring[i]);
                }
            }
        }
    } else if (warp < 8 && steps > 0) {
        // ------------------------------------------------ epilogue warps
        const int q = warp - 4;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q) << 16);
        int d_iter = 0;
        for (int tile = tb; tile < te; ++tile) {
            const int db = d_iter % ND;
            bool w_ok = mbar_wait(D_FULL(db), (d_iter / ND) & 1, abort_flag, status);
            w_ok = __all_sync(0xffffffffu, w_ok);
            if (!w_ok) break;
            tc_fence_after();
            const TcProb &P = B.p[tile_problem(B, tile)];
            const int n = (tile - P.tile_begin) * kTcTile + 32 * q + lane;
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
            ++d_iter;
        }
    } else if (warp == 8 && lane == 0 && steps > 0) {
        // ------------------------------------------------ activation copies
        Cursor c;
        c.init(B, tb);
        int last_phase[8];
        for (int i = 0; i < 8; ++i) last_phase[i] = -1;
        for (int it = 0; it < steps; ++it) {
            const int sb = it % SB;
            if (!mbar_wait(B_EMPTY(sb), ((it / SB) & 1) ^ 1, abort_flag, status)) break;
            const TcProb &P = B.p[c.pi];
            mbar_expect_tx(B_FULL(sb), stage_bytes);
            bulk_g2s(sbase + static_cast<uint32_t>(sb) * stage_bytes,
                     P.xs + static_cast<size_t>(c.kb) * (stage_bytes / 2), stage_bytes, B_FULL(sb));
            last_phase[sb] = (it / SB) & 1;
            c.next(B);
        }
        // every copy issued has landed before the CTA may exit
        for (int i = 0; i < SB && i < 8; ++i)
            if (last_phase[i] >= 0) {
                volatile int never = 0;
                mbar_wait(B_FULL(i), static_cast<uint32_t>(last_phase[i]), &never, status);
            }
    } else if (warp == 9 && lane == 0 && steps > 0) {
        // ------------------------------------------------ MMA issue
        const uint32_t idesc = f16_idesc(kTcTile, Npad);
        int a_iter = 0, d_iter = 0, it = 0;
        bool ok = true, issued = false;
        for (int tile = tb; ok && tile < te; ++tile) {
            const int nkb = B.p[tile_problem(B, tile)].k / kTcKB;
            const int db = d_iter % ND;
            if (!mbar_wait(D_EMPTY(db), ((d_iter / ND) & 1) ^ 1, abort_flag, status)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + dcol0 + static_cast<uint32_t>(db * Npad);
            for (int kb = 0; kb < nkb; ++kb, ++it, ++a_iter) {
                const int sa = a_iter % SA, sb = it % SB;
                if (!mbar_wait(A_FULL(sa), (a_iter / SA) & 1, abort_flag, status) ||
                    !mbar_wait(B_FULL(sb), (it / SB) & 1, abort_flag, status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t b0 = sbase + static_cast<uint32_t>(sb) * stage_bytes;
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const uint32_t a_tmem = tmem + static_cast<uint32_t>(64 * sa + 8 * t);
                    const uint64_t bd = sw128_desc(b0 + static_cast<uint32_t>((t >> 2) * Npad * 128 + (t & 3) * 32));
                    tc_mma(d_tmem, a_tmem, bd, idesc, (kb | t) != 0 ? 1u : 0u);
                }
                issued = true;
                tc_commit(A_EMPTY(sa));
                tc_commit(B_EMPTY(sb));
            }
            if (!ok) break;
            tc_commit(D_FULL(db));
            ++d_iter;
        }
        if (issued) {
            // all MMAs issued by this thread have completed before tensor memory is freed
            tc_commit(DONE);
            volatile int never = 0;
            mbar_wait(DONE, 0, &never, status);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 8) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
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

template <typename F>
cudaError_t set_smem(F kernel, int bytes, std::atomic<int> &done)
{
    if (done.load() >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.store(bytes);
    return e;
}

template <int PLANES, int G>
cudaError_t launch_tc(TcBatch &b, int smem, cudaStream_t s, unsigned int *status)
{
    auto k = tc_kernel<PLANES, G>;
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
    TcBatch b{};
    for (int m0 = 0; m0 < M; m0 += kTcMaxN) {
        const int Mc = std::min(kTcMaxN, M - m0);
        const int npad = npad_of(Mc);
        const uint32_t stage_bytes = 256u * npad;
        const int sb = std::max(2, std::min(8, static_cast<int>((200u * 1024u) / stage_bytes)));
        const int sa = (4 * 64 + 2 * npad <= kTmemCols) ? 4 : 3;
        const int nd = (sa * 64 + 2 * npad <= kTmemCols) ? 2 : 1;
        // 1 CTA per SM: the kernel allocates all 512 tensor-memory columns
        const int smem = std::max<int>(static_cast<int>(sb * stage_bytes) + 8 * 32 + 64 + 1024, 120 * 1024);
        for (int i0 = 0; i0 < count; i0 += kTcMaxP) {
            const int cnt = std::min(kTcMaxP, count - i0);
            long long tiles = 0, cost = 0;
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
                p.cost_begin = cost;
                p.pad = 0;
                const long long nt = (L.n_out + kTcTile - 1) / kTcTile;
                tiles += nt;
                cost += nt * L.k_in;
                off += stage_region_bytes(L.k_in, npad);
                kmax = std::max(kmax, L.k_in);
            }
            if (tiles > 0x7fffffffLL) return NQ_ERR_SHAPE;
            b.total_cost = cost;
            b.count = cnt;
            b.total_tiles = static_cast<int>(tiles);
            b.M = Mc;
            b.Npad = npad;
            b.group = group;
            b.sb = sb;
            b.sa = sa;
            b.nd = nd;
            const long long chunks = static_cast<long long>(kmax / 8) * npad;
            const int gx = static_cast<int>(std::min<long long>((chunks + 255) / 256, 4096));
            tc_stage_kernel<<<dim3(gx, cnt), 256, 0, stream>>>(b, status);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return NQ_ERR_CUDA;
            if (planes == 2) e = group == 128 ? launch_tc<2, 128>(b, smem, stream, status) : launch_tc<2, 64>(b, smem, stream, status);
            else e = group == 128 ? launch_tc<1, 128>(b, smem, stream, status) : launch_tc<1, 64>(b, smem, stream, status);
            if (e != cudaSuccess) return NQ_ERR_CUDA;
        }
    }
    return NQ_OK;
}

bool tc_route(int count, const nq_weights *w, int M, bool verify) { return tc_routable(count, w, M, verify); }
size_t tc_workspace_bytes(int count, const nq_weights *w, int M) { return tc_workspace(count, w, M); }

}  // namespace nq
