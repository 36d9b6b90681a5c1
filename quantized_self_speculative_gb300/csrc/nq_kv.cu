// nq_kv.cu -- the nested KV cache: appending quantised K/V rows, and decode
// attention that reads the 4-bit base view (draft) or the full 8-bit view
// (verify) of the same cache.
//
// BitNest, Fig. 4 ("KV nesting during speculative decoding"): the draft stage
// reads only the low-bit base view of the cache, verification reads the full
// b_kv + r_kv-bit view, accepted entries stay and the rejected suffix is
// discarded; Fig. 5 and Tables 9-11: reading the KV4 base while drafting is
// what pays at long context.  Each K or V row of head_dim values is quantised
// exactly like a NESTED44 weight row (groups of `group` values along the head
// dimension, s = fp16(absmax / 7), base q4 and refinement r), so the draft
// value of an element is s q4 and the target value (s / 16)(16 q4 + r).
//
// Attention (one launch + a combine): the cache rows of a (sequence, kv head)
// are cut into splits of 256 to 1024 rows (chosen per call); a CTA of four
// warps takes one split and a tile of 16 query vectors (query heads sharing
// the kv head, times query rows), each warp a quarter of the split in blocks
// of 16 rows, streamed through a four-stage cp.async ring, with its own
// online softmax.  Both
// products run on the tensor cores (warp MMA m16n8k16, fp16 operands, fp32
// accumulators), in the manner of FlashAttention-2: S = Q K^T with the query
// tile as the A rows and a block of K as two B tiles, then O += P V with P
// taken straight from the S accumulators as the A operand.  The cache codes
// enter the MMAs undequantised: an offset-binary nibble (q4 + 8) or byte
// (16 q4 + r + 136) sits in the low bits of an fp16 half, i.e. code * 2^-24,
// placed with integer masks and byte permutes only.  The offset leaves S
// through the accumulator's initial value and O through a running sum of P;
// the group scales multiply S after its MMA and P before the V product.  The
// warps' states merge in shared memory, the splits' in a second kernel (a
// dependent launch).
#include "nq_internal.cuh"

#include <atomic>
#include <type_traits>

namespace nq {
namespace {

constexpr int kKvWarps = 4;
constexpr int kBlk = 16;                    // cache rows per MMA block
constexpr int kStages = 4;                  // cp.async ring per warp (blocks in flight)
constexpr int kMinBlkPerWarp = 4;           // blocks per warp: 4 .. 16 (chosen per call)
constexpr int kMaxBlkPerWarp = 16;
constexpr int kQTile = 16;                  // query vectors per CTA (MMA rows)
constexpr int kAppendWarps = 8;

struct Cache {
    int B, H, d, G, L;
    const uint8_t *kb, *kr, *vb, *vr;
    const __half *ks, *vs;
};

// Quantise row (b, h, i) of the new K or V rows (one warp per (row, group)).
template <int G>
__global__ void __launch_bounds__(kAppendWarps * 32)
kv_append_kernel(const float *__restrict__ src, int B, int H, int n_new, int d, int L, const int32_t *__restrict__ pos,
                 uint8_t *__restrict__ base, uint8_t *__restrict__ resid, __half *__restrict__ scales,
                 unsigned int *status)
{
    constexpr int E = G / 32;
    const int gpr = d / G;
    const long long job = static_cast<long long>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
    if (job >= static_cast<long long>(B) * H * n_new * gpr) return;
    const int lane = threadIdx.x & 31;
    const int grp = static_cast<int>(job % gpr);
    const long long rowi = job / gpr;                     // (b, h, i)
    const int i = static_cast<int>(rowi % n_new);
    const int h = static_cast<int>((rowi / n_new) % H);
    const int b = static_cast<int>(rowi / (static_cast<long long>(n_new) * H));
    const int t = pos[b] + i;
    if (t < 0 || t >= L) {
        if (lane == 0) set_status(status, NQ_DEV_SEQ_FULL);
        return;
    }
    const float *w = src + rowi * d + static_cast<size_t>(grp) * G + lane * E;
    float v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = w[e];
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
    const size_t row = (static_cast<size_t>(b) * H + h) * L + t;
    const size_t off = row * (d / 2) + static_cast<size_t>(grp) * (G / 2) + lane * (E / 2);
    if (E == 4) {
        *reinterpret_cast<uint16_t *>(base + off) = static_cast<uint16_t>(bb);
        *reinterpret_cast<uint16_t *>(resid + off) = static_cast<uint16_t>(rr);
    } else {
        base[off] = static_cast<uint8_t>(bb);
        resid[off] = static_cast<uint8_t>(rr);
    }
    if (lane == 0) scales[row * gpr + grp] = sh;
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t h2_pack(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// 2^x by the multi-function unit (about 2 ulp; the probabilities enter the
// products as fp16 anyway)
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Codes of nibbles i (low half) and i + 4 (high half) of a word of eight
// elements, as fp16 subnormals: KV4 (q4 + 8), where an odd i leaves the
// nibbles in bits 4-7 of each half (16 (q4 + 8): one shift per two pairs
// instead of one per pair; the other operand or the output carries the
// 1/16); KV8 from the base and refinement words, 16 (q4 + 8) + (r + 8) =
// q8 + 136: the code bytes of the even nibbles (0, 2, 4, 6) and of the odd
// ones are formed first (one shift and one bit-select each, shared by two
// pairs), then each pair is one mask or one byte permute.
template <int PLANES>
__device__ __forceinline__ uint32_t code_pair(uint32_t xb, uint32_t xr, int i)
{
    if constexpr (PLANES == 1) {
        (void)xr;
        const uint32_t x = i >= 2 ? xb >> 8 : xb;
        return (i & 1) ? ((x & 0x00F000F0u) ^ 0x00800080u) : ((x & 0x000F000Fu) ^ 0x00080008u);
    } else {
        // xb, xr already have every nibble's sign bit flipped (offset binary);
        // byte j of x is the code of nibble 2 j + (i & 1)
        const uint32_t x = (i & 1) ? ((xb & 0xF0F0F0F0u) | ((xr >> 4) & 0x0F0F0F0Fu))
                                   : (((xb << 4) & 0xF0F0F0F0u) | (xr & 0x0F0F0F0Fu));
        return i >= 2 ? __byte_perm(x, 0u, 0x4341) : (x & 0x00FF00FFu);
    }
}
// Scale of the codes code_pair returns for pair index i (1 or 16).
template <int PLANES>
__host__ __device__ constexpr float code_scale(int i) { return PLANES == 1 && (i & 1) ? 16.0f : 1.0f; }

// Byte offset of (row r, byte o) of a 16-row tile of rows of RB bytes in
// shared memory: 16-byte chunks, chunk q = r RB / 16 + o / 16 stored at
// position (q mod 8) xor (q / 8 mod 8) of its 128-byte line (the MMA operand
// reads of both products are then free of bank conflicts).
template <int RB>
__device__ __forceinline__ uint32_t swz(int r, int o)
{
    const int q = r * (RB / 16) + (o >> 4), line = q >> 3;
    return static_cast<uint32_t>((line << 7) + (((q & 7) ^ (line & 7)) << 4) + (o & 15));
}

template <int PLANES, int D>
struct AttnGeo {
    static constexpr int RB = D / 2;                          // bytes per row and plane
    static constexpr int TILE = kBlk * RB;                    // one plane of one block
    static constexpr int STAGE = 2 * PLANES * TILE;           // K and V planes of one block
    static constexpr int SCALES = 2 * kBlk * 2 * (D / 64);    // K and V scales of one block (fp16, up to 2 groups)
    static constexpr int WARP = kStages * STAGE + kMaxBlkPerWarp * SCALES;
    static constexpr int MERGE = kKvWarps * kQTile * (D + 2) * 4;
    static constexpr int SMEM = kKvWarps * WARP > MERGE ? kKvWarps * WARP : MERGE;
};

// Scales of a warp's blocks into its shared-memory slice, [block][K / V][row]
// [group] fp16: every load first, then the stores (one exposed latency, not
// one per load); rows past the warp's blocks are not read.
template <int NG>
__device__ __forceinline__ void stage_scales(unsigned short *ssm, const Cache &C, size_t rowbase, int key_w, int nblk,
                                             int lane)
{
    constexpr int PER_BLK = 2 * kBlk * NG, NSC = kMaxBlkPerWarp * PER_BLK / 32;
    unsigned short sv[NSC];
#pragma unroll
    for (int k = 0; k < NSC; ++k) {
        const int e = lane + 32 * k;
        const int bi = e / PER_BLK, rem = e % PER_BLK, which = rem / (kBlk * NG), idx = rem % (kBlk * NG);
        const int key = min(key_w + bi * kBlk + idx / NG, C.L - 1);
        const unsigned short *src = reinterpret_cast<const unsigned short *>(which ? C.vs : C.ks);
        sv[k] = bi < nblk ? ld_nc_u16(src + (rowbase + key) * NG + idx % NG) : static_cast<unsigned short>(0);
    }
#pragma unroll
    for (int k = 0; k < NSC; ++k) ssm[lane + 32 * k] = sv[k];
}

// The CTA's partials of query vectors v0 .. v0 + nqv - 1: the four warps'
// states (red_m, red_l: [warp][row]; red_o: [warp][row][D], NQT rows per
// warp) merged to one running maximum M2, sum and output per vector, stored
// as part[b][m][hq][split][D + 2] = (o[0..D-1], M2, l).
template <int D, int NQT>
__device__ __forceinline__ void store_partials(const float *red_m, const float *red_l, const float *red_o, int nqv,
                                               int v0, int g8, int kvh, int b, int M, int Hq, int nsplit, int split,
                                               float *__restrict__ part)
{
    for (int i = threadIdx.x; i < nqv * (D + 2); i += kKvWarps * 32) {
        const int r = i / (D + 2), j = i % (D + 2);
        float M2 = -INFINITY;
#pragma unroll
        for (int w = 0; w < kKvWarps; ++w) M2 = fmaxf(M2, red_m[w * NQT + r]);
        float val = 0.0f;
        if (j == D) {
            val = M2;
        } else {
#pragma unroll
            for (int w = 0; w < kKvWarps; ++w) {
                const float mw = red_m[w * NQT + r];
                const float f = mw == -INFINITY ? 0.0f : exp2f(mw - M2);
                val = fmaf(f, j == D + 1 ? red_l[w * NQT + r] : red_o[(w * NQT + r) * D + j], val);
            }
        }
        const int v = v0 + r, m = v / g8, hq = kvh * g8 + v % g8;
        part[((((static_cast<size_t>(b) * M + m) * Hq + hq) * nsplit) + split) * (D + 2) + j] = val;
    }
}

// Partial attention of one split of cache rows for one tile of 16 query
// vectors.  Query vector v = 16 z' + r (z' the tile index) = (query row m,
// query head hq) with m = v / g, hq = kvh g + v % g.  NG = D / G groups per
// row (1, or 2 when G = 64 < D = 128).  RR = 1 when the call has at most 8
// query vectors per kv head (rows 8..15 of the tile stay empty), else 2.
template <int PLANES, int D, int NG, int RR>
__global__ void __launch_bounds__(kKvWarps * 32, 3)
attn_split_kernel(Cache C, const float *__restrict__ q, int M, int Hq, const int32_t *__restrict__ len, float scale,
                  float *__restrict__ part, int nsplit, int qtiles, int nbw)
{
    using Geo = AttnGeo<PLANES, D>;
    constexpr int RB = Geo::RB, TILE = Geo::TILE, HALVES = D / 64;
    constexpr int OFF = PLANES == 2 ? 136 : 8;
    constexpr float FK = PLANES == 2 ? 1048576.0f : 16777216.0f;   // 2^24 undoes the code scale; s/16 for KV8
    static_assert(NG == 1 || (NG == 2 && D == 128), "groups");
    extern __shared__ __align__(128) unsigned char sm[];
    const int g8 = C.H == 0 ? 1 : Hq / C.H, nq_all = M * g8;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z / qtiles, qt = blockIdx.z % qtiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    // the combine may be scheduled now; it waits (griddepcontrol.wait) for
    // this grid to complete before it reads the partials
    asm volatile("griddepcontrol.launch_dependents;");
    const int Lb = min(len[b], C.L);
    const int t_begin = split * kKvWarps * kBlk * nbw, t_end = min(t_begin + kKvWarps * kBlk * nbw, Lb);
    if (t_begin >= Lb) return;                // past the sequence: the combine does not read this split
    const size_t rowbase = (static_cast<size_t>(b) * C.H + kvh) * C.L;

    // ---- this warp's blocks: K and V planes through a ring of kStages
    // shared-memory stages (cp.async), all of its scales up front (by lanes)
    unsigned char *wsm = sm + warp * Geo::WARP;
    const int key_w = t_begin + warp * nbw * kBlk;               // first cache row of the warp
    const int nblk = t_end > key_w ? min(nbw, (t_end - key_w + kBlk - 1) / kBlk) : 0;
    const uint8_t *planes[4] = {C.kb, C.vb, C.kr, C.vr};
    auto issue = [&](int bi) {
        const uint32_t st = static_cast<uint32_t>(__cvta_generic_to_shared(wsm + (bi % kStages) * Geo::STAGE));
#pragma unroll
        for (int pl = 0; pl < 2 * PLANES; ++pl) {
#pragma unroll
            for (int qq = lane; qq < TILE / 16; qq += 32) {
                const int r = qq / (RB / 16), c = qq % (RB / 16);
                const int key = min(key_w + bi * kBlk + r, C.L - 1);
                const uint8_t *src = planes[pl] + (rowbase + key) * RB + 16 * c;
                const uint32_t dst = st + pl * TILE + swz<RB>(r, 16 * c);
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
            }
        }
    };
#pragma unroll
    for (int bi = 0; bi < kStages; ++bi) {
        if (bi < nblk) issue(bi);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    unsigned short *ssm = reinterpret_cast<unsigned short *>(wsm + kStages * Geo::STAGE);
    stage_scales<NG>(ssm, C, rowbase, key_w, nblk, lane);

    // ---- query fragments (A operand): rows g and g + 8 of the tile, scaled by
    // scale log2(e) (scores in base 2), fp16, in the dimension order of the
    // K fragments; and per group the offset term of the scores
    uint32_t qa[HALVES][4][4];
    float cinit[NG][2];
    int lim[2];
    {
        float qsum[NG][2];
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) qsum[gr][0] = qsum[gr][1] = 0.0f;
        const float qs = scale * 1.4426950408889634f;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int v = qt * kQTile + g + 8 * rr;
            const bool valid = v < nq_all;
            const int m = valid ? v / g8 : 0, hq = kvh * g8 + (valid ? v % g8 : 0);
            lim[rr] = valid ? Lb - (M - 1 - m) : Lb;
            const float *qrow = q + ((static_cast<size_t>(b) * M + m) * Hq + hq) * D;
#pragma unroll
            for (int h = 0; h < HALVES; ++h) {
                float x[16];
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4) {
                    float4 f = valid ? *reinterpret_cast<const float4 *>(qrow + 64 * h + 16 * t + 4 * j4)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                    x[4 * j4] = __half2float(__float2half_rn(__fmul_rn(f.x, qs)));
                    x[4 * j4 + 1] = __half2float(__float2half_rn(__fmul_rn(f.y, qs)));
                    x[4 * j4 + 2] = __half2float(__float2half_rn(__fmul_rn(f.z, qs)));
                    x[4 * j4 + 3] = __half2float(__float2half_rn(__fmul_rn(f.w, qs)));
                }
                float sum = 0.0f;
#pragma unroll
                for (int j = 0; j < 16; ++j) sum += x[j];
                qsum[NG == 2 ? h : 0][rr] += sum;
                // slice sl: word w = sl / 2 of the lane's 16 dimensions, nibbles
                // i0, i0 + 4 (k = 2t, 2t + 1) and i0 + 1, i0 + 5 (k = 2t + 8, 2t + 9)
#pragma unroll
                for (int sl = 0; sl < 4; ++sl) {
                    const int w = sl >> 1, i0 = 2 * (sl & 1);
                    // A-fragment registers: (row g, k 2t..2t+1), (row g + 8, same),
                    // (row g, k 2t+8..2t+9), (row g + 8, same)
                    // (the second pair's codes come 16 times too large at KV4: x / 16 there, exact in fp16)
                    constexpr float kInv = 1.0f / code_scale<PLANES>(1);
                    qa[h][sl][rr] = h2_pack(x[8 * w + i0], x[8 * w + i0 + 4]);
                    qa[h][sl][2 + rr] = h2_pack(x[8 * w + i0 + 1] * kInv, x[8 * w + i0 + 5] * kInv);
                }
            }
        }
#pragma unroll
        for (int gr = 0; gr < NG; ++gr)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                float v = qsum[gr][rr];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                cinit[gr][rr] = -static_cast<float>(OFF) * 5.9604644775390625e-08f * v;
            }
    }

    float o[HALVES * 8][4];
#pragma unroll
    for (int nt = 0; nt < HALVES * 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.0f;
    float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.0f, 0.0f}, sig[NG][4];
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) sig[gr][0] = sig[gr][1] = sig[gr][2] = sig[gr][3] = 0.0f;
    // the lowest row limit of the warp's query rows: blocks below it need no mask
    int limw = min(t_end, RR == 2 ? min(lim[0], lim[1]) : lim[0]);
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) limw = min(limw, __shfl_xor_sync(0xffffffffu, limw, o2));
    for (int bi = 0; bi < nblk; ++bi) {
        // kStages groups are outstanding here; block bi's is the oldest
        asm volatile("cp.async.wait_group %0;" :: "n"(kStages - 1) : "memory");
        __syncwarp();
        const unsigned char *st = wsm + (bi % kStages) * Geo::STAGE;
        const int key0 = key_w + bi * kBlk;
        // ---- S = Q K^T: key tile kt holds cache rows kappa(8 kt + n) = 4 (n / 2) + 2 kt + n % 2
        // one accumulator per (half, key tile): four independent MMA chains;
        // the offset term enters through the first half of each group
        float acc[HALVES][2][4];
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
#pragma unroll
            for (int kt = 0; kt < 2; ++kt) {
                const bool first = NG == 2 || h == 0;
                acc[h][kt][0] = acc[h][kt][1] = first ? cinit[NG == 2 ? h : 0][0] : 0.0f;
                acc[h][kt][2] = acc[h][kt][3] = first ? cinit[NG == 2 ? h : 0][1] : 0.0f;
            }
        uint32_t xb[2][HALVES][2], xr[2][HALVES][2];
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
            const int kr = 4 * (g >> 1) + 2 * kt + (g & 1);
#pragma unroll
            for (int h = 0; h < HALVES; ++h) {
                const uint2 wb = *reinterpret_cast<const uint2 *>(st + swz<RB>(kr, 32 * h + 8 * t));
                uint2 wr = make_uint2(0u, 0u);
                if constexpr (PLANES == 2) wr = *reinterpret_cast<const uint2 *>(st + 2 * TILE + swz<RB>(kr, 32 * h + 8 * t));
                xb[kt][h][0] = PLANES == 2 ? wb.x ^ 0x88888888u : wb.x;
                xb[kt][h][1] = PLANES == 2 ? wb.y ^ 0x88888888u : wb.y;
                xr[kt][h][0] = wr.x ^ 0x88888888u;
                xr[kt][h][1] = wr.y ^ 0x88888888u;
            }
        }
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
            const int w = sl >> 1, i0 = 2 * (sl & 1);
#pragma unroll
            for (int h = 0; h < HALVES; ++h)
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const uint32_t b0 = code_pair<PLANES>(xb[kt][h][w], xr[kt][h][w], i0);
                    const uint32_t b1 = code_pair<PLANES>(xb[kt][h][w], xr[kt][h][w], i0 + 1);
                    mma16816(acc[h][kt], qa[h][sl], b0, b1);
                }
        }
        // ---- scores of rows (g, g + 8) x cache rows 4t + kk, kk = 0..3, then the
        // online softmax (base 2) and P' = p times the V row's group scale.
        // Masking (rows past the split or past a query row's causal limit)
        // is only needed where the block reaches the warp's lowest limit.
        float sk[4][NG], sv[4][NG];
        {
            const unsigned short *sc = ssm + bi * 2 * kBlk * NG;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int gr = 0; gr < NG; ++gr) {
                    sk[kk][gr] = __fmul_rn(__half2float(__ushort_as_half(sc[(4 * t + kk) * NG + gr])), FK);
                    const float v = __half2float(__ushort_as_half(sc[kBlk * NG + (4 * t + kk) * NG + gr]));
                    sv[kk][gr] = PLANES == 2 ? __fmul_rn(v, 0.0625f) : v;
                }
        }
        float alpha[2] = {1.0f, 1.0f};
        uint32_t pa[NG][4];
        auto softmax_block = [&](auto mask_c) {
            constexpr bool MASK = decltype(mask_c)::value;
#pragma unroll
            for (int rr = 0; rr < RR; ++rr) {
                float sr[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    float v = 0.0f;
#pragma unroll
                    for (int h = 0; h < HALVES; ++h)
                        v = fmaf(sk[kk][NG == 2 ? h : 0], acc[h][kk >> 1][(kk & 1) + 2 * rr], v);
                    if constexpr (MASK) {
                        const int key = key0 + 4 * t + kk;
                        v = (key < t_end && key < lim[rr]) ? v : -INFINITY;
                    }
                    sr[kk] = v;
                }
                float mx = fmaxf(fmaxf(sr[0], sr[1]), fmaxf(sr[2], sr[3]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float mn = fmaxf(mrun[rr], mx);
                // no earlier row: the state is all zeros, any factor does
                alpha[rr] = mrun[rr] == -INFINITY ? 0.0f : ex2(mrun[rr] - mn);
                mrun[rr] = mn;
                float pr[4], ps = 0.0f;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    pr[kk] = MASK ? (sr[kk] == -INFINITY ? 0.0f : ex2(sr[kk] - mn)) : ex2(sr[kk] - mn);
                    ps += pr[kk];
                }
                lrun[rr] = fmaf(lrun[rr], alpha[rr], ps);
#pragma unroll
                for (int gr = 0; gr < NG; ++gr) {
                    float pw[4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)     // masked rows may hold any scale bits: keep them out
                        pw[kk] = MASK ? (pr[kk] > 0.0f ? __fmul_rn(pr[kk], sv[kk][gr]) : 0.0f) : __fmul_rn(pr[kk], sv[kk][gr]);
                    pa[gr][rr] = h2_pack(pw[0], pw[1]);       // (row, cache rows 4t, 4t + 1) = k 2t, 2t + 1
                    pa[gr][2 + rr] = h2_pack(pw[2], pw[3]);   // (row, cache rows 4t + 2, 4t + 3) = k 2t + 8, 2t + 9
                }
            }
            if constexpr (RR == 1) {
#pragma unroll
                for (int gr = 0; gr < NG; ++gr) pa[gr][1] = pa[gr][3] = 0u;   // rows 8..15 hold no query
            }
        };
        if (key0 + kBlk <= limw) softmax_block(std::false_type{});
        else softmax_block(std::true_type{});
        if (__any_sync(0xffffffffu, alpha[0] != 1.0f || alpha[1] != 1.0f)) {
#pragma unroll
            for (int nt = 0; nt < HALVES * 8; ++nt) {
                o[nt][0] *= alpha[0]; o[nt][1] *= alpha[0];
                o[nt][2] *= alpha[1]; o[nt][3] *= alpha[1];
            }
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) {
                sig[gr][0] *= alpha[0]; sig[gr][1] *= alpha[0];
                sig[gr][2] *= alpha[1]; sig[gr][3] *= alpha[1];
            }
        }
        // sum of P' per row and group through the tensor cores: B = all ones
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) mma16816(sig[gr], pa[gr], 0x3C003C00u, 0x3C003C00u);
        // ---- O += P' V: n-tile (h, i) holds dimension 64 h + 8 n + i in column n
#pragma unroll
        for (int h = 0; h < HALVES; ++h) {
            uint32_t vb[4], vr[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                vb[kk] = *reinterpret_cast<const uint32_t *>(st + TILE + swz<RB>(4 * t + kk, 32 * h + 4 * g));
                if constexpr (PLANES == 2) {
                    vr[kk] = *reinterpret_cast<const uint32_t *>(st + 3 * TILE + swz<RB>(4 * t + kk, 32 * h + 4 * g)) ^ 0x88888888u;
                    vb[kk] ^= 0x88888888u;
                } else {
                    vr[kk] = 0u;
                }
            }
            // byte-interleave cache rows (4t, 4t + 1) and (4t + 2, 4t + 3): nibble i
            // of the first row of a pair lands at bit 4 i, of the second at 16 + 4 i
            const uint32_t u0[2] = {__byte_perm(vb[0], vb[1], 0x5410), __byte_perm(vb[0], vb[1], 0x7632)};
            const uint32_t u1[2] = {__byte_perm(vb[2], vb[3], 0x5410), __byte_perm(vb[2], vb[3], 0x7632)};
            uint32_t r0[2] = {0u, 0u}, r1[2] = {0u, 0u};
            if constexpr (PLANES == 2) {
                r0[0] = __byte_perm(vr[0], vr[1], 0x5410); r0[1] = __byte_perm(vr[0], vr[1], 0x7632);
                r1[0] = __byte_perm(vr[2], vr[3], 0x5410); r1[1] = __byte_perm(vr[2], vr[3], 0x7632);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t b0 = code_pair<PLANES>(u0[i >> 2], r0[i >> 2], i & 3);
                const uint32_t b1 = code_pair<PLANES>(u1[i >> 2], r1[i >> 2], i & 3);
                mma16816(o[8 * h + i], pa[NG == 2 ? h : 0], b0, b1);
            }
        }
        __syncwarp();                           // every lane is done with this stage: refill it
        if (bi + kStages < nblk) issue(bi + kStages);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    // finish the pipeline (blocks past this warp's range were committed empty)
    asm volatile("cp.async.wait_group 0;" ::: "memory");

    // ---- the warp's state: l summed over the four lanes of a row; the P'
    // sums (every column of sig holds its row's sum); O = 2^24 acc - off sum(P')
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        lrun[rr] += __shfl_xor_sync(0xffffffffu, lrun[rr], 1);
        lrun[rr] += __shfl_xor_sync(0xffffffffu, lrun[rr], 2);
    }
    __syncthreads();                           // every warp is done with its stages
    float *red_m = reinterpret_cast<float *>(sm);                 // [warp][row]
    float *red_l = red_m + kKvWarps * kQTile;                     // [warp][row]
    float *red_o = red_l + kKvWarps * kQTile;                     // [warp][row][D]
#pragma unroll
    for (int rr = 0; rr < RR; ++rr) {
        const int row = g + 8 * rr;
        if (t == 0) {
            red_m[warp * kQTile + row] = mrun[rr];
            red_l[warp * kQTile + row] = lrun[rr];
        }
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int n = 2 * t + cc, dim = 64 * h + 8 * n + i;
                    const float val = fmaf(16777216.0f / code_scale<PLANES>(i & 3), o[8 * h + i][2 * rr + cc],
                                           -static_cast<float>(OFF) * sig[NG == 2 ? h : 0][2 * rr]);
                    red_o[(warp * kQTile + row) * D + dim] = val;
                }
    }
    __syncthreads();
    store_partials<D, kQTile>(red_m, red_l, red_o, min(kQTile, nq_all - qt * kQTile), qt * kQTile, g8, kvh, b, M, Hq,
                              nsplit, split, part);
}

// ---- keys as rows, at most 8 query vectors per kv head (D = 128)
//
// S^T = K Q^T and O^T = V^T P'^T: the 16 cache rows of a block are the MMA's
// M dimension and the query vectors (up to 8) its N dimension, so no MMA row
// is empty: half the products and half the output accumulators of the
// query-tile kernel above when that tile would hold 8 or fewer vectors.  P'
// reaches the second product's B operand through a 256-byte shared tile per
// group (two 32-bit stores per lane, one ldmatrix.trans).  Same partials
// layout as the kernel above, merged by the same combine.
constexpr int kNQ = 8;

// Byte offset of (row r, byte o) of a 16-row block of 64-byte rows: 16-byte
// chunk c = o / 16 of row r at slot (4 (r mod 2) + c) xor 2 (r / 2 mod 4) of
// 128-byte line r / 2.  The K fragment reads (rows g and g + 8, 8 bytes at
// 32 h + 8 t) and the V fragment reads (rows 2 t + {0, 1, 8, 9}, 4 bytes at
// 32 h + 4 g) are then free of bank conflicts.
__device__ __forceinline__ uint32_t swz_kt(int r, int o)
{
    const int line = r >> 1, slot = ((4 * (r & 1)) + (o >> 4)) ^ (2 * (line & 3));
    return static_cast<uint32_t>((line << 7) + (slot << 4) + (o & 15));
}

// Four CTAs per SM: the KV8 read keeps three stages (the same bytes in
// flight per SM as four stages at three CTAs) and its one-group form fits
// 4 x (53 KB + 1 KB reserved) in the SM's 228 KB; the two-group KV8 form stays at three.
template <int PLANES, int NG>
struct AttnKtGeo {
    static constexpr int STAGES = PLANES == 2 ? 3 : kStages;
    static constexpr int CTAS = PLANES == 2 && NG == 2 ? 3 : 4;
    static constexpr int TILE = kBlk * 64;                    // one plane of one block
    static constexpr int STAGE = 2 * PLANES * TILE;           // K and V planes of one block
    static constexpr int SCALES = 2 * kBlk * NG * 2;          // K and V scales of one block (fp16)
    static constexpr int PT = NG * kBlk * kNQ * 2;            // P' tiles [group][cache row][query] fp16
    static constexpr int WARP = STAGES * STAGE + kMaxBlkPerWarp * SCALES + PT;
    static constexpr int MERGE = kKvWarps * kNQ * (128 + 2) * 4;
    static constexpr int SMEM = kKvWarps * WARP > MERGE ? kKvWarps * WARP : MERGE;
};

template <int PLANES, int NG>
__global__ void __launch_bounds__(kKvWarps * 32, AttnKtGeo<PLANES, NG>::CTAS)
attn_split_kt_kernel(Cache C, const float *__restrict__ q, int M, int Hq, const int32_t *__restrict__ len,
                     float scale, float *__restrict__ part, int nsplit, int nbw)
{
    constexpr int D = 128, RB = 64, HALVES = 2;
    using Geo = AttnKtGeo<PLANES, NG>;
    constexpr int TILE = Geo::TILE, STG = Geo::STAGES;
    constexpr int OFF = PLANES == 2 ? 136 : 8;
    constexpr float FK = PLANES == 2 ? 1048576.0f : 16777216.0f;   // 2^24 undoes the code scale; s/16 for KV8
    extern __shared__ __align__(128) unsigned char sm[];
    const int g8 = C.H == 0 ? 1 : Hq / C.H, nq_all = M * g8;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    asm volatile("griddepcontrol.launch_dependents;");
    const int Lb = min(len[b], C.L);
    const int t_begin = split * kKvWarps * kBlk * nbw, t_end = min(t_begin + kKvWarps * kBlk * nbw, Lb);
    if (t_begin >= Lb) return;                // past the sequence: the combine does not read this split
    const size_t rowbase = (static_cast<size_t>(b) * C.H + kvh) * C.L;

    // ---- this warp's blocks through a ring of STG shared-memory stages
    unsigned char *wsm = sm + warp * Geo::WARP;
    const int key_w = t_begin + warp * nbw * kBlk;
    const int nblk = t_end > key_w ? min(nbw, (t_end - key_w + kBlk - 1) / kBlk) : 0;
    const uint8_t *planes[4] = {C.kb, C.vb, C.kr, C.vr};
    auto issue = [&](int bi) {
        const uint32_t st = static_cast<uint32_t>(__cvta_generic_to_shared(wsm + (bi % STG) * Geo::STAGE));
#pragma unroll
        for (int pl = 0; pl < 2 * PLANES; ++pl) {
#pragma unroll
            for (int qq = lane; qq < TILE / 16; qq += 32) {
                const int r = qq / (RB / 16), c = qq % (RB / 16);
                const int key = min(key_w + bi * kBlk + r, C.L - 1);
                const uint8_t *src = planes[pl] + (rowbase + key) * RB + 16 * c;
                const uint32_t dst = st + pl * TILE + swz_kt(r, 16 * c);
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
            }
        }
    };
#pragma unroll
    for (int bi = 0; bi < STG; ++bi) {
        if (bi < nblk) issue(bi);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    unsigned short *ssm = reinterpret_cast<unsigned short *>(wsm + STG * Geo::STAGE);
    stage_scales<NG>(ssm, C, rowbase, key_w, nblk, lane);
    unsigned char *ptile = wsm + STG * Geo::STAGE + kMaxBlkPerWarp * Geo::SCALES;

    // ---- query fragments (B operand of S^T): query vector g, scaled by
    // scale log2(e), fp16, dimensions 64 h + 16 t .. + 15 in the order of the
    // K fragments; the offset term of the scores for columns 2t, 2t + 1
    uint32_t qb[HALVES][4][2];
    float cinit[NG][2];
    int lim[2];
    {
        float qsum[NG] = {};
        const float qs = scale * 1.4426950408889634f;
        const bool valid = g < nq_all;
        const int m = valid ? g / g8 : 0, hq = kvh * g8 + (valid ? g % g8 : 0);
        const float *qrow = q + ((static_cast<size_t>(b) * M + m) * Hq + hq) * D;
#pragma unroll
        for (int h = 0; h < HALVES; ++h) {
            float x[16];
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
                float4 f = valid ? *reinterpret_cast<const float4 *>(qrow + 64 * h + 16 * t + 4 * j4)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                x[4 * j4] = __half2float(__float2half_rn(__fmul_rn(f.x, qs)));
                x[4 * j4 + 1] = __half2float(__float2half_rn(__fmul_rn(f.y, qs)));
                x[4 * j4 + 2] = __half2float(__float2half_rn(__fmul_rn(f.z, qs)));
                x[4 * j4 + 3] = __half2float(__float2half_rn(__fmul_rn(f.w, qs)));
            }
            float sum = 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j) sum += x[j];
            qsum[NG == 2 ? h : 0] += sum;
            // k-step sl: word w = sl / 2 of the lane's 16 dimensions, nibbles
            // i0, i0 + 4 (slots 2t, 2t + 1) and i0 + 1, i0 + 5 (slots 2t + 8, 2t + 9);
            // the second pair's codes come 16 times too large at KV4: x / 16 there
#pragma unroll
            for (int sl = 0; sl < 4; ++sl) {
                const int w = sl >> 1, i0 = 2 * (sl & 1);
                constexpr float kInv = 1.0f / code_scale<PLANES>(1);
                qb[h][sl][0] = h2_pack(x[8 * w + i0], x[8 * w + i0 + 4]);
                qb[h][sl][1] = h2_pack(x[8 * w + i0 + 1] * kInv, x[8 * w + i0 + 5] * kInv);
            }
        }
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) {
            float v = qsum[gr];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);                 // query g's sum, in lanes 4g .. 4g + 3
#pragma unroll
            for (int c = 0; c < 2; ++c)
                cinit[gr][c] = -static_cast<float>(OFF) * 5.9604644775390625e-08f *
                               __shfl_sync(0xffffffffu, v, 4 * (2 * t + c));
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int n = 2 * t + c;
            lim[c] = n < nq_all ? Lb - (M - 1 - n / g8) : Lb;
        }
    }

    // O^T tile (h, i): row g = dimension 64 h + 8 g + i, row g + 8 = 64 h + 8 g + 4 + i;
    // columns 2t, 2t + 1 = queries
    float o[HALVES * 4][4];
#pragma unroll
    for (int ti = 0; ti < HALVES * 4; ++ti) o[ti][0] = o[ti][1] = o[ti][2] = o[ti][3] = 0.0f;
    float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.0f, 0.0f}, sig[NG][4];
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) sig[gr][0] = sig[gr][1] = sig[gr][2] = sig[gr][3] = 0.0f;
    int limw = min(t_end, min(lim[0], lim[1]));
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) limw = min(limw, __shfl_xor_sync(0xffffffffu, limw, o2));
    const uint32_t pt_s = static_cast<uint32_t>(__cvta_generic_to_shared(ptile));
    for (int bi = 0; bi < nblk; ++bi) {
        asm volatile("cp.async.wait_group %0;" :: "n"(STG - 1) : "memory");
        __syncwarp();
        const unsigned char *st = wsm + (bi % STG) * Geo::STAGE;
        const int key0 = key_w + bi * kBlk;
        // ---- S^T: rows g, g + 8 = cache rows key0 + g, key0 + g + 8; four
        // independent chains (half, word); the offset term enters the first
        // chain of each group
        float acc[HALVES][2][4];
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const bool first = w == 0 && (NG == 2 || h == 0);
                acc[h][w][0] = acc[h][w][2] = first ? cinit[NG == 2 ? h : 0][0] : 0.0f;
                acc[h][w][1] = acc[h][w][3] = first ? cinit[NG == 2 ? h : 0][1] : 0.0f;
            }
        uint32_t xb[HALVES][2][2], xr[HALVES][2][2];
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const uint2 wb = *reinterpret_cast<const uint2 *>(st + swz_kt(g + 8 * rr, 32 * h + 8 * t));
                uint2 wr = make_uint2(0u, 0u);
                if constexpr (PLANES == 2) wr = *reinterpret_cast<const uint2 *>(st + 2 * TILE + swz_kt(g + 8 * rr, 32 * h + 8 * t));
                xb[h][rr][0] = PLANES == 2 ? wb.x ^ 0x88888888u : wb.x;
                xb[h][rr][1] = PLANES == 2 ? wb.y ^ 0x88888888u : wb.y;
                xr[h][rr][0] = wr.x ^ 0x88888888u;
                xr[h][rr][1] = wr.y ^ 0x88888888u;
            }
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
            const int w = sl >> 1, i0 = 2 * (sl & 1);
#pragma unroll
            for (int h = 0; h < HALVES; ++h) {
                const uint32_t a[4] = {code_pair<PLANES>(xb[h][0][w], xr[h][0][w], i0),
                                       code_pair<PLANES>(xb[h][1][w], xr[h][1][w], i0),
                                       code_pair<PLANES>(xb[h][0][w], xr[h][0][w], i0 + 1),
                                       code_pair<PLANES>(xb[h][1][w], xr[h][1][w], i0 + 1)};
                mma16816(acc[h][w], a, qb[h][sl][0], qb[h][sl][1]);
            }
        }
        // ---- scores of cache rows (g, g + 8) x queries (2t, 2t + 1), the
        // online softmax (base 2) and P' = p times the V row's group scale,
        // stored as [cache row][query] for the transposing load
        float sk[2][NG], sv[2][NG];
        {
            const unsigned short *sc = ssm + bi * 2 * kBlk * NG;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int gr = 0; gr < NG; ++gr) {
                    sk[rr][gr] = __fmul_rn(__half2float(__ushort_as_half(sc[(g + 8 * rr) * NG + gr])), FK);
                    const float v = __half2float(__ushort_as_half(sc[kBlk * NG + (g + 8 * rr) * NG + gr]));
                    sv[rr][gr] = PLANES == 2 ? __fmul_rn(v, 0.0625f) : v;
                }
        }
        float alpha[2];
        auto softmax_block = [&](auto mask_c) {
            constexpr bool MASK = decltype(mask_c)::value;
            float s[2][2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float v = 0.0f;
#pragma unroll
                    for (int h = 0; h < HALVES; ++h)
                        v = fmaf(sk[rr][NG == 2 ? h : 0], acc[h][0][2 * rr + c] + acc[h][1][2 * rr + c], v);
                    if constexpr (MASK) {
                        const int key = key0 + g + 8 * rr;
                        v = (key < t_end && key < lim[c]) ? v : -INFINITY;
                    }
                    s[rr][c] = v;
                }
            float p[2][2];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float mx = fmaxf(s[0][c], s[1][c]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mn = fmaxf(mrun[c], mx);
                alpha[c] = mrun[c] == -INFINITY ? 0.0f : ex2(mrun[c] - mn);
                mrun[c] = mn;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
                    p[rr][c] = MASK ? (s[rr][c] == -INFINITY ? 0.0f : ex2(s[rr][c] - mn)) : ex2(s[rr][c] - mn);
                lrun[c] = fmaf(lrun[c], alpha[c], p[0][c] + p[1][c]);
            }
#pragma unroll
            for (int gr = 0; gr < NG; ++gr)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    float pw[2];
#pragma unroll
                    for (int c = 0; c < 2; ++c)      // masked rows may hold any scale bits: keep them out
                        pw[c] = MASK ? (p[rr][c] > 0.0f ? __fmul_rn(p[rr][c], sv[rr][gr]) : 0.0f)
                                     : __fmul_rn(p[rr][c], sv[rr][gr]);
                    *reinterpret_cast<uint32_t *>(ptile + gr * (kBlk * kNQ * 2) + (g + 8 * rr) * (kNQ * 2) + 4 * t) =
                        h2_pack(pw[0], pw[1]);
                }
        };
        if (key0 + kBlk <= limw) softmax_block(std::false_type{});
        else softmax_block(std::true_type{});
        if (__any_sync(0xffffffffu, alpha[0] != 1.0f || alpha[1] != 1.0f)) {
#pragma unroll
            for (int ti = 0; ti < HALVES * 4; ++ti) {
                o[ti][0] *= alpha[0]; o[ti][1] *= alpha[1];
                o[ti][2] *= alpha[0]; o[ti][3] *= alpha[1];
            }
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) {
                sig[gr][0] *= alpha[0]; sig[gr][1] *= alpha[1];
                sig[gr][2] *= alpha[0]; sig[gr][3] *= alpha[1];
            }
        }
        __syncwarp();                           // P' tiles written by every lane
        // B operand of O^T: (cache rows 2t, 2t + 1; query g) and (2t + 8, 2t + 9; g)
        uint32_t pb[NG][2];
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) {
            const uint32_t addr = pt_s + gr * (kBlk * kNQ * 2) + (lane & 15) * (kNQ * 2);
            asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                         : "=r"(pb[gr][0]), "=r"(pb[gr][1]) : "r"(addr) : "memory");
        }
        // sum of P' per query and group through the tensor cores: A = all ones
        {
            const uint32_t ones[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) mma16816(sig[gr], ones, pb[gr][0], pb[gr][1]);
        }
        // ---- O^T += V^T P'^T
#pragma unroll
        for (int h = 0; h < HALVES; ++h) {
            uint32_t vb[4], vr[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int row = 2 * t + (kk & 1) + 8 * (kk >> 1);
                vb[kk] = *reinterpret_cast<const uint32_t *>(st + TILE + swz_kt(row, 32 * h + 4 * g));
                if constexpr (PLANES == 2) {
                    vr[kk] = *reinterpret_cast<const uint32_t *>(st + 3 * TILE + swz_kt(row, 32 * h + 4 * g)) ^ 0x88888888u;
                    vb[kk] ^= 0x88888888u;
                } else {
                    vr[kk] = 0u;
                }
            }
            // byte-interleave cache rows (2t, 2t + 1) and (2t + 8, 2t + 9): nibble i
            // of the first row of a pair lands at bit 4 i, of the second at 16 + 4 i
            const uint32_t u0[2] = {__byte_perm(vb[0], vb[1], 0x5410), __byte_perm(vb[0], vb[1], 0x7632)};
            const uint32_t u1[2] = {__byte_perm(vb[2], vb[3], 0x5410), __byte_perm(vb[2], vb[3], 0x7632)};
            uint32_t r0[2] = {0u, 0u}, r1[2] = {0u, 0u};
            if constexpr (PLANES == 2) {
                r0[0] = __byte_perm(vr[0], vr[1], 0x5410); r0[1] = __byte_perm(vr[0], vr[1], 0x7632);
                r1[0] = __byte_perm(vr[2], vr[3], 0x5410); r1[1] = __byte_perm(vr[2], vr[3], 0x7632);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t a[4] = {code_pair<PLANES>(u0[0], r0[0], i), code_pair<PLANES>(u0[1], r0[1], i),
                                       code_pair<PLANES>(u1[0], r1[0], i), code_pair<PLANES>(u1[1], r1[1], i)};
                mma16816(o[4 * h + i], a, pb[NG == 2 ? h : 0][0], pb[NG == 2 ? h : 0][1]);
            }
        }
        __syncwarp();                           // every lane is done with this stage and the P' tiles
        if (bi + STG < nblk) issue(bi + STG);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");

    // ---- the warp's state: l summed over the eight lanes of a query; O =
    // 2^24 acc - off sum(P') (every row of sig holds its query's sum)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        lrun[c] += __shfl_xor_sync(0xffffffffu, lrun[c], 4);
        lrun[c] += __shfl_xor_sync(0xffffffffu, lrun[c], 8);
        lrun[c] += __shfl_xor_sync(0xffffffffu, lrun[c], 16);
    }
    __syncthreads();                           // every warp is done with its stages
    float *red_m = reinterpret_cast<float *>(sm);                 // [warp][query]
    float *red_l = red_m + kKvWarps * kNQ;                        // [warp][query]
    float *red_o = red_l + kKvWarps * kNQ;                        // [warp][query][D]
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int n = 2 * t + c;
        if (g == 0) {
            red_m[warp * kNQ + n] = mrun[c];
            red_l[warp * kNQ + n] = lrun[c];
        }
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int dim = 64 * h + 8 * g + 4 * rr + i;
                    const float val = fmaf(16777216.0f / code_scale<PLANES>(i), o[4 * h + i][2 * rr + c],
                                           -static_cast<float>(OFF) * sig[NG == 2 ? h : 0][c]);
                    red_o[(warp * kNQ + n) * D + dim] = val;
                }
    }
    __syncthreads();
    store_partials<D, kNQ>(red_m, red_l, red_o, min(kNQ, nq_all), 0, g8, kvh, b, M, Hq, nsplit, split, part);
}

// out[b][m][hq][:] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the
// splits that hold rows of the sequence (maxima in base 2).  One CTA per
// output vector: warp w merges splits w, w + 8, ... (lane l holds dimensions
// l, l + 32, ...), then the eight warps merge in shared memory.
constexpr int kCombWarps = 8;

template <int D>
__global__ void __launch_bounds__(kCombWarps * 32)
attn_combine_kernel(const float *__restrict__ part, int nsplit, int split_rows, const int32_t *__restrict__ len,
                    int L, int MHq, float *__restrict__ out)
{
    constexpr int DPL = D / 32;
    __shared__ float sm_m[kCombWarps], sm_l[kCombWarps], sm_o[kCombWarps][D];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t vec = blockIdx.x;            // (b, m, hq)
    const int b = static_cast<int>(vec / MHq);
    const int Lb = min(len[b], L);
    const int ns = min(nsplit, (Lb + split_rows - 1) / split_rows);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float m = -INFINITY, l = 0.0f, o[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = 0.0f;
    // four splits per step, all their loads issued before the first merge
    constexpr int U = 4;
    for (int sp0 = warp; sp0 < ns; sp0 += kCombWarps * U) {
        float ms[U], ls[U], ov[U][DPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int sp = sp0 + u * kCombWarps;
            ms[u] = -INFINITY;
            ls[u] = 0.0f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) ov[u][e] = 0.0f;
            if (sp < ns) {
                const float *p = part + (vec * nsplit + sp) * (D + 2);
                ms[u] = p[D];
                ls[u] = p[D + 1];
#pragma unroll
                for (int e = 0; e < DPL; ++e) ov[u][e] = p[lane + 32 * e];
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (ms[u] == -INFINITY) continue;     // no visible row in this split (warp-uniform)
            const float mn = fmaxf(m, ms[u]);
            const float a = m == -INFINITY ? 0.0f : exp2f(m - mn), f = exp2f(ms[u] - mn);
            l = fmaf(l, a, f * ls[u]);
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[e] = fmaf(o[e], a, f * ov[u][e]);
            m = mn;
        }
    }
    if (lane == 0) {
        sm_m[warp] = m;
        sm_l[warp] = l;
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e) sm_o[warp][lane + 32 * e] = o[e];
    __syncthreads();
    for (int j = threadIdx.x; j < D; j += kCombWarps * 32) {
        float M2 = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCombWarps; ++w) M2 = fmaxf(M2, sm_m[w]);
        float num = 0.0f, den = 0.0f;
#pragma unroll
        for (int w = 0; w < kCombWarps; ++w) {
            if (sm_m[w] == -INFINITY) continue;
            const float f = exp2f(sm_m[w] - M2);
            num = fmaf(f, sm_o[w][j], num);
            den = fmaf(f, sm_l[w], den);
        }
        out[vec * D + j] = den > 0.0f ? num / den : 0.0f;
    }
}

template <int PLANES, int D, int NG, int RR>
cudaError_t launch_attn_t(dim3 grid, cudaStream_t s, Cache C, const float *q, int M, int Hq, const int32_t *len,
                          float scale, float *part, int nsplit, int qtiles, int nbw)
{
    constexpr int smem = AttnGeo<PLANES, D>::SMEM;
    static std::atomic<bool> done[64];          // per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!done[dev].load()) {
        e = cudaFuncSetAttribute(attn_split_kernel<PLANES, D, NG, RR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem);
        if (e != cudaSuccess) return e;
        done[dev].store(true);
    }
    attn_split_kernel<PLANES, D, NG, RR><<<grid, kKvWarps * 32, smem, s>>>(C, q, M, Hq, len, scale, part, nsplit,
                                                                           qtiles, nbw);
    return cudaGetLastError();
}
template <int PLANES, int D, int NG>
cudaError_t launch_attn_r(int rr, dim3 grid, cudaStream_t s, Cache C, const float *q, int M, int Hq,
                          const int32_t *len, float scale, float *part, int nsplit, int qtiles, int nbw)
{
    return rr == 1 ? launch_attn_t<PLANES, D, NG, 1>(grid, s, C, q, M, Hq, len, scale, part, nsplit, qtiles, nbw)
                   : launch_attn_t<PLANES, D, NG, 2>(grid, s, C, q, M, Hq, len, scale, part, nsplit, qtiles, nbw);
}
template <int PLANES, int NG>
cudaError_t launch_attn_kt(dim3 grid, cudaStream_t s, Cache C, const float *q, int M, int Hq, const int32_t *len,
                           float scale, float *part, int nsplit, int nbw)
{
    constexpr int smem = AttnKtGeo<PLANES, NG>::SMEM;
    static std::atomic<bool> done[64];          // per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!done[dev].load()) {
        e = cudaFuncSetAttribute(attn_split_kt_kernel<PLANES, NG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        done[dev].store(true);
    }
    attn_split_kt_kernel<PLANES, NG><<<grid, kKvWarps * 32, smem, s>>>(C, q, M, Hq, len, scale, part, nsplit, nbw);
    return cudaGetLastError();
}
// D = 128 with at most 8 query vectors per kv head: keys as rows; otherwise
// the query-tile kernel
cudaError_t launch_attn(int planes, int d, int ng, int rr, dim3 grid, cudaStream_t s, Cache C, const float *q, int M,
                        int Hq, const int32_t *len, float scale, float *part, int nsplit, int qtiles, int nbw)
{
    if (d == 128) {
        if (rr == 1) {
            if (ng == 2)
                return planes == 1 ? launch_attn_kt<1, 2>(grid, s, C, q, M, Hq, len, scale, part, nsplit, nbw)
                                   : launch_attn_kt<2, 2>(grid, s, C, q, M, Hq, len, scale, part, nsplit, nbw);
            return planes == 1 ? launch_attn_kt<1, 1>(grid, s, C, q, M, Hq, len, scale, part, nsplit, nbw)
                               : launch_attn_kt<2, 1>(grid, s, C, q, M, Hq, len, scale, part, nsplit, nbw);
        }
        if (ng == 2)
            return planes == 1 ? launch_attn_t<1, 128, 2, 2>(grid, s, C, q, M, Hq, len, scale, part, nsplit, qtiles, nbw)
                               : launch_attn_t<2, 128, 2, 2>(grid, s, C, q, M, Hq, len, scale, part, nsplit, qtiles, nbw);
        return planes == 1 ? launch_attn_t<1, 128, 1, 2>(grid, s, C, q, M, Hq, len, scale, part, nsplit, qtiles, nbw)
                           : launch_attn_t<2, 128, 1, 2>(grid, s, C, q, M, Hq, len, scale, part, nsplit, qtiles, nbw);
    }
    return planes == 1 ? launch_attn_r<1, 64, 1>(rr, grid, s, C, q, M, Hq, len, scale, part, nsplit, qtiles, nbw)
                       : launch_attn_r<2, 64, 1>(rr, grid, s, C, q, M, Hq, len, scale, part, nsplit, qtiles, nbw);
}

nq_status check_cache(const nq_kv_cache *c)
{
    if (!c || c->batch < 1 || c->heads_kv < 1 || c->max_len < 1) return NQ_ERR_ARG;
    if (!(c->head_dim == 64 || c->head_dim == 128) || !(c->group == 64 || c->group == 128) || c->group > c->head_dim)
        return NQ_ERR_SHAPE;
    if (!c->k_base || !c->k_resid || !c->k_scales || !c->v_base || !c->v_resid || !c->v_scales) return NQ_ERR_ARG;
    if (!aligned16(c->k_base) || !aligned16(c->k_resid) || !aligned16(c->k_scales) || !aligned16(c->v_base) ||
        !aligned16(c->v_resid) || !aligned16(c->v_scales))
        return NQ_ERR_ALIGN;
    return NQ_OK;
}

// splits of a call with nbw blocks per warp; the workspace is sized for the
// smallest split (most of them)
int n_splits(int max_len, int nbw = kMinBlkPerWarp) { return (max_len + kKvWarps * kBlk * nbw - 1) / (kKvWarps * kBlk * nbw); }

}  // namespace
}  // namespace nq

extern "C" nq_status nq_kv_cache_bytes(int batch, int heads_kv, int head_dim, int group, int max_len,
                                       size_t *plane_bytes, size_t *scale_bytes)
{
    if (batch < 1 || heads_kv < 1 || max_len < 1) return NQ_ERR_ARG;
    if (!(head_dim == 64 || head_dim == 128) || !(group == 64 || group == 128) || group > head_dim) return NQ_ERR_SHAPE;
    const size_t rows = static_cast<size_t>(batch) * heads_kv * max_len;
    if (plane_bytes) *plane_bytes = rows * (head_dim / 2);
    if (scale_bytes) *scale_bytes = rows * (head_dim / group) * 2;
    return NQ_OK;
}

extern "C" nq_status nq_kv_append(const nq_kv_cache *cache, const float *k_new, const float *v_new, int n_new,
                                  const int32_t *pos, cudaStream_t stream)
{
    nq_status st = nq::check_cache(cache);
    if (st != NQ_OK) return st;
    if (!k_new || !v_new || !pos || n_new < 1 || n_new > cache->max_len) return NQ_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(k_new) & 15u) || (reinterpret_cast<uintptr_t>(v_new) & 15u) ||
        (reinterpret_cast<uintptr_t>(pos) & 3u))
        return NQ_ERR_ALIGN;
    unsigned int *status = nq::device_status_ptr();
    if (!status) return NQ_ERR_CUDA;
    const nq_kv_cache &c = *cache;
    const long long jobs = static_cast<long long>(c.batch) * c.heads_kv * n_new * (c.head_dim / c.group);
    const int grid = static_cast<int>((jobs + nq::kAppendWarps - 1) / nq::kAppendWarps);
    for (int which = 0; which < 2; ++which) {
        const float *src = which ? v_new : k_new;
        auto *base = static_cast<uint8_t *>(which ? c.v_base : c.k_base);
        auto *resid = static_cast<uint8_t *>(which ? c.v_resid : c.k_resid);
        auto *sc = static_cast<__half *>(which ? c.v_scales : c.k_scales);
        if (c.group == 128)
            nq::kv_append_kernel<128><<<grid, nq::kAppendWarps * 32, 0, stream>>>(
                src, c.batch, c.heads_kv, n_new, c.head_dim, c.max_len, pos, base, resid, sc, status);
        else
            nq::kv_append_kernel<64><<<grid, nq::kAppendWarps * 32, 0, stream>>>(
                src, c.batch, c.heads_kv, n_new, c.head_dim, c.max_len, pos, base, resid, sc, status);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return NQ_ERR_CUDA;
    }
    return NQ_OK;
}

extern "C" size_t nq_attn_workspace_bytes(int batch, int M, int heads_q, int head_dim, int max_len)
{
    if (batch < 1 || M < 1 || heads_q < 1 || max_len < 1 || !(head_dim == 64 || head_dim == 128)) return 0;
    return static_cast<size_t>(batch) * M * heads_q * nq::n_splits(max_len) * (head_dim + 2) * sizeof(float);
}

extern "C" nq_status nq_attn_decode(const nq_kv_cache *cache, const float *q, int M, int heads_q, const int32_t *len,
                                    int planes, float scale, float *out, void *ws, size_t ws_bytes,
                                    cudaStream_t stream)
{
    nq_status st = nq::check_cache(cache);
    if (st != NQ_OK) return st;
    const nq_kv_cache &c = *cache;
    if (!q || !len || !out || M < 1 || M > c.max_len || heads_q < c.heads_kv || heads_q % c.heads_kv != 0 ||
        (planes != 1 && planes != 2) || !(scale > 0.0f))
        return NQ_ERR_ARG;
    if (!nq::aligned16(q) || !nq::aligned16(out) || (reinterpret_cast<uintptr_t>(len) & 3u)) return NQ_ERR_ALIGN;
    if (!ws || ws_bytes < nq_attn_workspace_bytes(c.batch, M, heads_q, c.head_dim, c.max_len)) return NQ_ERR_WORKSPACE;
    if (!nq::aligned16(ws)) return NQ_ERR_ALIGN;
    const int g = heads_q / c.heads_kv, nq_all = M * g;
    const int qtiles = (nq_all + nq::kQTile - 1) / nq::kQTile;
    if (static_cast<long long>(c.batch) * qtiles > 65535 || c.heads_kv > 65535) return NQ_ERR_SHAPE;
    // the longest splits (fewest CTAs and partials, per-CTA work amortised),
    // shortened only below one CTA per SM.  Measured at 32K rows: LLaMA-2-7B
    // MHA draft / verify 53.7 / 76.2 us per layer at 1024-row splits against
    // 76.3 / 104.4 at 256; Qwen2.5-7B GQA 18.1 / 41.3 against 22.7 / 61.0.
    const long long units = static_cast<long long>(c.batch) * c.heads_kv * qtiles;
    int nbw = nq::kMaxBlkPerWarp;
    while (nbw > nq::kMinBlkPerWarp && units * nq::n_splits(c.max_len, nbw) < nq::sm_count()) nbw /= 2;
    const int nsplit = nq::n_splits(c.max_len, nbw);
    nq::Cache C{c.batch, c.heads_kv, c.head_dim, c.group, c.max_len,
                static_cast<const uint8_t *>(c.k_base), static_cast<const uint8_t *>(c.k_resid),
                static_cast<const uint8_t *>(c.v_base), static_cast<const uint8_t *>(c.v_resid),
                static_cast<const __half *>(c.k_scales), static_cast<const __half *>(c.v_scales)};
    float *part = static_cast<float *>(ws);
    dim3 grid(nsplit, c.heads_kv, c.batch * qtiles);
    cudaError_t e = nq::launch_attn(planes, c.head_dim, c.head_dim / c.group, nq_all <= 8 ? 1 : 2, grid, stream, C,
                                    q, M, heads_q, len, scale, part, nsplit, qtiles, nbw);
    if (e != cudaSuccess) return NQ_ERR_CUDA;
    const int nvec = c.batch * M * heads_q;
    const int rows = nq::kKvWarps * nq::kBlk * nbw;
    // the combine as a programmatic dependent launch: its launch overlaps the
    // split kernel's tail, griddepcontrol.wait orders its reads after it
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nvec);
    cfg.blockDim = dim3(nq::kCombWarps * 32);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float *cpart = part;
    const int mhq = M * heads_q;
    if (c.head_dim == 128)
        e = cudaLaunchKernelEx(&cfg, nq::attn_combine_kernel<128>, cpart, nsplit, rows, len, c.max_len, mhq, out);
    else
        e = cudaLaunchKernelEx(&cfg, nq::attn_combine_kernel<64>, cpart, nsplit, rows, len, c.max_len, mhq, out);
    return nq::cuda_status(e);
}
