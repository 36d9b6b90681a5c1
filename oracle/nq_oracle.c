/*
 * nq_oracle.c -- plain, slow, obviously correct CPU oracle for the hot path of
 * quantized self-speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library: every routine below is written from the definitions it cites.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (no SIMD intrinsics, no BLAS).  Floating point follows IEEE-754 with the
 * default round-to-nearest-even mode; `float` expressions are evaluated in
 * float (FLT_EVAL_METHOD == 0 on x86-64 SSE and on aarch64).
 *
 * Sources (cited by page title and section / table / equation):
 *   [BitNest]  "BitNest: Bit-Nested Speculative Decoding for Memory-Efficient
 *              LLM Inference Acceleration" -- abstract; Fig. 2 (b-bit base +
 *              r-bit refinement of the remaining error; drafting reads only
 *              the base, verification reads both planes); Fig. 3 (dual-plane
 *              storage: two independent 4-bit streams of N/2 bytes each, the
 *              target recovers the full 8-bit representation).
 *   [SpecQuant] "SpecQuant -- Speculative Decoding with Multi-Parent
 *              Quantization for Adaptive LLM Inference", Sec. III.A
 *              (Q4 = f(W16, 4) INT4, Q8 = f(W16, 8) FP8, Q16 = W16) and
 *              Sec. III.D.4 (token acceptance or correction).
 *   [Erge]     "How Speculative Decoding Speeds Up Inference" -- "Drafting
 *              and checking tokens" (the round), Table 1 (k = 4 worked
 *              round), "The same output as the large model alone" (greedy
 *              equivalence; speculative sampling of Leviathan et al. and Chen
 *              et al. follows the target distribution), Eq. (1).
 *   [Philox]   Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 *              as 1, 2, 3", SC'11 -- the Philox4x32-10 bijection.
 *
 * Readings where the pages are silent:
 *   R1  per (row, group of G consecutive inputs) symmetric scale
 *       s = fp16(fp32(absmax / 7)); base q4 = clamp(rint(w/s), -8, 7);
 *       refinement r = clamp(rint(16 (w/s - q4)), -8, 7); residual scale s/16;
 *       8-bit target code q8 = 16 q4 + r.  absmax == 0 (or s == 0) -> all 0.
 *   R2  two's-complement nibbles, element 2j in the low nibble of byte j,
 *       row-major planes [N][K/2]; scales fp16 [N][K/G].
 *   R3  FP8 tier: per-output-row scale s_n = absmax_row / 448 (fp32), code =
 *       E4M3FN(w / s_n) round-to-nearest-even, saturating at +-448.
 *   R4  greedy: argmax ties go to the lowest index; pads are -1.
 *   R5  sampled acceptance canonical arithmetic: see the block comment above
 *       orc_exp2c().
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "nq_oracle.h"

/* ======================================================================== */
/* Number formats, written from the IEEE-754 / OCP FP8 definitions.          */
/* ======================================================================== */

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bfloat16 is the top half of a binary32. */
float orc_bf16_to_f32(uint16_t b) { return bits_to_f32((uint32_t)b << 16); }

/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
float orc_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    float v;
    if (e == 0)       v = ldexpf((float)m, -24);                 /* subnormal */
    else if (e == 31) v = m ? NAN : INFINITY;
    else              v = ldexpf((float)(1024 + m), e - 25);     /* (1+m/1024) 2^(e-15) */
    return sign ? -v : v;
}

/* Round a finite non-negative value to a multiple of the quantum `q`
 * (a power of two), ties to even. a/q is exact (power-of-two scaling). */
static float round_to_quantum(float a, float q) { return rintf(a / q) * q; }

/* binary32 -> binary16, round to nearest even, overflow -> inf. */
uint16_t orc_f32_to_f16(float f)
{
    uint32_t sign = (f32_to_bits(f) >> 31) << 15;
    float a = fabsf(f);
    if (isnan(f)) return (uint16_t)(sign | 0x7E00);
    if (a >= 65520.0f) return (uint16_t)(sign | 0x7C00);         /* rounds past 65504 */
    float q;
    if (a < ldexpf(1.0f, -14)) q = ldexpf(1.0f, -24);            /* subnormal spacing */
    else { int e; frexpf(a, &e); q = ldexpf(1.0f, (e - 1) - 10); }
    float v = round_to_quantum(a, q);
    if (v == 0.0f) return (uint16_t)sign;
    if (v < ldexpf(1.0f, -14)) return (uint16_t)(sign | (uint32_t)(v / ldexpf(1.0f, -24)));
    int e; float fr = frexpf(v, &e);            /* v = fr 2^e, fr in [0.5,1) */
    uint32_t E = (uint32_t)(e - 1 + 15);
    uint32_t M = (uint32_t)((fr * 2.0f - 1.0f) * 1024.0f);
    return (uint16_t)(sign | (E << 10) | M);
}

/* E4M3FN (OCP 8-bit FP): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * no infinities; S.1111.111 is NaN; largest finite 448 = 1.75 * 2^8. */
float orc_e4m3_to_f32(uint8_t c)
{
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    float v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexpf((float)m, -9);                        /* subnormal */
    else        v = ldexpf((float)(8 + m), e - 10);              /* (1+m/8) 2^(e-7) */
    return sign ? -v : v;
}

/* binary32 -> E4M3FN, round to nearest even, saturate to +-448, NaN -> 0x7F. */
uint8_t orc_f32_to_e4m3(float f)
{
    uint8_t sign = (uint8_t)((f32_to_bits(f) >> 31) << 7);
    if (isnan(f)) return 0x7F;
    float a = fabsf(f);
    if (a >= 448.0f) return (uint8_t)(sign | 0x7E);
    float q;
    if (a < ldexpf(1.0f, -6)) q = ldexpf(1.0f, -9);
    else { int e; frexpf(a, &e); q = ldexpf(1.0f, (e - 1) - 3); }
    float v = round_to_quantum(a, q);
    if (v > 448.0f) v = 448.0f;
    if (v == 0.0f) return sign;
    if (v < ldexpf(1.0f, -6)) return (uint8_t)(sign | (uint8_t)(v / ldexpf(1.0f, -9)));
    int e; float fr = frexpf(v, &e);
    uint8_t E = (uint8_t)(e - 1 + 7);
    uint8_t M = (uint8_t)((fr * 2.0f - 1.0f) * 8.0f);
    return (uint8_t)(sign | (E << 3) | M);
}

/* ======================================================================== */
/* C1: nested quantise / pack / unpack  [BitNest Fig. 2, Fig. 3; R1, R2]     */
/* ======================================================================== */

static int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* Signed value of a two's-complement nibble. */
int orc_nibble_value(unsigned nib) { nib &= 15u; return nib >= 8 ? (int)nib - 16 : (int)nib; }

static void put_nibble(uint8_t *plane, size_t idx, int code)
{
    uint8_t nib = (uint8_t)(code & 15);
    if (idx % 2 == 0) plane[idx / 2] = (uint8_t)((plane[idx / 2] & 0xF0) | nib);
    else              plane[idx / 2] = (uint8_t)((plane[idx / 2] & 0x0F) | (nib << 4));
}

int orc_get_code(const uint8_t *plane, size_t idx)
{
    uint8_t byte = plane[idx / 2];
    return orc_nibble_value(idx % 2 == 0 ? byte & 15 : byte >> 4);
}

/*
 * Quantise one weight given its group's scale (R1): the b = 4-bit base code
 * first, then the remaining error w/s - q4 quantised to the r = 4-bit
 * refinement at a sixteenth of the base step [BitNest Fig. 2].
 */
void orc_quantise_weight(float w, float s, int *q4, int *r)
{
    if (s == 0.0f) { *q4 = 0; *r = 0; return; }
    float x = w / s;
    int b = clampi((int)rintf(x), -8, 7);
    float err = (x - (float)b) * 16.0f;
    *q4 = b;
    *r = clampi((int)rintf(err), -8, 7);
}

/*
 * Pack W [n][k] (fp32) into the base plane, the refinement plane (may be NULL
 * for the INT4 tier, which is exactly the base plane [SpecQuant III.A Q4]) and
 * fp16 group scales.  Returns 0, or -1 on bad arguments / non-finite weights.
 */
int orc_pack_nested(const float *w, int n, int k, int g,
                    uint8_t *base, uint8_t *resid, uint16_t *scales)
{
    if (n < 0 || k <= 0 || g <= 0 || k % g != 0 || k % 2 != 0) return -1;
    for (int row = 0; row < n; row++) {
        for (int grp = 0; grp < k / g; grp++) {
            const float *wg = w + (size_t)row * k + (size_t)grp * g;
            float amax = 0.0f;
            for (int i = 0; i < g; i++) {
                if (!isfinite(wg[i])) return -1;
                if (fabsf(wg[i]) > amax) amax = fabsf(wg[i]);
            }
            uint16_t sh = orc_f32_to_f16(amax / 7.0f);
            float s = orc_f16_to_f32(sh);
            scales[(size_t)row * (k / g) + grp] = sh;
            for (int i = 0; i < g; i++) {
                int q4, r;
                orc_quantise_weight(wg[i], s, &q4, &r);
                size_t idx = (size_t)row * k + (size_t)grp * g + i;
                put_nibble(base, idx, q4);
                if (resid) put_nibble(resid, idx, r);
            }
        }
    }
    return 0;
}

/* FP8 tier [SpecQuant III.A Q8 = f(W16, 8); R3]. */
int orc_pack_fp8(const float *w, int n, int k, uint8_t *codes, float *row_scale)
{
    for (int row = 0; row < n; row++) {
        const float *wr = w + (size_t)row * k;
        float amax = 0.0f;
        for (int i = 0; i < k; i++) {
            if (!isfinite(wr[i])) return -1;
            if (fabsf(wr[i]) > amax) amax = fabsf(wr[i]);
        }
        float s = amax / 448.0f;
        row_scale[row] = s;
        for (int i = 0; i < k; i++)
            codes[(size_t)row * k + i] = s == 0.0f ? 0 : orc_f32_to_e4m3(wr[i] / s);
    }
    return 0;
}

/* FP16 tier [SpecQuant III.A Q16 = W16]. */
int orc_pack_fp16(const float *w, int n, int k, uint16_t *w16)
{
    for (size_t i = 0; i < (size_t)n * k; i++) {
        if (!isfinite(w[i])) return -1;
        w16[i] = orc_f32_to_f16(w[i]);
    }
    return 0;
}

/* ======================================================================== */
/* C2: dequantised linear, fp64 accumulation                                 */
/*   draft : y[m,n] = sum_g s[n,g]      sum_{k in g} q4[n,k]          x[m,k] */
/*   verify: y[m,n] = sum_g (s[n,g]/16) sum_{k in g} (16 q4 + r)[n,k] x[m,k] */
/* [BitNest Fig. 2: drafting reads only the base, verification reads both]   */
/* ======================================================================== */

static double linear_row_nested(const nq_oracle_weights *W, int use_resid,
                                const uint16_t *xm, int row)
{
    int ng = W->k / W->group;
    double acc = 0.0;
    for (int grp = 0; grp < ng; grp++) {
        double part = 0.0;
        for (int i = 0; i < W->group; i++) {
            size_t idx = (size_t)row * W->k + (size_t)grp * W->group + i;
            int code = orc_get_code(W->base, idx);
            if (use_resid) code = 16 * code + orc_get_code(W->resid, idx);
            part += (double)code * (double)orc_bf16_to_f32(xm[grp * W->group + i]);
        }
        double s = (double)orc_f16_to_f32(((const uint16_t *)W->scales)[(size_t)row * ng + grp]);
        acc += (use_resid ? s / 16.0 : s) * part;
    }
    return acc;
}

static double linear_row_fp8(const nq_oracle_weights *W, const uint16_t *xm, int row)
{
    double acc = 0.0;
    for (int i = 0; i < W->k; i++)
        acc += (double)orc_e4m3_to_f32(W->base[(size_t)row * W->k + i]) * (double)orc_bf16_to_f32(xm[i]);
    return (double)((const float *)W->scales)[row] * acc;
}

static double linear_row_fp16(const nq_oracle_weights *W, const uint16_t *xm, int row)
{
    const uint16_t *w16 = (const uint16_t *)W->base;
    double acc = 0.0;
    for (int i = 0; i < W->k; i++)
        acc += (double)orc_f16_to_f32(w16[(size_t)row * W->k + i]) * (double)orc_bf16_to_f32(xm[i]);
    return acc;
}

/*
 * y[m][j] for the listed output rows (rows == NULL: all n rows, j == row).
 * `use_resid` selects the verify pass (both planes) for ORC_FMT_NESTED44.
 */
int orc_linear(const nq_oracle_weights *W, int use_resid, const uint16_t *x, int M,
               const int32_t *rows, int nrows, double *y)
{
    if (!rows) nrows = W->n;
    for (int m = 0; m < M; m++) {
        const uint16_t *xm = x + (size_t)m * W->k;
        for (int j = 0; j < nrows; j++) {
            int row = rows ? rows[j] : j;
            if (row < 0 || row >= W->n) return -1;
            double v;
            switch (W->format) {
            case ORC_FMT_NESTED44: v = linear_row_nested(W, use_resid, xm, row); break;
            case ORC_FMT_INT4:     if (use_resid) return -1; v = linear_row_nested(W, 0, xm, row); break;
            case ORC_FMT_FP8:      v = linear_row_fp8(W, xm, row); break;
            case ORC_FMT_FP16:     v = linear_row_fp16(W, xm, row); break;
            default: return -1;
            }
            y[(size_t)m * nrows + j] = v;
        }
    }
    return 0;
}

/* ======================================================================== */
/* W4A8 -> W8A8: int8 activations [BitNest Table 1 "W4A8 -> W8A8", Table 12]. */
/* ======================================================================== */

/* Per activation row: s_x = fp32(absmax / 127) (IEEE division), codes
 * x_q = clamp(rint(x / s_x), -127, 127); a zero row gives s_x = 0, codes 0. */
int orc_quantize_act_int8(const uint16_t *x, int M, int K, int8_t *xq, float *sx)
{
    for (int m = 0; m < M; m++) {
        float amax = 0.0f;
        for (int i = 0; i < K; i++) {
            float v = fabsf(orc_bf16_to_f32(x[(size_t)m * K + i]));
            if (!(v <= 3.0e38f)) return -1;
            if (v > amax) amax = v;
        }
        float s = amax / 127.0f;
        sx[m] = s;
        for (int i = 0; i < K; i++) {
            int q = 0;
            if (s > 0.0f) {
                float r = rintf(orc_bf16_to_f32(x[(size_t)m * K + i]) / s);
                q = r < -127.0f ? -127 : (r > 127.0f ? 127 : (int)r);
            }
            xq[(size_t)m * K + i] = (int8_t)q;
        }
    }
    return 0;
}

/* y[m][n] = s_x[m] * sum_g S_g * sum_{k in g} code[n][k] * x_q[m][k] with
 * code = q4 and S = s (draft), or code = 16 q4 + r and S = s / 16 (verify);
 * the group dot products are exact integers, the scaling fp64. */
int orc_linear_a8(const nq_oracle_weights *W, int use_resid, const int8_t *xq, const float *sx, int M, double *y)
{
    if (W->format != ORC_FMT_NESTED44 && W->format != ORC_FMT_INT4) return -1;
    if (use_resid && W->format != ORC_FMT_NESTED44) return -1;
    int ng = W->k / W->group;
    for (int m = 0; m < M; m++)
        for (int row = 0; row < W->n; row++) {
            double acc = 0.0;
            for (int grp = 0; grp < ng; grp++) {
                long long dot = 0;
                for (int i = 0; i < W->group; i++) {
                    size_t idx = (size_t)row * W->k + (size_t)grp * W->group + i;
                    int code = orc_get_code(W->base, idx);
                    if (use_resid) code = 16 * code + orc_get_code(W->resid, idx);
                    dot += (long long)code * xq[(size_t)m * W->k + (size_t)grp * W->group + i];
                }
                double sc = (double)orc_f16_to_f32(((const uint16_t *)W->scales)[(size_t)row * ng + grp]);
                acc += (use_resid ? sc / 16.0 : sc) * (double)dot;
            }
            y[(size_t)m * W->n + row] = (double)sx[m] * acc;
        }
    return 0;
}

/* ======================================================================== */
/* C3: greedy acceptance  [Erge, "Drafting and checking tokens", Table 1;    */
/*     SpecQuant III.D.4; R4]                                                */
/* ======================================================================== */

/* Index of the largest value, lowest index on ties; -1 if any value is not finite. */
static int argmax_lowest(const float *v, int V)
{
    int best = 0;
    for (int x = 0; x < V; x++) {
        if (!isfinite(v[x])) return -1;
        if (v[x] > v[best]) best = x;
    }
    return best;
}

/*
 * For each row b: t_j = argmax of the target logits at position j (j = 0..k);
 * keep the draft tokens while they equal the target's choice; at the first
 * mismatch n the target's choice t_n replaces the draft token and the rest is
 * discarded; if all k match, the target's choice t_k after the last draft
 * token is added.  Emits n + 1 tokens (1..k+1), pads -1.
 */
int orc_accept_greedy(const int32_t *draft, const float *tgt_logits, int B, int k, int V,
                      int32_t *out_tok, int32_t *out_cnt)
{
    for (int b = 0; b < B; b++) {
        int t[64];
        if (k + 1 > 64) return -1;
        for (int j = 0; j <= k; j++) {
            t[j] = argmax_lowest(tgt_logits + ((size_t)b * (k + 1) + j) * V, V);
            if (t[j] < 0) return -1;
        }
        int n = k;
        for (int j = 0; j < k; j++)
            if (draft[b * k + j] != t[j]) { n = j; break; }
        for (int j = 0; j <= k; j++)
            out_tok[b * (k + 1) + j] = j < n ? draft[b * k + j] : (j == n ? t[n] : -1);
        out_cnt[b] = n + 1;
    }
    return 0;
}

/* ======================================================================== */
/* Round bookkeeping [Erge, "Drafting and checking tokens"; BitNest Fig. 4]. */
/* ======================================================================== */

/* The draft model's greedy choice of each of M rows (lowest index on ties). */
int orc_draft_argmax(const float *logits, int M, int V, int32_t *tok)
{
    for (int m = 0; m < M; m++) {
        tok[m] = argmax_lowest(logits + (size_t)m * V, V);
        if (tok[m] < 0) return -1;
    }
    return 0;
}

/* Append each row's emitted tokens (the first out_cnt[b] of out_tok[b]) to
 * its sequence, up to max_len; the last emitted token is the next round's
 * first input.  Returns 1 if some sequence ran out of room, -1 on a count
 * outside 1..k+1 (that row is left unchanged), else 0. */
int orc_round_commit(const int32_t *out_tok, const int32_t *out_cnt, int B, int k, int32_t *seq,
                     int32_t *seq_len, int max_len, int32_t *x0)
{
    int rc = 0;
    for (int b = 0; b < B; b++) {
        int c = out_cnt[b];
        if (c < 1 || c > k + 1) { rc = -1; continue; }
        for (int i = 0; i < c; i++) {
            if (seq_len[b] >= max_len) { if (rc == 0) rc = 1; break; }
            seq[(size_t)b * max_len + seq_len[b]] = out_tok[(size_t)b * (k + 1) + i];
            seq_len[b] += 1;
        }
        x0[b] = out_tok[(size_t)b * (k + 1) + c - 1];
    }
    return rc;
}

/* ======================================================================== */
/* C4: sampled acceptance (Leviathan et al.; Chen et al.)  [Erge, "The same  */
/*     output as the large model alone"]; canonical fp32 arithmetic (R5).    */
/* ======================================================================== */

/* Philox4x32-10 [Philox]: ten rounds of two 32x32->64 multiplies with the
 * round key bumped by the Weyl constants between rounds. */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; round++) {
        uint64_t p0 = (uint64_t)M0 * c0, p1 = (uint64_t)M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += W0; k1 += W1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The uniform for (row seed, position j, purpose, round): key = seed halves,
 * counter = (j, purpose, round_lo, round_hi), word 0, top 24 bits * 2^-24. */
float orc_uniform(uint64_t seed, uint32_t j, uint32_t purpose, uint64_t round)
{
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {j, purpose, (uint32_t)round, (uint32_t)(round >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return (float)(out[0] >> 8) * ldexpf(1.0f, -24);
}

/*
 * R5 -- canonical arithmetic.  Softmax probabilities decide integers (accept
 * or not, which token), so both the oracle and the GPU take those decisions
 * on the same fp32 values, computed by this fixed recipe:
 *
 *   c      = fp32(log2(e)) / T                       (IEEE division)
 *   leaf   = 16 consecutive vocabulary entries in index order: leaf i holds
 *            entries 16 i .. 16 i + 15; entries >= V are absent
 *   lsum   = the sum of the 16 values w_0..w_15 of a leaf as two serial
 *            chains, E = (..((w_0 + w_2) + w_4) ..) + w_14 and
 *            O = (..((w_1 + w_3) + w_5) ..) + w_15, then E + O; absent
 *            entries count as 0
 *   segment = 1024 consecutive entries (64 leaves): segment s holds entries
 *            1024 s .. 1024 s + 1023; mx = its maximum raw logit
 *   mz     = RN(mx * c);  t(x) = fma(l(x), c, -mz of x's segment)  (<= ~0)
 *   e2(t)  = 0 if t < -125, else P(f) * 2^n with n = rint(t), f = t - n and
 *            P the degree-6 Taylor polynomial of 2^f (coefficients
 *            RN(ln2^i / i!)), evaluated by Horner with fma
 *   segment s = pairwise sum tree over its 64 leaves' lsum of e2(t(x))
 *   merge  (m1,s1),(m2,s2): the larger m survives; s = fma(s_small,
 *            e2(m_small - m_large), s_large); a (-inf, 0) pad is the identity
 *   valid  = every logit finite and every segment's mz finite (a logit whose
 *            scaled value underflows gets probability 0)
 *   tree   = segments padded to a power of two with (-inf, 0), merged
 *            pairwise, left operand first, level by level -> (M, S)
 *   p(x)   = RN(e2(t(x)) * F_seg), F_seg = RN(e2(mz_seg - M) * RN(1/S))
 *   accept position j  <=>  u_j < RN(p_j(d_j) / q_j(d_j))
 *   residual r(x) = max(0, RN(p(x) - q(x))); sampling from a non-negative w:
 *            leaf sums lsum, pairwise power-of-two tree (pads 0), root R,
 *            t = RN(u R), descend (left if t < L or the right sum is 0, else
 *            t -= L and go right), then scan the leaf for the first x whose
 *            running sum exceeds t (fallback: last x of the leaf with w > 0).
 *            R == 0 for the residual -> sample from p_j instead.
 *   sampling from p (the bonus draw, and the residual's fallback): the first
 *            level picks a segment by the pairwise tree over the segment
 *            weights W = RN(s_seg * F_seg) (the (max, sum) pass's own
 *            segment sums rescaled to p; pads 0), t = RN(u R_W); the second
 *            level descends the chosen segment's pairwise tree over its 64
 *            leaf sums of p with the remaining t and scans the leaf as above.
 *   uniforms: purpose 0 = accept test at j, 1 = resample at j, 2 = bonus at k.
 */
static const float ORC_LOG2E = 1.44269504088896340736f;

/* RN(ln2^i / i!) for i = 0..6: the Taylor series of 2^f = e^(f ln 2). */
static float exp2_coef[7];
static int exp2_coef_ready = 0;

static void init_exp2_coef(void)
{
    if (exp2_coef_ready) return;
    double ln2 = 0.69314718055994530941723212145818, term = 1.0;
    for (int i = 0; i <= 6; i++) {
        exp2_coef[i] = (float)term;              /* round the exact-enough double once */
        term = term * ln2 / (double)(i + 1);
    }
    exp2_coef_ready = 1;
}

float orc_exp2_coef(int i) { init_exp2_coef(); return (i >= 0 && i <= 6) ? exp2_coef[i] : 0.0f; }

float orc_exp2c(float t)
{
    init_exp2_coef();
    if (t < -125.0f) return 0.0f;
    float n = rintf(t);
    float f = t - n;
    float p = exp2_coef[6];
    for (int i = 5; i >= 0; i--) p = fmaf(p, f, exp2_coef[i]);
    return ldexpf(p, (int)n);
}

float orc_temper_coef(float T) { return ORC_LOG2E / T; }

typedef struct { float m, s; } ms_t;

static ms_t ms_merge(ms_t a, ms_t b)
{
    if (b.m == -INFINITY) return a;
    if (a.m == -INFINITY) return b;
    ms_t r;
    if (a.m >= b.m) { r.m = a.m; r.s = fmaf(b.s, orc_exp2c(b.m - a.m), a.s); }
    else            { r.m = b.m; r.s = fmaf(a.s, orc_exp2c(a.m - b.m), b.s); }
    return r;
}

/* Number of 16-entry leaves and the entry held at position e (0..15) of
 * leaf i; -1 if that entry lies at or beyond V. */
static int n_leaves(int V) { return (V + ORC_LEAF - 1) / ORC_LEAF; }
static int leaf_entry(int V, int i, int e)
{
    int x = ORC_LEAF * i + e;
    return x < V ? x : -1;
}

/* lsum of R5: two serial chains over the even and the odd entries, then E + O. */
static float leaf_sum(const float w[ORC_LEAF])
{
    float E = w[0], O = w[1];
    for (int e = 2; e < ORC_LEAF; e += 2) { E = E + w[e]; O = O + w[e + 1]; }
    return E + O;
}
static int pow2_at_least(int n) { int p = 1; while (p < n) p *= 2; return p; }

/* Number of 1024-entry segments of a vector. */
static int n_segments(int V) { return (V + ORC_SEG - 1) / ORC_SEG; }

/* Plain pairwise sum of n (a power of two) values, left operand first. */
static float pairwise_sum(float *v, int n)
{
    for (int width = n; width > 1; width /= 2)
        for (int i = 0; i < width / 2; i++) v[i] = v[2 * i] + v[2 * i + 1];
    return v[0];
}

/* Per-segment (mz, s) for one logits vector; returns the number of segments.
 * Every segment holds at least one present entry. */
static int seg_stats(const float *l, int V, float c, ms_t *seg)
{
    const int NS = n_segments(V), LPS = ORC_SEG / ORC_LEAF;
    for (int sg = 0; sg < NS; sg++) {
        float mx = -INFINITY;
        int any = 0;
        for (int x = ORC_SEG * sg; x < ORC_SEG * (sg + 1) && x < V; x++)
            if (!any || l[x] > mx) { mx = l[x]; any = 1; }
        float mz = mx * c, ls[ORC_SEG / ORC_LEAF];
        for (int i = 0; i < LPS; i++) {
            float w[ORC_LEAF];
            for (int e = 0; e < ORC_LEAF; e++) {
                int x = leaf_entry(V, LPS * sg + i, e);
                w[e] = x >= 0 ? orc_exp2c(fmaf(l[x], c, -mz)) : 0.0f;
            }
            ls[i] = leaf_sum(w);
        }
        seg[sg].m = mz;
        seg[sg].s = pairwise_sum(ls, LPS);
    }
    return NS;
}

/* Root (M, S) of the power-of-two (max, sum) tree over the segments. */
static ms_t ms_tree(const ms_t *leaf, int L)
{
    int P = pow2_at_least(L);
    ms_t *node = malloc(sizeof(ms_t) * P);
    for (int i = 0; i < P; i++) {
        if (i < L) node[i] = leaf[i];
        else { node[i].m = -INFINITY; node[i].s = 0.0f; }
    }
    for (int width = P; width > 1; width /= 2)
        for (int i = 0; i < width / 2; i++) node[i] = ms_merge(node[2 * i], node[2 * i + 1]);
    ms_t root = node[0];
    free(node);
    return root;
}

/* Canonical probabilities p(x) of one logits vector at temperature T. */
int orc_softmax_canonical(const float *l, int V, float T, float *p)
{
    float c = orc_temper_coef(T);
    for (int x = 0; x < V; x++) if (!isfinite(l[x])) return -1;
    ms_t *seg = malloc(sizeof(ms_t) * n_segments(V));
    int NS = seg_stats(l, V, c, seg);
    for (int i = 0; i < NS; i++)
        if (!isfinite(seg[i].m)) { free(seg); return -1; }
    ms_t root = ms_tree(seg, NS);
    float inv_s = 1.0f / root.s;
    for (int i = 0; i < NS; i++) {
        float F = orc_exp2c(seg[i].m - root.m) * inv_s;
        for (int x = ORC_SEG * i; x < ORC_SEG * (i + 1) && x < V; x++)
            p[x] = orc_exp2c(fmaf(l[x], c, -seg[i].m)) * F;
    }
    free(seg);
    return 0;
}

/* The intermediate values of the recipe for one logits vector (for tests):
 * per segment (mz, s), and the root (M, S).  Returns the number of segments,
 * or -1 if the vector is not valid. */
int orc_softmax_stats(const float *l, int V, float T, float *seg_mz, float *seg_s, float *M, float *S)
{
    float c = orc_temper_coef(T);
    for (int x = 0; x < V; x++) if (!isfinite(l[x])) return -1;
    ms_t *seg = malloc(sizeof(ms_t) * n_segments(V));
    int NS = seg_stats(l, V, c, seg);
    for (int i = 0; i < NS; i++) { seg_mz[i] = seg[i].m; seg_s[i] = seg[i].s; }
    ms_t root = ms_tree(seg, NS);
    *M = root.m;
    *S = root.s;
    free(seg);
    return NS;
}

/* Draw an index from the non-negative weights w (not necessarily normalised)
 * with uniform u, by the power-of-two sum-tree descent of R5.
 * Returns -1 if the total is not positive. */
int orc_tree_sample(const float *w, int V, float u)
{
    int L = n_leaves(V), P = pow2_at_least(L), levels = 0;
    while ((1 << levels) < P) levels++;
    /* level[0] = leaf sums (P entries), level[l] has P >> l entries */
    float **level = malloc(sizeof(float *) * (levels + 1));
    for (int l = 0; l <= levels; l++) level[l] = calloc((size_t)(P >> l), sizeof(float));
    for (int i = 0; i < L; i++) {
        float wl[ORC_LEAF];
        for (int e = 0; e < ORC_LEAF; e++) {
            int x = leaf_entry(V, i, e);
            wl[e] = x >= 0 ? w[x] : 0.0f;
        }
        level[0][i] = leaf_sum(wl);
    }
    for (int l = 1; l <= levels; l++)
        for (int i = 0; i < (P >> l); i++) level[l][i] = level[l - 1][2 * i] + level[l - 1][2 * i + 1];
    float R = level[levels][0];
    int result = -1;
    if (R > 0.0f) {
        float t = u * R;
        int node = 0;
        for (int l = levels; l >= 1; l--) {
            float left = level[l - 1][2 * node], right = level[l - 1][2 * node + 1];
            if (t < left || !(right > 0.0f)) node = 2 * node;
            else { t = t - left; node = 2 * node + 1; }
        }
        float run = 0.0f;
        for (int e = 0; e < ORC_LEAF && result < 0; e++) {
            int x = leaf_entry(V, node, e);
            if (x < 0) continue;
            run = run + w[x];
            if (t < run) result = x;
        }
        for (int e = ORC_LEAF - 1; e >= 0 && result < 0; e--) {
            int x = leaf_entry(V, node, e);
            if (x >= 0 && w[x] > 0.0f) result = x;
        }
    }
    for (int l = 0; l <= levels; l++) free(level[l]);
    free(level);
    return result;
}

/* Descend a pairwise sum tree level by level: node i of level l is
 * level[l][i]; at each level go left if t < left or the right sum is not
 * positive, else t -= left.  Returns the leaf index; *t is updated. */
static int tree_descend(float **level, int levels, float *t)
{
    int node = 0;
    for (int l = levels; l >= 1; l--) {
        float left = level[l - 1][2 * node], right = level[l - 1][2 * node + 1];
        if (*t < left || !(right > 0.0f)) node = 2 * node;
        else { *t = *t - left; node = 2 * node + 1; }
    }
    return node;
}

/* Pairwise tree levels over n values (padded with zeros to a power of two). */
static int tree_build(const float *v, int n, float ***out)
{
    int P = pow2_at_least(n), levels = 0;
    while ((1 << levels) < P) levels++;
    float **level = malloc(sizeof(float *) * (levels + 1));
    for (int l = 0; l <= levels; l++) level[l] = calloc((size_t)(P >> l), sizeof(float));
    for (int i = 0; i < n; i++) level[0][i] = v[i];
    for (int l = 1; l <= levels; l++)
        for (int i = 0; i < (P >> l); i++) level[l][i] = level[l - 1][2 * i] + level[l - 1][2 * i + 1];
    *out = level;
    return levels;
}
static void tree_free(float **level, int levels)
{
    for (int l = 0; l <= levels; l++) free(level[l]);
    free(level);
}

/* Draw from p of one logits vector with uniform u by the two-level rule of
 * R5 (segment weights from the (max, sum) pass, then the chosen segment's
 * leaf tree).  Returns -1 if the vector is not valid. */
int orc_sample_p(const float *l, int V, float T, float u)
{
    float c = orc_temper_coef(T);
    for (int x = 0; x < V; x++) if (!isfinite(l[x])) return -1;
    int NS = n_segments(V), LPS = ORC_SEG / ORC_LEAF;
    ms_t *seg = malloc(sizeof(ms_t) * NS);
    seg_stats(l, V, c, seg);
    for (int i = 0; i < NS; i++) if (!isfinite(seg[i].m)) { free(seg); return -1; }
    ms_t root = ms_tree(seg, NS);
    float inv_s = 1.0f / root.s;
    float *W = malloc(sizeof(float) * NS), *F = malloc(sizeof(float) * NS);
    for (int i = 0; i < NS; i++) {
        F[i] = orc_exp2c(seg[i].m - root.m) * inv_s;
        W[i] = seg[i].s * F[i];
    }
    float **lv;
    int levels = tree_build(W, NS, &lv);
    float t = u * lv[levels][0];
    int sg = tree_descend(lv, levels, &t);
    tree_free(lv, levels);
    /* the chosen segment: p(x), leaf sums, leaf tree, scan */
    float pw[ORC_SEG], ls[ORC_SEG / ORC_LEAF];
    for (int e = 0; e < ORC_SEG; e++) {
        int x = ORC_SEG * sg + e;
        pw[e] = x < V ? orc_exp2c(fmaf(l[x], c, -seg[sg].m)) * F[sg] : 0.0f;
    }
    for (int i = 0; i < LPS; i++) ls[i] = leaf_sum(pw + ORC_LEAF * i);
    levels = tree_build(ls, LPS, &lv);
    int leaf = tree_descend(lv, levels, &t);
    tree_free(lv, levels);
    int result = -1;
    float run = 0.0f;
    for (int e = 0; e < ORC_LEAF && result < 0; e++) {
        int x = ORC_SEG * sg + ORC_LEAF * leaf + e;
        if (x >= V) continue;
        run = run + pw[ORC_LEAF * leaf + e];
        if (t < run) result = x;
    }
    for (int e = ORC_LEAF - 1; e >= 0 && result < 0; e--) {
        int x = ORC_SEG * sg + ORC_LEAF * leaf + e;
        if (x < V && pw[ORC_LEAF * leaf + e] > 0.0f) result = x;
    }
    free(seg); free(W); free(F);
    return result;
}

/*
 * Speculative sampling for B rows: draft tokens d_0..d_{k-1} drawn from q,
 * draft logits [B][k][V], target logits [B][k+1][V].  For j = 0..k-1 accept
 * d_j when u_j < p_j(d_j) / q_j(d_j); at the first rejection draw the
 * replacement from normalise(max(0, p_j - q_j)) and stop; if all k are
 * accepted draw one more token from p_k.  Emits 1..k+1 tokens, pads -1.
 * `accepted` (may be NULL) receives the number of accepted draft tokens.
 */
int orc_accept_sample(const int32_t *draft, const float *draft_logits, const float *tgt_logits,
                      int B, int k, int V, float T, const uint64_t *seeds, uint64_t round,
                      int32_t *out_tok, int32_t *out_cnt)
{
    if (!(T > 0.0f) || k < 1 || V < 1) return -1;
    float *p = malloc(sizeof(float) * V), *q = malloc(sizeof(float) * V), *r = malloc(sizeof(float) * V);
    int rc = 0;
    for (int b = 0; b < B && rc == 0; b++) {
        int n = k, tok = -1;
        for (int j = 0; j < k; j++) {
            int d = draft[b * k + j];
            if (d < 0 || d >= V) { rc = -1; break; }
            if (orc_softmax_canonical(tgt_logits + ((size_t)b * (k + 1) + j) * V, V, T, p) ||
                orc_softmax_canonical(draft_logits + ((size_t)b * k + j) * V, V, T, q)) { rc = -1; break; }
            float ratio = p[d] / q[d];
            float u = orc_uniform(seeds[b], (uint32_t)j, 0, round);
            if (u < ratio) continue;                     /* accepted */
            for (int x = 0; x < V; x++) { float dlt = p[x] - q[x]; r[x] = dlt > 0.0f ? dlt : 0.0f; }
            float u1 = orc_uniform(seeds[b], (uint32_t)j, 1, round);
            tok = orc_tree_sample(r, V, u1);
            if (tok < 0) tok = orc_sample_p(tgt_logits + ((size_t)b * (k + 1) + j) * V, V, T, u1);
            n = j;
            break;
        }
        if (rc) break;
        if (n == k) {
            tok = orc_sample_p(tgt_logits + ((size_t)b * (k + 1) + k) * V, V, T,
                               orc_uniform(seeds[b], (uint32_t)k, 2, round));
            if (tok < 0) { rc = -1; break; }
        }
        for (int j = 0; j <= k; j++)
            out_tok[b * (k + 1) + j] = j < n ? draft[b * k + j] : (j == n ? tok : -1);
        out_cnt[b] = n + 1;
    }
    free(p); free(q); free(r);
    return rc;
}

/*
 * The same round in plain fp64 (libm exp, serial sums, the textbook inverse
 * CDF over the vocabulary in index order), for checking the canonical fp32
 * recipe against textbook arithmetic: the recipe's sum tree over index-order
 * leaves, descended by u * R, is that inverse CDF up to rounding.  Also
 * reports per row the smallest distance between a uniform and the boundary
 * it was compared with (|u - ratio| and, for the drawn token, the distance
 * of u*R to the nearest cumulative boundary) so that callers can separate
 * genuine disagreements from near-ties.
 */
static void softmax_f64(const float *l, int V, double T, double *p)
{
    double mx = -INFINITY, s = 0.0;
    for (int x = 0; x < V; x++) if ((double)l[x] / T > mx) mx = (double)l[x] / T;
    for (int x = 0; x < V; x++) { p[x] = exp((double)l[x] / T - mx); s += p[x]; }
    for (int x = 0; x < V; x++) p[x] /= s;
}

/* Textbook inverse CDF in fp64 over the vocabulary in index order: the first
 * x whose cumulative weight exceeds u * total (the last x with positive
 * weight if rounding leaves none).  *margin receives the distance of u * total
 * to the nearer boundary of the chosen entry, relative to the total. */
static int cdf_sample_f64(const double *w, int V, double u, double *margin)
{
    double tot = 0.0;
    for (int x = 0; x < V; x++) tot += w[x];
    if (!(tot > 0.0)) return -1;
    double t = u * tot, run = 0.0;
    int pick = -1, last = -1;
    for (int x = 0; x < V; x++) {
        double prev = run;
        run += w[x];
        if (w[x] > 0.0) last = x;
        if (w[x] > 0.0 && pick < 0 && t < run) {
            pick = x;
            double d0 = (t - prev) / tot, d1 = (run - t) / tot;
            *margin = d0 < d1 ? d0 : d1;
        }
    }
    if (pick < 0) { pick = last; *margin = 0.0; }
    return pick;
}

int orc_accept_sample_f64(const int32_t *draft, const float *draft_logits, const float *tgt_logits,
                          int B, int k, int V, float T, const uint64_t *seeds, uint64_t round,
                          int32_t *out_tok, int32_t *out_cnt, double *margin)
{
    double *p = malloc(sizeof(double) * V), *q = malloc(sizeof(double) * V), *r = malloc(sizeof(double) * V);
    for (int b = 0; b < B; b++) {
        int n = k, tok = -1;
        double mrg = INFINITY, sm = INFINITY;
        for (int j = 0; j < k; j++) {
            int d = draft[b * k + j];
            softmax_f64(tgt_logits + ((size_t)b * (k + 1) + j) * V, V, T, p);
            softmax_f64(draft_logits + ((size_t)b * k + j) * V, V, T, q);
            double ratio = p[d] / q[d];
            double u = (double)orc_uniform(seeds[b], (uint32_t)j, 0, round);
            if (fabs(u - ratio) < mrg) mrg = fabs(u - ratio);
            if (u < ratio) continue;
            double tot = 0.0;
            for (int x = 0; x < V; x++) { r[x] = p[x] > q[x] ? p[x] - q[x] : 0.0; tot += r[x]; }
            double u1 = (double)orc_uniform(seeds[b], (uint32_t)j, 1, round);
            tok = tot > 0.0 ? cdf_sample_f64(r, V, u1, &sm) : cdf_sample_f64(p, V, u1, &sm);
            n = j;
            break;
        }
        if (n == k) {
            softmax_f64(tgt_logits + ((size_t)b * (k + 1) + k) * V, V, T, p);
            tok = cdf_sample_f64(p, V, (double)orc_uniform(seeds[b], (uint32_t)k, 2, round), &sm);
        }
        for (int j = 0; j <= k; j++)
            out_tok[b * (k + 1) + j] = j < n ? draft[b * k + j] : (j == n ? tok : -1);
        out_cnt[b] = n + 1;
        if (margin) margin[b] = mrg < sm ? mrg : sm;
    }
    free(p); free(q); free(r);
    return 0;
}

/* ======================================================================== */
/* Nested KV cache attention [BitNest Fig. 4: the draft reads the low-bit    */
/* base view, verification the full view of the same cache].                */
/* ======================================================================== */

/* Element j of cache row `row` (head_dim d, group G): draft s q4, target
 * (s/16)(16 q4 + r), in fp64 (exact). */
static double kv_value(const uint8_t *base, const uint8_t *resid, const uint16_t *sc, size_t row, int d, int G,
                       int j, int planes)
{
    uint8_t bb = base[row * (d / 2) + j / 2];
    int q4 = (j & 1) ? (bb >> 4) : (bb & 15);
    if (q4 > 7) q4 -= 16;
    double s = (double)orc_f16_to_f32(sc[row * (d / G) + j / G]);
    if (planes == 1) return s * q4;
    uint8_t rb = resid[row * (d / 2) + j / 2];
    int r = (j & 1) ? (rb >> 4) : (rb & 15);
    if (r > 7) r -= 16;
    return s / 16.0 * (16 * q4 + r);
}

/* out[b][m][h] = softmax_t(scale q . K_t) V_t over t = 0 .. len[b] - M + m,
 * kv head h / (Hq / Hkv); plain fp64. */
int orc_attn_decode(const float *q, int B, int M, int Hq, int Hkv, int d, int G, int L,
                    const uint8_t *kb, const uint8_t *kr, const uint16_t *ks,
                    const uint8_t *vb, const uint8_t *vr, const uint16_t *vs,
                    const int32_t *len, int planes, float scale, float *out)
{
    if (Hq % Hkv != 0 || (planes != 1 && planes != 2)) return -1;
    int g = Hq / Hkv;
    double *w = malloc(sizeof(double) * (L > 0 ? L : 1));
    for (int b = 0; b < B; b++)
        for (int m = 0; m < M; m++)
            for (int h = 0; h < Hq; h++) {
                int kvh = h / g, lim = len[b] - (M - 1 - m);
                if (lim > L) lim = L;
                const float *qv = q + (((size_t)b * M + m) * Hq + h) * d;
                float *o = out + (((size_t)b * M + m) * Hq + h) * d;
                double mx = -INFINITY;
                for (int t = 0; t < lim; t++) {
                    size_t row = ((size_t)b * Hkv + kvh) * L + t;
                    double sc = 0.0;
                    for (int j = 0; j < d; j++) sc += (double)qv[j] * kv_value(kb, kr, ks, row, d, G, j, planes);
                    w[t] = sc * scale;
                    if (w[t] > mx) mx = w[t];
                }
                double den = 0.0;
                for (int t = 0; t < lim; t++) { w[t] = exp(w[t] - mx); den += w[t]; }
                for (int j = 0; j < d; j++) {
                    double acc = 0.0;
                    for (int t = 0; t < lim; t++) {
                        size_t row = ((size_t)b * Hkv + kvh) * L + t;
                        acc += w[t] * kv_value(vb, vr, vs, row, d, G, j, planes);
                    }
                    o[j] = lim > 0 ? (float)(acc / den) : 0.0f;
                }
            }
    free(w);
    return 0;
}

/* ======================================================================== */
/* Draft features [SpecKV, "How it works": mean and maximum draft entropy,    */
/* mean and minimum draft confidence over a step's drafted positions].       */
/* ======================================================================== */

/* Per row b: H_j = entropy (nats) of q_j = softmax(draft_logits[b][j] / T)
 * and c_j = q_j(draft[b][j]) (the drafted token's probability under the
 * draft) for j = 0..k-1; out[b] = (mean H, mean c, max H, min c).  Plain
 * fp64 with libm exp and log. */
int orc_draft_features(const int32_t *draft, const float *draft_logits, int B, int k, int V, float T, double *out)
{
    if (!(T > 0.0f) || k < 1 || V < 1) return -1;
    double *q = malloc(sizeof(double) * V);
    for (int b = 0; b < B; b++) {
        double sh = 0.0, sc = 0.0, mh = -INFINITY, mc = INFINITY;
        for (int j = 0; j < k; j++) {
            const float *l = draft_logits + ((size_t)b * k + j) * V;
            int d = draft[b * k + j];
            if (d < 0 || d >= V) { free(q); return -1; }
            double mx = -INFINITY, s = 0.0, h = 0.0;
            for (int x = 0; x < V; x++) {
                if (!isfinite(l[x])) { free(q); return -1; }
                if ((double)l[x] / T > mx) mx = (double)l[x] / T;
            }
            for (int x = 0; x < V; x++) { q[x] = exp((double)l[x] / T - mx); s += q[x]; }
            for (int x = 0; x < V; x++) {
                q[x] /= s;
                if (q[x] > 0.0) h -= q[x] * log(q[x]);
            }
            sh += h; sc += q[d];
            if (h > mh) mh = h;
            if (q[d] < mc) mc = q[d];
        }
        out[4 * b] = sh / k; out[4 * b + 1] = sc / k; out[4 * b + 2] = mh; out[4 * b + 3] = mc;
    }
    free(q);
    return 0;
}

/* ======================================================================== */
/* Array helpers so that callers need not loop per element.                 */
/* ======================================================================== */
void orc_exp2c_n(const float *t, float *out, int n) { for (int i = 0; i < n; i++) out[i] = orc_exp2c(t[i]); }
void orc_f32_to_f16_n(const float *f, uint16_t *out, int n) { for (int i = 0; i < n; i++) out[i] = orc_f32_to_f16(f[i]); }
void orc_f16_to_f32_n(const uint16_t *h, float *out, int n) { for (int i = 0; i < n; i++) out[i] = orc_f16_to_f32(h[i]); }
void orc_f32_to_e4m3_n(const float *f, uint8_t *out, int n) { for (int i = 0; i < n; i++) out[i] = orc_f32_to_e4m3(f[i]); }
void orc_e4m3_to_f32_n(const uint8_t *c, float *out, int n) { for (int i = 0; i < n; i++) out[i] = orc_e4m3_to_f32(c[i]); }
void orc_uniform_n(const uint64_t *seed, const uint32_t *j, const uint32_t *purpose, const uint64_t *round,
                   float *out, int n)
{
    for (int i = 0; i < n; i++) out[i] = orc_uniform(seed[i], j[i], purpose[i], round[i]);
}
