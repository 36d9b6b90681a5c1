/*
 * nq.h -- C ABI of libnq.so: the weight-streaming linears and the acceptance
 * step of quantized self-speculative decoding, as hand-written CUDA for
 * sm_103a (GB300).
 *
 * Method sources (page title; section / figure / table / equation):
 *   "BitNest: Bit-Nested Speculative Decoding for Memory-Efficient LLM
 *    Inference Acceleration" -- Fig. 2 (a b-bit base plus an r-bit
 *    refinement of the remaining error; drafting reads only the base,
 *    verification reads both planes to recover the (b+r)-bit target) and
 *    Fig. 3 (dual-plane storage: two independent 4-bit streams of N/2 bytes
 *    for N weights; the target recovers the full 8-bit representation).
 *   "SpecQuant -- Speculative Decoding with Multi-Parent Quantization for
 *    Adaptive LLM Inference" -- Sec. III.A (Q4 = f(W16,4) INT4, Q8 =
 *    f(W16,8) FP8, Q16 = W16, all from one FP16 base) and Sec. III.D.3-4
 *    (parent verification; token acceptance or correction).
 *   "How Speculative Decoding Speeds Up Inference" -- "Drafting and checking
 *    tokens" (draft k tokens, check all k positions in one target pass, keep
 *    the matching prefix, the target's token replaces the first mismatch,
 *    1..k+1 tokens per pass), Table 1 (k = 4 worked round), "The same output
 *    as the large model alone" (greedy equivalence; speculative sampling of
 *    Leviathan et al. / Chen et al.), Eq. (1).
 *
 * Conventions (all entry points):
 *   - Every pointer argument is caller-owned DEVICE memory unless stated
 *     otherwise; the library allocates nothing and keeps no per-call state.
 *   - Every call is asynchronous on `stream`; outputs are valid once the
 *     stream reaches the call.  Arguments are validated on the host before
 *     any launch; a rejected call launches nothing and returns a status.
 *   - Device pointers must be 16-byte aligned (NQ_ERR_ALIGN otherwise).
 *   - Data-dependent faults that only the device can see (non-finite logits,
 *     out-of-range draft ids) set bits in a sticky per-device status word,
 *     read (and cleared) with nq_get_device_status().
 *   - Activations are bfloat16, passed as their uint16_t bit patterns.
 *   - Results are deterministic: the same inputs give the same bits, and a
 *     linear's output row for one activation row does not depend on M or on
 *     the other rows of the batch (batch invariance).
 */
#ifndef NQ_H
#define NQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(NQ_BUILDING) && defined(__GNUC__)
#define NQ_API __attribute__((visibility("default")))
#else
#define NQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NQ_OK = 0,
    NQ_ERR_ARG = 1,        /* null pointer, unknown format, bad k / M / temperature */
    NQ_ERR_SHAPE = 2,      /* k_in % group, k_in % 64, group not in {64,128}, sizes too large */
    NQ_ERR_ALIGN = 3,      /* a device pointer is not 16-byte aligned */
    NQ_ERR_CUDA = 4,       /* a CUDA runtime call failed (launch error, bad device) */
    NQ_ERR_NONFINITE = 5,  /* reported by nq_get_device_status(): non-finite logits */
    NQ_ERR_TIMEOUT = 6,    /* reserved (a bounded device wait that gives up sets NQ_DEV_TIMEOUT) */
    NQ_ERR_WORKSPACE = 7,  /* workspace NULL or smaller than the *_workspace_bytes() size */
    NQ_ERR_TOKEN = 8       /* reported by nq_get_device_status(): draft id outside [0, V) */
} nq_status;

/* Bits of the sticky device status word. */
#define NQ_DEV_NONFINITE 0x1u
#define NQ_DEV_BAD_TOKEN 0x2u
#define NQ_DEV_TIMEOUT   0x4u
#define NQ_DEV_ACT_RANGE 0x8u   /* an activation exceeded the fp16 range (|x| > 65504) */
#define NQ_DEV_SEQ_FULL  0x10u  /* spec_round_commit: a sequence buffer was full, tokens dropped */

/*
 * Weight formats (SpecQuant Sec. III.A tiers; BitNest Fig. 3 planes).
 *   NESTED44    base = 4-bit codes [n_out][k_in/2], resid = 4-bit refinement
 *               codes [n_out][k_in/2], scales = fp16 [n_out][k_in/group].
 *               Two's-complement nibbles, element 2j in the low nibble of
 *               byte j.  Draft value s*q4; target value (s/16)*(16*q4 + r).
 *   INT4        base + scales exactly as NESTED44, no refinement plane.
 *   FP8E4M3_ROW base = E4M3FN codes [n_out][k_in], scales = fp32 [n_out]
 *               (value = scale[n] * e4m3), resid unused, group ignored.
 *   FP16        base = fp16 weights [n_out][k_in], resid/scales unused.
 * Valid pairs: draft (nq_draft_gemv*) takes NESTED44 (base plane only) and
 * INT4; verify (nq_verify_gemm*) takes NESTED44 (both planes), FP8E4M3_ROW
 * and FP16.  Any other pair returns NQ_ERR_ARG.
 */
typedef enum {
    NQ_FMT_NESTED44 = 0,
    NQ_FMT_INT4 = 1,
    NQ_FMT_FP8E4M3_ROW = 2,
    NQ_FMT_FP16 = 3
} nq_format;

/* One packed linear layer, W [n_out][k_in] (y = x W^T).  The struct itself is
 * host memory; the three buffers are device memory owned by the caller. */
typedef struct {
    int32_t n_out;
    int32_t k_in;     /* multiple of 64; for NESTED44/INT4 also of group */
    int32_t group;    /* 64 or 128 (NESTED44 / INT4); ignored otherwise */
    int32_t format;   /* nq_format */
    void *base;
    void *resid;
    void *scales;
} nq_weights;

/* Byte sizes of the three buffers of a packed layer (host-only; no CUDA).
 * Any output pointer may be NULL.  NQ_ERR_SHAPE / NQ_ERR_ARG on bad shapes. */
NQ_API nq_status nq_packed_bytes(int n_out, int k_in, int group, int format,
                          size_t *base_bytes, size_t *resid_bytes, size_t *scale_bytes);

/*
 * Quantise and pack fp32 weights w [n_out][k_in] (device, row-major) into the
 * caller-allocated buffers of `out` (sizes from nq_packed_bytes()).
 * NESTED44 / INT4 (BitNest Fig. 2): per (row, group of `group` inputs)
 * s = fp16(absmax/7); q4 = clamp(rint(w/s), -8, 7); r = clamp(rint(16 (w/s -
 * q4)), -8, 7); a group with s == 0 packs to zeros.  FP8E4M3_ROW: s_n =
 * absmax_row/448, code = E4M3FN(w/s_n), round to nearest even, saturating.
 * FP16: round to nearest even.  Weights must be finite (non-finite input
 * gives unspecified codes).  Offline step, not part of a decoding round.
 */
NQ_API nq_status nq_pack_weights(const float *w, const nq_weights *out, cudaStream_t stream);

/*
 * Draft pass linear (BitNest Fig. 2: drafting reads only the base plane):
 *   y[m][n] = sum_g s[n][g] * sum_{k in g} q4[n][k] * x[m][k]
 * x: bf16 bits [M][k_in]; y: fp32 [M][n_out]; 1 <= M <= 4096 (the kernel
 * streams the weights once per 16 activation rows).  Formats: NESTED44, INT4.
 * Arithmetic: the 4-bit codes are exact in fp16; activations are rounded
 * bf16 -> fp16 (exact for 2^-14 <= |x| <= 65504; |x| > 65504 sets
 * NQ_DEV_ACT_RANGE), products accumulate in fp32, the group scale is applied
 * once per group in fp32.
 */
NQ_API nq_status nq_draft_gemv(const nq_weights *w, const uint16_t *x, int M, float *y, cudaStream_t stream);

/*
 * Verify pass linear over the k+1 candidate positions (BitNest Fig. 2 and
 * Fig. 3: both planes rebuild the 8-bit target; SpecQuant Sec. III.D.3):
 *   NESTED44:    y[m][n] = sum_g (s[n][g]/16) sum_{k in g} (16 q4 + r)[n][k] x[m][k]
 *   FP8E4M3_ROW: y[m][n] = s[n] sum_k e4m3[n][k] x[m][k]
 *   FP16:        y[m][n] = sum_k w16[n][k] x[m][k]
 * Same layouts, limits and fp16/fp32 arithmetic as nq_draft_gemv (E4M3 and
 * fp16 weights are exact in fp16).
 */
NQ_API nq_status nq_verify_gemm(const nq_weights *w, const uint16_t *x, int M, float *y, cudaStream_t stream);

/*
 * Many independent linears in one persistent launch (e.g. every linear of a
 * model pass), all at the same M.  w, x and y are HOST arrays of `count`
 * entries (x[i], y[i] device pointers, layouts as for the single calls).
 * Equivalent to `count` single calls in order; bit-identical results.
 * All layers must share the format class of the call (draft or verify).
 */
NQ_API nq_status nq_draft_gemv_batch(int count, const nq_weights *w, const uint16_t *const *x, int M,
                              float *const *y, cudaStream_t stream);
NQ_API nq_status nq_verify_gemm_batch(int count, const nq_weights *w, const uint16_t *const *x, int M,
                               float *const *y, cudaStream_t stream);

/*
 * Batched speculative rounds (many sequences, M = B (k+1) of a few tens to
 * hundreds of rows) turn the same linears into dense contractions.  These two
 * calls take a device workspace and, when M >= 16 and every layer is NESTED44
 * (or INT4 for the draft) with k_in % 128 == 0, run the contraction on the
 * tensor cores with the decoded weights in tensor memory: one pre-pass writes
 * the activations as fp16 into the workspace, then each CTA decodes 128
 * weight rows to fp16(q8 * s/16) (verify) or fp16(q4 * s) (draft), each
 * weight rounded once to fp16, and accumulates in fp32 (activations rounded
 * bf16 -> fp16 as above).  Results agree with nq_*_batch to fp16 weight
 * rounding (well inside the 2e-3 normwise bound) but are not bit-identical
 * to them, and M >= 16 rows are not batch-invariant with respect to M < 16.
 * Other cases run exactly as nq_draft_gemv_batch / nq_verify_gemm_batch and
 * ignore ws.  M > 256 is processed in chunks of 256 rows.
 *
 * nq_linear_workspace_bytes() gives the workspace size in bytes (host-only;
 * 0 when the tensor-core path is not taken or the arguments are invalid).
 * The workspace is caller-owned device memory, 16-byte aligned, needs no
 * initialisation and must not be used by another call that may run at the
 * same time.  NQ_ERR_WORKSPACE if ws is NULL or smaller than that size.
 * A bounded internal wait that gives up sets NQ_DEV_TIMEOUT.
 */
NQ_API size_t nq_linear_workspace_bytes(int count, const nq_weights *w, int M, int verify);
NQ_API nq_status nq_draft_gemv_batch_ws(int count, const nq_weights *w, const uint16_t *const *x, int M,
                                 float *const *y, void *ws, size_t ws_bytes, cudaStream_t stream);
NQ_API nq_status nq_verify_gemm_batch_ws(int count, const nq_weights *w, const uint16_t *const *x, int M,
                                  float *const *y, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Device workspace for the acceptance calls, in bytes (host-only).  The
 * workspace must be zero-filled once before its first use; every call leaves
 * it ready for the next one.  Calls that share a workspace must not overlap
 * on the GPU (use one stream, or one workspace per stream).
 * Limits: 1 <= B <= 65535, 1 <= k <= 16, 1 <= V <= 524288; k = 0 gives the
 * workspace of spec_draft_argmax over B rows.  Returns 0 on bad sizes.
 */
NQ_API size_t spec_accept_workspace_bytes(int B, int k, int V);

/*
 * Greedy acceptance ("Drafting and checking tokens"; Table 1; "The same
 * output as the large model alone"):
 *   t_j = argmax_x tgt_logits[b][j][x] (lowest index on ties), j = 0..k;
 *   n   = first j < k with draft[b][j] != t_j, else k;
 *   out_tok[b] = draft[b][0..n-1], t_n, then -1 pads;  out_cnt[b] = n + 1.
 * draft: int32 [B][k]; tgt_logits: fp32 [B][k+1][V]; out_tok: int32 [B][k+1];
 * out_cnt: int32 [B].  Non-finite logits set NQ_DEV_NONFINITE and out-of-range
 * draft ids NQ_DEV_BAD_TOKEN (that row's output is then unspecified).
 */
NQ_API nq_status spec_accept_greedy(const int32_t *draft, const float *tgt_logits, int B, int k, int V,
                             int32_t *out_tok, int32_t *out_cnt, void *ws, size_t ws_bytes,
                             cudaStream_t stream);

/*
 * Speculative sampling (Leviathan et al.; Chen et al.; "The same output as
 * the large model alone"), p = softmax(tgt/T), q = softmax(draft_logits/T):
 *   for j = 0..k-1: accept draft[b][j] iff u_j < p_j(d_j) / q_j(d_j);
 *   at the first rejection j draw from normalise(max(0, p_j - q_j)) (from p_j
 *   if that is all zero) and stop; if all k are accepted draw a bonus token
 *   from p_k.  Emits 1..k+1 tokens: out_tok / out_cnt as for greedy.
 * draft_logits: fp32 [B][k][V]; tgt_logits: fp32 [B][k+1][V]; temperature > 0;
 * seeds: uint64 [B] (device); round: caller's round counter.  Uniforms come
 * from Philox4x32-10 with key = seeds[b], counter = (j, purpose, round) --
 * purpose 0 accept test, 1 resample, 2 bonus -- so a (seed, round) pair
 * replays exactly.  The fp32 arithmetic follows a fixed recipe so that every
 * decision is reproducible bit for bit: an own base-2 exponential; exponents
 * taken against the maximum of each 1024-entry segment of the vocabulary;
 * sums of 16-entry leaves as two serial chains (even and odd entries); a
 * pairwise tree over each segment's leaves and a pairwise (max, sum) tree
 * over the segments; sampling by descending the pairwise sum tree over the
 * leaves, all in vocabulary index order.
 */
NQ_API nq_status spec_accept_sample(const int32_t *draft, const float *draft_logits, const float *tgt_logits,
                             int B, int k, int V, float temperature, const uint64_t *seeds,
                             uint64_t round, int32_t *out_tok, int32_t *out_cnt, void *ws,
                             size_t ws_bytes, cudaStream_t stream);

/*
 * spec_accept_sample plus the draft features SpecKV feeds its acceptance-rate
 * predictor (SpecKV, "How it works": mean and maximum draft entropy, mean and
 * minimum draft confidence over a step's drafted positions), taken from the
 * same pass over the draft logits at no extra read:
 *   features[b] = (mean_j H(q_j), mean_j q_j(d_j), max_j H(q_j), min_j q_j(d_j)),
 * j = 0..k-1, H in nats of q_j = softmax(draft_logits[b][j] / T), q_j(d_j)
 * the drafted token's draft probability (its canonical fp32 value, the one the
 * acceptance test uses).  features: fp32 [B][4] device, 16-byte aligned.
 * Token outputs are bit-identical to spec_accept_sample's; the features are
 * floating-point values, accurate to about 1e-5 relative.
 */
NQ_API nq_status spec_accept_sample_features(const int32_t *draft, const float *draft_logits,
                                             const float *tgt_logits, int B, int k, int V, float temperature,
                                             const uint64_t *seeds, uint64_t round, int32_t *out_tok,
                                             int32_t *out_cnt, float *features, void *ws, size_t ws_bytes,
                                             cudaStream_t stream);

/*
 * Round bookkeeping ("Drafting and checking tokens": the draft proposes k
 * tokens one at a time, each from the previous one; the target checks the
 * k+1 positions in one pass; the kept prefix plus the target's token extend
 * the sequence and that last token starts the next round).  These four calls
 * keep a whole round on the device, so that it can be queued (or captured in
 * a CUDA graph) with no host round trip.  Token arrays are int32 and need
 * 4-byte alignment only; tables and activations 16-byte alignment.
 *
 * spec_draft_argmax: the draft model's greedy choice per row,
 *   tok[m * tok_stride] = argmax_x logits[m][x] (lowest index on ties).
 *   logits fp32 [M][V]; workspace spec_accept_workspace_bytes(M, 0, V),
 *   zero-filled once (calls leave it ready).  Non-finite logits set
 *   NQ_DEV_NONFINITE.  1 <= M <= 65535.
 */
NQ_API nq_status spec_draft_argmax(const float *logits, int M, int V, int32_t *tok, int tok_stride, void *ws,
                                   size_t ws_bytes, cudaStream_t stream);

/*
 * nq_embed_rows: input rows of a pass from token ids,
 *   out[m][:] = table[ids[m * ids_stride]][:],  m = 0..M-1.
 * nq_embed_round: the verify pass's k+1 input rows per sequence b, position 0
 *   the last committed token x0[b], positions 1..k the drafted tokens:
 *   out[b][j][:] = table[j == 0 ? x0[b] : draft[b][j-1]][:].
 * table: bf16 bits [V][d], d a multiple of 8; out: bf16 bits, rows of d.  An
 * id outside [0, V) writes a zero row and sets NQ_DEV_BAD_TOKEN.
 */
NQ_API nq_status nq_embed_rows(const uint16_t *table, int V, int d, const int32_t *ids, int ids_stride, int M,
                               uint16_t *out, cudaStream_t stream);
NQ_API nq_status nq_embed_round(const uint16_t *table, int V, int d, const int32_t *x0, const int32_t *draft,
                                int B, int k, uint16_t *out, cudaStream_t stream);

/*
 * spec_round_commit: after an acceptance call (out_tok [B][k+1], out_cnt [B]),
 *   seq[b][L .. L + c - 1] = out_tok[b][0 .. c - 1]   (c = out_cnt[b], L = seq_len[b])
 *   seq_len[b] = L + c;   x0[b] = out_tok[b][c - 1]   (the next round's first input).
 * seq: int32 [B][max_len]; seq_len, x0: int32 [B] (in/out).  Tokens beyond
 * max_len are dropped and set NQ_DEV_SEQ_FULL; a count outside 1..k+1 appends
 * nothing and sets NQ_DEV_BAD_TOKEN.  The verify pass computed KV entries for
 * its k+1 positions x0, d_0 .. d_{k-1}; the first c of them stay and the
 * rejected suffix (positions c .. k) is discarded (BitNest, Fig. 4), so a
 * caller's cache length becomes seq_len[b] - 1.
 */
NQ_API nq_status spec_round_commit(const int32_t *out_tok, const int32_t *out_cnt, int B, int k, int32_t *seq,
                                   int32_t *seq_len, int max_len, int32_t *x0, cudaStream_t stream);

/*
 * Int8-activation linears (BitNest, Table 1 "W4A8 -> W8A8" and Table 12: the
 * draft multiplies the 4-bit base codes, the target the 8-bit codes, both
 * against 8-bit activations).
 *
 * nq_quantize_act_int8: per activation row, s_x = fp32(absmax / 127) (IEEE
 *   division), x_q = clamp(rint(x / s_x), -127, 127); a zero row gives
 *   s_x = 0 and zero codes.  x bf16 bits [M][K]; xq int8 [M][K]; sx fp32 [M].
 *   A non-finite row sets NQ_DEV_NONFINITE (its codes are then zero).
 * nq_linear_a8_batch: `count` linears at M activation rows (w, xq, sx, y are
 *   host arrays of device pointers, as for nq_draft_gemv_batch):
 *     draft  (verify = 0, NESTED44 base plane or INT4):
 *       y[m][n] = s_x[m] sum_g s[n][g] sum_{k in g} q4[n][k] x_q[m][k]
 *     verify (verify = 1, NESTED44, both planes):
 *       y[m][n] = s_x[m] sum_g (s[n][g] / 16) sum_{k in g} (16 q4 + r)[n][k] x_q[m][k]
 *   The products of codes are exact integers (dp4a); the group scales are
 *   applied in fp32, 32 inputs at a time.  All layers share one group size.
 */
NQ_API nq_status nq_quantize_act_int8(const uint16_t *x, int M, int K, int8_t *xq, float *sx, cudaStream_t stream);
NQ_API nq_status nq_linear_a8_batch(int count, const nq_weights *w, const int8_t *const *xq, const float *const *sx,
                                    int M, int verify, float *const *y, cudaStream_t stream);

/*
 * The nested KV cache (BitNest, Fig. 4 "KV nesting during speculative
 * decoding": the draft stage reads only the low-bit base view of the cache,
 * verification reads the full b_kv + r_kv-bit view of the same cache, the
 * accepted entries stay and the rejected suffix is discarded).  One layer:
 * for each of `batch` sequences and `heads_kv` heads, `max_len` rows of
 * `head_dim` values (64 or 128); each K or V row is quantised like a NESTED44
 * weight row, in groups of `group` (64 or 128, <= head_dim) values along the
 * head dimension: base and refinement planes uint8
 * [batch][heads_kv][max_len][head_dim/2], scales fp16
 * [batch][heads_kv][max_len][head_dim/group].  An element's draft value is
 * s q4 (4-bit view), its target value (s/16)(16 q4 + r) (8-bit view).  The
 * struct is host memory; the six buffers are caller-owned device memory
 * (sizes from nq_kv_cache_bytes), 16-byte aligned.  Discarding a rejected
 * suffix is only a length: rows at or beyond a sequence's length are never read.
 */
typedef struct {
    int32_t batch, heads_kv, head_dim, group, max_len, pad;
    void *k_base, *k_resid, *k_scales;
    void *v_base, *v_resid, *v_scales;
} nq_kv_cache;

/* Bytes of one plane buffer and of one scale buffer (host-only). */
NQ_API nq_status nq_kv_cache_bytes(int batch, int heads_kv, int head_dim, int group, int max_len,
                                   size_t *plane_bytes, size_t *scale_bytes);

/*
 * Quantise and store n_new new K and V rows per (sequence, head) at rows
 * pos[b] .. pos[b] + n_new - 1 (the positions a pass has just computed):
 * k_new, v_new fp32 [batch][heads_kv][n_new][head_dim] (device, 16-byte
 * aligned); pos int32 [batch] device.  Rows that would land at or beyond
 * max_len are dropped and set NQ_DEV_SEQ_FULL.  Codes are bit-identical to
 * nq_pack_weights' NESTED44 codes of the same rows.
 */
NQ_API nq_status nq_kv_append(const nq_kv_cache *cache, const float *k_new, const float *v_new, int n_new,
                              const int32_t *pos, cudaStream_t stream);

/*
 * Decode attention of M new query rows per sequence over the nested cache:
 *   out[b][m][h][:] = softmax_t(scale q[b][m][h] . K[b][kv(h)][t]) V[b][kv(h)][t]
 * over rows t = 0 .. len[b] - M + m (causal: len[b] counts the M new rows,
 * already appended), kv(h) = h / (heads_q / heads_kv) (grouped-query
 * attention).  planes = 1 reads the 4-bit base view (draft), 2 both planes
 * (the 8-bit target view).  q, out fp32 [batch][M][heads_q][head_dim]; len
 * int32 [batch] device.  Both products run on the tensor cores with fp16
 * operands (the scaled queries, the cache codes, the probabilities times the
 * value rows' scales) and fp32 accumulation; exponentials and sums in fp32:
 * agrees with an fp64 evaluation over the same dequantised rows within the
 * linears' 2e-3 normwise tolerance (about 5e-4 measured).  Workspace
 * (caller-owned, no initialisation) of nq_attn_workspace_bytes() bytes; 0 on
 * bad sizes.
 */
NQ_API size_t nq_attn_workspace_bytes(int batch, int M, int heads_q, int head_dim, int max_len);
NQ_API nq_status nq_attn_decode(const nq_kv_cache *cache, const float *q, int M, int heads_q, const int32_t *len,
                                int planes, float scale, float *out, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Greedy acceptance that allocates nothing and takes no workspace: the same
 * computation and results as spec_accept_greedy, for callers that cannot
 * allocate device memory where they decide tokens (their device memory is
 * owned by another component, such as a serving runtime with a fixed budget,
 * or an allocation must not fail or block inside the decode loop).  The pages
 * have no counterpart; this is a deployment variant.
 * Scratch: a fixed 1 MiB array inside the library, held on every GPU that
 * loads the library until the process exits.  Sizes needing more than that,
 * 256*ceil(4B/256) + B*(k+1)*ceil(V/16384)*8 bytes > 1 MiB, return
 * NQ_ERR_WORKSPACE (e.g. B = 64, k = 8, V = 152064 needs 46,336 bytes).
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  Every
 * call clears the part of the array that must start at zero.  All calls share
 * the one array: calls that overlap on the GPU race and give wrong results.
 */
NQ_API nq_status spec_accept_greedy_noalloc(const int32_t *draft, const float *tgt_logits, int B, int k, int V,
                                            int32_t *out_tok, int32_t *out_cnt, cudaStream_t stream);

/*
 * Diagnostic for the failure path of the library's bounded device waits (the
 * tensor-core linears hand stages between warp roles through mbarriers, each
 * wait limited to 2 s).  Launches one warp that waits, through the same
 * bounded wait, on an mbarrier that nothing ever completes; after limit_us
 * microseconds (1 .. 1,000,000) the wait gives up, sets NQ_DEV_TIMEOUT in the
 * sticky status word and the kernel returns.  Nothing else is in flight, so
 * the CUDA context stays usable: read the bit with nq_get_device_status().
 * Returns NQ_ERR_ARG for a limit outside that range, NQ_ERR_CUDA if the launch
 * fails, else NQ_OK (asynchronous on `stream`).
 */
NQ_API nq_status nq_selftest_bounded_wait(uint32_t limit_us, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
NQ_API const char *nq_status_string(int status);

/* Read, then clear, the sticky device status word of the current device
 * (NQ_DEV_* bits), ordered after all work already queued on `stream`
 * (blocks the host until then). */
NQ_API nq_status nq_get_device_status(cudaStream_t stream, uint32_t *out);

#ifdef __cplusplus
}
#endif
#endif /* NQ_H */
