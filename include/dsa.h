/*
 * dsa.h -- C ABI of libdsa: the DeepSeek sparse-attention (DSA) hot path on
 * one GB300 (sm_103a).
 *
 * The path has three stages, as the DeepSeek-V3.2-Exp atlas page states them
 * (MoE transformer block, "All 43 steps"):
 *
 *   1. the lightning indexer
 *        S^I_{t,s} = 1/(sqrt(H_I) sqrt(D_I)) sum_h w_{t,h} ReLU(q^I_{h,t} . k^I_s)
 *      plus the causal mask M (S~^I = S^I + M),
 *   2. the top-k selection M^sel (top_2048 of S~^I_t per query), and
 *   3. multi-head latent attention over the selected keys, computed in the
 *      absorbed form: q~_h = q^C_h W_UK,h scores against the shared latent
 *      row [c^KV | k^R] (d_c + d_r values per key), an online softmax runs
 *      over the selected keys, and W_UV maps the latent context back to the
 *      per-head values (the output before the output projection wo).
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers unless the comment says "host".  The
 *     caller owns every buffer.  The library never allocates device or host
 *     memory and never synchronises the stream; scratch memory comes from a
 *     caller buffer whose size the matching *_workspace_size call returns.
 *   - Every launch goes on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Every call returns a dsa_status.  Arguments are validated on the host
 *     before anything is launched; an invalid call launches nothing.
 *     Nothing aborts the process.
 *   - A batch is a set of sequences (dsa_seqs).  Query rows of all sequences
 *     are stacked: rows cu_q[b] .. cu_q[b+1]-1 belong to sequence b, and
 *     query t of sequence b sits at absolute position p = start_pos[b] + t.
 *     Keys of sequence b are rows cu_k[b] .. cu_k[b+1]-1 of the key caches
 *     and are numbered 0 .. S_b-1 within the sequence (S_b = cu_k[b+1]-cu_k[b]).
 *     Causality: key s is visible to the query at position p iff s <= p.
 *     Every sequence must satisfy start_pos[b] + T_b <= S_b.
 *   - Element types: DSA_F32 (fp32), DSA_BF16 (bf16), DSA_E4M3 (FP8 e4m3 codes,
 *     one byte each, with fp32 power-of-two block scales).
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dsa_status {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,  /* null pointer, bad size / stride / alignment, inconsistent sequences */
    DSA_ERR_UNSUPPORTED = 2,  /* a dtype / shape combination no kernel handles */
    DSA_ERR_CUDA = 3,         /* a CUDA call or launch failed: dsa_last_cuda_error() gives the code */
    DSA_ERR_TIMEOUT = 4,      /* a device-side wait gave up (reported by dsa_check_device_error) */
    DSA_ERR_WORKSPACE = 5     /* workspace pointer NULL, misaligned (256 B) or smaller than required */
} dsa_status;

typedef enum dsa_dtype {
    DSA_F32 = 0,
    DSA_BF16 = 1,
    DSA_E4M3 = 2
} dsa_dtype;

/* Largest number of sequences in one call. */
#define DSA_MAX_SEQS 1024

/* A batch of sequences.  All three arrays are HOST memory, read during the
 * call only (the library copies what the kernels need into their launch
 * parameters, so the arrays may be freed when the call returns). */
typedef struct dsa_seqs {
    int32_t B;                 /* number of sequences, 1 .. DSA_MAX_SEQS */
    const int32_t *cu_q;       /* host [B+1]: cumulative query rows, cu_q[0] = 0 */
    const int32_t *cu_k;       /* host [B+1]: cumulative keys in the caches, cu_k[0] = 0 */
    const int32_t *start_pos;  /* host [B]: absolute position of each sequence's first query */
} dsa_seqs;

/* ------------------------------------------------------------------------
 * FP8 quantisation of indexer inputs.
 * Source: config_671B_v3.2.json excerpt on the "DeepSeek-V3.2-Exp - Block
 * input" atlas page (dtype fp8, scale_fmt ue8m0).  The block recipe is a
 * reading of that: a block is 128 consecutive values; its scale is 2^e with
 * e the smallest integer such that amax <= 448 * 2^e, clamped to [-127, 127]
 * (amax = 0 gives e = 0); codes are x / 2^e rounded to nearest-even e4m3,
 * saturating at +-448.
 *
 *   x        [n_blocks * 128] values of x_dtype (DSA_F32 or DSA_BF16)
 *   codes    out [n_blocks * 128] e4m3 codes (4-byte aligned)
 *   scales   out [n_blocks] fp32 scales 2^e
 * Inf and NaN inputs are not supported.
 * Errors: DSA_ERR_INVALID_ARG (null pointer, n_blocks < 0, misaligned codes),
 * DSA_ERR_UNSUPPORTED (x_dtype not F32/BF16), DSA_ERR_CUDA.  n_blocks = 0
 * launches nothing.
 * ---------------------------------------------------------------------- */
int dsa_quant_e4m3_ue8m0(const void *x, int x_dtype, int64_t n_blocks, uint8_t *codes, float *scales,
                         void *stream);

/* ------------------------------------------------------------------------
 * Lightning-indexer scores with the causal mask.
 * Source: DeepSeek-V3.2-Exp atlas page, MoE transformer block, equations
 * S^I_{t,s} and S~^I = S^I + M; the indexer's 64 heads x 128 (nnterp
 * deepseek_v32 page, "Up to 2048 tokens ..." note and printout).
 *
 *   q_idx    [sum T, H_I, D_I] of idx_dtype (F32, BF16, or E4M3 codes)
 *   q_scale  [sum T, H_I] fp32 block scales of q_idx (E4M3 only, else NULL)
 *   k_idx    [sum S, D_I] of idx_dtype
 *   k_scale  [sum S] fp32 block scales of k_idx (E4M3 only, else NULL)
 *   w        [sum T, H_I] fp32 per-head weights
 *   scores   out [sum T, ld_scores] fp32.  Row r (query t of sequence b at
 *            position p) receives columns 0 .. S_b-1: the score for s <= p
 *            and -inf for p < s < S_b.  Columns >= S_b are not written.
 *   ld_scores >= max_b S_b, a multiple of 4 (16-byte rows); scores 16-byte aligned.
 * With E4M3 the factorisation sum_h w s_q ReLU(s_k cq.ck) = s_k sum_h (w s_q)
 * ReLU(cq.ck) holds exactly for positive power-of-two scales, so D_I must be
 * 128 (one block per head row).
 * Errors: DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED (H_I > 128 or D_I > 256,
 * E4M3 with D_I != 128), DSA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int dsa_indexer_scores(const void *q_idx, const float *q_scale, const void *k_idx, const float *k_scale,
                       int idx_dtype, const float *w, int H_I, int D_I, const dsa_seqs *seqs,
                       float *scores, int64_t ld_scores, void *stream);

/* ------------------------------------------------------------------------
 * Top-k selection per query row.
 * Source: DeepSeek-V3.2-Exp atlas page, M^sel_{t,s} = M_{t,s} if
 * s in top_k(S~^I_t); the selection tensor is int32 key indices
 * [batch, query, min(index_topk, seq)] (nnterp deepseek_v32 page).
 *
 *   scores   [sum T, ld_scores] fp32 as written by dsa_indexer_scores; only
 *            columns 0 .. p of row r are read (the causal keys).
 *   k        1 .. 16384
 *   idx      out [sum T, k] int32: the n = min(k, p + 1) causal keys with the
 *            largest scores, then -1 padding.  The exact top-n set is returned;
 *            among keys whose score equals the n-th largest the lower key
 *            indices win.  Order within the row: keys above the threshold
 *            in increasing key order, then the tied keys in increasing order.
 *            NaN scores are not supported.
 * Errors: DSA_ERR_INVALID_ARG, DSA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int dsa_topk_select(const float *scores, int64_t ld_scores, const dsa_seqs *seqs, int k, int32_t *idx,
                    void *stream);

/* ------------------------------------------------------------------------
 * Sparse multi-head latent attention over selected keys (absorbed form).
 * Source: DeepSeek-V3.2-Exp atlas page (q^C, k^C = c^KV W_UK, K_i =
 * [K^C_i; k^R], v = c^KV W_UV, M^sel); nnterp deepseek_v32 page (unselected
 * keys masked before the softmax; one rotary key shared by all heads);
 * "DeepSeek-V3.2-Exp - Attention input" page (softmax scale).
 *
 *   q_nope   [sum T, H, d_n]  (dtype)
 *   q_pe     [sum T, H, d_r]  (dtype)
 *   kv_cache latent rows c^KV: row j at kv_cache + j * ld_kv, d_c values (dtype)
 *   k_pe     rotary keys: row j at k_pe + j * ld_pe, d_r values (dtype).  A packed
 *            [sum S, d_c + d_r] cache is k_pe = kv_cache + d_c, ld_pe = ld_kv.
 *   W_UK     [H, d_n, d_c] (dtype): K^C[s,h,d] = sum_c W_UK[h,d,c] c[s,c]
 *   W_UV     [H, d_c, d_v] (dtype): V[s,h,e] = sum_c c[s,c] W_UV[h,c,e]
 *   idx      [sum T, k] int32 key indices local to the row's sequence.  Entries
 *            outside 0 .. min(p, S_b-1) (e.g. the -1 padding) are masked.
 *            Each listed index counts once per occurrence.  NULL selects the
 *            dense causal pattern: entry e of every row is key e (so a row
 *            attends to keys 0 .. min(k, p + 1, S_b) - 1).
 *   softmax_scale  multiplies q.k before the softmax (1/sqrt(d_n + d_r), or the
 *            YaRN-scaled 0.1352 of the released model)
 *   out      out [sum T, H, d_v] (dtype)
 *   lse      out [sum T, H] fp32 natural-log log-sum-exp of the scaled logits,
 *            may be NULL; a row with no live key gets out = 0, lse = -inf.
 *   workspace / ws_bytes  caller scratch, >= dsa_sparse_mla_workspace_size(),
 *            256-byte aligned.
 * Strides are in elements and must keep rows 16-byte aligned.
 * Errors: DSA_ERR_INVALID_ARG, DSA_ERR_WORKSPACE, DSA_ERR_UNSUPPORTED
 * (dtype E4M3, or dims beyond H <= 256, d_n <= 256, d_r <= 128, d_c <= 1024,
 * d_v <= 256), DSA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
size_t dsa_sparse_mla_workspace_size(int dtype, int H, int d_n, int d_r, int d_c, int d_v, int k,
                                     const dsa_seqs *seqs);
int dsa_sparse_mla_fwd(const void *q_nope, const void *q_pe, int dtype, const void *kv_cache, int64_t ld_kv,
                       const void *k_pe, int64_t ld_pe, const void *W_UK, const void *W_UV, int H, int d_n,
                       int d_r, int d_c, int d_v, const int32_t *idx, int k, const dsa_seqs *seqs,
                       float softmax_scale, void *out, float *lse, void *workspace, size_t ws_bytes,
                       void *stream);

/* ------------------------------------------------------------------------
 * Sparse latent attention over an FP8 latent cache.
 * Source: the "DeepSeek-V3.2-Exp - Block input" page, config_671B_v3.2.json
 * excerpt (dtype fp8, scale_fmt ue8m0), read as the storage format of the
 * latent rows c^KV: e4m3 codes with one power-of-two scale per 128 values,
 * the same block recipe as dsa_quant_e4m3_ue8m0 (which produces them).  The
 * rotary keys k_pe stay bf16.
 *
 * Computes what dsa_sparse_mla_fwd computes on the dequantised latent rows
 * c[s, j] = code[s, j] * kv_scale[s, j / 128] (exact in bf16), with the same
 * arguments except:
 *   kv_codes  [sum S, ld_kv] uint8 e4m3 codes (d_c per row; ld_kv in bytes, a
 *             multiple of 16; 16-byte aligned)
 *   kv_scale  [sum S, d_c / 128] fp32 power-of-two scales
 *   k_pe      [sum S, ld_pe] bf16
 * Only the tensor-core kernel's shapes (H = 128, d_n = 128, d_r = 64,
 * d_c = 512, d_v = 128, bf16 queries and weights) are supported.
 * Errors: DSA_ERR_INVALID_ARG, DSA_ERR_WORKSPACE, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int dsa_sparse_mla_fwd_fp8kv(const void *q_nope, const void *q_pe, const uint8_t *kv_codes, int64_t ld_kv,
                             const float *kv_scale, const void *k_pe, int64_t ld_pe, const void *W_UK, const void *W_UV,
                             int H, int d_n, int d_r, int d_c, int d_v, const int32_t *idx, int k,
                             const dsa_seqs *seqs, float softmax_scale, void *out, float *lse, void *workspace,
                             size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Sparse latent attention without a caller workspace.
 * The pages have no counterpart to this entry point: it exists for callers
 * that cannot obtain device memory when they run the attention, e.g. a
 * serving runtime that has already handed all of HBM to its own KV-cache
 * pool (a late cudaMalloc would fail or stall every stream), or a plugin
 * called from such a runtime that receives only its input and output
 * tensors.  It computes exactly what dsa_sparse_mla_fwd computes, with the
 * same arguments minus the workspace, using scratch memory that is part of
 * the library's device code (DSA_NOALLOC_SCRATCH_BYTES per device, held until
 * the process exits) instead of a caller buffer.  It allocates nothing.
 *
 *   - Limit: the call needs the same scratch as dsa_sparse_mla_workspace_size()
 *     reports; a call needing more than DSA_NOALLOC_SCRATCH_BYTES returns
 *     DSA_ERR_WORKSPACE and launches nothing.  With the 671B head shapes and
 *     this version's scratch layout that is up to 128 query rows per call,
 *     e.g. one decode step of up to 128 sequences.
 *   - When the scratch is reserved: CUDA loads the library's device code on a
 *     device lazily by default, at the first call of this entry point on that
 *     device, and the scratch is reserved then.  A call with zero query rows
 *     (cu_q[B] = 0) does this set-up and launches nothing.  A caller that
 *     hands the rest of HBM to its own pool makes that first call before
 *     carving the pool (or runs with CUDA_MODULE_LOADING=EAGER, which loads
 *     it with the context); make it before any stream capture as well.
 *   - Every call looks up the scratch's device address for the current
 *     device (a host-side lookup once loaded), so it stays right across a
 *     device reset.
 *   - Every call on a device shares the one scratch array, which keeps the
 *     previous call's contents (the attention writes every scratch byte it
 *     reads, so nothing needs clearing).  Calls that overlap on the GPU --
 *     on different streams, or from several host threads without ordering --
 *     race on it and give wrong results.
 * Errors: as dsa_sparse_mla_fwd, plus DSA_ERR_WORKSPACE beyond the limit.
 * ---------------------------------------------------------------------- */
#define DSA_NOALLOC_SCRATCH_BYTES (64u << 20)
int dsa_sparse_mla_fwd_noalloc(const void *q_nope, const void *q_pe, int dtype, const void *kv_cache,
                               int64_t ld_kv, const void *k_pe, int64_t ld_pe, const void *W_UK, const void *W_UV,
                               int H, int d_n, int d_r, int d_c, int d_v, const int32_t *idx, int k,
                               const dsa_seqs *seqs, float softmax_scale, void *out, float *lse, void *stream);

/* ------------------------------------------------------------------------
 * The step before the path: the key side of the new tokens, appended to the
 * caches.
 * Sources: "DeepSeek-V3.2-Exp - Attention input" page, mla-init and mla-kv
 * excerpts (kv = wkv_a(x); split into kv_lora_rank + qk_rope_head_dim;
 * kv_norm; apply_rotary_emb on k_pe with freqs_cis); "DeepSeek-V3.2-Exp -
 * Block input" page, RMSNorm excerpt (float32 compute, one gain per feature,
 * eps 1e-6); nnterp deepseek_v32 printout (indexer wk 7168 -> 128, k_norm
 * LayerNorm(128, eps 1e-6, gain and bias), weights_proj 7168 -> 64) and its
 * note that the rotary part is served de-interleaved.
 *
 * For token t of sequence b (position p = start_pos[b] + t, cache row
 * j = cu_k[b] + p), with Y = x . W_proj^T kept in fp32:
 *   kv_cache[j, 0 .. d_c-1]       = bf16(kv_gain * Y[0:d_c] / sqrt(mean(Y[0:d_c]^2) + 1e-6))
 *   kv_cache[j, d_c + i]          = bf16(a cos_i - b sin_i)   with (a, b) = Y[d_c + 2i], Y[d_c + 2i + 1]
 *   kv_cache[j, d_c + d_r/2 + i]  = bf16(a sin_i + b cos_i)   (cos_i, sin_i of position p)
 *   k^I = bf16(LayerNorm(Y[d_c+d_r : +D_I]) * k_gain + k_bias)  (mean, biased variance, eps 1e-6)
 *   k_cache[j] = k^I (bf16), or its e4m3 codes with k_scale[j] as
 *                dsa_quant_e4m3_ue8m0 computes them from the bf16 k^I
 *   w[r, :]    = Y[d_c+d_r+D_I : +H_I]   (r = cu_q[b] + t, the indexer's weights)
 *
 *   x          [sum T, dim] bf16: the new tokens as the attention receives them
 *   W_proj     [d_c + d_r + D_I + H_I, dim] bf16: the rows of wkv_a, then of
 *              wk, then of weights_proj (nn.Linear layout, stacked)
 *   kv_gain    [d_c] fp32; k_gain, k_bias [D_I] fp32
 *   rope_cos, rope_sin  [n_pos, d_r/2] fp32: cos and sin of the angle of
 *              frequency i at position p (row p); every appended position
 *              must be < n_pos
 *   kv_cache   [sum S, ld_kv] bf16, ld_kv >= d_c + d_r (rows written: the
 *              appended ones only)
 *   k_cache    [sum S, D_I] of k_dtype (DSA_BF16, or DSA_E4M3 with D_I = 128
 *              and k_scale [sum S] fp32)
 *   w          out [sum T, H_I] fp32
 *   workspace  >= dsa_kv_prologue_workspace_size(), 256-byte aligned (the fp32 Y)
 * Errors: DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED (dim or the stacked width
 * not a multiple of 64, odd d_r, D_I > 256), DSA_ERR_WORKSPACE, DSA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
size_t dsa_kv_prologue_workspace_size(int dim, int d_c, int d_r, int D_I, int H_I, const dsa_seqs *seqs);
int dsa_kv_prologue(const void *x, int dim, const void *W_proj, const float *kv_gain, const float *k_gain,
                    const float *k_bias, const float *rope_cos, const float *rope_sin, int n_pos, int d_c, int d_r,
                    int D_I, int H_I, const dsa_seqs *seqs, void *kv_cache, int64_t ld_kv, void *k_cache, int k_dtype,
                    float *k_scale, float *w, void *workspace, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * The step after the path: the output projection y = out . wo^T.
 * Source: "DeepSeek-V3.2-Exp - Attention input" page, mla-init excerpt (wo maps
 * n_heads * v_head_dim to dim); nnterp deepseek_v32 printout (o_proj,
 * 16384 -> 7168, reading every head's output side by side).
 *
 *   out   [M, in_features] bf16: the attention output [M, H, d_v] viewed as
 *         [M, H * d_v]
 *   wo    [d_model, in_features] bf16 (nn.Linear layout)
 *   y     out [M, d_model] bf16
 * in_features and d_model multiples of 64; pointers 16-byte aligned.  fp32
 * accumulation on the tensor cores.
 * Errors: DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int dsa_output_proj(const void *out, const void *wo, int M, int in_features, int d_model, void *y, void *stream);

/* ------------------------------------------------------------------------
 * The whole path: [quantise] -> indexer -> top-k -> sparse latent attention.
 * Sources: as for the three stages above.  Rows are processed in chunks so
 * that the fp32 score buffer stays bounded; the workspace size covers one
 * chunk of scores, the selection (unless idx_out is given), the FP8 copies
 * of q^I / k^I (idx_fp8) and the attention scratch.
 * When every row's causal prefix holds at most top_k keys (k >= S, the case
 * the deepseek_v32 note on the nnterp page calls plain causal attention), the
 * selection is every causal key and is known without scores: the quantiser,
 * indexer and top-k are not launched, the attention reads the dense causal
 * pattern, and idx_out (when given) is filled with 0 .. n-1 and -1 padding,
 * exactly what the top-k writes for such rows.
 * ---------------------------------------------------------------------- */
typedef struct dsa_problem {
    /* shapes */
    int32_t H_I, D_I, top_k;          /* indexer heads, head dim, k */
    int32_t H, d_n, d_r, d_c, d_v;    /* MLA heads and widths */
    int32_t dtype;                    /* DSA_F32 or DSA_BF16: storage type of every tensor below but w */
    int32_t idx_fp8;                  /* 1: quantise q^I, k^I to e4m3 + ue8m0 before the indexer */
    float softmax_scale;
    /* indexer inputs */
    const void *q_idx;                /* [sum T, H_I, D_I] */
    const void *k_idx;                /* [sum S, D_I] */
    const float *w;                   /* [sum T, H_I] fp32 */
    /* attention inputs (layouts as in dsa_sparse_mla_fwd) */
    const void *q_nope, *q_pe;
    const void *kv_cache;
    int64_t ld_kv;
    const void *k_pe;
    int64_t ld_pe;
    const void *W_UK, *W_UV;
    /* outputs */
    void *out;                        /* [sum T, H, d_v] (dtype) */
    float *lse;                       /* [sum T, H] or NULL */
    int32_t *idx_out;                 /* [sum T, top_k] or NULL (then kept in the workspace) */
    /* The step after the path, optional (NULL wo: not applied): the output
     * projection y = out wo^T ("DeepSeek-V3.2-Exp - Attention input" page,
     * mla-init excerpt, wo: n_heads * v_head_dim -> dim).  W_UV and wo run
     * chunk by chunk (2048 rows), so each chunk of the attention output is read
     * back from L2 right after it is written.  `out` may then be NULL (the
     * chunks live in the workspace).  bf16 only; d_model and H * d_v multiples
     * of 64. */
    const void *wo;                   /* [d_model, H * d_v] */
    int32_t d_model;
    void *y;                          /* out [sum T, d_model] */
    /* FP8 latent cache (as dsa_sparse_mla_fwd_fp8kv): kv_fp8 = 1 makes kv_cache
     * e4m3 codes with ld_kv in bytes (a multiple of 16) and kv_scale their
     * [sum S, d_c / 128] fp32 block scales; k_pe stays bf16.  bf16 only, at
     * the tensor-core kernel's head shapes. */
    int32_t kv_fp8;
    const float *kv_scale;
} dsa_problem;

size_t dsa_forward_workspace_size(const dsa_problem *p, const dsa_seqs *seqs);
int dsa_forward(const dsa_problem *p, const dsa_seqs *seqs, void *workspace, size_t ws_bytes, void *stream);

/* The forward from HOST buffers: the end-to-end call of one step.  On `stream`
 * it copies the step's inputs from host memory into the device buffers that
 * `p` names, runs dsa_forward, and copies the results back: one
 * cudaMemcpyAsync per input and output; the appended cache rows of each array
 * go in one copy to the start of `workspace` and a small kernel puts them in
 * their rows (the workspace is free until the forward starts) -- or, when that
 * staging does not fit the workspace or a row is not a multiple of 16 bytes,
 * one copy per sequence and array.  q_nope and q_pe, which only the attention
 * stage reads, are copied last and on a side stream of the library's (one per
 * host thread and device, created on first use and kept): their transfer
 * overlaps the quantiser, indexer and top-k, and the attention stage waits for
 * it on `stream`.  Everything else is enqueued on `stream`.  With
 * page-locked (pinned) host buffers every copy is asynchronous and the call
 * returns once all the work is enqueued; the caller synchronises `stream`
 * before reading the host outputs.  Pageable host memory also works, but then
 * the copies block the calling thread.
 *
 * Host inputs (NULL: the device buffer already holds that data):
 *   q_idx, w, q_nope, q_pe   the step's queries, laid out as the device tensors
 *                            of `p` ([sum T, ...] rows, dense);
 *   kv_new                   the cache rows the step appends: for every
 *                            sequence b in order, its rows start_pos[b] ..
 *                            S_b - 1 (S_b = cu_k[b+1] - cu_k[b]), each a full
 *                            row of ld_kv elements (bytes for an e4m3 cache),
 *                            written to cache rows cu_k[b] + start_pos[b] ..;
 *   k_pe_new                 the same rows of k_pe (ld_pe elements each); NULL
 *                            when k_pe lies inside the kv_cache rows that
 *                            kv_new already carries;
 *   k_idx_new                the same rows of the indexer key cache (D_I each);
 *   kv_scale_new             e4m3 cache: the same rows' d_c / 128 scales.
 * Host outputs (NULL: not copied back): out (y when p->wo is set: the
 * projected output), lse, idx (requires p->idx_out).
 * Pipelining (all NULL: none), four cudaEvent_t handles: copy_after, which
 * the input copies wait for (cudaStreamWaitEvent before the first of them);
 * copy_done, recorded once the input copies (on both streams) and the append
 * kernel are enqueued; compute_after, which the forward waits for after that;
 * and compute_done, recorded once the forward's kernels are enqueued, before
 * the output copies.  Calls on two streams with their own device buffers can
 * so chain their forwards (each waits for the previous call's compute_done)
 * while one call's copies overlap the other's kernels, and chain their input
 * copies (each waits for the previous call's copy_done) so that two calls'
 * inputs do not share the host-to-device bandwidth: the first forward then
 * waits for one call's inputs instead of two calls'.
 * Every check dsa_forward makes runs before the first copy is enqueued, so a
 * refused call changes no device buffer.
 * Returns what dsa_forward returns, DSA_ERR_INVALID_ARG when a sequence has
 * start_pos[b] > S_b with kv_new, k_pe_new, k_idx_new or kv_scale_new given, or
 * when a requested output has no device buffer in `p`, and DSA_ERR_CUDA when
 * a copy cannot be enqueued. */
typedef struct dsa_host_io {
    const void *q_idx, *w, *q_nope, *q_pe;
    const void *kv_new, *k_pe_new, *k_idx_new;
    const float *kv_scale_new;
    void *out;
    float *lse;
    int32_t *idx;
    void *compute_after, *compute_done;
    void *copy_after, *copy_done;
} dsa_host_io;
int dsa_forward_host(const dsa_problem *p, const dsa_seqs *seqs, const dsa_host_io *io, void *workspace,
                     size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Status and diagnostics.
 * ---------------------------------------------------------------------- */
/* Human-readable name of a dsa_status. */
const char *dsa_status_string(int status);
/* The cudaError_t behind the most recent DSA_ERR_CUDA on this host thread. */
int dsa_last_cuda_error(void);
/* Waits for `stream`, then reads and clears the device error word that the
 * kernels' bounded waits set.  Returns DSA_OK, DSA_ERR_TIMEOUT (and stores
 * the recorded site in *site when non-NULL), or DSA_ERR_CUDA.  This is the
 * only entry point that synchronises. */
int dsa_check_device_error(void *stream, int *site);
/* Self-test of the failure-detection path (no counterpart on the pages: a
 * diagnostic of this library).  Launches, on `stream`, one CTA that waits on an
 * mbarrier phase that nothing completes, through the same bounded wait every
 * tensor-core kernel here uses, with a limit of `limit_cycles` SM clock cycles
 * (1 .. 2^32) instead of the kernels' ~2 s.  The wait gives up, records site 90
 * in the device error word and returns; the CTA then completes the phase and
 * checks that a second wait on it succeeds, writing 1 to *completed_ok (a device
 * int, may be NULL) when both behaved.  The GPU does not fault or hang: the
 * caller reads the outcome with dsa_check_device_error (DSA_ERR_TIMEOUT, site
 * 90), after which the context is usable as before.  Returns DSA_ERR_INVALID_ARG
 * for a limit out of range. */
int dsa_selftest_bounded_wait(int64_t limit_cycles, int *completed_ok, void *stream);
/* Wait limit of the tensor-core kernels (no counterpart on the pages: a
 * diagnostic of this library).  Every wait of the indexer, absorption and
 * attention kernels on a barrier phase gives up after this many SM clock cycles
 * (default, and `cycles` = 0: 2^32, about two seconds), records its site in the
 * device error word, and the CTA drains its copies and MMAs already in flight
 * (those drain waits keep the default limit), frees its tensor memory and exits.
 * A short limit makes the failure path of the production kernels run without a
 * fault: the next dsa_check_device_error returns DSA_ERR_TIMEOUT with the site,
 * the outputs of the calls made meanwhile are undefined, and calls made after
 * the limit is restored behave normally.  The setting is process-wide and read
 * when a kernel is launched.  Returns DSA_ERR_INVALID_ARG for cycles < 0 or
 * above the default. */
int dsa_set_wait_limit(int64_t cycles);
/* Selects, for dsa_forward calls that follow, between the two implementations
 * of the indexer + top-k on batches of at least 304 groups of 4 query rows
 * (no counterpart on the pages: a choice of this library).  Fused: one
 * persistent kernel scores a group into a per-SM slot and selects its rows'
 * top-k from it while the next group is scored, with no [rows, S] score
 * buffer; two kernels: the indexer writes chunks of fp32 score rows and a
 * separate top-k kernel selects from them.  Both give identical selections.
 * mode 1: fused wherever it applies; 0: never; -1 (default): where it measured
 * faster, the FP8 indexer over rows that see on average >= 16384 keys.
 * Process-wide.  Returns DSA_ERR_INVALID_ARG for another mode. */
int dsa_set_fused_topk(int mode);
/* Bit mask of the kernels the last entry point launched on this host thread
 * (DSA_KERNEL_* bits), and how many kernel launches it made. */
uint32_t dsa_last_kernels(void);
int dsa_last_launch_count(void);

/* Optional timing hook.  When `events` is non-NULL, dsa_forward records
 * events[i] (cudaEvent_t handles created by the caller) on its stream at
 * these stage boundaries:
 *   0 start, 1 after FP8 quantisation, 2 after the indexer + top-k loop,
 *   3 after q~ = q_nope W_UK, 4 after the sparse attention (and its
 *   split-key combine), 5 after o_lat W_UV (the end).
 * n_events must be DSA_STAGE_EVENTS.  Pass NULL to switch it off.  The setting
 * is per host thread.  Returns DSA_ERR_INVALID_ARG for a wrong count. */
#define DSA_STAGE_EVENTS 6
int dsa_set_stage_events(void *const *events, int n_events);

#define DSA_KERNEL_QUANT        (1u << 0)
#define DSA_KERNEL_INDEXER_SIMT (1u << 1)
#define DSA_KERNEL_INDEXER_TC   (1u << 2)
#define DSA_KERNEL_INDEXER_FP8  (1u << 3)
#define DSA_KERNEL_TOPK         (1u << 4)
#define DSA_KERNEL_ABSORB_SIMT  (1u << 5)
#define DSA_KERNEL_ABSORB_TC    (1u << 6)
#define DSA_KERNEL_MLA_SIMT     (1u << 7)
#define DSA_KERNEL_MLA_TC       (1u << 8)
#define DSA_KERNEL_COMBINE      (1u << 9)
#define DSA_KERNEL_SELFTEST     (1u << 10)
#define DSA_KERNEL_DENSE_IDX    (1u << 11)
#define DSA_KERNEL_GEMM_TC      (1u << 12)
#define DSA_KERNEL_PROLOGUE     (1u << 13)
#define DSA_KERNEL_INDEXER_TOPK (1u << 14)  /* the indexer launch also selected the top-k (fused) */
#define DSA_KERNEL_APPEND       (1u << 15)  /* dsa_forward_host put staged cache rows in place */

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
