/*
 * dflash.h — C ABI of the GB300 speculative-decoding draft-round library (libdflash.so).
 *
 * One draft round, as hf2q 0.1.1's `spec_decode/dflash/qwen35_orchestrator.rs` runs it
 * (module doc, "Per-round loop", steps 1-9): a drafter forward over a block of K+1
 * positions, a per-position argmax over the vocabulary, the greedy accept-prefix walk
 * against the verifier's argmaxes and the KV rollback of the rejected positions. The
 * Qwen3.5 MTP (NextN) draft step of `models/qwen35/mtp.rs` (`forward_draft_with_hidden`)
 * is the second drafter.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer is caller-owned. Device pointers are CUDA global memory on the current
 *    device; "host" is marked where a pointer is host memory. The library allocates no
 *    tensor memory; besides the thread-local error text it keeps only executable CUDA graphs
 *    of df_generate and df_draft_round_host (keyed by every argument they bake in) and the
 *    streams it captures them on.
 *  - BF16 tensors are passed as `const uint16_t *` holding BF16 bit patterns (little-endian,
 *    row-major `[out, in]`, as tensors.rs `upload_bf16` copies them: no transpose, no
 *    dequantisation). RMSNorm weights are F32 (tensors.rs `upload_bf16_as_f32`: a BF16 buffer
 *    read as F32 is the misinterpretation bug that file's tests guard against).
 *    Activations, residuals, logits and the KV cache are F32.
 *  - Calls are asynchronous on `stream` (a `cudaStream_t`; NULL = legacy default stream). A
 *    call returns after host-side validation and kernel launches; nothing synchronises except
 *    `df_draft_round_host`. Return value: DF_OK or a negative `df_status`; `df_last_error()`
 *    then holds a message. Host-detected errors launch nothing and modify nothing.
 *  - Conditions only the device can see (a sequence's `n_new` above `n_new_max`, a cache that
 *    would overflow, a token id outside [0, vocab), a rollback longer than the cache) are
 *    clamped so no access leaves its buffer, and the failing `df_status` code is written to the
 *    optional device word `d_status` (int32, may be NULL). A kernel never traps.
 *  - `ws` is a device workspace of at least the size the matching `*_workspace_bytes` query
 *    returns (256-byte aligned). Its counter region must be zero before the first call that
 *    uses it (allocate it zeroed); every call leaves it zero again. Calls sharing one workspace
 *    must be ordered on the GPU (the same stream, or events).
 *  - Dimensions: every K dimension of a projection (hidden, intermediate, n_q_heads*head_dim,
 *    n_target_layers*hidden) must be a multiple of 8; head_dim a multiple of 32 and <= 256;
 *    rotary_dim even and <= head_dim; n_q_heads a multiple of n_kv_heads.
 *  - Weights (row-major or tiled) are read-only inputs that must be complete when a call is
 *    enqueued: a projection requests its first weight tiles before it waits for the kernel ahead
 *    of it on the stream (programmatic dependent launch), so weights written by kernels on the
 *    same stream need a stream synchronisation or an event wait before the call.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *df_stream_t; /* same type as cudaStream_t */

typedef enum {
    DF_OK = 0,
    DF_EINVAL = -1,      /* null pointer, bad flag, id outside [0, vocab) */
    DF_ESHAPE = -2,      /* dimension out of range or misaligned; n_new above n_new_max */
    DF_ECAPACITY = -3,   /* KV cache would overflow, or a rollback exceeds seq_len */
    DF_EWORKSPACE = -4,  /* workspace missing, misaligned or too small */
    DF_ECUDA = -5,       /* a CUDA runtime call or launch failed */
    DF_ETIMEOUT = -6     /* a bounded device-side wait gave up */
} df_status;

/* Thread-local text of the last error returned on this thread ("" if none). */
const char *df_last_error(void);

/* Library ABI version (major * 100 + minor). */
int df_version(void);

/* Number of kernels this process has launched through the library so far (all threads).
 * Launches recorded into a CUDA graph count once, at capture. */
uint64_t df_kernel_launches(void);

/* Per-kernel GPU time of the library's own launches (the analogue of the pages'
 * HF2Q_MTP_PROFILE / HF2Q_DFLASH_PROFILE sub-step timers, without their forced syncs): while
 * enabled, an event pair brackets every kernel on its launching stream; launches recorded into
 * a CUDA graph capture are not timed. df_profile_enable(1) clears the record (room for 4096
 * kernels) and starts recording, df_profile_enable(0) stops. df_profile_read synchronises and
 * writes up to max_entries durations (microseconds) into us and their kernel names, one per
 * line, into names; it returns the number of entries. */
int df_profile_enable(int on);
int df_profile_read(float *us, int max_entries, char *names, size_t names_bytes);

/* Trace builds only (libdflash_trace.so, built with build.py --trace; other builds return
 * DF_EINVAL): every CTA of every kernel records its kernel id (TK_* of the library's internal
 * list; projections 100 + 2 * epilogue + stream-K), its SM and the global-timer nanoseconds at
 * which it started and its thread 0 left, into one device buffer of 2^20 records, so the
 * launches of a CUDA graph replay can be timed one by one with their overlaps.
 * df_trace_reset clears the buffer (synchronous); df_trace_read synchronises the device and
 * copies up to max_records records out, returning their number. */
int df_trace_reset(void);
int df_trace_read(uint32_t *kid, uint32_t *sm, unsigned long long *t0, unsigned long long *t1,
                  int max_records);

/* ------------------------------------------------------------------------------------------
 * DFlash drafter (tensors.rs `DFlashLayerTensors`, `DFlashModelTensors`; dflash config fields
 * seen in qwen35_orchestrator.rs: target_layer_ids, mask_token_id, hidden_size, head_dim).
 * ---------------------------------------------------------------------------------------- */
typedef struct {
    int32_t hidden;           /* H */
    int32_t n_layers;         /* decoder layers */
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t head_dim;         /* d */
    int32_t intermediate;     /* SwiGLU I */
    int32_t vocab;            /* V (shared embed / lm_head rows) */
    int32_t n_target_layers;  /* fc input = n_target_layers * H */
    int32_t rotary_dim;       /* 0 = head_dim */
    int32_t mask_token_id;    /* id of the K mask positions of the block */
    int32_t causal_block;     /* 0: block positions attend to each other freely; 1: causal */
    float rms_eps;
    float rope_theta;
    float embed_scale;        /* multiplies gathered embedding rows (1.0) */
    int32_t kv_bf16;          /* 0: F32 KV cache; 1: BF16 KV cache (k[l], v[l] hold BF16 bit
                                 patterns in the same layout; every K/V value the attention reads
                                 is rounded to BF16 when produced). Needs head_dim 128 or 256 and
                                 at most 32 query rows per KV head (block x n_q / n_kv). */
} df_dflash_config;

typedef struct {
    const float *input_norm;      /* [H] F32, before attention */
    const float *post_attn_norm;  /* [H] F32, before the SwiGLU */
    const float *q_norm;          /* [d] F32, per-head RMSNorm of q */
    const float *k_norm;          /* [d] F32, per-head RMSNorm of k */
    const uint16_t *wq;           /* [n_q*d, H] BF16 */
    const uint16_t *wk;           /* [n_kv*d, H] BF16 */
    const uint16_t *wv;           /* [n_kv*d, H] BF16 */
    const uint16_t *wo;           /* [H, n_q*d] BF16 */
    const uint16_t *w_gate;       /* [I, H] BF16 */
    const uint16_t *w_up;         /* [I, H] BF16 */
    const uint16_t *w_down;       /* [H, I] BF16 */
} df_layer_weights;

typedef struct {
    const uint16_t *fc;              /* [H, n_target_layers*H] BF16 */
    const float *hidden_norm;        /* [H] F32, RMSNorm of the fc output */
    const float *final_norm;         /* [H] F32 */
    const df_layer_weights *layers;  /* HOST array [n_layers] */
    const uint16_t *embed;           /* [V, H] BF16 token embedding (the target's, borrowed) */
    const uint16_t *lm_head;         /* [V, H] BF16 (the target's, borrowed) */
    const void *tiled;               /* NULL, or the projection and lm_head weights re-laid out by
                                        df_dflash_tile_weights from these same matrices: the
                                        projections then read their weights from it (the matrices
                                        above must stay valid: they still describe the shapes) */
} df_dflash_weights;

/*
 * Tiled weights. The projections read their weights as 128-row x 64-column BF16 tiles; from the
 * row-major [out, in] matrices each tile arrives as 128 strided 128-byte rows, from a tiled copy
 * as one contiguous block laid out exactly as the tensor cores read it (the 128-byte-swizzled
 * image: row r of a tile at byte r * 128, its 16-byte piece j at (j ^ (r % 8)) * 16; tile
 * (m, kb) of a matrix at byte (m * kbt + kb) * 16384, kbt = ceil(in / 64); rows and columns past
 * the matrix zero). Two K blocks are then moved per bulk copy, which on this part streams at the
 * HBM rate where 16 KB tensor-map copies do not. A one-time device-to-device conversion at model
 * load; the copy takes as many bytes as the matrices (padded to whole tiles).
 *
 * df_dflash_tiled_bytes: bytes of a DFlash model's tiled copy (fc, every layer's QKV, O,
 *   gate/up (gate and up rows paired 64 + 64 per tile), down, then the lm_head); 0 on an invalid
 *   config.
 * df_dflash_tile_weights: fills `tiled` (device, >= df_dflash_tiled_bytes, 1024-byte aligned,
 *   owned by the caller) from w's matrices on `stream`; set w->tiled = tiled afterwards, and
 *   synchronise `stream` before the first call that reads it (see the weights convention above).
 *   DF_EWORKSPACE when too small, DF_EINVAL on a bad pointer.
 * df_tiled_matrix_bytes / df_tile_matrix: the same for one [N, K] matrix (K a multiple of 8),
 *   e.g. an lm_head for lm_head_argmax_tiled.
 */
size_t df_dflash_tiled_bytes(const df_dflash_config *cfg);
int df_dflash_tile_weights(const df_dflash_config *cfg, const df_dflash_weights *w, void *tiled,
                           size_t tiled_bytes, df_stream_t stream);
size_t df_tiled_matrix_bytes(int N, int K);
int df_tile_matrix(const uint16_t *W, int N, int K, void *tiled, size_t tiled_bytes,
                   df_stream_t stream);

/* Per-layer KV cache, F32 (or BF16 with cfg->kv_bf16). Row p of sequence b, KV head h lives at
 * element ((b * n_kv + h) * cap + p) * head_dim of k[l]. seq_len[b] counts the valid rows. */
typedef struct {
    float *const *k;     /* HOST array [n_layers] of device pointers [batch, n_kv, cap, d] */
    float *const *v;     /* HOST array [n_layers], same layout */
    int32_t *seq_len;    /* device [batch] */
    int32_t cap;         /* rows per sequence and head */
    int32_t batch;
    int32_t n_layers;
} df_kv_cache;

/* Workspace bytes for dflash_block_forward / df_draft_round at batch B, block = K+1 and
 * at most n_new_max new context rows per sequence. 0 on invalid arguments. */
size_t df_dflash_workspace_bytes(const df_dflash_config *cfg, int B, int block, int n_new_max);

/*
 * dflash_block_forward — the drafter forward of one round (qwen35_orchestrator.rs steps 2-4,
 * `dispatch_dflash_model_forward`; tensors.rs for the tensors it reads).
 *   block_ids          device int32 [B, block]: [last_token, mask_token_id x K] per sequence
 *   target_hidden_new  device F32 [B, n_new_max, n_target_layers*H]: the target hidden rows of
 *                      the n_new[b] context positions committed since the last round
 *   n_new              device int32 [B], each in [0, n_new_max]
 *   h_final            device F32 [B, block, H] out: final-normed hidden of every block row
 * For every layer the n_new[b] context rows' K/V (per-head k-norm, RoPE at their absolute
 * positions seq_len[b] + j) are appended at cache rows seq_len[b] + j; the block rows (at
 * positions seq_len[b] + n_new[b] + i) attend over the whole cache plus the block and their
 * own K/V are not kept. On return seq_len[b] has advanced by n_new[b].
 * Device status: DF_ESHAPE (n_new out of range), DF_ECAPACITY (append beyond cap),
 * DF_EINVAL (block id outside [0, vocab)).
 */
int dflash_block_forward(const df_dflash_config *cfg, const df_dflash_weights *w,
                         const df_kv_cache *cache, const int32_t *block_ids,
                         const float *target_hidden_new, const int32_t *n_new, int n_new_max,
                         int B, int block, float *h_final, void *ws, size_t ws_bytes,
                         int32_t *d_status, df_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * lm_head + per-row argmax (qwen35_orchestrator.rs step 5,
 * `per_position_argmax_from_normed_hidden`; mtp.rs `forward_shared_head`), fused so the
 * logits never reach global memory.
 * ---------------------------------------------------------------------------------------- */
size_t df_lm_head_workspace_bytes(int rows, int H, int V);

/*   W     device BF16 [V, H];  X device F32 [rows, H] (already normed)
 *   idx   device int32 [rows] out: argmax, the lowest index among exactly equal maxima
 *   top1  device F32 [rows] out or NULL: the largest logit
 *   top2  device F32 [rows] out or NULL: the second largest (== top1 when the max is tied) */
int lm_head_argmax(const uint16_t *W, const float *X, int rows, int H, int V, int32_t *idx,
                   float *top1, float *top2, void *ws, size_t ws_bytes, df_stream_t stream);

/* lm_head_argmax reading the tiled copy of W (df_tile_matrix, V x H): same outputs, same
 * workspace; W_tiled device, 1024-byte aligned. */
int lm_head_argmax_tiled(const void *W_tiled, const float *X, int rows, int H, int V,
                         int32_t *idx, float *top1, float *top2, void *ws, size_t ws_bytes,
                         df_stream_t stream);

/*
 * lm_head_argmax_noalloc — lm_head_argmax for callers that cannot allocate device memory:
 * host code that runs inside an engine or plug-in which owns every allocation, or a loop that
 * may not take cudaMalloc's implicit synchronisation. The source pages have no counterpart;
 * the arithmetic and outputs are those of lm_head_argmax.
 * It takes no workspace: its scratch (about 3.5 MB) is one fixed array in the library's device
 * memory, which every GPU that loads the library holds until the process exits. Limits:
 * rows <= 16, H <= 8192 (a multiple of 8), V <= 524288; larger sizes return DF_ESHAPE.
 * The first call on a device looks up the array's device address with that device current, so
 * make that first call before any stream capture. All calls share the one array and it keeps
 * the last call's contents: the call clears the part that must start at zero itself, and calls
 * that overlap on the GPU (other streams, other host threads) race — order them.
 */
int lm_head_argmax_noalloc(const uint16_t *W, const float *X, int rows, int H, int V,
                           int32_t *idx, float *top1, float *top2, df_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * One BF16-weight x F32-activation projection (mtp.rs `apply_linear_projection_f32`;
 * tensors.rs: row-major [out, in] BF16 weights consumed with F32 activations):
 *   Y[t, n] = sum_k X[t, k] * W[n, k],  W device BF16 [N, K], X device F32 [T, K],
 *   Y device F32 [T, N]; K a multiple of 8. F32 accumulation.
 * ---------------------------------------------------------------------------------------- */
size_t df_linear_workspace_bytes(int T, int N, int K);

int df_linear(const uint16_t *W, const float *X, int T, int N, int K, float *Y, void *ws,
              size_t ws_bytes, df_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Split-KV scaled dot-product attention on its own (the attention step of every drafter layer
 * and of the MTP step: softmax(q k^T / sqrt(d)) v with grouped KV heads, mtp.rs
 * `forward_full_attention`; the DFlash block attends to the context rows and to all block rows,
 * qwen35_orchestrator.rs step 4). The same kernels run inside dflash_block_forward and
 * mtp_forward_draft.
 * ---------------------------------------------------------------------------------------- */
/* Workspace for the per-chunk partial outputs; 0 for unsupported sizes. */
size_t df_attention_workspace_bytes(int B, int blk, int nq, int nkv, int d, int cap);

/*   q            device F32 [B, blk, nq, d]: query rows (RoPE and norms already applied)
 *   cache_k/v    device F32 [B, nkv, cap, d]; sequence b sees cache rows [0, seq_len[b])
 *   seq_len      device int32 [B], clamped to [0, cap]
 *   kb, vb       device F32 [B, nkv, blk, d] block keys/values seen after the cache rows, or
 *                both NULL
 *   causal_block 0: every query row sees all block rows; 1: block row i sees block rows <= i
 *   out          device F32 [B, blk, nq, d] out
 * Query head h reads KV head h / (nq / nkv). d is 32, 64, 128 or 256; q, the caches and the
 * block buffers are 16-byte aligned. A row with no visible key gets zeros. */
int df_attention(const float *q, const float *cache_k, const float *cache_v, int cap,
                 const int32_t *seq_len, const float *kb, const float *vb, int B, int blk, int nq,
                 int nkv, int d, int causal_block, float *out, void *ws, size_t ws_bytes,
                 int32_t *d_status, df_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Greedy accept walk (qwen35_orchestrator.rs module doc "Greedy accept-walk consistency
 * invariant" and steps 7-9: `step_round_from_argmaxes`, rollback = K - accept_count).
 * ---------------------------------------------------------------------------------------- */
/*   drafts       device int32, row b at drafts + b*drafts_ld, K entries (block positions 1..K)
 *   target       device int32 [B, K+1]: verifier argmaxes over [last_token, drafts...]
 *   eos          device int32 [n_eos] (may be NULL when n_eos == 0)
 *   committed    device int32 [B, K+1] out: accepted drafts + the free token, cut after the
 *                first EOS id; entries past n_committed[b] are set to -1
 *   n_committed, accept_count, hit_eos, rollback   device int32 [B] out
 * accept_count = longest prefix with drafts == target; rollback = K - accept_count
 * (independent of the EOS cut); 1 <= n_committed <= K+1. */
int accept_prefix_argmax(const int32_t *drafts, int drafts_ld, const int32_t *target, int B,
                         int K, const int32_t *eos, int n_eos, int32_t *committed,
                         int32_t *n_committed, int32_t *accept_count, int32_t *hit_eos,
                         int32_t *rollback, df_stream_t stream);

/* Same walk on the host for one sequence (all pointers HOST memory). Synchronous. */
int accept_prefix_argmax_host(const int32_t *drafts, const int32_t *target, int K,
                              const int32_t *eos, int n_eos, int32_t *committed,
                              int32_t *n_committed, int32_t *accept_count, int32_t *hit_eos,
                              int32_t *rollback);

/* ------------------------------------------------------------------------------------------
 * Non-greedy accept step: speculative sampling at temperature T > 0. qwen35_orchestrator.rs,
 * module doc "Non-greedy (Metropolis-Hastings) is out of scope here": stochastic acceptance is
 * wired through the MTP K=1 path and would take the place of `step_round_from_argmaxes` at
 * step 11 of the DFlash loop. The page gives no formula; the rule is read as the standard
 * speculative-sampling test. With p_i = softmax(target_logits[b, i] / T) and
 * q_i = softmax(draft_logits[b, i] / T):
 *   draft x_i is accepted while u_accept[b, i] * q_i(x_i) < p_i(x_i);
 *   at the first rejection a the committed token is drawn from max(0, p_a - q_a) (normalised),
 *   after K acceptances from p_K;
 *   a draw from weights w with uniform u is the smallest j with w_0 + ... + w_j > u * sum(w).
 * committed / n_committed / hit_eos / rollback follow the greedy walk: accepted drafts then the
 * drawn token, cut after the first EOS id, -1 past n_committed, rollback = K - accept_count.
 * ---------------------------------------------------------------------------------------- */
/* Workspace (chunk statistics, per-sequence state, draw partial sums, counters); allocate it
 * zeroed. 0 for unsupported sizes. */
size_t df_accept_stochastic_workspace_bytes(int B, int K, int V);

/*   draft_logits   device F32 [B, K, V]: drafter logits of block positions 1..K, 16-byte aligned
 *   target_logits  device F32 [B, K+1, V]: verifier logits at positions 0..K, 16-byte aligned
 *   V              vocabulary, a positive multiple of 4
 *   drafts         device int32 [B, K]: the drafted tokens (ids outside [0, V) are clamped and
 *                  set DF_EINVAL in d_status)
 *   temperature    > 0 (DF_EINVAL otherwise; temperature 0 is accept_prefix_argmax)
 *   u_accept       device F32 [B, K] uniforms in [0, 1); u_sample device F32 [B] the same
 *   eos            device int32 [n_eos] (NULL when n_eos == 0)
 *   committed      device int32 [B, K+1] out; n_committed, accept_count, hit_eos, rollback
 *                  device int32 [B] out
 * 1 <= K <= 64. A draw whose weights sum to zero sets DF_EINVAL in d_status. */
int accept_stochastic(const float *draft_logits, const float *target_logits, int V,
                      const int32_t *drafts, int B, int K, float temperature,
                      const float *u_accept, const float *u_sample, const int32_t *eos, int n_eos,
                      int32_t *committed, int32_t *n_committed, int32_t *accept_count,
                      int32_t *hit_eos, int32_t *rollback, void *ws, size_t ws_bytes,
                      int32_t *d_status, df_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Sampled drafts: one token per row drawn from q = softmax(logits[r] / T) with the uniform
 * u[r]: the smallest j whose running sum q_0 + ... + q_j exceeds u[r] (the drafter's side of
 * the non-greedy path of qwen35_orchestrator.rs's module doc, "Non-greedy (Metropolis-Hastings)
 * is out of scope here": each drafted position is a sample of the drafter's distribution, which
 * the accept step above then divides by). The weights are computed to ~1e-14 relative and summed
 * as float-float pairs, so a draw differs from a float64 reference only where u * total is
 * within ~1e-12 of a cumulative boundary.
 * ---------------------------------------------------------------------------------------- */
/* Workspace (chunk statistics, draw partial sums, counters); allocate it zeroed. */
size_t df_sample_softmax_workspace_bytes(int R, int V);

/*   logits       device F32 [R, V], 16-byte aligned; V a positive multiple of 4, V <= 2^21
 *   temperature  > 0 (DF_EINVAL otherwise)
 *   u            device F32 [R] uniforms in [0, 1)
 *   tokens       device int32 [R] out
 * A row whose weights sum to zero (all logits -inf) sets DF_EINVAL in d_status. */
int sample_softmax(const float *logits, int R, int V, float temperature, const float *u,
                   int32_t *tokens, void *ws, size_t ws_bytes, int32_t *d_status,
                   df_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Failure-detection test hook (no counterpart on the pages). Every barrier wait of the
 * tensor-core projection kernel is bounded: after the limit it raises the CTA's abort flag,
 * writes DF_ETIMEOUT to the call's status word, lets every role leave, waits (bounded) for the
 * TMA loads it issued and frees its tensor memory, so the context stays usable. This call sets,
 * for the projections launched after it from any thread, the limit in SM cycles (0 restores the
 * default of ~2 s) and, with withhold_first != 0, makes every CTA's TMA producer skip the load of
 * its first pipeline stage, so the MMA warp's wait runs out. Outputs of calls made while
 * withholding are meaningless. Returns DF_EINVAL for a negative limit, or for withholding without
 * a positive limit. Reset with (0, 0).
 * ---------------------------------------------------------------------------------------- */
int df_test_wait_hook(long long wait_cycles, int withhold_first);

/* ------------------------------------------------------------------------------------------
 * KV rollback (qwen35_orchestrator.rs step 8, `rollback_kv`): seq_len[b] -= n[b]. Cache rows
 * are not touched. If n[b] < 0 or n[b] > seq_len[b], seq_len[b] is left unchanged and
 * DF_ECAPACITY is written to d_status.
 * ---------------------------------------------------------------------------------------- */
int kv_rollback(int32_t *seq_len, const int32_t *n, int B, int32_t *d_status,
                df_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Whole DFlash draft round on the device: the benchmark unit. Steps: block build
 * [last_token, mask x K] + embed gather, dflash_block_forward, lm_head argmax of every block
 * row, drafts = argmax[1..K], accept walk against target_argmax, rollback of the verifier's
 * KV length target_seq_len[b] by K - accept_count[b].
 *   last_token      device int32 [B]
 *   target_argmax   device int32 [B, K+1]
 *   target_seq_len  device int32 [B] in/out (verifier cache length after its K+1 positions)
 *   argmax_out      device int32 [B, K+1] out (position 0 = the drafter's own guess for
 *                   last_token's successor; 1..K = the drafts)
 *   committed, n_committed, accept_count, hit_eos, rollback: as accept_prefix_argmax
 * The drafter cache advances by n_new[b] exactly as in dflash_block_forward.
 * ---------------------------------------------------------------------------------------- */
int df_draft_round(const df_dflash_config *cfg, const df_dflash_weights *w,
                   const df_kv_cache *cache, const int32_t *last_token,
                   const float *target_hidden_new, const int32_t *n_new, int n_new_max, int B,
                   int K, const int32_t *target_argmax, const int32_t *eos, int n_eos,
                   int32_t *target_seq_len, int32_t *argmax_out, int32_t *committed,
                   int32_t *n_committed, int32_t *accept_count, int32_t *hit_eos,
                   int32_t *rollback, void *ws, size_t ws_bytes, int32_t *d_status,
                   df_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Non-greedy DFlash draft round (temperature T > 0): the drafter forward of df_draft_round, the
 * lm_head logits of every block row, draft i = 1..K drawn from softmax(logits_i / T)
 * (sample_softmax's rule) with u_draft[b, i-1], then accept_stochastic against the verifier's
 * logits and the rollback of target_seq_len by K - accept_count (qwen35_orchestrator.rs, module
 * doc "Non-greedy (Metropolis-Hastings) is out of scope here": the stochastic acceptance takes
 * the place of the greedy walk at step 11).
 *   target_logits   device F32 [B, K+1, V]: verifier logits at positions 0..K (16-byte aligned)
 *   u_draft, u_accept device F32 [B, K]; u_sample device F32 [B]: uniforms in [0, 1)
 *   logits_out      device F32 [B, K+1, V] out: the drafter's logits of every block row
 *                   (row 0 = last_token's position; rows 1..K are the drafts' q)
 *   drafts_out      device int32 [B, K] out: the sampled drafts
 *   committed, n_committed, accept_count, hit_eos, rollback, target_seq_len: as df_draft_round
 * 1 <= K <= 64; V a multiple of 4. The drafter cache advances as in df_draft_round.
 * ---------------------------------------------------------------------------------------- */
size_t df_draft_round_stochastic_workspace_bytes(const df_dflash_config *cfg, int B, int K,
                                                 int n_new_max);
int df_draft_round_stochastic(const df_dflash_config *cfg, const df_dflash_weights *w,
                              const df_kv_cache *cache, const int32_t *last_token,
                              const float *target_hidden_new, const int32_t *n_new,
                              int n_new_max, int B, int K, const float *target_logits,
                              float temperature, const float *u_draft, const float *u_accept,
                              const float *u_sample, const int32_t *eos, int n_eos,
                              int32_t *target_seq_len, float *logits_out, int32_t *drafts_out,
                              int32_t *committed, int32_t *n_committed, int32_t *accept_count,
                              int32_t *hit_eos, int32_t *rollback, void *ws, size_t ws_bytes,
                              int32_t *d_status, df_stream_t stream);

/* Bytes of the host-buffer round's staging area (device), in addition to the round's own. */
size_t df_draft_round_host_workspace_bytes(const df_dflash_config *cfg, int B, int K,
                                           int n_new_max, int n_eos);

/*
 * df_draft_round_host — the same round with HOST inputs and outputs: copies last_token,
 * target_hidden_new, n_new, target_argmax, eos and target_seq_len into device staging carved
 * from `ws`, runs df_draft_round, copies the results back, and synchronises `stream`.
 * Host buffers should be pinned for asynchronous copies. Outputs (host): target_seq_len
 * (in/out), argmax_out [B, K+1], committed [B, K+1], n_committed, accept_count, hit_eos,
 * rollback [B], status (the device status word). ws must hold
 * df_dflash_workspace_bytes(cfg, B, K+1, n_new_max) + df_draft_round_host_workspace_bytes().
 * When every host buffer is page-locked, the copies and kernels of the call are captured once
 * into a CUDA graph cached under all of the call's arguments (pointers, sizes, stream and the
 * weight and cache pointers they reach; up to 16 argument sets, least recently used dropped),
 * and a repeated call launches that graph: the buffers' contents are read at each launch, so
 * only their addresses are fixed. The cache holds graphs, not data; pageable buffers take the
 * stream path. Not thread-safe against a concurrent call on the same buffers (as any stream
 * use of them).
 */
int df_draft_round_host(const df_dflash_config *cfg, const df_dflash_weights *w,
                        const df_kv_cache *cache, const int32_t *last_token,
                        const float *target_hidden_new, const int32_t *n_new, int n_new_max,
                        int B, int K, const int32_t *target_argmax, const int32_t *eos,
                        int n_eos, int32_t *target_seq_len, int32_t *argmax_out,
                        int32_t *committed, int32_t *n_committed, int32_t *accept_count,
                        int32_t *hit_eos, int32_t *rollback, int32_t *status, void *ws,
                        size_t ws_bytes, df_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Multi-round generate loop on the device (qwen35_orchestrator.rs, `dispatch_qwen35_dflash_
 * generate`, "Multi-round loop (Option A)", steps 1-10 and the final truncation) with a
 * synthetic verifier standing in for the target model. Per round, for every sequence still
 * running: n_new = prior_len - drafter cache length new context rows, gathered from the
 * captured verifier states as the concatenation of the drafter's target layers
 * (`extract_drafter_concat`); the draft round (df_draft_round's steps); the verifier's greedy
 * tokens for [last_token, drafts]; the greedy accept walk; the committed tokens appended and
 * last_token updated; the sequence stops on EOS, when out_len - prompt_len >= max_new_tokens
 * (then out_len is truncated to prompt_len + max_new_tokens) or when the next round would not
 * fit max_len; otherwise the first n_committed verify positions are appended to the captured
 * prefix (`append_capture_positions`). Before the first round a sequence whose last token is an
 * EOS id, or any sequence when max_new_tokens == 0, is done (the page returns prompt + first
 * token). The whole loop is one CUDA graph: a while node repeats the round until no sequence is
 * running or max_rounds rounds have run; no host synchronisation happens in between.
 * ---------------------------------------------------------------------------------------- */
typedef struct {
    const int32_t *ref;     /* device [B, max_len]: the verifier's greedy token after position p
                               is ref[b, p + 1] ... */
    const uint8_t *agree;   /* ... unless agree[b, p] != 0 (device [B, max_len], or NULL) for a
                               drafted position p < p0 + K of a verify starting at p0, where it
                               is the draft itself */
    const float *table;     /* device [B, n_comb, max_len, H]: the verifier's captured hidden
                               state of capture layer c at position p */
    int32_t n_comb;         /* capture layers */
    int32_t sel[16];        /* the drafter's target layer l is capture layer sel[l] */
    int32_t max_len;        /* positions per sequence in ref, agree, table, prior_cap, out */
} df_synthetic_verifier;

/* Workspace: the round's (df_dflash_workspace_bytes(cfg, B, K+1, n_new_max)) plus the loop's
 * round scratch; allocate it zeroed. 0 on invalid arguments (n_new_max < K + 1). */
size_t df_generate_workspace_bytes(const df_dflash_config *cfg, int B, int K, int n_new_max);

/*   prior_cap      device F32 [B, n_comb, max_len, H] in/out: captured verifier states of the
 *                  committed prefix, positions [0, prior_len[b])
 *   prior_len      device int32 [B] in/out: must equal out_len - 1 on entry
 *   out_tokens     device int32 [B, max_len] in/out: prompt + first token on entry (out_len[b]
 *                  of them), the generated tokens appended
 *   out_len        device int32 [B] in/out
 *   prompt_len     device int32 [B]
 *   rounds         device int32 [B] out: rounds each sequence ran
 *   accept_hist    device int32 [max_rounds, B] out (or NULL): accept count of round r, for the
 *                  sequences that ran it
 *   n_new_max      >= K + 1 and >= the first round's prior_len - cache length (the drafter's
 *                  initial catch-up); at most cache->cap
 * The drafter cache advances as in df_draft_round. The first call with a given set of
 * arguments builds and keeps the loop graph; later calls with the same arguments relaunch it. */
int df_generate(const df_dflash_config *cfg, const df_dflash_weights *w, const df_kv_cache *cache,
                const df_synthetic_verifier *v, float *prior_cap, int32_t *prior_len,
                int32_t *out_tokens, int32_t *out_len, const int32_t *prompt_len,
                int max_new_tokens, int max_rounds, int B, int K, int n_new_max,
                const int32_t *eos, int n_eos, int32_t *rounds, int32_t *accept_hist, void *ws,
                size_t ws_bytes, int32_t *d_status, df_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * MTP (NextN) draft step, mtp.rs `MtpWeights::forward_draft_with_hidden`, chained n_steps
 * times (the returned hidden feeds the next step with the embedding of the step's argmax).
 * ---------------------------------------------------------------------------------------- */
typedef struct {
    int32_t hidden, n_q_heads, n_kv_heads, head_dim, vocab;
    int32_t intermediate;   /* dense SwiGLU I (0 when MoE) */
    int32_t n_experts;      /* 0 = dense FFN */
    int32_t top_k;          /* experts chosen per token (MoE) */
    int32_t expert_inter;   /* per-expert SwiGLU intermediate (MoE) */
    int32_t shared_inter;   /* shared-expert SwiGLU intermediate (MoE) */
    int32_t rotary_dim;     /* 0 = head_dim */
    float rms_eps, rope_theta;
} df_mtp_config;

typedef struct {
    const float *enorm, *hnorm;             /* [H] F32 (eps fixed at 1e-6) */
    const uint16_t *eh_embed, *eh_hidden;   /* [H, H] BF16 each (eh_proj halves) */
    const float *attn_norm, *post_attn_norm, *q_norm, *k_norm;   /* F32 */
    const uint16_t *wq, *wk, *wv;           /* [n_q*d, H], [n_kv*d, H], [n_kv*d, H] */
    const uint16_t *w_gate;                 /* [n_q*d, H] or NULL (no output gate) */
    const uint16_t *wo;                     /* [H, n_q*d] */
    const float *shared_head_norm;          /* [H] */
    const uint16_t *embed, *lm_head;        /* [V, H] */
    /* dense FFN */
    const uint16_t *w_gate_mlp, *w_up, *w_down;   /* [I, H], [I, H], [H, I] */
    /* MoE FFN */
    const uint16_t *router;                 /* [E, H] */
    const uint16_t *exp_gate, *exp_up;      /* [E, Ie, H] */
    const uint16_t *exp_down;               /* [E, H, Ie] */
    const uint16_t *sh_gate_mlp, *sh_up;    /* [Is, H] */
    const uint16_t *sh_down;                /* [H, Is] */
    const uint16_t *sh_expert_gate;         /* [1, H]: sigmoid gate of the shared expert */
    const void *tiled;                      /* NULL, or the tiled copy by df_mtp_tile_weights */
} df_mtp_weights;

/* Tiled weights of an MTP block (the layout of the DFlash tiled weights above): eh_proj (its two
 * halves as one K range), QKV with the output gate rows, O, the dense gate/up (paired) and down
 * when there are no experts, and the lm_head. The experts and the router stay row-major.
 * df_mtp_tiled_bytes: 0 on an invalid config or weights. df_mtp_tile_weights: fills `tiled`
 * (device, 1024-byte aligned, >= df_mtp_tiled_bytes) on `stream`; set w->tiled = tiled and
 * synchronise before the first call that reads it. DF_EWORKSPACE / DF_EINVAL as above. */
size_t df_mtp_tiled_bytes(const df_mtp_config *cfg, const df_mtp_weights *w);
int df_mtp_tile_weights(const df_mtp_config *cfg, const df_mtp_weights *w, void *tiled,
                        size_t tiled_bytes, df_stream_t stream);

size_t df_mtp_workspace_bytes(const df_mtp_config *cfg, int B);

/*   cache        one-layer KV slot (n_layers = 1); step s of sequence b writes row
 *                seq_len[b] + s and attends over rows [0, seq_len[b] + s]; seq_len advances
 *                by n_steps
 *   prev_hidden  device F32 [B, H]: hidden state of the verifier for the previous token
 *   token        device int32 [B]: the just-accepted token (its embedding is embed[token])
 *   hidden_out   device F32 [n_steps, B, H] out: pre-head hidden of every step
 *   argmax_out   device int32 [n_steps, B] out: the draft token of every step
 *   logits_out   device F32 [B, V] or NULL: dense logits of the last step, only if asked */
int mtp_forward_draft(const df_mtp_config *cfg, const df_mtp_weights *w,
                      const df_kv_cache *cache, const float *prev_hidden, const int32_t *token,
                      int B, int n_steps, float *hidden_out, int32_t *argmax_out,
                      float *logits_out, void *ws, size_t ws_bytes, int32_t *d_status,
                      df_stream_t stream);

/* The MTP K=1 path at temperature T > 0 (qwen35_orchestrator.rs module doc, "Non-greedy
 * (Metropolis-Hastings) is out of scope here": the stochastic acceptance is wired through the
 * MTP K=1 path): as mtp_forward_draft, but every step's token is drawn from
 * softmax(logits / T) with u_draft[s, b] (sample_softmax's rule) and fed to the next step.
 *   temperature  > 0 (DF_EINVAL otherwise)
 *   u_draft      device F32 [n_steps, B] uniforms in [0, 1)
 *   draft_out    device int32 [n_steps, B] out: the drawn tokens
 *   logits_out   device F32 [n_steps, B, V] out (required): every step's logits, the q of the
 *                accept step; V a multiple of 4
 * Workspace: df_mtp_workspace_bytes. */
int mtp_forward_draft_sampled(const df_mtp_config *cfg, const df_mtp_weights *w,
                              const df_kv_cache *cache, const float *prev_hidden,
                              const int32_t *token, int B, int n_steps, float temperature,
                              const float *u_draft, float *hidden_out, int32_t *draft_out,
                              float *logits_out, void *ws, size_t ws_bytes, int32_t *d_status,
                              df_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Mixture-of-experts FFN of the MTP block on its own (mtp.rs `MtpFfnWeightsGpu::Moe`; the
 * same kernels run inside mtp_forward_draft when cfg->n_experts > 0). The page names the
 * router, the experts and the shared expert with its scalar gate; the routing rule is read as
 *   p = softmax(x . router^T) over all E experts; sel = the top_k largest p (the lower expert
 *   index first on equal values), largest first; w_j = p[sel_j] / sum_i p[sel_i]
 *   out = sum_j w_j * SwiGLU_{sel_j}(x) + sigmoid(x . sh_expert_gate) * SwiGLU_shared(x)
 * with SwiGLU_e(x) = down_e( silu(gate_e x) * (up_e x) ).
 * ---------------------------------------------------------------------------------------- */
/* Workspace of df_moe_ffn for T rows; 0 when cfg has no experts or T is outside 1..16. */
size_t df_moe_workspace_bytes(const df_mtp_config *cfg, int T);

/*   cfg          n_experts <= 512, top_k <= 16; hidden, expert_inter and shared_inter
 *                multiples of 8 (attention fields are checked but unused)
 *   w            only router, exp_*, sh_gate_mlp, sh_up, sh_down and sh_expert_gate are read
 *   x            device F32 [T, H], 16-byte aligned: the FFN input (already normalised)
 *   T            1..16 rows
 *   out          device F32 [T, H] out: the FFN output (no residual)
 *   expert_ids   device int32 [T, top_k] out, or NULL: the chosen experts, largest weight first
 *   expert_w     device F32 [T, top_k + 1] out, or NULL: the renormalised weights, then the
 *                shared expert's sigmoid gate
 * Errors: DF_ESHAPE for sizes outside the limits, DF_EINVAL for NULL pointers; a NaN router
 * logit sets *d_status to DF_EINVAL. */
int df_moe_ffn(const df_mtp_config *cfg, const df_mtp_weights *w, const float *x, int T,
               float *out, int32_t *expert_ids, float *expert_w, void *ws, size_t ws_bytes,
               int32_t *d_status, df_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H */
