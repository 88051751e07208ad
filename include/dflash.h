/*
 * dflash.h - C ABI of the DFlash 2 draft cycle on one GPU (sm_103a).
 *
 * One draft cycle, as the serving sequence on the DFlash 2 Architecture page
 * ("One Cycle, Step by Step") orders it:
 *   1. dflash_inject_context   target hidden states -> every draft layer's K/V cache
 *   2. dflash_draft_block      one non-causal drafter pass over a block of K slots,
 *                              per-position top-k candidates
 *      dflash_draft_block_inject   1 and 2 in one pass (each layer's K/V
 *                              weights read once)
 *   3. dflash_select_path      one coherent candidate path (Viterbi over the lattice)
 *      dflash_sample_path      ... or a temperature-1 walk drawn from the same scores
 *   4. dflash_accept_greedy    longest prefix that matches the target's argmax + bonus
 *      dflash_accept_sample    ... or lossless speculative rejection sampling
 *
 * Conventions shared by every call
 *  - Every buffer belongs to the caller.  The library never allocates, frees or
 *    synchronises device memory, except dflash_read_device_status, which waits
 *    for the stream.  All pointers named "device" are device addresses.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL =
 *    the legacy default stream) and may be captured in a CUDA graph.
 *  - Return value: DFLASH_OK (0) or a negative DFLASH_ERR_* code for errors the
 *    host can see (NULL pointer, bad dimension, block size out of range,
 *    workspace too small, misaligned pointer, launch failure).  Nothing is
 *    launched when a host check fails.
 *  - Data-dependent errors (token id >= vocab, page id out of the pool, a
 *    position beyond the page table, a bounded wait that expired) are found on
 *    the device: the value is clamped, a bit is OR-ed into the sticky status
 *    word at the start of the workspace, and the call continues.  Read it with
 *    dflash_read_device_status.  Kernels never trap or assert.
 *  - Weights are row-major [out, in] (the nn.Linear layout), in the dtype of
 *    the config (norm gains and conv base kernels too).  Pointers passed to
 *    tensor-memory-accelerator loads (fc, wqkv, wo, w_gate_up, w_down, conv_w,
 *    lm_head, sel_pu, sel_pv, the workspace) must be 16-byte aligned.
 *  - The workspace must be zero-filled once before its first use (the status
 *    word lives at offset 0); after that it may be reused by any call of the
 *    same or smaller shape.  Calls that share a workspace must not overlap.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH_MAX_LAYERS 16
#define DFLASH_MAX_BLOCK 32   /* K, block slots (anchor + K-1 masks)            */
#define DFLASH_MAX_TOPK 32    /* candidates kept per position                   */

/* storage dtypes */
#define DFLASH_F32 0
#define DFLASH_BF16 1

/* host-side status codes */
#define DFLASH_OK 0
#define DFLASH_ERR_NULL (-1)       /* a required pointer is NULL                */
#define DFLASH_ERR_DIMS (-2)       /* a dimension breaks the shape rules        */
#define DFLASH_ERR_BLOCK (-3)      /* K outside 2..DFLASH_MAX_BLOCK, or B < 0   */
#define DFLASH_ERR_WORKSPACE (-4)  /* ws_bytes below dflash_workspace_bytes     */
#define DFLASH_ERR_DTYPE (-5)      /* unsupported dtype                         */
#define DFLASH_ERR_CUDA (-6)       /* a CUDA runtime/driver call failed         */
#define DFLASH_ERR_ALIGN (-7)      /* a pointer is not 16-byte aligned          */
#define DFLASH_ERR_DEVICE (-8)     /* no usable sm_103 device                   */

/* device-side sticky status bits (dflash_read_device_status) */
#define DFLASH_DEV_TOKEN_RANGE 1   /* a token id was outside [0, vocab)         */
#define DFLASH_DEV_PAGE_RANGE 2    /* a page id was outside [0, num_pages)      */
#define DFLASH_DEV_POS_RANGE 4     /* a position fell outside the page table    */
#define DFLASH_DEV_TIMEOUT 8       /* a bounded on-chip wait expired            */
#define DFLASH_DEV_REQ_RANGE 16    /* an inject request row was out of range    */

/* Drafter dimensions.  Shape rules (checked by every call):
 *   d_model, d_ff, n_taps*d_target, n_q_heads*head_dim multiples of 64;
 *   head_dim 64 or 128; n_q_heads a multiple of n_kv_heads;
 *   d_model a multiple of conv_group; 1 <= top_k <= 32, top_k <= vocab,
 *   vocab <= 1048576 (8192 vocab tiles of 128 entries for the top-k);
 *   sel_rank a multiple of 16 and <= 1024; window >= 1; page_size >= 1;
 *   1 <= n_layers <= DFLASH_MAX_LAYERS; 0 <= mask_token_id < vocab.         */
typedef struct dflash_config {
  int32_t d_model;      /* D, draft width                                   */
  int32_t n_layers;     /* L                                                */
  int32_t n_q_heads;    /* Hq                                               */
  int32_t n_kv_heads;   /* Hkv                                              */
  int32_t head_dim;     /* d                                                */
  int32_t d_ff;         /* F, SwiGLU width                                  */
  int32_t vocab;        /* V                                                */
  int32_t n_taps;       /* tapped target layers                             */
  int32_t d_target;     /* target width per tap                             */
  int32_t window;       /* context keys read per pass (sliding window)      */
  int32_t page_size;    /* tokens per KV page                               */
  int32_t top_k;        /* candidates per position                          */
  int32_t sel_rank;     /* selector rank r                                  */
  int32_t conv_group;   /* channels sharing one conv gate correction        */
  int32_t mask_token_id;
  int32_t dtype;        /* DFLASH_F32 or DFLASH_BF16                        */
  float rms_eps;        /* RMSNorm epsilon                                  */
  float rope_theta;     /* RoPE base; 0 disables RoPE                       */
  int32_t weight_bits;  /* 0: every weight in the storage dtype; 4: the
                           projections fc, wqkv, wo, w_gate_up, w_down and
                           lm_head in the 4-bit format below (bf16 storage) */
} dflash_config;

/* 4-bit weights (README mirror, MLX section: the drafter runs with 4-bit
 * weights).  A matrix W [N, K] (K a multiple of 64) is kept as 4-bit codes q
 * and, per row and group of 64 consecutive input features, a bf16 scale s and
 * bias b; the products use w = bf16(s*q + b) (s*q + b rounded once, to
 * nearest even), activations stay bf16.
 *   data   device, 16-byte aligned: ceil(N/128)*2 row blocks of 64 rows, each
 *          cut into K/64 records of 2304 bytes, records ordered (row block,
 *          group): record (r, g) is the codes of rows 64r..64r+63 for input
 *          features 64g..64g+63 (64 rows x 32 bytes), then their (scale, bias)
 *          words (64 x 4 bytes: bf16 scale in the low 16 bits, bf16 bias in
 *          the high 16 bits).  In a row's 32 bytes, the 32-bit little-endian
 *          word holding features 64g+8j..64g+8j+7 keeps their codes, from the
 *          least significant nibble up, in the order 8j, 8j+2, 8j+4, 8j+6,
 *          8j+1, 8j+3, 8j+5, 8j+7.  Rows past N (padding) may hold anything.
 * One k-block of a 128-row weight tile is then two contiguous records. */
typedef struct dflash_q4 {
  const void *data;
} dflash_q4;

/* One draft layer.  All device pointers, dtype of the config. */
typedef struct dflash_layer_weights {
  const void *attn_norm;   /* [D]   pre-attention RMSNorm gain                      */
  const void *mlp_norm;    /* [D]   pre-MLP RMSNorm gain                            */
  const void *wqkv;        /* [(Hq+2Hkv)*d, D] rows = [Wq; Wk; Wv]                  */
  const void *wo;          /* [D, Hq*d]                                             */
  const void *q_norm;      /* [d]   per-head RMSNorm gain on q                      */
  const void *k_norm;      /* [d]   per-head RMSNorm gain on k (block and injected) */
  const void *w_gate_up;   /* [2F, D] rows = [Wgate; Wup]                           */
  const void *w_down;      /* [D, F]                                                */
  const void *conv_w[4];   /* [2D/conv_group, D] gate linear [G_a; G_b] of the four
                              two-tap convs: 0 before attention, 1 after attention,
                              2 before the MLP, 3 after the MLP                     */
  const void *conv_base[4];/* [2D] base kernels [base_a; base_b] of the same convs  */
  /* weight_bits == 4: the 4-bit forms of wqkv, wo, w_gate_up and w_down (their
   * storage-dtype pointers above are then unused and may be NULL) */
  dflash_q4 wqkv_q4, wo_q4, w_gate_up_q4, w_down_q4;
} dflash_layer_weights;

typedef struct dflash_weights {
  const void *fc_norm;     /* [n_taps*d_target] RMSNorm gain on the concatenated taps */
  const void *fc;          /* [D, n_taps*d_target] injection projection              */
  const void *embed;       /* [V, D] token embeddings                                 */
  const void *lm_head;     /* [V, D]                                                  */
  const void *final_norm;  /* [D]                                                     */
  const void *sel_pu;      /* [r, D] selector projection of the predecessor token     */
  const void *sel_pv;      /* [r, D] selector projection of the successor token       */
  dflash_layer_weights layer[DFLASH_MAX_LAYERS];
  /* optional: f32 [2][V][r] = (P_u e_v, P_v e_v) for every vocabulary row v, as
   * written by dflash_prepare_selector; NULL: dflash_select_path gathers the
   * candidates' embedding rows and projects them on every call */
  const float *sel_table;
  /* optional: [r, D] W_H of the context gate H(h) = sigmoid(W_H h) of the
   * gated selector (dflash_select_greedy); unused by the other calls */
  const void *sel_gate;
  /* weight_bits == 4: the 4-bit forms of fc and lm_head (fc and lm_head above
   * then unused) */
  dflash_q4 fc_q4, lm_head_q4;
} dflash_weights;

/* Paged per-layer draft KV cache.
 * k, v: device, each [L][num_pages][Hkv][page_size][d] in the config dtype.
 * page_table: device int32 [num_rows][max_pages_per_req]; row b serves request
 *   b of a draft call and request row req[n] of an inject call; absolute
 *   position p of that request lives in page page_table[row][p / page_size],
 *   slot p % page_size.                                                        */
typedef struct dflash_kv {
  void *k;
  void *v;
  const int32_t *page_table;
  int32_t num_pages;
  int32_t max_pages_per_req;
  int32_t num_rows;
} dflash_kv;

/* Bytes of workspace needed by every call below for up to B requests, block
 * size K and up to max_inject_tokens tokens per inject call.  Returns 0 when
 * the config or sizes are invalid. */
size_t dflash_workspace_bytes(const dflash_config *cfg, int32_t B, int32_t K,
                              int32_t max_inject_tokens);

/* Target-KV injection (KV-injection post, "Persistent Conditioning Through
 * Target KV Injection"; Architecture page, Component Breakdown, "KV injection
 * path", and "Internals Worth Knowing": immediate projection into draft KV,
 * norm + RoPE post-processing).  For each token n:
 *   c = W_fc RMSNorm_{fc_norm}(target_hidden[n])
 *   for every layer l: K = RoPE(pos[n], RMSNorm_{k_norm,l}(W_k,l c)) per head,
 *                      V = W_v,l c
 * stored at request row req[n], absolute position pos[n].
 *   target_hidden  device [N, n_taps*d_target], config dtype, row-major
 *   req, pos       device int32 [N]
 *   N              0 (no-op) .. max_inject_tokens of the workspace            */
int dflash_inject_context(const dflash_config *cfg, const dflash_weights *w,
                          const dflash_kv *kv, const void *target_hidden,
                          const int32_t *req, const int32_t *pos, int32_t N,
                          void *ws, size_t ws_bytes, void *stream);

/* One drafter pass over B blocks of K slots (Architecture page, Component
 * Breakdown: block attention mask, 5-layer backbone with sliding window,
 * shared lm_head, top-16; "Problem 2": two-tap dynamic convs).  Slot 0 of
 * request b holds anchor[b] at absolute position ctx_len[b]; slots 1..K-1
 * hold mask_token_id at positions ctx_len[b]+i.  Attention keys = the last
 * min(window, ctx_len[b]) injected positions plus all K block slots (no mask
 * inside the block).  Block K/V are not written to the cache.
 *   anchor, ctx_len  device int32 [B]
 *   topk_ids         device int32 [B, K-1, top_k]   out, larger logit first
 *   topk_logp        device f32   [B, K-1, top_k]   out, logit - logsumexp
 *   logits_opt       device f32   [B, K-1, V] out, or NULL                     */
int dflash_draft_block(const dflash_config *cfg, const dflash_weights *w,
                       const dflash_kv *kv, const int32_t *anchor,
                       const int32_t *ctx_len, int32_t B, int32_t K,
                       int32_t *topk_ids, float *topk_logp, float *logits_opt,
                       void *ws, size_t ws_bytes, void *stream);

/* Injection and drafter pass in one call: the same results as
 * dflash_inject_context(target_hidden, req, pos, N) followed by
 * dflash_draft_block(anchor, ctx_len, B, K), with the new rows' K/V
 * projections done inside each layer's QKV projection of the pass, so that
 * every layer's K/V weights are read once per cycle instead of twice
 * (Architecture page, "Internals Worth Knowing": the accepted tokens'
 * target features are projected into draft KV right away, and the serving
 * loop overlaps that with the next draft).  Layer l's injected K/V are
 * written just before layer l's block attention reads the window, so rows
 * at positions below ctx_len[b] are attended in this same pass.
 *   target_hidden, req, pos, N   as dflash_inject_context (N <= the
 *                                workspace's max_inject_tokens; N = 0: the
 *                                pass alone); (req, pos) pairs must differ
 *   anchor .. logits_opt          as dflash_draft_block
 * B = 0 with N > 0 is the injection alone.  float32 storage runs the two
 * calls in sequence.  Device-side checks of req, pos and pages as
 * dflash_inject_context (the row is skipped, a status bit set).          */
int dflash_draft_block_inject(const dflash_config *cfg, const dflash_weights *w,
                              const dflash_kv *kv, const void *target_hidden,
                              const int32_t *req, const int32_t *pos, int32_t N,
                              const int32_t *anchor, const int32_t *ctx_len,
                              int32_t B, int32_t K, int32_t *topk_ids,
                              float *topk_logp, float *logits_opt, void *ws,
                              size_t ws_bytes, void *stream);

/* Candidate-path selector (Architecture page, "Problem 1", eq. S_t, in the
 * low-rank form (P_u e_a).(P_v e_b) with e = embedding rows, walked by
 * max-sum Viterbi from the anchor; the projections are read from
 * w->sel_table when it is set, else formed from the gathered rows):
 *   delta_1(j) = logp_1(j) + u(anchor).v(c_1j)
 *   delta_t(j) = logp_t(j) + max_i [delta_{t-1}(i) + u(c_{t-1,i}).v(c_tj)]
 * Ties go to the lower candidate rank.  B <= 16384 (else DFLASH_ERR_DIMS).
 *   anchor      device int32 [B]
 *   topk_ids    device int32 [B, K-1, top_k];  topk_logp device f32 [B, K-1, top_k]
 *   path        device int32 [B, K-1] out;     path_score device f32 [B] out     */
int dflash_select_path(const dflash_config *cfg, const dflash_weights *w,
                       const int32_t *anchor, const int32_t *topk_ids,
                       const float *topk_logp, int32_t B, int32_t K,
                       int32_t *path, float *path_score, void *ws, size_t ws_bytes,
                       void *stream);

/* Selector tables (Architecture page, "Problem 1": the pair score
 * (P_u e_a).(P_v e_b) is bilinear in fixed projections of vocabulary rows, so
 * both projections of every row can be formed once per weight set):
 *   table[0][v][:] = P_u e_v,   table[1][v][:] = P_v e_v    (f32 [2][V][r])
 * from w->embed, w->sel_pu, w->sel_pv, on `stream`.  The caller owns `table`
 * (2*V*r floats, 16-byte aligned; 311 MB for V = 151936, r = 256) and then
 * sets w->sel_table = table, after which dflash_select_path reads the
 * candidates' rows from it instead of projecting them.  ws: any workspace of
 * dflash_workspace_bytes (only its status word is used). */
int dflash_prepare_selector(const dflash_config *cfg, const dflash_weights *w, float *table,
                            void *ws, size_t ws_bytes, void *stream);

/* Greedy acceptance (Architecture page, "Speculative Decoding Context" and
 * "One Cycle, Step by Step"): row i of the target logits predicts the token
 * after slot i; draft token path[i] (slot i+1) is accepted while it equals
 * argmax(target_logits[b, i]) (lower id on ties; NaN counts as larger than
 * every number, so a row's first NaN is its argmax).  With m accepted drafts,
 *   accept_len[b] = m + 1,  tokens[b] = path[0..m-1], argmax(row m), -1 ...
 *   path           device int32 [B, K-1]
 *   target_logits  device [B, K, V] f32 (logits_dtype DFLASH_F32) or bf16
 * B * K <= 65535 (else DFLASH_ERR_DIMS).                                      */
int dflash_accept_greedy(const int32_t *path, const void *target_logits,
                         int32_t logits_dtype, int32_t B, int32_t K, int32_t V,
                         int32_t *accept_len, int32_t *tokens, void *ws,
                         size_t ws_bytes, void *stream);

/* Temperature-1 sampling walk (Architecture page, "Problem 1": only the final
 * walk over the precomputed pair scores is sequential, and sampling draws from
 * the same scores as the greedy walk).  From the anchor, position t draws one
 * of its top_k candidates with probability
 *   q_t(j) = softmax_j( logp_t(j) + u(prev) . v(c_tj) ),   prev = token drawn at t-1,
 * with u, v the selector projections (from w->sel_table when set, else formed
 * from the gathered embedding rows) and the inverse CDF over candidate ranks
 * (the smallest j whose running sum of q exceeds uniforms[b][t]).
 *   anchor     device int32 [B]
 *   topk_ids   device int32 [B, K-1, top_k];  topk_logp device f32 [B, K-1, top_k]
 *   uniforms   device f32 [B, K-1], values in [0, 1) (the caller's random numbers)
 *   path       device int32 [B, K-1] out: the drawn tokens
 *   path_q     device f32 [B, K-1, top_k] out: q_t over position t's candidates
 *              given the token drawn before it (the proposal dflash_accept_sample
 *              needs).  Workspace and errors as for dflash_select_path. */
int dflash_sample_path(const dflash_config *cfg, const dflash_weights *w, const int32_t *anchor,
                       const int32_t *topk_ids, const float *topk_logp, int32_t B, int32_t K,
                       const float *uniforms, int32_t *path, float *path_q, void *ws,
                       size_t ws_bytes, void *stream);

/* The pages' selector form with its greedy walk (Architecture page, "Problem
 * 1", eq. S_t, and "greedy follows the best successor"):
 *   S_t(a, b) = logp_t(b) + < (P_u e_a) * sigmoid(W_H h_t), P_v e_b >
 * with h_t the drafter's final-normed hidden state of draft position t (the
 * lm_head's input; dflash_draft_hidden gives the rows the last draft pass left
 * in the workspace) and W_H = w->sel_gate; from the anchor each position takes
 * the candidate of largest S_t given the token taken before it (the lower
 * rank on ties).  logp in place of the raw logit shifts every S_t by the same
 * amount per position, so the walk is the same.
 *   hidden      device [B, K-1, D] in the config dtype, 16-byte aligned
 *   path        device int32 [B, K-1] out;  path_score device f32 [B] out: sum
 *               of the chosen S_t.  Other arguments, workspace and errors as
 *               for dflash_select_path; w->sel_gate is required. */
int dflash_select_greedy(const dflash_config *cfg, const dflash_weights *w,
                         const int32_t *anchor, const int32_t *topk_ids, const float *topk_logp,
                         const void *hidden, int32_t B, int32_t K, int32_t *path,
                         float *path_score, void *ws, size_t ws_bytes, void *stream);

/* Device address, inside `ws`, of the final-normed hidden states [B*(K-1), D]
 * (config dtype; request b's draft position t at row b*(K-1) + t-1) that the
 * last dflash_draft_block on this workspace wrote, valid until the next call
 * that uses the workspace; NULL for invalid arguments.  Reads nothing on the
 * device. */
const void *dflash_draft_hidden(const dflash_config *cfg, int32_t B, int32_t K, const void *ws,
                                size_t ws_bytes);

/* Lossless speculative rejection sampling (Architecture page, "Speculative
 * Decoding Context": rejection sampling makes the scheme lossless; "Problem 1":
 * it restores the exact target distribution).  Row i of the target logits
 * gives p_i = softmax(row i) for the token after slot i.  Draft i (token
 * x = path[b][i], proposed with q_i: path_q over the candidates topk_ids[b][i],
 * zero for other tokens) is accepted while u0 * q_i(x) < p_i(x), with
 * u0 = uniforms[b][i][0].  At the first rejection the replacement is drawn from
 * max(0, p_i - q_i) with uniforms[b][i][1] and the block ends; when every draft
 * is accepted a bonus token is drawn from p_{K-1} with uniforms[b][K-1][1].
 * Draws take the smallest token id whose running sum (in id order) exceeds
 * u times the total.  The committed tokens follow the target's distribution
 * exactly, whatever the proposal.
 *   path           device int32 [B, K-1];  topk_ids device int32 [B, K-1, top_k]
 *   path_q         device f32 [B, K-1, top_k] (from dflash_sample_path)
 *   target_logits  device [B, K, V] f32 (logits_dtype DFLASH_F32) or bf16
 *   uniforms       device f32 [B, K, 2], values in [0, 1)
 *   accept_len     device int32 [B] out: committed tokens, 1..K
 *   tokens         device int32 [B, K] out: the committed tokens, then -1
 * B * K <= 65535 (else DFLASH_ERR_DIMS).  ws: any workspace of
 * dflash_workspace_bytes for these B and K (scratch after its fixed header:
 * B*K*ceil(V/8192)*16 bytes). */
int dflash_accept_sample(const int32_t *path, const int32_t *topk_ids, const float *path_q,
                         const void *target_logits, int32_t logits_dtype, int32_t B, int32_t K,
                         int32_t V, int32_t top_k, const float *uniforms, int32_t *accept_len,
                         int32_t *tokens, void *ws, size_t ws_bytes, void *stream);

/* Greedy acceptance for callers that cannot provide a workspace.  (The DFlash
 * pages have no counterpart: this is a deployment variant of
 * dflash_accept_greedy, with the same inputs, outputs and results.)
 * Some callers cannot allocate device memory where acceptance runs: a runtime
 * whose device memory is planned once at start-up and may not grow, a host
 * binding without a device allocator, or code that must not call cudaMalloc
 * at that point.  This entry point takes no workspace and allocates nothing:
 * its scratch (argmax partials) is a fixed 256 KiB array in the library's own
 * device memory, held by every GPU that loads the library until exit.
 *   Limit: B * K * ceil(V / 8192) <= 32768, else DFLASH_ERR_WORKSPACE
 *   (for V = 151936: B * K <= 1724).
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture.
 *   Every call shares the one array: calls that overlap on the GPU (different
 *   streams, or different host threads on one device) race and must be
 *   serialised by the caller.  Each call writes every partial it reads, so no
 *   clearing is needed between calls. */
int dflash_accept_greedy_noalloc(const int32_t *path, const void *target_logits,
                                 int32_t logits_dtype, int32_t B, int32_t K, int32_t V,
                                 int32_t *accept_len, int32_t *tokens, void *stream);

/* The projection GEMM every call above is built on (the drafter's dense
 * layers: nn.Linear without bias).  Slice s of `out` receives
 *   out[s][t][n] = sum over the s-th of `splits` equal K ranges of X[t][k] W[n][k]
 * so Y = X W^T = sum_s out[s].  bf16 operands run on the tcgen05 tensor cores
 * fed by TMA; f32 operands on CUDA cores.
 *   dtype   DFLASH_BF16 or DFLASH_F32 (both W and X)
 *   W       device [N_out, K_in] row-major, 16-byte aligned
 *   X       device [T, K_in] row-major, 16-byte aligned
 *   splits  >= 1 and dividing K_in/64 (dflash_linear_splits gives the
 *           library's own choice for the shape)
 *   out     device f32 [splits, T, N_out]
 * K_in must be a multiple of 64. */
int dflash_linear(int32_t dtype, const void *W, int32_t N_out, int32_t K_in, const void *X,
                  int32_t T, int32_t splits, float *out, void *stream);
/* The same product with W in the 4-bit format (w = bf16(s*q + b)) and bf16 X:
 * tensor-core GEMM whose weight tiles are dequantized into tensor memory.
 *   W       the records of W [N_out, K_in]; K_in a multiple of 64
 *   X, splits, out   as dflash_linear                                       */
int dflash_linear_q4(dflash_q4 W, int32_t N_out, int32_t K_in, const void *X, int32_t T,
                     int32_t splits, float *out, void *stream);
int32_t dflash_linear_splits(int32_t N_out, int32_t T, int32_t K_in);

/* Test hook for the failure-detection path of the projection GEMM (no
 * counterpart in the pages).  Every on-chip wait of the GEMM is bounded: when
 * one runs out, the kernel stops issuing, waits for the copies and matrix
 * operations it already issued, frees its tensor memory, sets
 * DFLASH_DEV_TIMEOUT in the status word and returns, leaving the context
 * usable.  This call runs dflash_linear's GEMM (bf16, one K slice:
 * out[t][n] = sum_k X[t][k] W[n][k]) with its status word at the start of
 * `ws`.  With stall_wait_us > 0 the tensor-core issuer first waits on a
 * barrier that nothing arrives on, with every wait of the launch limited to
 * stall_wait_us microseconds, so that the give-up path runs and out is not
 * written; with 0 it is an ordinary launch.  W [N_out, K_in], X [T, K_in]
 * bf16, 16-byte aligned; out f32 [T, N_out]; ws at least 256 bytes, zeroed. */
int dflash_test_linear_wait(const void *W, int32_t N_out, int32_t K_in, const void *X, int32_t T,
                            float *out, void *ws, size_t ws_bytes, uint32_t stall_wait_us,
                            void *stream);

/* Waits for `stream`, then returns the sticky device status bits (>= 0) of
 * the workspace, or a negative DFLASH_ERR_* code. */
int dflash_read_device_status(const void *ws, void *stream);
/* Clears the sticky device status word (asynchronous). */
int dflash_clear_device_status(void *ws, void *stream);
/* Static description of a status code (host or device bit). */
const char *dflash_status_string(int code);
/* Number of kernels the library launched on this thread since the last reset
 * (a counter kept by the host code; for measurement). */
int64_t dflash_launch_count(int reset);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
