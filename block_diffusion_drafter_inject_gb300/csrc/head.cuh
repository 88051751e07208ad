// Per-position top-k + logsumexp, candidate-path selector, greedy acceptance.
#pragma once
#include "common.cuh"

namespace dflh {

// top-k works on 128-entry vocab tiles (the projection's weight tiles)
constexpr int kTopkMaxTiles = 8192;  // vocab <= 8192 * 128
inline int topk_tiles(int V) { return (V + 127) / 128; }

// ids / logp [rows][k]; stats: per row the (max, sum e^(z - max)) of each
// 128-entry tile [rows][topk_tiles(V)], or nullptr (formed from the logits)
int launch_topk(const float *logits, const float2 *stats, int rows, int V, int k, int32_t *ids,
                float *logp, cudaStream_t st);

template <typename S>
int launch_sel_gather(const S *E, const int32_t *anchor, const int32_t *topk_ids, int B, int K,
                      int k, int V, int D, S *rows, int *err, cudaStream_t st);

// U, Vp: reduced selector projections [B*R, r] fp32 (R = 1 + (K-1)*k rows per
// request: anchor, then candidates by (position, rank)); or, with tab non-null,
// the projections of every vocabulary row [2][V][r] fp32, read by token (the
// anchor and the candidates; tokens out of range raise a status bit in err and
// are clamped).  pair: B*(K-1)*k*k scratch; tickets: B ints, zero on entry and on exit
int launch_viterbi(const float *U, const float *Vp, const int32_t *topk_ids,
                   const float *topk_logp, int B, int K, int k, int r, float *pair, int *tickets,
                   int32_t *path, float *score, const float *tab, int V, const int32_t *anchor,
                   int *err, cudaStream_t st);

constexpr int kArgmaxChunk = 8192;
inline int argmax_chunks(int V) { return (V + kArgmaxChunk - 1) / kArgmaxChunk; }
// partial: B*K*chunks*2 words
int launch_accept(const int32_t *path, const void *logits, int dtype, int B, int K, int V,
                  float *partial, int32_t *accept_len, int32_t *tokens, cudaStream_t st);

// Temperature-1 sampling walk over the pair scores (projections as for
// launch_viterbi); uniforms [B][K-1]; path [B][K-1]; path_q [B][K-1][k]: the
// proposal over position t's candidates given the token drawn before it.
int launch_sample_walk(const float *U, const float *Vp, const int32_t *topk_ids,
                       const float *topk_logp, int B, int K, int k, int r, const float *tab, int V,
                       const int32_t *anchor, const float *uniforms, int32_t *path, float *path_q,
                       int *err, cudaStream_t st);

// Greedy walk over the pair scores with the context gate: gate [B*(K-1)][r]
// pre-activations (sigmoid applied here), or nullptr; score [B].
int launch_greedy_walk(const float *U, const float *Vp, const int32_t *topk_ids,
                       const float *topk_logp, int B, int K, int k, int r, const float *tab, int V,
                       const int32_t *anchor, const float *gate, int32_t *path, float *score,
                       int *err, cudaStream_t st);

// Speculative rejection sampling; uniforms [B][K][2]; scratch of
// accept_sample_floats(B, K, V) floats.
size_t accept_sample_floats(int B, int K, int V);
int launch_accept_sample(const int32_t *path, const int32_t *topk_ids, const float *path_q,
                         const void *logits, int dtype, int B, int K, int V, int k,
                         const float *uniforms, float *scratch, int32_t *accept_len,
                         int32_t *tokens, cudaStream_t st);

}  // namespace dflh
