// Row-wise kernels of the draft pass and injection.  Templates over the
// storage dtype S (float or bf16); arithmetic is fp32.
#pragma once
#include "common.cuh"

namespace dflh {

struct LayerPtrs {
  const void *p[DFLASH_MAX_LAYERS];
};

// RoPE frequencies theta^(-2i/d), i < d/2, computed once on the host in fp64.
struct RopeTable {
  double inv_freq[64];
  int enabled;
};
RopeTable rope_table(float theta, int head_dim);

// Both also write the RoPE (cos, sin) row of each row's absolute position
// (embed: ctx_len[b] + slot; rows_norm: pos[row], skipped when rope_cs is null).
// embed with ssq_out: row r's sum of squares to ssq_out[r] (one partial a row,
// the form the fused pre-sublayer conv reads).
template <typename S>
int launch_embed_norm(const S *E, const int32_t *anchor, int mask_id, int V, int B, int K, int D,
                      const S *gain, float eps, float *x, S *un, int *err, const int32_t *ctx_len,
                      const RopeTable &rope, int half, float2 *rope_cs, cudaStream_t st,
                      float *ssq_out = nullptr);
// Cache place of each injected row (rows_norm, optional): slot[n] = element
// offset of (page, position within the page) for head 0, feature 0 inside one
// layer of the caches [L][num_pages][Hkv][P][dh], or -1 (and a status bit) when
// req[n], pos[n] or the page fails the checks.
struct CacheSlots {
  const int32_t *req = nullptr, *table = nullptr;
  int max_pages = 0, num_rows = 0, num_pages = 0, P = 0, Hkv = 0, dh = 0;
  long long *slot = nullptr;
  int *err = nullptr;
};
template <typename S>
int launch_rows_norm(const S *in, int rows, int cols, const S *gain, float eps, S *out,
                     const int32_t *pos, const RopeTable &rope, int half, float2 *rope_cs,
                     cudaStream_t st, const CacheSlots &slots = CacheSlots());
// gate: the conv's gate linear as nsl K slices, fp32 [nsl][rows][2D/group],
// summed by the conv in slice order
template <typename S>
int launch_conv_pre(const S *un, const float *gate, int nsl, int rows, int K, int D, int group,
                    const S *base, S *ub, cudaStream_t st);
template <typename S>
int launch_conv_post_norm(const float *rf, const float *gate, int nsl, int rows, int K, int D,
                          int group, const S *base, float *x, const S *gain, float eps, S *un,
                          S *zf, cudaStream_t st);
// Two-tap conv with its gate linear fused, for T <= kGconvMaxT block rows
// (one launch per conv).  PRE: ub = conv(u) with u = R(rmsnorm(x, gain)) formed
// here from the fp32 residual x.  POST: x += conv(rf) with the gates of gin.
constexpr int kGconvMaxT = 16;
// whether the fused conv takes T rows of width D with channel groups of `group`
bool gconv_fits(int T, int D, int group, int dtype);
// Row sums of squares handed from the kernel that updates the residual stream
// to the next PRE conv: the POST conv (bf16) writes one partial per CTA and row
// into [slots][16] floats; 0 when this shape does not write them.
int gconv_ssq_slots(int T, int D, int group, int dtype);
// PRE with ssq_in: the n_ssq partials [n_ssq][16] of each row's sum of squares
// (from the POST conv or the embedding kernel) replace the cluster's own.
template <typename S>
int launch_gconv_pre(const float *x, int T, int K, int D, int group, const S *G, const S *base,
                     const S *gain, float eps, S *ub, cudaStream_t st,
                     const float *ssq_in = nullptr, int n_ssq = 0);
// POST with ssq_out (when gconv_ssq_slots > 0): writes the partials described above.
template <typename S>
int launch_gconv_post(const float *rf, const S *gin, int T, int K, int D, int group, const S *G,
                      const S *base, float *x, cudaStream_t st, float *ssq_out = nullptr);
// zf: RMSNorm of the rows of slots 1..K-1, written compactly [B*(K-1), D].
template <typename S>
int launch_final_norm(const float *x, int B, int K, int D, const S *gain, float eps, S *zf,
                      cudaStream_t st);
template <typename S>
int launch_qkv_post(const float *qkv, int rows, int K, int Hq, int Hkv, int dh, const S *qn,
                    const S *kn, const float2 *rope_cs, float eps, S *qb, S *kb, S *vb,
                    cudaStream_t st);
template <typename S>
int launch_inject_store(const float *kvf, int N, int L, int Hkv, int dh, LayerPtrs knorm,
                        const int32_t *req, const int32_t *pos, const int32_t *page_table,
                        int num_rows, int max_pages, int num_pages, int page_size,
                        const float2 *rope_cs, float eps, S *kc, S *vc, int *err,
                        cudaStream_t st);

}  // namespace dflh
