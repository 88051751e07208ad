// Row-wise kernels: RMSNorm, two-tap conv gates, split-K reductions, SwiGLU,
// q/k head norm + RoPE, and the paged K/V store of injection.
//
// Each kernel sums the K slices of its producer GEMM in slice order, so a
// result does not depend on timing.  Every kernel signals its dependents
// early and waits for its predecessor before reading (programmatic launch).
#include <string.h>

#include <math.h>

#include "pointwise.cuh"

namespace dfl {

__device__ __forceinline__ float sigmoidf_(float t) { return 1.f / (1.f + expf(-t)); }

// x[r] = E[token of r]; un[r] = gain * x / rms(x).  Row r = b*K + i; slot 0 holds
// the anchor, the other slots the mask token.  Requires D % 8 == 0 and
// 16-byte aligned rows (8 elements per access).
// cos/sin of the rotate-half RoPE angles of absolute position `pos` for the
// d/2 frequencies: the angle pos * theta^(-2i/d) is formed and reduced modulo
// 2*pi in fp64, its sine and cosine taken in fp32.  Written once per row so
// that the kernels applying RoPE stay in fp32.
__device__ __forceinline__ void rope_row(float2 *__restrict__ cs, int pos,
                                         const dflh::RopeTable &rope, int half) {
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    float2 v = make_float2(1.f, 0.f);
    if (rope.enabled) {
      const double two_pi = 6.283185307179586476925286766559;
      const double a = (double)pos * rope.inv_freq[i];
      const float ar = (float)(a - two_pi * floor(a * (1.0 / two_pi)));
      sincosf(ar, &v.y, &v.x);
    }
    cs[i] = v;
  }
}

template <typename S>
__global__ void __launch_bounds__(512) k_embed_norm(const S *__restrict__ E,
                                                    const int32_t *__restrict__ anchor,
                                                    int mask_id, int V, int K, int D,
                                                    const S *__restrict__ gain, float eps,
                                                    float *__restrict__ x, S *__restrict__ un,
                                                    int *err, const int32_t *__restrict__ ctx_len,
                                                    const dflh::RopeTable rope, int half,
                                                    float2 *__restrict__ rope_cs) {
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  const int r = blockIdx.x, b = r / K, i = r % K;
  rope_row(rope_cs + (size_t)r * half, ctx_len[b] + i, rope, half);
  int tok = i == 0 ? anchor[b] : mask_id;
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) set_err(err, DFLASH_DEV_TOKEN_RANGE);
    tok = tok < 0 ? 0 : V - 1;
  }
  const S *e = E + (size_t)tok * D;
  float ss = 0.f;
  for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
    float v[8];
    load8(e + c, v);
    store8(x + (size_t)r * D + c, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += v[j] * v[j];
  }
  const float inv = rsqrtf(block_sum(ss, red) / D + eps);
  for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
    float v[8], g[8];
    load8(e + c, v);
    load8(gain + c, g);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = v[j] * inv * g[j];
    store8(un + (size_t)r * D + c, v);
  }
}

// out[r] = gain * in[r] / rms(in[r]); cols % 8 == 0, 16-byte aligned rows.
template <typename S>
__global__ void __launch_bounds__(1024) k_rows_norm(const S *__restrict__ in, int cols,
                                                    const S *__restrict__ gain, float eps,
                                                    S *__restrict__ out,
                                                    const int32_t *__restrict__ pos,
                                                    const dflh::RopeTable rope, int half,
                                                    float2 *__restrict__ rope_cs) {
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  if (rope_cs) rope_row(rope_cs + (size_t)blockIdx.x * half, pos[blockIdx.x], rope, half);
  const S *row = in + (size_t)blockIdx.x * cols;
  float ss = 0.f;
  for (int c = threadIdx.x * 8; c < cols; c += blockDim.x * 8) {
    float v[8];
    load8(row + c, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += v[j] * v[j];
  }
  const float inv = rsqrtf(block_sum(ss, red) / cols + eps);
  for (int c = threadIdx.x * 8; c < cols; c += blockDim.x * 8) {
    float v[8], g[8];
    load8(row + c, v);
    load8(gain + c, g);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = v[j] * inv * g[j];
    store8(out + (size_t)blockIdx.x * cols + c, v);
  }
}

// Pre-sublayer conv: ub[r] = a(r) * un[r] + b(r) * un[r-1] (zero before slot 0),
//   a_c(r) = sigmoid(base[c] + gate[r][c/g]),  b_c(r) = sigmoid(base[D+c] + gate[r][D/g + c/g])
// gate: the conv's gate linear of row r, fp32 [rows, 2D/g].  grid (rows, D/chunk).
template <typename S>
__global__ void __launch_bounds__(256) k_conv_pre(const S *__restrict__ un,
                                                  const float *__restrict__ gate, int K, int D,
                                                  int group, int chunk, const S *__restrict__ base,
                                                  S *__restrict__ ub) {
  pdl_launch();
  pdl_wait();
  const int r = blockIdx.x;
  const int c0 = blockIdx.y * chunk, c1 = min(D, c0 + chunk);
  const float *ga = gate + (size_t)r * (2 * D / group);
  const float *gb = ga + D / group;
  const bool first = (r % K) == 0;
  for (int c = c0 + threadIdx.x * 8; c < c1; c += blockDim.x * 8) {
    float cur[8], prev[8], ba[8], bb[8], y[8];
    load8(un + (size_t)r * D + c, cur);
    if (first) {
#pragma unroll
      for (int j = 0; j < 8; ++j) prev[j] = 0.f;
    } else {
      load8(un + (size_t)(r - 1) * D + c, prev);
    }
    load8(base + c, ba);
    load8(base + D + c, bb);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int g = (c + j) / group;
      const float a = sigmoidf_(ba[j] + ga[g]);
      const float b = sigmoidf_(bb[j] + gb[g]);
      y[j] = a * cur[j] + b * prev[j];
    }
    store8(ub + (size_t)r * D + c, y);
  }
}

// Post-sublayer conv + residual + the next pre-norm:
//   x[r] += a(r) * rf[r] + b(r) * rf[r-1];  un[r] = gain * x[r] / rms(x[r]).
// With zf != nullptr (after the last layer) the normed rows of slots 1..K-1
// are written compactly to zf[b*(K-1) + i-1] instead of un.
// One CTA per row; dynamic shared: D floats.
template <typename S>
__global__ void __launch_bounds__(512) k_conv_post_norm(
    const float *__restrict__ rf, const float *__restrict__ gate, int K, int D, int group,
    const S *__restrict__ base, float *__restrict__ x, const S *__restrict__ gain, float eps,
    S *__restrict__ un, S *__restrict__ zf) {
  extern __shared__ float xrow[];
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  const int r = blockIdx.x;
  const float *ga = gate + (size_t)r * (2 * D / group);
  const float *gb = ga + D / group;
  const bool first = (r % K) == 0;
  float ss = 0.f;
  for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
    float cur[8], prev[8], ba[8], bb[8], xv[8];
    load8(rf + (size_t)r * D + c, cur);
    if (first) {
#pragma unroll
      for (int j = 0; j < 8; ++j) prev[j] = 0.f;
    } else {
      load8(rf + (size_t)(r - 1) * D + c, prev);
    }
    load8(base + c, ba);
    load8(base + D + c, bb);
    load8(x + (size_t)r * D + c, xv);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int g = (c + j) / group;
      const float a = sigmoidf_(ba[j] + ga[g]);
      const float b = sigmoidf_(bb[j] + gb[g]);
      xv[j] += a * cur[j] + b * prev[j];
      xrow[c + j] = xv[j];
      ss += xv[j] * xv[j];
    }
    store8(x + (size_t)r * D + c, xv);
  }
  const float inv = rsqrtf(block_sum(ss, red) / D + eps);
  S *o;
  if (zf) {
    const int i = r % K, b = r / K;
    if (i == 0) return;
    o = zf + ((size_t)b * (K - 1) + (i - 1)) * D;
  } else {
    o = un + (size_t)r * D;
  }
  for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
    float g[8], y[8];
    load8(gain + c, g);
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = xrow[c + j] * inv * g[j];
    store8(o + c, y);
  }
}

// RMSNorm over one head (d values held as pairs (i, i + d/2) by d/2 threads)
// followed by rotate-half RoPE with the row's (cos, sin) table.
__device__ __forceinline__ void head_norm_rope(float &lo, float &hi, int i, int half,
                                               float gl, float gh, float eps, float2 cs,
                                               float *red) {
  float ss = lo * lo + hi * hi;
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (2 * half) + eps);
  lo = lo * inv * gl;
  hi = hi * inv * gh;
  const float x = lo * cs.x - hi * cs.y, y = hi * cs.x + lo * cs.y;
  lo = x;
  hi = y;
}

// q, k, v of the block from the QKV projection qkv [rows, (Hq+2Hkv)*d] (fp32).
// grid (rows, Hq + 2*Hkv), block d/2.
template <typename S>
__global__ void k_qkv_post(const float *__restrict__ qkv, int rows, int K, int Hq,
                           int Hkv, int dh, const S *__restrict__ qn, const S *__restrict__ kn,
                           const float2 *__restrict__ rope_cs, float eps,
                           S *__restrict__ qb, S *__restrict__ kb, S *__restrict__ vb) {
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  const int r = blockIdx.x, h = blockIdx.y, i = threadIdx.x, half = dh / 2;
  const int W = (Hq + 2 * Hkv) * dh;
  const size_t o = (size_t)r * W + (size_t)h * dh;
  float lo = qkv[o + i], hi = qkv[o + i + half];
  (void)rows;
  if (h < Hq + Hkv) {
    const S *g = h < Hq ? qn : kn;
    head_norm_rope(lo, hi, i, half, ldf(g + i), ldf(g + i + half), eps,
                   rope_cs[(size_t)r * half + i], red);
    S *dst = h < Hq ? qb + ((size_t)r * Hq + h) * dh : kb + ((size_t)r * Hkv + (h - Hq)) * dh;
    stf(dst + i, lo);
    stf(dst + i + half, hi);
  } else {
    S *dst = vb + ((size_t)r * Hkv + (h - Hq - Hkv)) * dh;
    stf(dst + i, lo);
    stf(dst + i + half, hi);
  }
}

// Injection epilogue: K = RoPE(k_norm(.)), V as is, into the paged caches.
// kvf holds, per layer, the K/V projection [N, 2*Hkv*d] (K heads then V heads).
// grid (N, L, 2*Hkv), block d/2.
template <typename S>
__global__ void k_inject_store(const float *__restrict__ kvf, int N, int L, int Hkv,
                               int dh, dflh::LayerPtrs knorm, const int32_t *__restrict__ req,
                               const int32_t *__restrict__ pos, const int32_t *__restrict__ table,
                               int num_rows, int max_pages, int num_pages, int P,
                               const float2 *__restrict__ rope_cs, float eps,
                               S *__restrict__ kc, S *__restrict__ vc, int *err) {
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  const int n = blockIdx.x, l = blockIdx.y, h = blockIdx.z, i = threadIdx.x, half = dh / 2;
  const int W = 2 * Hkv * dh;
  const size_t o = (size_t)l * N * W + (size_t)n * W + (size_t)h * dh;
  float lo = kvf[o + i], hi = kvf[o + i + half];
  const int row = req[n], p = pos[n];
  bool ok = true;
  if (row < 0 || row >= num_rows) {
    if (i == 0 && l == 0 && h == 0) set_err(err, DFLASH_DEV_REQ_RANGE);
    ok = false;
  }
  int page = -1;
  if (ok && (p < 0 || p / P >= max_pages)) {
    if (i == 0 && l == 0 && h == 0) set_err(err, DFLASH_DEV_POS_RANGE);
    ok = false;
  }
  if (ok) {
    page = table[(size_t)row * max_pages + p / P];
    if (page < 0 || page >= num_pages) {
      if (i == 0 && l == 0 && h == 0) set_err(err, DFLASH_DEV_PAGE_RANGE);
      ok = false;
    }
  }
  const bool is_k = h < Hkv;
  if (is_k) {
    const S *g = (const S *)knorm.p[l];
    // every thread of the block takes part in the norm's reduction
    head_norm_rope(lo, hi, i, half, ldf(g + i), ldf(g + i + half), eps,
                   rope_cs[(size_t)n * half + i], red);
  }
  if (!ok) return;
  const int hh = is_k ? h : h - Hkv;
  S *dst = (is_k ? kc : vc) +
           ((((size_t)l * num_pages + page) * Hkv + hh) * P + (p % P)) * (size_t)dh;
  stf(dst + i, lo);
  stf(dst + i + half, hi);
}

}  // namespace dfl

namespace dflh {

RopeTable rope_table(float theta, int head_dim) {
  RopeTable t;
  memset(&t, 0, sizeof(t));
  t.enabled = theta > 0.f;
  for (int i = 0; i < head_dim / 2 && i < 64; ++i)
    t.inv_freq[i] = t.enabled ? pow((double)theta, -2.0 * i / (double)head_dim) : 0.0;
  return t;
}

template <typename S>
int launch_embed_norm(const S *E, const int32_t *anchor, int mask_id, int V, int B, int K, int D,
                      const S *gain, float eps, float *x, S *un, int *err, const int32_t *ctx_len,
                      const RopeTable &rope, int half, float2 *rope_cs, cudaStream_t st) {
  DFL_CHECK_LAUNCH(launch(dfl::k_embed_norm<S>, dim3(B * K), dim3(D >= 4096 ? 512 : 128), 0, st, E,
                          anchor, mask_id, V, K, D, gain, eps, x, un, err, ctx_len, rope, half,
                          rope_cs));
  return DFLASH_OK;
}
template <typename S>
int launch_rows_norm(const S *in, int rows, int cols, const S *gain, float eps, S *out,
                     const int32_t *pos, const RopeTable &rope, int half, float2 *rope_cs,
                     cudaStream_t st) {
  if (rows <= 0) return DFLASH_OK;
  const int threads = cols >= 8192 ? 1024 : cols >= 2048 ? 256 : 64;
  DFL_CHECK_LAUNCH(launch(dfl::k_rows_norm<S>, dim3(rows), dim3(threads), 0, st, in, cols, gain,
                          eps, out, pos, rope, half, rope_cs));
  return DFLASH_OK;
}
template <typename S>
int launch_conv_pre(const S *un, const float *gate, int rows, int K, int D, int group,
                    const S *base, S *ub, cudaStream_t st) {
  const int chunk = D >= 2048 ? 1024 : D;
  DFL_CHECK_LAUNCH(launch(dfl::k_conv_pre<S>, dim3(rows, (D + chunk - 1) / chunk), dim3(128), 0,
                          st, un, gate, K, D, group, chunk, base, ub));
  return DFLASH_OK;
}
template <typename S>
int launch_conv_post_norm(const float *rf, const float *gate, int rows, int K, int D, int group,
                          const S *base, float *x, const S *gain, float eps, S *un, S *zf,
                          cudaStream_t st) {
  const size_t smem = (size_t)D * sizeof(float);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(dfl::k_conv_post_norm<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return DFLASH_ERR_CUDA;
  }
  const int threads = D >= 4096 ? 512 : D >= 1024 ? 128 : 32;
  DFL_CHECK_LAUNCH(launch(dfl::k_conv_post_norm<S>, dim3(rows), dim3(threads), smem, st, rf, gate,
                          K, D, group, base, x, gain, eps, un, zf));
  return DFLASH_OK;
}
template <typename S>
int launch_qkv_post(const float *qkv, int rows, int K, int Hq, int Hkv, int dh, const S *qn,
                    const S *kn, const float2 *rope_cs, float eps, S *qb, S *kb, S *vb,
                    cudaStream_t st) {
  DFL_CHECK_LAUNCH(launch(dfl::k_qkv_post<S>, dim3(rows, Hq + 2 * Hkv), dim3(dh / 2), 0, st, qkv,
                          rows, K, Hq, Hkv, dh, qn, kn, rope_cs, eps, qb, kb, vb));
  return DFLASH_OK;
}
template <typename S>
int launch_inject_store(const float *kvf, int N, int L, int Hkv, int dh, LayerPtrs knorm,
                        const int32_t *req, const int32_t *pos, const int32_t *page_table,
                        int num_rows, int max_pages, int num_pages, int page_size,
                        const float2 *rope_cs, float eps, S *kc, S *vc, int *err,
                        cudaStream_t st) {
  DFL_CHECK_LAUNCH(launch(dfl::k_inject_store<S>, dim3(N, L, 2 * Hkv), dim3(dh / 2), 0, st, kvf, N,
                          L, Hkv, dh, knorm, req, pos, page_table, num_rows, max_pages, num_pages,
                          page_size, rope_cs, eps, kc, vc, err));
  return DFLASH_OK;
}

#define DFL_INST(S)                                                                              \
  template int launch_embed_norm<S>(const S *, const int32_t *, int, int, int, int, int, const S *, \
                                    float, float *, S *, int *, const int32_t *,                 \
                                    const RopeTable &, int, float2 *, cudaStream_t);             \
  template int launch_rows_norm<S>(const S *, int, int, const S *, float, S *, const int32_t *,  \
                                   const RopeTable &, int, float2 *, cudaStream_t);              \
  template int launch_conv_pre<S>(const S *, const float *, int, int, int, int, const S *, S *,  \
                                  cudaStream_t);                                                 \
  template int launch_conv_post_norm<S>(const float *, const float *, int, int, int, int,        \
                                        const S *, float *, const S *, float, S *, S *,          \
                                        cudaStream_t);                                           \
  template int launch_qkv_post<S>(const float *, int, int, int, int, int, const S *, const S *,  \
                                  const float2 *, float, S *, S *, S *, cudaStream_t);           \
  template int launch_inject_store<S>(const float *, int, int, int, int, LayerPtrs,              \
                                      const int32_t *, const int32_t *, const int32_t *, int,    \
                                      int, int, int, const float2 *, float, S *, S *, int *,     \
                                      cudaStream_t);
DFL_INST(float)
DFL_INST(dfl::bf16)

}  // namespace dflh
