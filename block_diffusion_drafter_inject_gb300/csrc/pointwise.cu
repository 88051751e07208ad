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
template <typename S>
__global__ void __launch_bounds__(512) k_embed_norm(const S *__restrict__ E,
                                                    const int32_t *__restrict__ anchor,
                                                    int mask_id, int V, int K, int D,
                                                    const S *__restrict__ gain, float eps,
                                                    float *__restrict__ x, S *__restrict__ un,
                                                    int *err) {
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  const int r = blockIdx.x, b = r / K, i = r % K;
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
                                                    S *__restrict__ out) {
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
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

// Gate corrections of row r for gate rows [j0, j0 + n) of each half (a and b):
// the K slices of the gate GEMM summed in slice order into shared memory
// (ga[j] for a, gb[j] for b).  One pass over the slices per gate row.
__device__ __forceinline__ void gate_sums(const float *__restrict__ gpart, int nsplit, int rows,
                                          int GW, int r, int j0, int n, float *ga, float *gb) {
  const int half = GW / 2;
  for (int e = threadIdx.x; e < 2 * n; e += blockDim.x) {
    const int j = e < n ? j0 + e : half + j0 + (e - n);
    const float *p = gpart + (size_t)r * GW + j;
    float s = 0.f;
    for (int k = 0; k < nsplit; ++k) s += p[(size_t)k * rows * GW];
    if (e < n)
      ga[e] = s;
    else
      gb[e - n] = s;
  }
  __syncthreads();
}

// Pre-sublayer conv: ub[r] = a(r) * un[r] + b(r) * un[r-1] (zero before slot 0).
// grid (rows, channel chunks of `chunk`), dynamic shared: 2 * chunk/group floats.
template <typename S>
__global__ void __launch_bounds__(256) k_conv_pre(const S *__restrict__ un,
                                                  const float *__restrict__ gpart, int nsplit,
                                                  int rows, int K, int D, int group, int chunk,
                                                  const S *__restrict__ base,
                                                  S *__restrict__ ub) {
  extern __shared__ float gs[];
  pdl_launch();
  pdl_wait();
  const int r = blockIdx.x;
  const int c0 = blockIdx.y * chunk, c1 = min(D, c0 + chunk);
  const int GW = 2 * D / group;
  const int g0 = c0 / group, ng = (c1 - 1) / group - g0 + 1;
  float *ga = gs, *gb = gs + ng;
  gate_sums(gpart, nsplit, rows, GW, r, g0, ng, ga, gb);
  const bool first = (r % K) == 0;
  for (int c = c0 + threadIdx.x; c < c1; c += blockDim.x) {
    const int g = c / group - g0;
    const float a = sigmoidf_(ldf(base + c) + ga[g]);
    const float bg = sigmoidf_(ldf(base + D + c) + gb[g]);
    const float cur = ldf(un + (size_t)r * D + c);
    const float prev = first ? 0.f : ldf(un + (size_t)(r - 1) * D + c);
    stf(ub + (size_t)r * D + c, a * cur + bg * prev);
  }
}

// Post-sublayer conv + residual + the next pre-norm:
//   x[r] += a(r) * rf[r] + b(r) * rf[r-1];  un[r] = gain * x[r] / rms(x[r]).
// With zf != nullptr (after the last layer) the normed rows of slots 1..K-1
// are written compactly to zf[b*(K-1) + i-1] instead of un.
// One CTA per row; dynamic shared: D + 2*D/group floats.
template <typename S>
__global__ void __launch_bounds__(1024) k_conv_post_norm(
    const float *__restrict__ rf, const float *__restrict__ gpart, int nsplit, int rows, int K,
    int D, int group, const S *__restrict__ base, float *__restrict__ x,
    const S *__restrict__ gain, float eps, S *__restrict__ un, S *__restrict__ zf) {
  extern __shared__ float sm[];
  __shared__ float red[32];
  float *xrow = sm;
  float *ga = sm + D, *gb = ga + D / group;
  pdl_launch();
  pdl_wait();
  const int r = blockIdx.x;
  const int GW = 2 * D / group;
  gate_sums(gpart, nsplit, rows, GW, r, 0, D / group, ga, gb);
  const bool first = (r % K) == 0;
  float ss = 0.f;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    const int g = c / group;
    const float a = sigmoidf_(ldf(base + c) + ga[g]);
    const float bg = sigmoidf_(ldf(base + D + c) + gb[g]);
    const float cur = rf[(size_t)r * D + c];
    const float prev = first ? 0.f : rf[(size_t)(r - 1) * D + c];
    const float v = x[(size_t)r * D + c] + (a * cur + bg * prev);
    x[(size_t)r * D + c] = v;
    xrow[c] = v;
    ss += v * v;
  }
  const float inv = rsqrtf(block_sum(ss, red) / D + eps);
  if (zf) {
    const int i = r % K, b = r / K;
    if (i == 0) return;
    S *o = zf + ((size_t)b * (K - 1) + (i - 1)) * D;
    for (int c = threadIdx.x; c < D; c += blockDim.x) stf(o + c, xrow[c] * inv * ldf(gain + c));
  } else {
    for (int c = threadIdx.x; c < D; c += blockDim.x)
      stf(un + (size_t)r * D + c, xrow[c] * inv * ldf(gain + c));
  }
}

// rf = sum of slices (fp32, may be null); rb = rf rounded to storage
template <typename S>
__global__ void __launch_bounds__(256) k_reduce(const float *__restrict__ part, int nsplit,
                                                size_t n, float *__restrict__ rf,
                                                S *__restrict__ rb) {
  pdl_launch();
  pdl_wait();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int k = 0; k < nsplit; ++k) s += part[(size_t)k * n + i];
    if (rf) rf[i] = s;
    if (rb) stf(rb + i, s);
  }
}

// hb[r][j] = SiLU(gate) * up with [gate | up] the two halves of the gate/up GEMM row
template <typename S>
__global__ void __launch_bounds__(256) k_swiglu(const float *__restrict__ part, int nsplit,
                                                int rows, int F, S *__restrict__ hb) {
  pdl_launch();
  pdl_wait();
  const size_t n = (size_t)rows * F;
  const size_t slice = (size_t)rows * 2 * F;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / F, j = i % F;
    float g = 0.f, u = 0.f;
    for (int k = 0; k < nsplit; ++k) {
      g += part[k * slice + r * 2 * F + j];
      u += part[k * slice + r * 2 * F + F + j];
    }
    stf(hb + i, g * sigmoidf_(g) * u);
  }
}

// RMSNorm over one head (d values held as pairs (i, i + d/2) by d/2 threads)
// followed by rotate-half RoPE at absolute position `pos`.  The angle
// pos * theta^(-2i/d) is formed and reduced modulo 2*pi in fp64 (two fp64
// operations); sine and cosine of the reduced angle are taken in fp32.
__device__ __forceinline__ void head_norm_rope(float &lo, float &hi, int i, int half,
                                               float gl, float gh, float eps, int pos,
                                               const dflh::RopeTable &rope, float *red) {
  float ss = lo * lo + hi * hi;
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (2 * half) + eps);
  lo = lo * inv * gl;
  hi = hi * inv * gh;
  if (rope.enabled) {
    const double two_pi = 6.283185307179586476925286766559;
    const double a = (double)pos * rope.inv_freq[i];
    const float ar = (float)(a - two_pi * floor(a * (1.0 / two_pi)));
    float s, c;
    sincosf(ar, &s, &c);
    const float x = lo * c - hi * s, y = hi * c + lo * s;
    lo = x;
    hi = y;
  }
}

// q, k, v of the block from the QKV GEMM slices.  grid (rows, Hq + 2*Hkv), block d/2.
template <typename S>
__global__ void k_qkv_post(const float *__restrict__ part, int nsplit, int rows, int K, int Hq,
                           int Hkv, int dh, const S *__restrict__ qn, const S *__restrict__ kn,
                           const int32_t *__restrict__ ctx_len, const dflh::RopeTable rope,
                           float eps, S *__restrict__ qb, S *__restrict__ kb,
                           S *__restrict__ vb) {
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  const int r = blockIdx.x, h = blockIdx.y, i = threadIdx.x, half = dh / 2;
  const int W = (Hq + 2 * Hkv) * dh;
  const size_t slice = (size_t)rows * W;
  const size_t o = (size_t)r * W + (size_t)h * dh;
  float lo = 0.f, hi = 0.f;
#pragma unroll 8
  for (int k = 0; k < nsplit; ++k) {
    lo += part[k * slice + o + i];
    hi += part[k * slice + o + i + half];
  }
  if (h < Hq + Hkv) {
    const S *g = h < Hq ? qn : kn;
    const int pos = ctx_len[r / K] + (r % K);
    head_norm_rope(lo, hi, i, half, ldf(g + i), ldf(g + i + half), eps, pos, rope, red);
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
// kvpart holds, per layer, nsplit slices of [N, 2*Hkv*d] (K heads then V heads).
// grid (N, L, 2*Hkv), block d/2.
template <typename S>
__global__ void k_inject_store(const float *__restrict__ kvpart, int nsplit, int N, int L, int Hkv,
                               int dh, dflh::LayerPtrs knorm, const int32_t *__restrict__ req,
                               const int32_t *__restrict__ pos, const int32_t *__restrict__ table,
                               int num_rows, int max_pages, int num_pages, int P,
                               const dflh::RopeTable rope, float eps, S *__restrict__ kc,
                               S *__restrict__ vc, int *err) {
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  const int n = blockIdx.x, l = blockIdx.y, h = blockIdx.z, i = threadIdx.x, half = dh / 2;
  const int W = 2 * Hkv * dh;
  const size_t slice = (size_t)N * W;
  const size_t layer_off = (size_t)l * nsplit * slice;
  const size_t o = (size_t)n * W + (size_t)h * dh;
  float lo = 0.f, hi = 0.f;
#pragma unroll 8
  for (int k = 0; k < nsplit; ++k) {
    lo += kvpart[layer_off + k * slice + o + i];
    hi += kvpart[layer_off + k * slice + o + i + half];
  }
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
    head_norm_rope(lo, hi, i, half, ldf(g + i), ldf(g + i + half), eps, p, rope, red);
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

static int grid_for(size_t n) {
  const Dev *d = device();
  size_t g = (n + 255) / 256;
  size_t cap = (size_t)(d ? d->num_sms : 152) * 8;
  return (int)(g < cap ? (g > 0 ? g : 1) : cap);
}

template <typename S>
int launch_embed_norm(const S *E, const int32_t *anchor, int mask_id, int V, int B, int K, int D,
                      const S *gain, float eps, float *x, S *un, int *err, cudaStream_t st) {
  DFL_CHECK_LAUNCH(launch(dfl::k_embed_norm<S>, dim3(B * K), dim3(D >= 4096 ? 512 : 128), 0, st, E,
                          anchor, mask_id, V, K, D, gain, eps, x, un, err));
  return DFLASH_OK;
}
template <typename S>
int launch_rows_norm(const S *in, int rows, int cols, const S *gain, float eps, S *out,
                     cudaStream_t st) {
  if (rows <= 0) return DFLASH_OK;
  const int threads = cols >= 8192 ? 1024 : cols >= 2048 ? 256 : 64;
  DFL_CHECK_LAUNCH(
      launch(dfl::k_rows_norm<S>, dim3(rows), dim3(threads), 0, st, in, cols, gain, eps, out));
  return DFLASH_OK;
}
template <typename S>
int launch_conv_pre(const S *un, const float *gpart, int nsplit, int rows, int K, int D,
                    int group, const S *base, S *ub, cudaStream_t st) {
  // channel chunks: a multiple of the group, about 1024 channels
  int chunk = ((1024 + group - 1) / group) * group;
  if (chunk > D) chunk = D;
  const int nchunk = (D + chunk - 1) / chunk;
  const size_t smem = 2 * (size_t)(chunk / group + 2) * sizeof(float);
  DFL_CHECK_LAUNCH(launch(dfl::k_conv_pre<S>, dim3(rows, nchunk), dim3(256), smem, st, un, gpart,
                          nsplit, rows, K, D, group, chunk, base, ub));
  return DFLASH_OK;
}
template <typename S>
int launch_conv_post_norm(const float *rf, const float *gpart, int nsplit, int rows, int K, int D,
                          int group, const S *base, float *x, const S *gain, float eps, S *un,
                          S *zf, cudaStream_t st) {
  const size_t smem = ((size_t)D + 2 * (size_t)(D / group)) * sizeof(float);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(dfl::k_conv_post_norm<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return DFLASH_ERR_CUDA;
  }
  const int threads = D >= 4096 ? 1024 : D >= 1024 ? 512 : 256;
  DFL_CHECK_LAUNCH(launch(dfl::k_conv_post_norm<S>, dim3(rows), dim3(threads), smem, st, rf,
                          gpart, nsplit, rows, K, D, group, base, x, gain, eps, un, zf));
  return DFLASH_OK;
}
template <typename S>
int launch_reduce(const float *part, int nsplit, int rows, int N, float *rf, S *rb,
                  cudaStream_t st) {
  const size_t n = (size_t)rows * N;
  DFL_CHECK_LAUNCH(
      launch(dfl::k_reduce<S>, dim3(grid_for(n)), dim3(256), 0, st, part, nsplit, n, rf, rb));
  return DFLASH_OK;
}
template <typename S>
int launch_swiglu(const float *part, int nsplit, int rows, int F, S *hb, cudaStream_t st) {
  const size_t n = (size_t)rows * F;
  DFL_CHECK_LAUNCH(
      launch(dfl::k_swiglu<S>, dim3(grid_for(n)), dim3(256), 0, st, part, nsplit, rows, F, hb));
  return DFLASH_OK;
}
template <typename S>
int launch_qkv_post(const float *part, int nsplit, int rows, int K, int Hq, int Hkv, int dh,
                    const S *qn, const S *kn, const int32_t *ctx_len, const RopeTable &rope,
                    float eps, S *qb, S *kb, S *vb, cudaStream_t st) {
  DFL_CHECK_LAUNCH(launch(dfl::k_qkv_post<S>, dim3(rows, Hq + 2 * Hkv), dim3(dh / 2), 0, st, part,
                          nsplit, rows, K, Hq, Hkv, dh, qn, kn, ctx_len, rope, eps, qb, kb, vb));
  return DFLASH_OK;
}
template <typename S>
int launch_inject_store(const float *kvpart, int nsplit, int N, int L, int Hkv, int dh,
                        LayerPtrs knorm, const int32_t *req, const int32_t *pos,
                        const int32_t *page_table, int num_rows, int max_pages, int num_pages,
                        int page_size, const RopeTable &rope, float eps, S *kc, S *vc, int *err,
                        cudaStream_t st) {
  DFL_CHECK_LAUNCH(launch(dfl::k_inject_store<S>, dim3(N, L, 2 * Hkv), dim3(dh / 2), 0, st, kvpart,
                          nsplit, N, L, Hkv, dh, knorm, req, pos, page_table, num_rows, max_pages,
                          num_pages, page_size, rope, eps, kc, vc, err));
  return DFLASH_OK;
}

#define DFL_INST(S)                                                                              \
  template int launch_embed_norm<S>(const S *, const int32_t *, int, int, int, int, int, const S *, \
                                    float, float *, S *, int *, cudaStream_t);                   \
  template int launch_rows_norm<S>(const S *, int, int, const S *, float, S *, cudaStream_t);    \
  template int launch_conv_pre<S>(const S *, const float *, int, int, int, int, int, const S *,  \
                                  S *, cudaStream_t);                                            \
  template int launch_conv_post_norm<S>(const float *, const float *, int, int, int, int, int,   \
                                        const S *, float *, const S *, float, S *, S *,          \
                                        cudaStream_t);                                           \
  template int launch_reduce<S>(const float *, int, int, int, float *, S *, cudaStream_t);       \
  template int launch_swiglu<S>(const float *, int, int, int, S *, cudaStream_t);                \
  template int launch_qkv_post<S>(const float *, int, int, int, int, int, int, const S *,        \
                                  const S *, const int32_t *, const RopeTable &, float, S *, S *, \
                                  S *, cudaStream_t);                                            \
  template int launch_inject_store<S>(const float *, int, int, int, int, int, LayerPtrs,         \
                                      const int32_t *, const int32_t *, const int32_t *, int,    \
                                      int, int, int, const RopeTable &, float, S *, S *, int *,  \
                                      cudaStream_t);
DFL_INST(float)
DFL_INST(dfl::bf16)

}  // namespace dflh
