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

// 8-element chunks of a row a thread keeps in registers between the two
// passes of a row norm
constexpr int kNormCache = 4;

template <typename S>
__global__ void __launch_bounds__(512) k_embed_norm(const S *__restrict__ E,
                                                    const int32_t *__restrict__ anchor,
                                                    int mask_id, int V, int K, int D,
                                                    const S *__restrict__ gain, float eps,
                                                    float *__restrict__ x, S *__restrict__ un,
                                                    int *err, const int32_t *__restrict__ ctx_len,
                                                    const dflh::RopeTable rope, int half,
                                                    float2 *__restrict__ rope_cs,
                                                    float *__restrict__ ssq_out) {
  __shared__ float red[32];
  // The first kernel of a draft pass releases its dependents only once its
  // own wait has returned: every later kernel of the pass therefore starts
  // after all work queued before the pass (the injection of context K/V above
  // all) has completed, and may read the caches before its own wait.
  pdl_wait();
  pdl_launch();
  const int r = blockIdx.x, b = r / K, i = r % K;
  int tok = i == 0 ? anchor[b] : mask_id;
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) set_err(err, DFLASH_DEV_TOKEN_RANGE);
    tok = tok < 0 ? 0 : V - 1;
  }
  // the thread's first kNormCache chunks of the embedding row stay in
  // registers for the normed output; the RoPE row is formed while they load
  const S *e = E + (size_t)tok * D;
  const int step = blockDim.x * 8, c0 = threadIdx.x * 8;
  float v[kNormCache][8];
#pragma unroll
  for (int q = 0; q < kNormCache; ++q)
    if (c0 + q * step < D) load8(e + c0 + q * step, v[q]);
  rope_row(rope_cs + (size_t)r * half, ctx_len[b] + i, rope, half);
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < kNormCache; ++q)
    if (c0 + q * step < D) {
      store8(x + (size_t)r * D + c0 + q * step, v[q]);
#pragma unroll
      for (int j = 0; j < 8; ++j) ss += v[q][j] * v[q][j];
    }
  for (int c = c0 + kNormCache * step; c < D; c += step) {
    float w[8];
    load8(e + c, w);
    store8(x + (size_t)r * D + c, w);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += w[j] * w[j];
  }
  const float tot = block_sum(ss, red);
  if (ssq_out && threadIdx.x == 0) ssq_out[r] = tot;  // the row's sum of squares (slot 0)
  const float inv = rsqrtf(tot / D + eps);
  if (!un) return;
#pragma unroll
  for (int q = 0; q < kNormCache; ++q) {
    const int c = c0 + q * step;
    if (c < D) {
      float g[8];
      load8(gain + c, g);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[q][j] = v[q][j] * inv * g[j];
      store8(un + (size_t)r * D + c, v[q]);
    }
  }
  for (int c = c0 + kNormCache * step; c < D; c += step) {
    float w[8], g[8];
    load8(e + c, w);
    load8(gain + c, g);
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = w[j] * inv * g[j];
    store8(un + (size_t)r * D + c, w);
  }
}

// out[r] = gain * in[r] / rms(in[r]); cols % 8 == 0, 16-byte aligned rows.
// A thread's first few 8-element chunks of the row (kNormCache, two for
// float32 rows) are loaded at once and kept in registers for the output pass
// (the chunks past them, if any, are read again); the RoPE row and the
// cache-slot lookup run while those loads are in flight, the slot's page-table
// read after the row is written.
template <typename S>
__global__ void __launch_bounds__(1024) k_rows_norm(const S *__restrict__ in, int cols,
                                                    const S *__restrict__ gain, float eps,
                                                    S *__restrict__ out,
                                                    const int32_t *__restrict__ pos,
                                                    const dflh::RopeTable rope, int half,
                                                    float2 *__restrict__ rope_cs,
                                                    const dflh::CacheSlots cs) {
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  const S *row = in + (size_t)blockIdx.x * cols;
  // float32 rows: two cached chunks (64 registers a thread at 1024 threads)
  constexpr int NC = sizeof(S) == 2 ? kNormCache : 2;
  const int step = blockDim.x * 8, c0 = threadIdx.x * 8;
  float v[NC][8];
#pragma unroll
  for (int q = 0; q < NC; ++q)
    if (c0 + q * step < cols) load8(row + c0 + q * step, v[q]);
  int srow = 0, spos = 0;
  const bool slot_thread = cs.slot && threadIdx.x == 0;
  if (slot_thread) srow = cs.req[blockIdx.x], spos = pos[blockIdx.x];
  if (rope_cs) rope_row(rope_cs + (size_t)blockIdx.x * half, pos[blockIdx.x], rope, half);
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < NC; ++q)
    if (c0 + q * step < cols) {
#pragma unroll
      for (int j = 0; j < 8; ++j) ss += v[q][j] * v[q][j];
    }
  for (int c = c0 + NC * step; c < cols; c += step) {
    float w[8];
    load8(row + c, w);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += w[j] * w[j];
  }
  const float inv = rsqrtf(block_sum(ss, red) / cols + eps);
  S *o = out + (size_t)blockIdx.x * cols;
#pragma unroll
  for (int q = 0; q < NC; ++q) {
    const int c = c0 + q * step;
    if (c < cols) {
      float g[8];
      load8(gain + c, g);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[q][j] = v[q][j] * inv * g[j];
      store8(o + c, v[q]);
    }
  }
  for (int c = c0 + NC * step; c < cols; c += step) {
    float w[8], g[8];
    load8(row + c, w);
    load8(gain + c, g);
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = w[j] * inv * g[j];
    store8(o + c, w);
  }
  if (slot_thread) {
    long long sl = -1;
    if (srow < 0 || srow >= cs.num_rows) {
      set_err(cs.err, DFLASH_DEV_REQ_RANGE);
    } else if (spos < 0 || spos / cs.P >= cs.max_pages) {
      set_err(cs.err, DFLASH_DEV_POS_RANGE);
    } else {
      const int page = cs.table[(size_t)srow * cs.max_pages + spos / cs.P];
      if (page < 0 || page >= cs.num_pages)
        set_err(cs.err, DFLASH_DEV_PAGE_RANGE);
      else
        sl = ((long long)page * cs.Hkv * cs.P + spos % cs.P) * cs.dh;
    }
    cs.slot[blockIdx.x] = sl;
  }
}

// Sum of the nsl K slices p[0], p[stride], ... in slice order; the first
// kGateSlices loads are all issued before the first add (one round trip).
constexpr int kGateSlices = 16;
__device__ __forceinline__ float sum_slices(const float *p, int nsl, size_t stride) {
  float t[kGateSlices];
#pragma unroll
  for (int q = 0; q < kGateSlices; ++q)
    if (q < nsl) t[q] = p[(size_t)q * stride];
  float v = t[0];
#pragma unroll
  for (int q = 1; q < kGateSlices; ++q)
    if (q < nsl) v += t[q];
  for (int q = kGateSlices; q < nsl; ++q) v += p[(size_t)q * stride];
  return v;
}

// Pre-sublayer conv: ub[r] = a(r) * un[r] + b(r) * un[r-1] (zero before slot 0),
//   a_c(r) = sigmoid(base[c] + gate[r][c/g]),  b_c(r) = sigmoid(base[D+c] + gate[r][D/g + c/g])
// gate: the conv's gate linear of row r as nsl K slices, fp32 [nsl][rows][2D/g],
// summed here in slice order.  grid (rows, D/chunk); dynamic shared: the
// summed gates of the chunk's groups.
template <typename S>
__global__ void __launch_bounds__(256) k_conv_pre(const S *__restrict__ un,
                                                  const float *__restrict__ gate, int nsl, int K,
                                                  int D, int group, int chunk,
                                                  const S *__restrict__ base, S *__restrict__ ub) {
  extern __shared__ float sg[];  // [2][ng]: the a gates, then the b gates
  pdl_launch();
  pdl_wait();
  const int r = blockIdx.x, rows = gridDim.x;
  const int c0 = blockIdx.y * chunk, c1 = min(D, c0 + chunk);
  const int GW = 2 * D / group, gl0 = c0 / group, ng = (c1 - 1) / group - gl0 + 1;
  const bool first = (r % K) == 0;
  float cur[8], prev[8], ba[8], bb[8];
  auto load_at = [&](int c) {
    load8(un + (size_t)r * D + c, cur);
    if (first) {
#pragma unroll
      for (int j = 0; j < 8; ++j) prev[j] = 0.f;
    } else {
      load8(un + (size_t)(r - 1) * D + c, prev);
    }
    load8(base + c, ba);
    load8(base + D + c, bb);
  };
  const int cA = c0 + threadIdx.x * 8;
  for (int i = threadIdx.x; i < 2 * ng; i += blockDim.x) {
    const int col = i < ng ? gl0 + i : D / group + gl0 + (i - ng);
    sg[i] = sum_slices(gate + (size_t)r * GW + col, nsl, (size_t)rows * GW);
  }
  __syncthreads();
  const float *ga = sg - gl0, *gb = sg + ng - gl0;
  for (int c = cA; c < c1; c += blockDim.x * 8) {
    float y[8];
    load_at(c);
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
// gate: as for the pre-sublayer conv, nsl K slices [nsl][rows][2D/g].
// One CTA per row; dynamic shared: D + 2D/g floats.
template <typename S>
__global__ void __launch_bounds__(512) k_conv_post_norm(
    const float *__restrict__ rf, const float *__restrict__ gate, int nsl, int K, int D,
    int group, const S *__restrict__ base, float *__restrict__ x, const S *__restrict__ gain,
    float eps, S *__restrict__ un, S *__restrict__ zf) {
  extern __shared__ float xrow[];  // [D] the updated row, then [2D/g] the summed gates
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  const int r = blockIdx.x, rows = gridDim.x, GW = 2 * D / group;
  float *sg = xrow + D;
  const bool first = (r % K) == 0;
  float cur[8], prev[8], ba[8], bb[8], xv[8];
  auto load_at = [&](int c) {
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
  };
  const int cA = threadIdx.x * 8;
  for (int i = threadIdx.x; i < GW; i += blockDim.x) {
    sg[i] = sum_slices(gate + (size_t)r * GW + i, nsl, (size_t)rows * GW);
  }
  __syncthreads();
  const float *ga = sg, *gb = sg + D / group;
  float ss = 0.f;
  for (int c = cA; c < D; c += blockDim.x * 8) {
    load_at(c);
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
  for (int c = cA; c < D; c += blockDim.x * 8) {
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
__global__ void __launch_bounds__(256) k_inject_store(
    const float *__restrict__ kvf, int N, int L, int Hkv, int dh, dflh::LayerPtrs knorm,
    const int32_t *__restrict__ req, const int32_t *__restrict__ pos,
    const int32_t *__restrict__ table, int num_rows, int max_pages, int num_pages, int P,
    const float2 *__restrict__ rope_cs, float eps, S *__restrict__ kc, S *__restrict__ vc,
    int *err) {
  pdl_launch();
  pdl_wait();
  // one CTA per (token, layer); one warp per head, lanes on the pairs (i, i + dh/2)
  const int n = blockIdx.x, l = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = dh / 2, W = 2 * Hkv * dh, nw = blockDim.x >> 5;
  const int row = req[n], p = pos[n];
  int page = -1;
  if (row < 0 || row >= num_rows) {
    if (threadIdx.x == 0 && l == 0) set_err(err, DFLASH_DEV_REQ_RANGE);
    return;
  }
  if (p < 0 || p / P >= max_pages) {
    if (threadIdx.x == 0 && l == 0) set_err(err, DFLASH_DEV_POS_RANGE);
    return;
  }
  page = table[(size_t)row * max_pages + p / P];
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0 && l == 0) set_err(err, DFLASH_DEV_PAGE_RANGE);
    return;
  }
  const float *src = kvf + (size_t)l * N * W + (size_t)n * W;
  const S *g = (const S *)knorm.p[l];
  for (int h = warp; h < 2 * Hkv; h += nw) {
    const bool is_k = h < Hkv;
    const float *hs = src + (size_t)h * dh;
    float lo[2], hi[2];  // dh <= 128: at most two pairs per lane
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int i = lane + 32 * j;
      lo[j] = i < half ? hs[i] : 0.f;
      hi[j] = i < half ? hs[i + half] : 0.f;
      ss += lo[j] * lo[j] + hi[j] * hi[j];
    }
    if (is_k) {
      // per-head RMSNorm, then rotate-half RoPE at the token's position
      const float inv = rsqrtf(warp_sum(ss) / dh + eps);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int i = lane + 32 * j;
        if (i < half) {
          const float a = lo[j] * inv * ldf(g + i), b = hi[j] * inv * ldf(g + i + half);
          const float2 cs = rope_cs[(size_t)n * half + i];
          lo[j] = a * cs.x - b * cs.y;
          hi[j] = b * cs.x + a * cs.y;
        }
      }
    }
    const int hh = is_k ? h : h - Hkv;
    S *dst = (is_k ? kc : vc) +
             ((((size_t)l * num_pages + page) * Hkv + hh) * P + (p % P)) * (size_t)dh;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int i = lane + 32 * j;
      if (i < half) {
        stf(dst + i, lo[j]);
        stf(dst + i + half, hi[j]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Two-tap conv with its gate linear fused, for a few block rows (T <= 16).
//
// The gate linear s = G u (G [2D/g, D]) is tiny next to the projections, and
// at T <= 16 its cost is the latency of a GEMM launch plus its split-K
// reduction.  Here one CTA owns NG channel groups: it stages its 2*NG gate
// rows in shared memory before waiting for the producer, forms the T gate
// pre-activations of those rows itself (fp32 dot products of full rows), and
// applies the conv to its NG*g channels.  PRE also forms u = R(rmsnorm(x))
// from the fp32 residual stream (sums of squares over the full rows, then
// u = (x * inv) * gain rounded to storage).
// ---------------------------------------------------------------------------

// 8 consecutive storage elements, global -> shared, asynchronously (16-byte aligned)
__device__ __forceinline__ void copy8_async(bf16 *d, const bf16 *s) {
  cp_async16(smem_u32(d), s, 16);
}
__device__ __forceinline__ void copy8_async(float *d, const float *s) {
  cp_async16(smem_u32(d), s, 16);
  cp_async16(smem_u32(d + 4), s + 4, 16);
}

constexpr int kGcMaxT = 16;

template <typename S>
struct GconvArgs {
  int T, K, D, group;
  const S *G;        // gate linear [2D/group, D]
  const S *base;     // [2D]
  const float *x;    // residual stream [T, D]: PRE reads it; POST adds the conv to it
  float *xo;         // POST: the residual stream (same array as x)
  const S *gain;     // PRE: pre-norm weight [D]
  float eps;
  S *ub;             // PRE: conv output [T, D]
  const S *gin;      // POST: gate input R(r) [T, D]
  const float *rf;   // POST: conv input r [T, D]
  // bf16 (cluster kernel): POST writes, per CTA, the sums of squares of the
  // updated rows over its channels to ssq_out[cta][16]; PRE with ssq_in sums
  // the n_ssq partials of each row in slot order instead of forming them
  float *ssq_out;
  const float *ssq_in;
  int n_ssq;
};

// grid (2D/g / (2*NG)), block 256; dynamic shared: (R2 + PRE) * D elements of S.
template <typename S, int R2, bool PRE>
__global__ void __launch_bounds__(256) k_gconv(const GconvArgs<S> A) {
  constexpr int NG = R2 / 2, N = kGcMaxT * R2;
  extern __shared__ __align__(16) uint8_t gc_smem[];
  S *sG = (S *)gc_smem;   // [R2][D]: rows a_{j0..}, then b_{j0..}
  S *sGain = sG + (size_t)R2 * A.D;
  __shared__ float red[8][N];
  __shared__ float s_s[N];   // gate pre-activations [t][R2]
  __shared__ float s_inv[kGcMaxT];
  pdl_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int D = A.D, T = A.T, nv = D / 8, GW = D / A.group;
  const int j0 = blockIdx.x * NG;
  for (int e = tid; e < R2 * nv; e += blockDim.x) {
    const int r = e / nv, v = e % nv;
    const int grow = r < NG ? j0 + r : GW + j0 + (r - NG);
    copy8_async(sG + (size_t)r * D + 8 * v, A.G + (size_t)grow * D + 8 * v);
  }
  if (PRE)
    for (int v = tid; v < nv; v += blockDim.x) copy8_async(sGain + 8 * v, A.gain + 8 * v);
  cp_async_commit();
  pdl_wait();

  if (PRE) {  // inverse RMS of every row
    float ss[kGcMaxT];
#pragma unroll
    for (int t = 0; t < kGcMaxT; ++t) ss[t] = 0.f;
    for (int v = tid; v < nv; v += blockDim.x) {
#pragma unroll
      for (int t = 0; t < kGcMaxT; ++t) {
        if (t < T) {
          float xv[8];
          load8(A.x + (size_t)t * D + 8 * v, xv);
#pragma unroll
          for (int j = 0; j < 8; ++j) ss[t] += xv[j] * xv[j];
        }
      }
    }
    warp_reduce_scatter<kGcMaxT>(ss, lane);
    if ((lane & 1) == 0) red[warp][lane >> 1] = ss[0];
    __syncthreads();
    if (tid < kGcMaxT) {
      float s = 0.f;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w][tid];
      s_inv[tid] = rsqrtf(s / D + A.eps);
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // s_inv, the staged rows; red is reused below

  float acc[N];
#pragma unroll
  for (int i = 0; i < N; ++i) acc[i] = 0.f;
  for (int v = tid; v < nv; v += blockDim.x) {
    float gw[R2][8], gn[8];
#pragma unroll
    for (int r = 0; r < R2; ++r) load8(sG + (size_t)r * D + 8 * v, gw[r]);
    if (PRE) load8(sGain + 8 * v, gn);
#pragma unroll
    for (int t = 0; t < kGcMaxT; ++t) {
      if (t < T) {
        float u[8];
        if (PRE) {
          load8(A.x + (size_t)t * D + 8 * v, u);
          const float inv = s_inv[t];
#pragma unroll
          for (int j = 0; j < 8; ++j) u[j] = rnd(u[j] * inv * gn[j], (const S *)nullptr);
        } else {
          load8(A.gin + (size_t)t * D + 8 * v, u);
        }
#pragma unroll
        for (int r = 0; r < R2; ++r)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[t * R2 + r] += u[j] * gw[r][j];
      }
    }
  }
  warp_reduce_scatter<N>(acc, lane);
  {
    const int f = rs_first<N>(lane);
#pragma unroll
    for (int m = 0; m < N / 32; ++m) red[warp][f + m] = acc[m];
  }
  __syncthreads();
  if (tid < N) {
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w][tid];
    s_s[tid] = s;
  }
  __syncthreads();

  // the conv on this CTA's channels
  const int c0 = j0 * A.group, nc = NG * A.group;
  for (int e = tid; e < T * nc; e += blockDim.x) {
    const int t = e / nc, c = c0 + e % nc, gl = c / A.group - j0;
    const float a = sigmoidf_(ldf(A.base + c) + s_s[t * R2 + gl]);
    const float b = sigmoidf_(ldf(A.base + D + c) + s_s[t * R2 + NG + gl]);
    const bool first = (t % A.K) == 0;
    const size_t o = (size_t)t * D + c;
    if (PRE) {
      const float g = ldf(sGain + c);
      const float cur = rnd(A.x[o] * s_inv[t] * g, (const S *)nullptr);
      const float prev = first ? 0.f : rnd(A.x[o - D] * s_inv[t - 1] * g, (const S *)nullptr);
      stf(A.ub + o, a * cur + b * prev);
    } else {
      const float cur = A.rf[o], prev = first ? 0.f : A.rf[o - D];
      A.xo[o] = A.x[o] + (a * cur + b * prev);
    }
  }
}

// A float whose load is issued here, ahead of later memory operations
__device__ __forceinline__ float ld_ordered(const float *p) {
  float v;
  asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
// 8 floats (16-byte aligned) whose loads are issued here, ahead of later
// memory operations (the compiler may not sink them to their first use)
__device__ __forceinline__ void load8_ordered(const float *p, float *v) {
  asm volatile("ld.global.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
               : "l"(p)
               : "memory");
  asm volatile("ld.global.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
               : "l"(p + 4)
               : "memory");
}

// bf16 storage: the same op on tensor cores, one thread-block cluster of C
// CTAs per NGc (<= 8) channel groups.  CTA rank q takes the channel slice
// [q*D/C, (q+1)*D/C) of the gate products: it stages its slice of the
// cluster's 2*NGc gate rows (zero rows up to 16) and of the T input rows (zero
// rows up to 16) in XOR-swizzled shared memory and runs mma.sync m16n8k16
// (tokens x gate rows) over it.  The C partial 16x16 tiles (and, for PRE, the
// C partial sums of squares of the rows) are read through distributed shared
// memory and summed in rank order, so every CTA holds the same totals.  Rank
// q then applies the conv to its W = NGc*g/C channels of the cluster's groups.
// The slice is DS = D/C wide with DS/8 (a power of two, <= 128) 16-byte chunks.
// Dynamic shared: 64 * DS bytes (+ 2 * DS for PRE's gain slice).
template <bool PRE, int C>
__global__ void __launch_bounds__(256) k_gconv_cl(const GconvArgs<bf16> A, int NGc) {
  constexpr int MAXI = 8;  // PRE: input rows per thread (16 rows x DS/8 chunks / 256)
  extern __shared__ __align__(128) uint8_t gc_sm[];
  const int D = A.D, T = A.T, GW = D / A.group;
  const int DS = D / C, nvs = DS / 8, RBs = DS * 2;
  uint8_t *sG = gc_sm;                     // [16][DS], swizzled
  uint8_t *sU = sG + 16 * RBs;             // [16][DS], swizzled
  bf16 *sGain = (bf16 *)(sU + 16 * RBs);   // [DS] (PRE)
  __shared__ float red[8][256];            // per-warp partial tiles [t][16]
  __shared__ float s_part[256];            // this CTA's partial tile (read by the peers)
  __shared__ float s_tot[256];             // the cluster's sums
  __shared__ float s_ssw[4][16];
  __shared__ float s_ssq[16];              // this CTA's partial sums of squares (read by peers)
  __shared__ float s_inv[16];
  pdl_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = (int)cluster_rank(), cl = blockIdx.x / C;
  const int j0 = cl * NGc, R = 2 * NGc, d0 = q * DS;
  const uint32_t uG = smem_u32(sG), uU = smem_u32(sU);
  for (int e = tid; e < 16 * nvs; e += 256) {
    const int r = e / nvs, v = e % nvs;
    const bool ok = r < R;
    const int grow = r < NGc ? j0 + r : GW + j0 + (r - NGc);
    cp_async16(uG + swz(r, v, RBs),
               ok ? (const void *)(A.G + (size_t)grow * D + d0 + 8 * v) : (const void *)A.G,
               ok ? 16 : 0);
  }
  if (PRE)
    for (int v = tid; v < nvs; v += 256) cp_async16(smem_u32(sGain + 8 * v), A.gain + d0 + 8 * v, 16);
  cp_async_commit();
  // the conv applies to W channels of the cluster's groups from cb on; this
  // thread's first element (e = tid): its weights before the wait, its
  // activations right after it, in flight with the staging loads
  const int W = NGc * A.group / C;
  const int cb = j0 * A.group + q * W;
  const bool pe = tid < T * W;
  const int pt = pe ? tid / W : 0, pch = cb + (pe ? tid % W : 0);
  const bool pfirst = (pt % A.K) == 0;
  const size_t po = (size_t)pt * D + pch;
  float pba = 0.f, pbb = 0.f, pg = 0.f, pc = 0.f, pp = 0.f, px = 0.f;
  if (pe) {
    pba = ldf(A.base + pch);
    pbb = ldf(A.base + D + pch);
    if (PRE) pg = ldf(A.gain + pch);
  }
  pdl_wait();
  if (pe) {
    const float *src = PRE ? A.x : A.rf;
    pc = ld_ordered(src + po);
    if (!pfirst) pp = ld_ordered(src + po - D);
    if (!PRE) px = ld_ordered(A.x + po);
  }

  if (!PRE) {
    for (int e = tid; e < 16 * nvs; e += 256) {
      const int t = e / nvs, v = e % nvs;
      const bool ok = t < T;
      cp_async16(uU + swz(t, v, RBs),
                 ok ? (const void *)(A.gin + (size_t)t * D + d0 + 8 * v) : (const void *)A.gin,
                 ok ? 16 : 0);
    }
    cp_async_commit();
  } else {
    // this thread's chunk v of rows t0 + j * tstep (nvs divides 256)
    const int v = tid % nvs, tstep = 256 / nvs, t0 = tid / nvs;
    float xv[MAXI][8];
    float ss[MAXI];
#pragma unroll
    for (int j = 0; j < MAXI; ++j) {
      const int t = t0 + j * tstep;
      if (t < T) {
        load8_ordered(A.x + (size_t)t * D + d0 + 8 * v, xv[j]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) xv[j][k] = 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < MAXI; ++j) {
      ss[j] = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) ss[j] += xv[j][k] * xv[j][k];
    }
    if (A.ssq_in) {
      // the rows' sums of squares from the partials written with x: warp w
      // sums rows w, w + 8 (each lane its slots in order, then a fixed tree)
      for (int t = warp; t < T; t += 8) {
        float a = 0.f;
        for (int i = lane; i < A.n_ssq; i += 32) a += A.ssq_in[(size_t)i * 16 + t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) s_inv[t] = rsqrtf(a / D + A.eps);
      }
    } else {
    // sum over the lanes that hold the same row (aligned groups of min(nvs, 32))
    const int span = nvs < 32 ? nvs : 32;
    for (int o = span >> 1; o > 0; o >>= 1)
#pragma unroll
      for (int j = 0; j < MAXI; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], o);
    if (lane % span == 0)
#pragma unroll
      for (int j = 0; j < MAXI; ++j) {
        const int t = t0 + j * tstep;
        if (t < 16) s_ssw[v / span][t] = ss[j];
      }
    __syncthreads();
    if (tid < 16) {
      float a = 0.f;
      for (int g = 0; g < (nvs + 31) / 32; ++g) a += s_ssw[g][tid];
      s_ssq[tid] = a;
    }
    cluster_sync();  // partial sums of squares visible to the cluster
    if (tid < 16) {
      float a = 0.f;
      for (int r = 0; r < C; ++r) a += ld_dsmem(smem_u32(&s_ssq[tid]), (uint32_t)r);
      s_inv[tid] = rsqrtf(a / D + A.eps);
    }
    }
    cp_async_wait<0>();  // the gain slice
    __syncthreads();
#pragma unroll
    for (int j = 0; j < MAXI; ++j) {
      const int t = t0 + j * tstep;
      if (t < 16) {
        uint4 pk = make_uint4(0u, 0u, 0u, 0u);
        if (t < T) {
          float gn[8];
          load8(sGain + 8 * v, gn);
          const float inv = s_inv[t];
          pk.x = pack_bf16(xv[j][0] * inv * gn[0], xv[j][1] * inv * gn[1]);
          pk.y = pack_bf16(xv[j][2] * inv * gn[2], xv[j][3] * inv * gn[3]);
          pk.z = pack_bf16(xv[j][4] * inv * gn[4], xv[j][5] * inv * gn[5]);
          pk.w = pack_bf16(xv[j][6] * inv * gn[6], xv[j][7] * inv * gn[7]);
        }
        *(uint4 *)(sU + swz(t, v, RBs)) = pk;
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // partial s[t][r] over this slice: tokens are the mma rows, gate rows the columns
  float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int r8 = lane & 7, mi = lane >> 3;
    const int nks = DS / 16;
    for (int ks = warp * 2; ks < nks; ks += 16) {
      uint32_t a0[4], a1[4], b0[4], b1[4];
      ldsm_x4(uU + swz((mi & 1) * 8 + r8, 2 * ks + (mi >> 1), RBs), a0[0], a0[1], a0[2], a0[3]);
      ldsm_x4(uU + swz((mi & 1) * 8 + r8, 2 * ks + 2 + (mi >> 1), RBs), a1[0], a1[1], a1[2],
              a1[3]);
      ldsm_x4(uG + swz(r8, 2 * ks + mi, RBs), b0[0], b0[1], b0[2], b0[3]);
      ldsm_x4(uG + swz(8 + r8, 2 * ks + mi, RBs), b1[0], b1[1], b1[2], b1[3]);
      mma_bf16_16816(c0, a0, b0[0], b0[1]);
      mma_bf16_16816(c0, a1, b0[2], b0[3]);
      mma_bf16_16816(c1, a0, b1[0], b1[1]);
      mma_bf16_16816(c1, a1, b1[2], b1[3]);
    }
  }
  {
    const int g8 = lane >> 2, t4 = lane & 3;
    float *rw = red[warp];
    rw[g8 * 16 + 2 * t4] = c0[0];
    rw[g8 * 16 + 2 * t4 + 1] = c0[1];
    rw[(g8 + 8) * 16 + 2 * t4] = c0[2];
    rw[(g8 + 8) * 16 + 2 * t4 + 1] = c0[3];
    rw[g8 * 16 + 8 + 2 * t4] = c1[0];
    rw[g8 * 16 + 8 + 2 * t4 + 1] = c1[1];
    rw[(g8 + 8) * 16 + 8 + 2 * t4] = c1[2];
    rw[(g8 + 8) * 16 + 8 + 2 * t4 + 1] = c1[3];
  }
  __syncthreads();
  {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) a += red[w][tid];
    s_part[tid] = a;
  }
  cluster_sync();  // partial tiles visible to the cluster
  {
    float a = 0.f;
    for (int r = 0; r < C; ++r) a += ld_dsmem(smem_u32(&s_part[tid]), (uint32_t)r);
    s_tot[tid] = a;
  }
  // this CTA is done reading its peers' shared memory; it waits for their
  // reads of its own only before it exits
  cluster_arrive_relaxed();
  __syncthreads();

  // the conv on this CTA's channels (the first element's operands prefetched)
  for (int e = tid; e < T * W; e += 256) {
    const bool f0 = e == tid;
    const int t = e / W, ch = cb + e % W, gl = ch / A.group - j0;
    const float a = sigmoidf_((f0 ? pba : ldf(A.base + ch)) + s_tot[t * 16 + gl]);
    const float b = sigmoidf_((f0 ? pbb : ldf(A.base + D + ch)) + s_tot[t * 16 + NGc + gl]);
    const bool first = (t % A.K) == 0;
    const size_t o = (size_t)t * D + ch;
    if (PRE) {
      const float g = f0 ? pg : ldf(A.gain + ch);
      const float xc = f0 ? pc : A.x[o], xp = first ? 0.f : (f0 ? pp : A.x[o - D]);
      const float cur = rnd(xc * s_inv[t] * g, (const bf16 *)nullptr);
      const float prev = first ? 0.f : rnd(xp * s_inv[t - 1] * g, (const bf16 *)nullptr);
      stf(A.ub + o, a * cur + b * prev);
    } else {
      const float cur = f0 ? pc : A.rf[o], prev = first ? 0.f : (f0 ? pp : A.rf[o - D]);
      const float xn = (f0 ? px : A.x[o]) + (a * cur + b * prev);
      A.xo[o] = xn;
      if (A.ssq_out) (&red[0][0])[e] = xn * xn;  // free since s_part was formed; T * W <= 2048
    }
  }
  if (!PRE && A.ssq_out) {
    __syncthreads();
    if (tid < T) {
      float a = 0.f;
      for (int j = 0; j < W; ++j) a += (&red[0][0])[tid * W + j];
      A.ssq_out[(size_t)blockIdx.x * 16 + tid] = a;
    }
  }
  cluster_wait();  // the peers have read s_part (and s_ssq) before this CTA exits
}

// zf[b*(K-1) + i-1] = gain * x[b*K + i] / rms(x[b*K + i]) for slots i >= 1.
template <typename S>
__global__ void __launch_bounds__(512) k_final_norm(const float *__restrict__ x, int K, int D,
                                                    const S *__restrict__ gain, float eps,
                                                    S *__restrict__ zf) {
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  const int o = blockIdx.x, b = o / (K - 1), i = o % (K - 1) + 1;
  const float *row = x + ((size_t)b * K + i) * D;
  float ss = 0.f;
  for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
    float v[8];
    load8(row + c, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += v[j] * v[j];
  }
  const float inv = rsqrtf(block_sum(ss, red) / D + eps);
  for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
    float v[8], g[8];
    load8(row + c, v);
    load8(gain + c, g);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = v[j] * inv * g[j];
    store8(zf + (size_t)o * D + c, v);
  }
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
                      const RopeTable &rope, int half, float2 *rope_cs, cudaStream_t st,
                      float *ssq_out) {
  DFL_CHECK_LAUNCH(launch(dfl::k_embed_norm<S>, dim3(B * K), dim3(D >= 4096 ? 512 : 128), 0, st, E,
                          anchor, mask_id, V, K, D, gain, eps, x, un, err, ctx_len, rope, half,
                          rope_cs, ssq_out));
  return DFLASH_OK;
}
template <typename S>
int launch_rows_norm(const S *in, int rows, int cols, const S *gain, float eps, S *out,
                     const int32_t *pos, const RopeTable &rope, int half, float2 *rope_cs,
                     cudaStream_t st, const CacheSlots &slots) {
  if (rows <= 0) return DFLASH_OK;
  const int threads = cols >= 8192 ? 1024 : cols >= 2048 ? 256 : 64;
  DFL_CHECK_LAUNCH(launch(dfl::k_rows_norm<S>, dim3(rows), dim3(threads), 0, st, in, cols, gain,
                          eps, out, pos, rope, half, rope_cs, slots));
  return DFLASH_OK;
}
template <typename S>
int launch_conv_pre(const S *un, const float *gate, int nsl, int rows, int K, int D, int group,
                    const S *base, S *ub, cudaStream_t st) {
  const int chunk = D >= 2048 ? 1024 : D;
  const size_t smem = (size_t)2 * ((chunk + group - 1) / group + 1) * sizeof(float);
  if (smem > 48 * 1024) return DFLASH_ERR_DIMS;
  DFL_CHECK_LAUNCH(launch(dfl::k_conv_pre<S>, dim3(rows, (D + chunk - 1) / chunk), dim3(128),
                          smem, st, un, gate, nsl, K, D, group, chunk, base, ub));
  return DFLASH_OK;
}
template <typename S>
int launch_conv_post_norm(const float *rf, const float *gate, int nsl, int rows, int K, int D,
                          int group, const S *base, float *x, const S *gain, float eps, S *un,
                          S *zf, cudaStream_t st) {
  const size_t smem = (size_t)(D + 2 * D / group) * sizeof(float);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(dfl::k_conv_post_norm<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return DFLASH_ERR_CUDA;
  }
  const int threads = D >= 4096 ? 512 : D >= 1024 ? 128 : 32;
  DFL_CHECK_LAUNCH(launch(dfl::k_conv_post_norm<S>, dim3(rows), dim3(threads), smem, st, rf, gate,
                          nsl, K, D, group, base, x, gain, eps, un, zf));
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
  DFL_CHECK_LAUNCH(launch(dfl::k_inject_store<S>, dim3(N, L), dim3(256), 0, st, kvf, N, L, Hkv,
                          dh, knorm, req, pos, page_table, num_rows, max_pages, num_pages,
                          page_size, rope_cs, eps, kc, vc, err));
  return DFLASH_OK;
}

template <typename S, int R2, bool PRE>
static int launch_gconv_t(const dfl::GconvArgs<S> &a, cudaStream_t st) {
  const size_t smem = (size_t)(R2 + (PRE ? 1 : 0)) * a.D * sizeof(S);
  static int attr_done = 0;
  if (smem > 48 * 1024 && !attr_done) {
    if (cudaFuncSetAttribute(dfl::k_gconv<S, R2, PRE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    attr_done = 1;
  }
  const int groups = a.D / a.group;
  DFL_CHECK_LAUNCH(
      launch(dfl::k_gconv<S, R2, PRE>, dim3(groups / (R2 / 2)), dim3(256), smem, st, a));
  return DFLASH_OK;
}

// Cluster size C and groups per cluster NGc of the bf16 fused conv for width D
// and group size g; false when the shape does not fit it.
static bool gconv_cluster_shape(int D, int g, int *C, int *NGc) {
  const int groups = D / g;
  for (int c : {4, 8, 2}) {
    if (D % (32 * c)) continue;
    const int nvs = D / c / 8;
    if (nvs > 128 || (nvs & (nvs - 1))) continue;
    for (int n : {8, 4, 2, 1}) {
      if (groups % n || (n * g) % c) continue;
      *C = c;
      *NGc = n;
      return true;
    }
  }
  return false;
}

template <bool PRE, int C>
static int launch_gconv_cl_t(const dfl::GconvArgs<dfl::bf16> &a, int ngc, cudaStream_t st) {
  const int DS = a.D / C;
  const size_t smem = (size_t)64 * DS + (PRE ? (size_t)2 * DS : 0);
  static int attr_done = 0;
  if (!attr_done) {
    if (cudaFuncSetAttribute(dfl::k_gconv_cl<PRE, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             66 * 1024 /* DS <= 1024 */) !=
        cudaSuccess)
      return DFLASH_ERR_CUDA;
    attr_done = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.D / a.group / ngc) * C);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  count_launch();
  DFL_CHECK_LAUNCH(cudaLaunchKernelEx(&cfg, dfl::k_gconv_cl<PRE, C>, a, ngc));
  return DFLASH_OK;
}

template <bool PRE>
static int launch_gconv_cl(const dfl::GconvArgs<dfl::bf16> &a, cudaStream_t st) {
  int C = 0, ngc = 0;
  if (!gconv_cluster_shape(a.D, a.group, &C, &ngc)) return DFLASH_ERR_DIMS;
  if (C == 4) return launch_gconv_cl_t<PRE, 4>(a, ngc, st);
  if (C == 8) return launch_gconv_cl_t<PRE, 8>(a, ngc, st);
  return launch_gconv_cl_t<PRE, 2>(a, ngc, st);
}

template <typename S>
static int launch_gconv(bool pre, const dfl::GconvArgs<S> &a, cudaStream_t st) {
  if (!gconv_fits(a.T, a.D, a.group, sizeof(S) == 2 ? DFLASH_BF16 : DFLASH_F32))
    return DFLASH_ERR_DIMS;
  const int groups = a.D / a.group;
  if constexpr (sizeof(S) == 2) {
    return pre ? launch_gconv_cl<true>(a, st) : launch_gconv_cl<false>(a, st);
  } else {
    const bool two = groups % 2 == 0 && groups >= 256;  // two groups per CTA on wide models
    if (pre) return two ? launch_gconv_t<S, 4, true>(a, st) : launch_gconv_t<S, 2, true>(a, st);
    return two ? launch_gconv_t<S, 4, false>(a, st) : launch_gconv_t<S, 2, false>(a, st);
  }
}

int gconv_ssq_slots(int T, int D, int group, int dtype) {
  int C, ngc;
  if (dtype != DFLASH_BF16 || !gconv_fits(T, D, group, dtype) ||
      !gconv_cluster_shape(D, group, &C, &ngc))
    return 0;
  const int W = ngc * group / C;  // channels of one CTA
  if ((size_t)T * W > 2048) return 0;
  return (D / group / ngc) * C;
}

bool gconv_fits(int T, int D, int group, int dtype) {
  if (T < 1 || T > kGconvMaxT) return false;
  int C, ngc;
  if (dtype == DFLASH_BF16) return gconv_cluster_shape(D, group, &C, &ngc);
  return (size_t)5 * D * 4 <= 160 * 1024;
}

template <typename S>
int launch_gconv_pre(const float *x, int T, int K, int D, int group, const S *G, const S *base,
                     const S *gain, float eps, S *ub, cudaStream_t st, const float *ssq_in,
                     int n_ssq) {
  dfl::GconvArgs<S> a = {};
  a.T = T, a.K = K, a.D = D, a.group = group, a.G = G, a.base = base;
  a.x = x, a.gain = gain, a.eps = eps, a.ub = ub;
  if (ssq_in && n_ssq > 0) a.ssq_in = ssq_in, a.n_ssq = n_ssq;
  return launch_gconv<S>(true, a, st);
}
template <typename S>
int launch_gconv_post(const float *rf, const S *gin, int T, int K, int D, int group, const S *G,
                      const S *base, float *x, cudaStream_t st, float *ssq_out) {
  dfl::GconvArgs<S> a = {};
  a.T = T, a.K = K, a.D = D, a.group = group, a.G = G, a.base = base;
  a.x = x, a.xo = x, a.gin = gin, a.rf = rf;
  if (ssq_out && gconv_ssq_slots(T, D, group, sizeof(S) == 2 ? DFLASH_BF16 : DFLASH_F32) > 0)
    a.ssq_out = ssq_out;
  return launch_gconv<S>(false, a, st);
}
template <typename S>
int launch_final_norm(const float *x, int B, int K, int D, const S *gain, float eps, S *zf,
                      cudaStream_t st) {
  DFL_CHECK_LAUNCH(launch(dfl::k_final_norm<S>, dim3(B * (K - 1)),
                          dim3(D >= 4096 ? 512 : D >= 1024 ? 128 : 32), 0, st, x, K, D, gain, eps,
                          zf));
  return DFLASH_OK;
}

#define DFL_INST(S)                                                                              \
  template int launch_embed_norm<S>(const S *, const int32_t *, int, int, int, int, int, const S *, \
                                    float, float *, S *, int *, const int32_t *,                 \
                                    const RopeTable &, int, float2 *, cudaStream_t, float *);    \
  template int launch_rows_norm<S>(const S *, int, int, const S *, float, S *, const int32_t *,  \
                                   const RopeTable &, int, float2 *, cudaStream_t,               \
                                   const CacheSlots &);                                          \
  template int launch_conv_pre<S>(const S *, const float *, int, int, int, int, int, const S *,  \
                                  S *, cudaStream_t);                                            \
  template int launch_conv_post_norm<S>(const float *, const float *, int, int, int, int, int,   \
                                        const S *, float *, const S *, float, S *, S *,          \
                                        cudaStream_t);                                           \
  template int launch_qkv_post<S>(const float *, int, int, int, int, int, const S *, const S *,  \
                                  const float2 *, float, S *, S *, S *, cudaStream_t);           \
  template int launch_inject_store<S>(const float *, int, int, int, int, LayerPtrs,              \
                                      const int32_t *, const int32_t *, const int32_t *, int,    \
                                      int, int, int, const float2 *, float, S *, S *, int *,     \
                                      cudaStream_t);                                             \
  template int launch_gconv_pre<S>(const float *, int, int, int, int, const S *, const S *,      \
                                   const S *, float, S *, cudaStream_t, const float *, int);     \
  template int launch_gconv_post<S>(const float *, const S *, int, int, int, int, const S *,     \
                                    const S *, float *, cudaStream_t, float *);                  \
  template int launch_final_norm<S>(const float *, int, int, int, const S *, float, S *,         \
                                    cudaStream_t);
DFL_INST(float)
DFL_INST(dfl::bf16)

}  // namespace dflh
