// Per-position top-k + logsumexp, the Viterbi path selector, greedy acceptance.
//
// Order used by every selection here: larger value first; equal values by the
// lower index (token id, candidate rank).
#include <math.h>

#include "head.cuh"

namespace dfl {

struct VI {
  float v;
  int i;
};
__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}
__device__ __forceinline__ VI warp_best(VI a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v = __shfl_xor_sync(0xffffffffu, a.v, o);
    int i = __shfl_xor_sync(0xffffffffu, a.i, o);
    if (better(v, i, a.v, a.i)) a.v = v, a.i = i;
  }
  return a;
}
// best over the block; red: 2*32 words of shared scratch
__device__ __forceinline__ VI block_best(VI a, float *redv, int *redi) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  a = warp_best(a);
  __syncthreads();
  if (lane == 0) redv[wid] = a.v, redi[wid] = a.i;
  __syncthreads();
  VI b{-INFINITY, 0x7fffffff};
  if (lane < nw) b.v = redv[lane], b.i = redi[lane];
  return warp_best(b);
}

// One chunk of one logit row: local max, sum of exp, local top-k.
// partial layout per (row, chunk): [m, s, v_0..v_{k-1}, id_0..id_{k-1}]
__global__ void __launch_bounds__(256) k_topk_partial(const float *__restrict__ logits, int V,
                                                      int k, float *__restrict__ partial) {
  __shared__ float vals[dflh::kTopkChunk];
  __shared__ float redv[32];
  __shared__ int redi[32];
  pdl_launch();
  pdl_wait();
  const int chunk = blockIdx.x, row = blockIdx.y, nch = gridDim.x;
  const int c0 = chunk * dflh::kTopkChunk;
  const int n = min(dflh::kTopkChunk, V - c0);
  const float *z = logits + (size_t)row * V + c0;
  float mx = -INFINITY;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    float v = z[i];
    vals[i] = v;
    mx = fmaxf(mx, v);
  }
  mx = warp_max(mx);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) redv[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = (threadIdx.x & 31) < (blockDim.x >> 5) ? redv[threadIdx.x & 31] : -INFINITY;
  mx = warp_max(mx);
  float se = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) se += expf(vals[i] - mx);
  se = block_sum(se, redv);
  float *out = partial + ((size_t)row * nch + chunk) * (2 * k + 2);
  if (threadIdx.x == 0) out[0] = mx, out[1] = se;
  for (int it = 0; it < k; ++it) {
    VI best{-INFINITY, 0x7fffffff};
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      if (better(vals[i], c0 + i, best.v, best.i)) best.v = vals[i], best.i = c0 + i;
    best = block_best(best, redv, redi);
    if (threadIdx.x == 0) {
      out[2 + it] = best.v;
      out[2 + k + it] = __int_as_float(best.i);
      if (best.i != 0x7fffffff) vals[best.i - c0] = -INFINITY;
    }
    __syncthreads();
  }
}

// Merge the chunks of one row: top-k ids, logp = logit - logsumexp.
__global__ void __launch_bounds__(256) k_topk_merge(const float *__restrict__ partial, int nch,
                                                    int k, int32_t *__restrict__ ids,
                                                    float *__restrict__ logp) {
  extern __shared__ float cand[];  // [nch*k] values, then [nch*k] ids
  __shared__ float redv[32];
  __shared__ int redi[32];
  pdl_launch();
  pdl_wait();
  const int row = blockIdx.x, n = nch * k;
  int *cid = (int *)(cand + n);
  const float *pr = partial + (size_t)row * nch * (2 * k + 2);
  float M = -INFINITY;
  for (int c = threadIdx.x; c < nch; c += blockDim.x) M = fmaxf(M, pr[(size_t)c * (2 * k + 2)]);
  M = warp_max(M);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) redv[threadIdx.x >> 5] = M;
  __syncthreads();
  M = (threadIdx.x & 31) < (blockDim.x >> 5) ? redv[threadIdx.x & 31] : -INFINITY;
  M = warp_max(M);
  float s = 0.f;
  for (int c = threadIdx.x; c < nch; c += blockDim.x) {
    const float *p = pr + (size_t)c * (2 * k + 2);
    s += p[1] * expf(p[0] - M);
  }
  s = block_sum(s, redv);
  const float lse = M + logf(s);
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int c = e / k, j = e % k;
    const float *p = pr + (size_t)c * (2 * k + 2);
    cand[e] = p[2 + j];
    cid[e] = __float_as_int(p[2 + k + j]);
  }
  __syncthreads();
  for (int it = 0; it < k; ++it) {
    VI best{-INFINITY, 0x7fffffff};
    int where = -1;
    for (int e = threadIdx.x; e < n; e += blockDim.x)
      if (better(cand[e], cid[e], best.v, best.i)) best.v = cand[e], best.i = cid[e], where = e;
    VI b = block_best(best, redv, redi);
    if (best.i == b.i && where >= 0 && cand[where] == b.v) {
      cand[where] = -INFINITY;
      cid[where] = 0x7fffffff;
    }
    if (threadIdx.x == 0) {
      ids[(size_t)row * k + it] = b.i;
      logp[(size_t)row * k + it] = b.v - lse;
    }
    __syncthreads();
  }
}

// rows[b*R + j] = E[token j of request b]: j = 0 the anchor, j >= 1 the
// candidates in (position, rank) order.  R = 1 + (K-1)*k.
template <typename S>
__global__ void __launch_bounds__(256) k_sel_gather(const S *__restrict__ E,
                                                    const int32_t *__restrict__ anchor,
                                                    const int32_t *__restrict__ topk_ids, int K,
                                                    int k, int V, int D, S *__restrict__ rows,
                                                    int *err) {
  pdl_launch();
  pdl_wait();
  const int R = 1 + (K - 1) * k;
  const int b = blockIdx.x / R, j = blockIdx.x % R;
  int tok = j == 0 ? anchor[b] : topk_ids[(size_t)b * (K - 1) * k + (j - 1)];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) set_err(err, DFLASH_DEV_TOKEN_RANGE);
    tok = tok < 0 ? 0 : V - 1;
  }
  const S *e = E + (size_t)tok * D;
  S *o = rows + (size_t)blockIdx.x * D;
  if ((D % 8) == 0 && sizeof(S) == 2) {
    const uint4 *src = (const uint4 *)e;
    uint4 *dst = (uint4 *)o;
    for (int c = threadIdx.x; c < D / 8; c += blockDim.x) dst[c] = src[c];
  } else {
    for (int c = threadIdx.x; c < D; c += blockDim.x) o[c] = e[c];
  }
}

// One CTA per request: max-sum Viterbi over the K-1 positions of k candidates.
// u = P_u e and v = P_v e come from the selector GEMM slices (summed here).
__global__ void __launch_bounds__(256) k_viterbi(const float *__restrict__ upart,
                                                 const float *__restrict__ vpart, int nsu,
                                                 int nsv, const int32_t *__restrict__ topk_ids,
                                                 const float *__restrict__ topk_logp, int B, int K,
                                                 int k, int r, int32_t *__restrict__ path,
                                                 float *__restrict__ score) {
  extern __shared__ float sm[];
  const int LDR = r + 1;
  float *su = sm;                     // [k][LDR] predecessors' u
  float *sv = su + (size_t)k * LDR;   // [k][LDR] current candidates' v
  float *pair = sv + (size_t)k * LDR; // [k][k]
  float *delta = pair + k * k;        // [k]
  int *bp = (int *)(delta + k);       // [(K-1)][k]
  pdl_launch();
  pdl_wait();
  const int b = blockIdx.x;
  const int R = 1 + (K - 1) * k;
  const size_t rows = (size_t)B * R;
  auto urow = [&](int j, int c) {
    float s = 0.f;
    for (int q = 0; q < nsu; ++q) s += upart[((size_t)q * rows + (size_t)b * R + j) * r + c];
    return s;
  };
  auto vrow = [&](int j, int c) {
    float s = 0.f;
    for (int q = 0; q < nsv; ++q) s += vpart[((size_t)q * rows + (size_t)b * R + j) * r + c];
    return s;
  };
  // predecessor of position 0: the anchor (row 0)
  for (int c = threadIdx.x; c < r; c += blockDim.x) su[c] = urow(0, c);
  int n_prev = 1;
  for (int t = 0; t < K - 1; ++t) {
    for (int e = threadIdx.x; e < k * r; e += blockDim.x) {
      const int j = e / r, c = e % r;
      sv[j * LDR + c] = vrow(1 + t * k + j, c);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n_prev * k; e += blockDim.x) {
      const int i = e / k, j = e % k;
      float d = 0.f;
      for (int c = 0; c < r; ++c) d = fmaf(su[i * LDR + c], sv[j * LDR + c], d);
      pair[i * k + j] = d;
    }
    __syncthreads();
    const float *lp = topk_logp + ((size_t)b * (K - 1) + t) * k;
    float nd = 0.f;
    int arg = 0;
    if (threadIdx.x < k) {
      const int j = threadIdx.x;
      float best = -INFINITY;
      for (int i = 0; i < n_prev; ++i) {
        const float c = (t == 0 ? 0.f : delta[i]) + pair[i * k + j];
        if (c > best) best = c, arg = i;  // strict: the lower rank keeps ties
      }
      nd = lp[j] + best;
    }
    __syncthreads();
    if (threadIdx.x < k) {
      delta[threadIdx.x] = nd;
      bp[t * k + threadIdx.x] = arg;
    }
    // the current candidates become the predecessors
    if (t + 1 < K - 1)
      for (int e = threadIdx.x; e < k * r; e += blockDim.x) {
        const int j = e / r, c = e % r;
        su[j * LDR + c] = urow(1 + t * k + j, c);
      }
    n_prev = k;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int best = 0;
    for (int j = 1; j < k; ++j)
      if (delta[j] > delta[best]) best = j;
    score[b] = delta[best];
    int j = best;
    for (int t = K - 2; t >= 0; --t) {
      path[(size_t)b * (K - 1) + t] = topk_ids[((size_t)b * (K - 1) + t) * k + j];
      j = bp[t * k + j];
    }
  }
}

// argmax of one chunk of one target-logit row -> partial (value, id)
template <typename L>
__global__ void __launch_bounds__(256) k_argmax_partial(const L *__restrict__ logits, int V,
                                                        float *__restrict__ partial) {
  __shared__ float redv[32];
  __shared__ int redi[32];
  pdl_launch();
  pdl_wait();
  const int chunk = blockIdx.x, row = blockIdx.y, nch = gridDim.x;
  const int c0 = chunk * dflh::kArgmaxChunk, c1 = min(V, c0 + dflh::kArgmaxChunk);
  const L *z = logits + (size_t)row * V;
  VI best{-INFINITY, 0x7fffffff};
  for (int i = c0 + threadIdx.x; i < c1; i += blockDim.x) {
    const float v = ldf(z + i);
    if (better(v, i, best.v, best.i)) best.v = v, best.i = i;
  }
  best = block_best(best, redv, redi);
  if (threadIdx.x == 0) {
    partial[((size_t)row * nch + chunk) * 2] = best.v;
    partial[((size_t)row * nch + chunk) * 2 + 1] = __int_as_float(best.i);
  }
}

// per request: argmax of each row (one warp per row), then the longest matching prefix
__global__ void __launch_bounds__(1024) k_accept(const int32_t *__restrict__ path,
                                                 const float *__restrict__ partial, int B, int K,
                                                 int nch, int32_t *__restrict__ accept_len,
                                                 int32_t *__restrict__ tokens) {
  __shared__ int tgt[DFLASH_MAX_BLOCK];
  pdl_launch();
  pdl_wait();
  const int b = blockIdx.x, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (w < K) {
    const float *p = partial + (size_t)(b * K + w) * nch * 2;
    VI best{-INFINITY, 0x7fffffff};
    for (int c = lane; c < nch; c += 32) {
      const float v = p[2 * c];
      const int id = __float_as_int(p[2 * c + 1]);
      if (better(v, id, best.v, best.i)) best.v = v, best.i = id;
    }
    best = warp_best(best);
    if (lane == 0) tgt[w] = best.i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int m = 0;
    while (m < K - 1 && path[(size_t)b * (K - 1) + m] == tgt[m]) ++m;
    for (int i = 0; i < K; ++i)
      tokens[(size_t)b * K + i] = i < m ? tgt[i] : i == m ? tgt[m] : -1;
    accept_len[b] = m + 1;
  }
}

}  // namespace dfl

namespace dflh {

int launch_topk(const float *logits, int rows, int V, int k, float *partial, int32_t *ids,
                float *logp, cudaStream_t st) {
  if (rows <= 0) return DFLASH_OK;
  const int nch = topk_chunks(V);
  DFL_CHECK_LAUNCH(launch(dfl::k_topk_partial, dim3(nch, rows), dim3(256), 0, st, logits, V, k,
                          partial));
  const size_t smem = (size_t)nch * k * 2 * sizeof(float);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(dfl::k_topk_merge, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return DFLASH_ERR_CUDA;
  }
  DFL_CHECK_LAUNCH(launch(dfl::k_topk_merge, dim3(rows), dim3(256), smem, st,
                          (const float *)partial, nch, k, ids, logp));
  return DFLASH_OK;
}

template <typename S>
int launch_sel_gather(const S *E, const int32_t *anchor, const int32_t *topk_ids, int B, int K,
                      int k, int V, int D, S *rows, int *err, cudaStream_t st) {
  const int R = 1 + (K - 1) * k;
  DFL_CHECK_LAUNCH(launch(dfl::k_sel_gather<S>, dim3(B * R), dim3(256), 0, st, E, anchor,
                          topk_ids, K, k, V, D, rows, err));
  return DFLASH_OK;
}
template int launch_sel_gather<float>(const float *, const int32_t *, const int32_t *, int, int,
                                      int, int, int, float *, int *, cudaStream_t);
template int launch_sel_gather<dfl::bf16>(const dfl::bf16 *, const int32_t *, const int32_t *, int,
                                          int, int, int, int, dfl::bf16 *, int *, cudaStream_t);

int launch_viterbi(const float *upart, const float *vpart, int nsu, int nsv,
                   const int32_t *topk_ids, const float *topk_logp, int B, int K, int k, int r,
                   int32_t *path, float *score, cudaStream_t st) {
  const size_t smem = sizeof(float) * (2 * (size_t)k * (r + 1) + (size_t)k * k + k) +
                      sizeof(int) * (size_t)(K - 1) * k;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(dfl::k_viterbi, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return DFLASH_ERR_CUDA;
  }
  DFL_CHECK_LAUNCH(launch(dfl::k_viterbi, dim3(B), dim3(256), smem, st, upart, vpart, nsu, nsv,
                          topk_ids, topk_logp, B, K, k, r, path, score));
  return DFLASH_OK;
}

int launch_accept(const int32_t *path, const void *logits, int dtype, int B, int K, int V,
                  float *partial, int32_t *accept_len, int32_t *tokens, cudaStream_t st) {
  const int nch = argmax_chunks(V);
  if (dtype == DFLASH_F32) {
    DFL_CHECK_LAUNCH(launch(dfl::k_argmax_partial<float>, dim3(nch, B * K), dim3(256), 0, st,
                            (const float *)logits, V, partial));
  } else {
    DFL_CHECK_LAUNCH(launch(dfl::k_argmax_partial<dfl::bf16>, dim3(nch, B * K), dim3(256), 0, st,
                            (const dfl::bf16 *)logits, V, partial));
  }
  DFL_CHECK_LAUNCH(launch(dfl::k_accept, dim3(B), dim3(32 * K), 0, st,
                          (const int32_t *)path, (const float *)partial, B, K, nch, accept_len,
                          tokens));
  return DFLASH_OK;
}

}  // namespace dflh
