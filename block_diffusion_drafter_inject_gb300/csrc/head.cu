// Per-position top-k + logsumexp, the Viterbi path selector, greedy acceptance.
//
// Order used by every selection here: larger value first; equal values by the
// lower index (token id, candidate rank).
#include <math.h>

#include <algorithm>

#include "head.cuh"

namespace dfl {

struct VI {
  float v;
  int i;
};
__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}
// The argmax of a target-logit row orders NaN above every number (the row's
// first NaN wins, as numpy's argmax does), then by value, then by lower id.
__device__ __forceinline__ bool better_nan_max(float v1, int i1, float v2, int i2) {
  const bool n1 = v1 != v1, n2 = v2 != v2;
  if (n1 || n2) return n1 && (!n2 || i1 < i2);
  return v1 > v2 || (v1 == v2 && i1 < i2);
}
template <bool NAN_MAX = false>
__device__ __forceinline__ bool pick(float v1, int i1, float v2, int i2) {
  return NAN_MAX ? better_nan_max(v1, i1, v2, i2) : better(v1, i1, v2, i2);
}
template <bool NAN_MAX = false>
__device__ __forceinline__ VI warp_best(VI a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v = __shfl_xor_sync(0xffffffffu, a.v, o);
    int i = __shfl_xor_sync(0xffffffffu, a.i, o);
    if (pick<NAN_MAX>(v, i, a.v, a.i)) a.v = v, a.i = i;
  }
  return a;
}
// best over the block; red: 2*32 words of shared scratch
template <bool NAN_MAX = false>
__device__ __forceinline__ VI block_best(VI a, float *redv, int *redi) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  a = warp_best<NAN_MAX>(a);
  __syncthreads();
  if (lane == 0) redv[wid] = a.v, redi[wid] = a.i;
  __syncthreads();
  VI b{-INFINITY, 0x7fffffff};
  if (lane < nw) b.v = redv[lane], b.i = redi[lane];
  return warp_best<NAN_MAX>(b);
}

// Descending bitonic sort of one value per lane across the warp; returns this
// lane's value of the sorted sequence (lane 0 holds the largest).
__device__ __forceinline__ float warp_sort_desc(float x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float y = __shfl_xor_sync(0xffffffffu, x, stride);
      const bool lower = (lane & stride) == 0;
      const bool desc_block = (lane & size) == 0;
      x = (lower == desc_block) ? fmaxf(x, y) : fminf(x, y);
    }
  }
  return x;
}

constexpr int kNoId = 0x7fffffff;  // id of an empty slot (never better than a real one)

// Bitonic sort of 64 (value, id) pairs held two per lane, element e = 32*i + lane
// in (v[i], id[i]); afterwards element 0 is the best (larger value, then lower id).
__device__ __forceinline__ void warp_sort64(float (&v)[2], int (&id)[2], int lane) {
#pragma unroll
  for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j == 32) {  // partner is the lane's other element; element 0 is the lower one
        const bool up = ((lane & k) == 0);  // k == 64 here: always the descending half
        const bool swap = up ? better(v[1], id[1], v[0], id[0]) : better(v[0], id[0], v[1], id[1]);
        if (swap) {
          const float tv = v[0];
          const int ti = id[0];
          v[0] = v[1], id[0] = id[1], v[1] = tv, id[1] = ti;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int e = 32 * i + lane;
          const float pv = __shfl_xor_sync(0xffffffffu, v[i], j);
          const int pi = __shfl_xor_sync(0xffffffffu, id[i], j);
          const bool lower = (e & j) == 0, up = (e & k) == 0;
          // the lower element of a pair takes the better one in a descending run
          const bool take = (lower == up) ? better(pv, pi, v[i], id[i]) : better(v[i], id[i], pv, pi);
          if (take) v[i] = pv, id[i] = pi;
        }
      }
    }
  }
}

// Warp-wide top-k (larger value, then lower id) of the candidates v[j], id[j]
// (j < J) held by the lanes; results in ov[0..k), oi[0..k) (written by lane 0).
// Every top-k element is >= the k-th largest of the lane maxima t (k lanes each
// hold an element >= t), so when at most `cap` candidates reach t they are
// compacted into the warp's shared buffers cv/ci and ranked there; otherwise
// (heavy ties) all candidates are ranked in registers.
template <int J>
__device__ __forceinline__ void warp_topk(const float (&v)[J], const int (&id)[J], int k,
                                          float *cv, int *ci, int cap, float *ov, int *oi,
                                          int lane) {
  float lm = -INFINITY;
#pragma unroll
  for (int j = 0; j < J; ++j)
    if (id[j] != kNoId) lm = fmaxf(lm, v[j]);
  const float t = __shfl_sync(0xffffffffu, warp_sort_desc(lm), k - 1);
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < J; ++j) cnt += (id[j] != kNoId && v[j] >= t) ? 1 : 0;
  int pre = cnt;  // inclusive prefix over the lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, pre, o);
    if (lane >= o) pre += y;
  }
  const int total = __shfl_sync(0xffffffffu, pre, 31);
  if (total <= cap) {
    int w = pre - cnt;
#pragma unroll
    for (int j = 0; j < J; ++j)
      if (id[j] != kNoId && v[j] >= t) cv[w] = v[j], ci[w] = id[j], ++w;
    __syncwarp();
    float sv[2];
    int si[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int e = 32 * i + lane;
      sv[i] = e < total ? cv[e] : -INFINITY;
      si[i] = e < total ? ci[e] : kNoId;
    }
    warp_sort64(sv, si, lane);
    if (lane < k) ov[lane] = sv[0], oi[lane] = si[0];  // k <= 32
  } else {
    uint32_t taken = 0;
    for (int it = 0; it < k; ++it) {
      VI best{-INFINITY, kNoId};
      int bj = -1;
#pragma unroll
      for (int j = 0; j < J; ++j)
        if (!((taken >> j) & 1u) && id[j] != kNoId && better(v[j], id[j], best.v, best.i))
          best.v = v[j], best.i = id[j], bj = j;
      const VI win = warp_best(best);
      if (bj >= 0 && best.i == win.i) taken |= 1u << bj;
      if (lane == 0) ov[it] = win.v, oi[it] = win.i;
    }
  }
  __syncwarp();
}

constexpr int kTopkCap = 64;       // compacted candidates per warp (one 64-element sort)
constexpr int kTopkCandTiles = 64; // vocab tiles scanned on the direct path
constexpr int kTopkCand = 512;     // candidates kept on the direct path

// Top-k and logsumexp of logit rows, one CTA per row.  The row is cut into
// 128-entry vocab tiles with (m_i, s_i) = (max, sum e^(z - m_i)) per tile,
// given by the projection that wrote the logits (or formed here when
// stats == nullptr); logsumexp = M + log sum_i s_i e^(m_i - M).  The k-th
// largest tile maximum thr is a lower bound of the k-th largest logit (k tiles
// each hold an entry >= thr), so every top-k entry lies in a tile with
// m_i >= thr and is itself >= thr: those tiles are scanned and their entries
// >= thr ranked (larger value, then lower id).  Rows whose ties defeat the
// bounds (more than kTopkCandTiles tiles or kTopkCand entries at or above thr)
// are ranked by a scan of the whole row instead.
__global__ void __launch_bounds__(256) k_topk_rows(const float *__restrict__ logits,
                                                   const float2 *__restrict__ stats, int V, int k,
                                                   int32_t *__restrict__ ids,
                                                   float *__restrict__ logp) {
  extern __shared__ float tk_sm[];  // [nt] tile maxima, [nt] tile sums
  __shared__ float cv[kTopkCand];
  __shared__ int ci[kTopkCand];
  __shared__ int ctile[kTopkCandTiles];
  __shared__ float sc[8][kTopkCap];
  __shared__ int sci[8][kTopkCap];
  __shared__ float wv[8 * DFLASH_MAX_TOPK];
  __shared__ int wi[8 * DFLASH_MAX_TOPK];
  __shared__ float rv[DFLASH_MAX_TOPK];
  __shared__ int ri[DFLASH_MAX_TOPK];
  __shared__ float red[32];
  __shared__ float s_thr;
  __shared__ int n_tiles, n_cand;
  pdl_launch();
  pdl_wait();
  const int row = blockIdx.x, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int nt = (V + 127) / 128;
  float *sm_m = tk_sm, *sm_s = tk_sm + nt;
  const float *z = logits + (size_t)row * V;
  constexpr int LB = 8;  // loads in flight per thread in the staging loops
  if (tid == 0) n_tiles = 0, n_cand = 0;
  if (stats) {
    const float2 *st = stats + (size_t)row * nt;
    for (int i0 = 0; i0 < nt; i0 += LB * 256) {
      float2 q[LB];
#pragma unroll
      for (int j = 0; j < LB; ++j)
        if (i0 + j * 256 + tid < nt) q[j] = st[i0 + j * 256 + tid];
#pragma unroll
      for (int j = 0; j < LB; ++j)
        if (i0 + j * 256 + tid < nt) {
          sm_m[i0 + j * 256 + tid] = q[j].x;
          sm_s[i0 + j * 256 + tid] = q[j].y;
        }
    }
  } else {
    for (int i = tid; i < nt; i += blockDim.x) {
      const int e1 = min(V, 128 * i + 128);
      float m = -INFINITY, sum = 0.f;
      for (int e = 128 * i; e < e1; ++e) m = fmaxf(m, z[e]);
      for (int e = 128 * i; e < e1; ++e) sum += expf(z[e] - m);
      sm_m[i] = m;
      sm_s[i] = sum;
    }
  }
  __syncthreads();
  float mm = -INFINITY;
  for (int i = tid; i < nt; i += blockDim.x) mm = fmaxf(mm, sm_m[i]);
  const float M = block_max(mm, red);
  float ss = 0.f;
  for (int i = tid; i < nt; i += blockDim.x) ss += sm_s[i] * expf(sm_m[i] - M);
  const float lse = M + logf(block_sum(ss, red));

  // threshold: the k-th largest tile maximum (warp 0)
  if (w == 0) {
    float lm = -INFINITY;
    for (int i = lane; i < nt; i += 32) lm = fmaxf(lm, sm_m[i]);
    const float t0 = __shfl_sync(0xffffffffu, warp_sort_desc(lm), k - 1);
    int cnt = 0;
    for (int i = lane; i < nt; i += 32) cnt += sm_m[i] >= t0 ? 1 : 0;
    int pre = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, pre, o);
      if (lane >= o) pre += y;
    }
    const int total = __shfl_sync(0xffffffffu, pre, 31);
    float thr = t0;
    if (total <= kTopkCap) {  // rank the maxima >= t0 exactly: thr = the k-th of them
      int wpos = pre - cnt;
      for (int i = lane; i < nt; i += 32)
        if (sm_m[i] >= t0) sc[0][wpos++] = sm_m[i];
      __syncwarp();
      float sv[2];
      int si[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int e = 32 * q + lane;
        sv[q] = e < total ? sc[0][e] : -INFINITY;
        si[q] = e < total ? e : kNoId;
      }
      warp_sort64(sv, si, lane);  // element k-1 is in half 0 (k <= 32)
      thr = __shfl_sync(0xffffffffu, sv[0], k - 1);
    }
    if (lane == 0) s_thr = thr;
  }
  __syncthreads();
  const float thr = s_thr;
  for (int i = tid; i < nt; i += blockDim.x)
    if (sm_m[i] >= thr) {
      const int pos = atomicAdd(&n_tiles, 1);
      if (pos < kTopkCandTiles) ctile[pos] = i;
    }
  __syncthreads();
  bool direct = n_tiles <= kTopkCandTiles;
  if (direct) {
    // the candidate tiles' entries, flattened over the threads (entry f of
    // the list is entry f % 128 of tile ctile[f / 128]), LB loads in flight
    const int nf = n_tiles * 128;
    for (int f0 = 0; f0 < nf; f0 += LB * 256) {
      float x[LB];
      int e[LB];
#pragma unroll
      for (int j = 0; j < LB; ++j) {
        const int f = f0 + j * 256 + tid;
        e[j] = f < nf ? 128 * ctile[f >> 7] + (f & 127) : V;
        if (e[j] < V) x[j] = z[e[j]];
      }
#pragma unroll
      for (int j = 0; j < LB; ++j)
        if (e[j] < V && x[j] >= thr) {
          const int pos = atomicAdd(&n_cand, 1);
          if (pos < kTopkCand) cv[pos] = x[j], ci[pos] = e[j];
        }
    }
    __syncthreads();
    direct = n_cand <= kTopkCand;
  }
  if (direct) {
    if (w != 0) return;
    const int n = n_cand;
    if (n <= kTopkCap) {
      float sv[2];
      int si[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int e = 32 * q + lane;
        sv[q] = e < n ? cv[e] : -INFINITY;
        si[q] = e < n ? ci[e] : kNoId;
      }
      warp_sort64(sv, si, lane);
      if (lane < k) {
        ids[(size_t)row * k + lane] = si[0];
        logp[(size_t)row * k + lane] = sv[0] - lse;
      }
    } else {
      float v[kTopkCand / 32];
      int id[kTopkCand / 32];
#pragma unroll
      for (int q = 0; q < kTopkCand / 32; ++q) {
        const int e = 32 * q + lane;
        v[q] = e < n ? cv[e] : -INFINITY;
        id[q] = e < n ? ci[e] : kNoId;
      }
      warp_topk<kTopkCand / 32>(v, id, k, sc[0], sci[0], kTopkCap, rv, ri, lane);
      for (int it = lane; it < k; it += 32) {
        ids[(size_t)row * k + it] = ri[it];
        logp[(size_t)row * k + it] = rv[it] - lse;
      }
    }
    return;
  }

  // whole-row scan: 8192 entries per pass (8 warps x 1024); warp 0 merges the
  // warps' lists with the running list
  if (tid < k) rv[tid] = -INFINITY, ri[tid] = kNoId;
  __syncthreads();
  for (int base = 0; base < V; base += 8192) {
    float v[32];
    int id[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int e = base + w * 1024 + j * 32 + lane;
      v[j] = e < V ? z[e] : -INFINITY;
      id[j] = e < V ? e : kNoId;
    }
    warp_topk<32>(v, id, k, sc[w], sci[w], kTopkCap, wv + w * k, wi + w * k, lane);
    __syncthreads();
    if (w == 0) {
      float mv[9];
      int mi[9];
#pragma unroll
      for (int q = 0; q < 9; ++q) {
        const int e = 32 * q + lane;
        mv[q] = -INFINITY;
        mi[q] = kNoId;
        if (e < 8 * k) mv[q] = wv[e], mi[q] = wi[e];
        else if (e < 9 * k) mv[q] = rv[e - 8 * k], mi[q] = ri[e - 8 * k];
      }
      __syncwarp();
      warp_topk<9>(mv, mi, k, sc[0], sci[0], kTopkCap, rv, ri, lane);
    }
    __syncthreads();
  }
  for (int it = tid; it < k; it += blockDim.x) {
    ids[(size_t)row * k + it] = ri[it];
    logp[(size_t)row * k + it] = rv[it] - lse;
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

// Pair scores and the Viterbi walk.  CTA (t, b) stages the rows of request b's
// candidates at positions t and t+1 (U of position t, or of the anchor for
// t = 0; Vp of position t+1) and writes pair[b][t][i][j] = U_i . Vp_j, then
// takes a ticket on its request; the CTA that finishes the request's last
// position (no waiting) walks max-sum Viterbi over the K-1 positions of k
// candidates on all of them (staged in shared memory).  Ties go to the lower
// candidate rank.  tickets: B ints, zero on entry and on exit.
__global__ void __launch_bounds__(256) k_sel_pairs(const float *__restrict__ U,
                                                   const float *__restrict__ Vp, int K, int k,
                                                   int r, float *__restrict__ pair, int *tickets,
                                                   const int32_t *__restrict__ topk_ids,
                                                   const float *__restrict__ topk_logp,
                                                   int32_t *__restrict__ path,
                                                   float *__restrict__ score,
                                                   const float *__restrict__ tab, int V,
                                                   const int32_t *__restrict__ anchor, int *err) {
  extern __shared__ float sm[];
  const int LDR = r + 1;  // odd row stride: the threads of a warp hit distinct banks
  float *su = sm, *sv = sm + (size_t)k * LDR;
  __shared__ float delta[DFLASH_MAX_TOPK];
  __shared__ int bp[DFLASH_MAX_BLOCK][DFLASH_MAX_TOPK];
  __shared__ int s_last;
  __shared__ const float *s_src[2 * DFLASH_MAX_TOPK];
  pdl_launch();
  pdl_wait();
  const int t = blockIdx.x, b = blockIdx.y;
  const int R = 1 + (K - 1) * k;
  const int np = t == 0 ? 1 : k;
  const size_t ubase = (size_t)b * R + (t == 0 ? 0 : 1 + (size_t)(t - 1) * k);
  const size_t vbase = (size_t)b * R + 1 + (size_t)t * k;
  const int r4 = r / 4, nrow = np + k;
  // the source row of every staged row first (one round trip for the tokens),
  // then all of a thread's row loads in flight at once
  if (threadIdx.x < nrow) {
    const int row = threadIdx.x;
    const float *src;
    if (tab) {
      // the rows' tokens: the anchor or position t-1's candidates (P_u side),
      // position t's candidates (P_v side); their projections from the table
      int tok = row < np ? (t == 0 ? anchor[b] : topk_ids[((size_t)b * (K - 1) + t - 1) * k + row])
                         : topk_ids[((size_t)b * (K - 1) + t) * k + (row - np)];
      if (tok < 0 || tok >= V) {
        set_err(err, DFLASH_DEV_TOKEN_RANGE);
        tok = tok < 0 ? 0 : V - 1;
      }
      src = tab + ((row < np ? 0 : (size_t)V) + (size_t)tok) * r;
    } else {
      src = row < np ? U + (ubase + row) * r : Vp + (vbase + row - np) * r;
    }
    s_src[row] = src;
  }
  __syncthreads();
  constexpr int SB = 8;  // 16-byte loads in flight per thread
  for (int e0 = 0; e0 < nrow * r4; e0 += SB * 256) {
    float4 q[SB];
#pragma unroll
    for (int j = 0; j < SB; ++j) {
      const int e = e0 + j * 256 + threadIdx.x;
      if (e < nrow * r4) q[j] = ((const float4 *)s_src[e / r4])[e % r4];
    }
#pragma unroll
    for (int j = 0; j < SB; ++j) {
      const int e = e0 + j * 256 + threadIdx.x;
      if (e < nrow * r4) {
        const int row = e / r4, c = e % r4;
        float *dst = (row < np ? su + (size_t)row * LDR : sv + (size_t)(row - np) * LDR) + 4 * c;
        dst[0] = q[j].x, dst[1] = q[j].y, dst[2] = q[j].z, dst[3] = q[j].w;
      }
    }
  }
  __syncthreads();
  float *out = pair + ((size_t)b * (K - 1) + t) * k * k;
  for (int e = threadIdx.x; e < np * k; e += blockDim.x) {
    const int i = e / k, j = e % k;
    const float *a = su + (size_t)i * LDR, *c = sv + (size_t)j * LDR;
    float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
    for (int q = 0; q < r; q += 4) {
      d0 = fmaf(a[q], c[q], d0);
      d1 = fmaf(a[q + 1], c[q + 1], d1);
      d2 = fmaf(a[q + 2], c[q + 2], d2);
      d3 = fmaf(a[q + 3], c[q + 3], d3);
    }
    out[e] = (d0 + d1) + (d2 + d3);
  }
  // ticket: the last position of the request walks the lattice
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    s_last = atomicAdd(&tickets[b], 1) == K - 2;
    if (s_last) tickets[b] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int npair = (K - 1) * k * k, nlp = (K - 1) * k;
  float *sp = sm, *slp = sm + npair;  // the staged rows are no longer needed
  const float *pr = pair + (size_t)b * npair;
  const float *lp = topk_logp + (size_t)b * nlp;
  for (int e = threadIdx.x; e < npair; e += blockDim.x) sp[e] = __ldcg(pr + e);
  for (int e = threadIdx.x; e < nlp; e += blockDim.x) slp[e] = lp[e];
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int j = threadIdx.x;
  for (int tt = 0; tt < K - 1; ++tt) {
    const float *ps = sp + (size_t)tt * k * k;
    float nd = 0.f;
    int arg = 0;
    if (j < k) {
      if (tt == 0) {
        nd = slp[j] + ps[j];
      } else {
        float best = -INFINITY;
        for (int i = 0; i < k; ++i) {
          const float c = delta[i] + ps[i * k + j];
          if (c > best) best = c, arg = i;  // strict: the lower rank keeps ties
        }
        nd = slp[tt * k + j] + best;
      }
    }
    __syncwarp();
    if (j < k) {
      delta[j] = nd;
      bp[tt][j] = arg;
    }
    __syncwarp();
  }
  if (j == 0) {
    int best = 0;
    for (int i = 1; i < k; ++i)
      if (delta[i] > delta[best]) best = i;
    score[b] = delta[best];
    int c = best;
    for (int tt = K - 2; tt >= 0; --tt) {
      path[(size_t)b * (K - 1) + tt] = topk_ids[((size_t)b * (K - 1) + tt) * k + c];
      c = bp[tt][c];
    }
  }
}

// argmax of one chunk of one target-logit row -> partial (value, id); NaN ranks
// above every number (better_nan_max).  better_nan_max is a total order on
// (value, id), so the visiting order does not change the result: a 16-byte
// aligned row is read as 16-byte words, all of a thread's words issued before
// the first comparison (one memory round trip per chunk), the ragged end of
// the chunk element by element.
template <typename L>
__global__ void __launch_bounds__(256) k_argmax_partial(const L *__restrict__ logits, int V,
                                                        float *__restrict__ partial) {
  constexpr int NT = 256, VW = 16 / sizeof(L), NV = dflh::kArgmaxChunk / (NT * VW);
  static_assert(dflh::kArgmaxChunk % (NT * VW) == 0, "chunk is whole 16-byte words per thread");
  __shared__ float redv[32];
  __shared__ int redi[32];
  pdl_launch();
  pdl_wait();
  const int chunk = blockIdx.x, row = blockIdx.y, nch = gridDim.x, tid = threadIdx.x;
  const int c0 = chunk * dflh::kArgmaxChunk, c1 = min(V, c0 + dflh::kArgmaxChunk);
  const L *z = logits + (size_t)row * V;
  VI best{-INFINITY, 0x7fffffff};
  int tail = c0;  // first element left to the element-wise loop
  if ((reinterpret_cast<uintptr_t>(z + c0) & 15) == 0) {
    const int nw = (c1 - c0) / VW;  // whole words in the chunk
    const uint4 *zw = reinterpret_cast<const uint4 *>(z + c0);
    uint4 r[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j)
      if (j * NT + tid < nw) r[j] = __ldg(zw + j * NT + tid);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int q = j * NT + tid;
      if (q < nw) {
        const L *e = reinterpret_cast<const L *>(&r[j]);
#pragma unroll
        for (int u = 0; u < VW; ++u) {
          const float v = ldf(e + u);
          const int i = c0 + q * VW + u;
          if (better_nan_max(v, i, best.v, best.i)) best.v = v, best.i = i;
        }
      }
    }
    tail = c0 + nw * VW;
  }
  for (int i = tail + tid; i < c1; i += NT) {
    const float v = ldf(z + i);
    if (better_nan_max(v, i, best.v, best.i)) best.v = v, best.i = i;
  }
  best = block_best<true>(best, redv, redi);
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
      if (better_nan_max(v, id, best.v, best.i)) best.v = v, best.i = id;
    }
    best = warp_best<true>(best);
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

// ---------------------------------------------------------------------------
// sampling walk and speculative rejection sampling
// ---------------------------------------------------------------------------

// Inverse-CDF draw (as the oracle's draw_index): the smallest j whose running
// sum of w exceeds u * total, walking w[0..n) in order; the last positive
// weight when rounding leaves none.
__device__ __forceinline__ int draw_inv_cdf(const float *w, int n, float u, float total) {
  const float target = u * total;
  float c = 0.f;
  int last = -1;
  for (int j = 0; j < n; ++j) {
    if (w[j] > 0.f) last = j;
    c += w[j];
    if (target < c && w[j] > 0.f) return j;
  }
  return last < 0 ? 0 : last;
}

// One CTA per request: the temperature-1 walk from the anchor.  Position t's
// candidate j gets s_j = logp_t(j) + u(prev) . v(c_tj) with the projections
// from the selector table (tab, by token) or from the gathered rows (U, Vp
// [B*R][r], R = 1 + (K-1)*k: anchor first, then the candidates by position and
// rank); q_t = softmax(s) is written out and one candidate is drawn with the
// uniform uw[b][t].  prev = the token drawn at t-1 (the anchor at t = 0).
//
// Greedy mode (uw == nullptr): the walk takes argmax_j s_j (the lower rank on
// ties) and score[b] receives the summed chosen scores.  gate (optional,
// [B*(K-1)][r] pre-activations): the predecessor's projection is multiplied by
// sigmoid(gate row of position t) before the dot products (the context gate).
__global__ void __launch_bounds__(256) k_sample_walk(
    const float *__restrict__ U, const float *__restrict__ Vp, const int32_t *__restrict__ ids,
    const float *__restrict__ logp, int K, int k, int r, const float *__restrict__ tab, int V,
    const int32_t *__restrict__ anchor, const float *__restrict__ uw, int32_t *__restrict__ path,
    float *__restrict__ pq, const float *__restrict__ gate, float *__restrict__ score, int *err) {
  extern __shared__ float sw[];
  float *up = sw;  // [r] projection of the predecessor
  __shared__ float sc[DFLASH_MAX_TOPK];
  __shared__ int s_tok, s_row;
  pdl_launch();
  pdl_wait();
  const int b = blockIdx.x, T = K - 1, R = 1 + T * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) {
    int a = anchor[b];
    if (a < 0 || a >= V) {
      set_err(err, DFLASH_DEV_TOKEN_RANGE);
      a = a < 0 ? 0 : V - 1;
    }
    s_tok = a;
    s_row = 0;
  }
  __syncthreads();
  float total = 0.f;  // greedy: summed chosen scores (thread 0)
  for (int t = 0; t < T; ++t) {
    const float *usrc = tab ? tab + (size_t)s_tok * r : U + ((size_t)b * R + s_row) * r;
    const float *grow = gate ? gate + ((size_t)b * T + t) * r : nullptr;
    for (int i = threadIdx.x; i < r; i += blockDim.x)
      up[i] = grow ? usrc[i] * (1.f / (1.f + expf(-grow[i]))) : usrc[i];
    __syncthreads();
    const size_t cb = ((size_t)b * T + t) * k;
    for (int j = warp; j < k; j += nw) {
      int c = ids[cb + j];
      if (c < 0 || c >= V) {
        if (lane == 0) set_err(err, DFLASH_DEV_TOKEN_RANGE);
        c = c < 0 ? 0 : V - 1;
      }
      const float *vsrc = tab ? tab + ((size_t)V + c) * r : Vp + ((size_t)b * R + 1 + (size_t)t * k + j) * r;
      float acc = 0.f;
      for (int i = lane; i < r; i += 32) acc = fmaf(up[i], vsrc[i], acc);
      acc = warp_sum(acc);
      if (lane == 0) sc[j] = logp[cb + j] + acc;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int jd = 0;
      if (uw) {
        float m = -INFINITY;
        for (int j = 0; j < k; ++j) m = fmaxf(m, sc[j]);
        float e[DFLASH_MAX_TOPK], tot = 0.f;
        for (int j = 0; j < k; ++j) {
          e[j] = expf(sc[j] - m);
          tot += e[j];
        }
        for (int j = 0; j < k; ++j) pq[cb + j] = e[j] / tot;
        jd = draw_inv_cdf(e, k, uw[(size_t)b * T + t], tot);
      } else {
        for (int j = 1; j < k; ++j)
          if (sc[j] > sc[jd]) jd = j;
        total += sc[jd];
        if (t == T - 1) score[b] = total;
      }
      int c = ids[cb + jd];
      c = c < 0 ? 0 : c >= V ? V - 1 : c;
      path[(size_t)b * T + t] = c;
      s_tok = c;
      s_row = 1 + t * k + jd;
    }
    __syncthreads();
  }
}

// (max, sum e^(z - max)) of one chunk of one target row -> part[row][chunk]
template <typename L>
__global__ void __launch_bounds__(256) k_row_chunk_stats(const L *__restrict__ logits, int V,
                                                          float2 *__restrict__ part) {
  __shared__ float red[32];
  pdl_launch();
  pdl_wait();
  const int chunk = blockIdx.x, row = blockIdx.y, nch = gridDim.x;
  const int c0 = chunk * dflh::kArgmaxChunk, c1 = min(V, c0 + dflh::kArgmaxChunk);
  const L *z = logits + (size_t)row * V;
  float m = -INFINITY;
  for (int i = c0 + threadIdx.x; i < c1; i += blockDim.x) m = fmaxf(m, ldf(z + i));
  m = block_max(m, red);
  float s = 0.f;
  if (m > -INFINITY)
    for (int i = c0 + threadIdx.x; i < c1; i += blockDim.x) s += expf(ldf(z + i) - m);
  s = block_sum(s, red);
  if (threadIdx.x == 0) part[(size_t)row * nch + chunk] = make_float2(m, s);
}

// The row's softmax normaliser from its chunk partials, in chunk order (every
// caller forms exactly the same values).
__device__ __forceinline__ float2 row_norm(const float2 *part, int nch) {
  float M = -INFINITY;
  for (int c = 0; c < nch; ++c) M = fmaxf(M, part[c].x);
  float S = 0.f;
  for (int c = 0; c < nch; ++c)
    if (part[c].x > -INFINITY) S += part[c].y * expf(part[c].x - M);
  return make_float2(M, S);
}

// Residual weight of token v in target row i of request b: max(0, p_i(v) -
// q_i(v)) for draft rows (q from the proposal over the row's candidates),
// p_i(v) for the last row (the bonus draw).
struct RowQ {
  int id[DFLASH_MAX_TOPK];
  float q[DFLASH_MAX_TOPK];
  int n;
};
__device__ __forceinline__ float resid_w(float z, float2 MS, int v, const RowQ &rq) {
  const float p = MS.y > 0.f ? expf(z - MS.x) / MS.y : 0.f;
  float q = 0.f;
  for (int j = 0; j < rq.n; ++j)
    if (rq.id[j] == v) q += rq.q[j];
  return fmaxf(p - q, 0.f);
}

// Per (chunk, row): the row's residual weights summed over the chunk ->
// rsum[row][chunk], and its target probabilities -> psum[row][chunk].
template <typename L>
__global__ void __launch_bounds__(256) k_resid_chunks(const L *__restrict__ logits, int V, int K,
                                                       int k, const float2 *__restrict__ part,
                                                       const int32_t *__restrict__ ids,
                                                       const float *__restrict__ pq,
                                                       float *__restrict__ rsum,
                                                       float *__restrict__ psum) {
  __shared__ float red[32];
  __shared__ RowQ rq;
  pdl_launch();
  pdl_wait();
  const int chunk = blockIdx.x, row = blockIdx.y, nch = gridDim.x;
  const int b = row / K, i = row % K;
  if (threadIdx.x == 0) {
    rq.n = i < K - 1 ? k : 0;
    for (int j = 0; j < rq.n; ++j) {
      rq.id[j] = ids[((size_t)b * (K - 1) + i) * k + j];
      rq.q[j] = pq[((size_t)b * (K - 1) + i) * k + j];
    }
  }
  __syncthreads();
  const float2 MS = row_norm(part + (size_t)row * nch, nch);
  const int c0 = chunk * dflh::kArgmaxChunk, c1 = min(V, c0 + dflh::kArgmaxChunk);
  const L *z = logits + (size_t)row * V;
  float rs = 0.f, ps = 0.f;
  for (int v = c0 + threadIdx.x; v < c1; v += blockDim.x) {
    const float zv = ldf(z + v);
    ps += MS.y > 0.f ? expf(zv - MS.x) / MS.y : 0.f;
    rs += resid_w(zv, MS, v, rq);
  }
  rs = block_sum(rs, red);
  ps = block_sum(ps, red);
  if (threadIdx.x == 0) {
    rsum[(size_t)row * nch + chunk] = rs;
    psum[(size_t)row * nch + chunk] = ps;
  }
}

// One CTA per request: accept draft i while u0 q_i(x) < p_i(x); at the first
// rejection draw the replacement from the residual max(0, p_i - q_i) (from p_i
// when that is zero everywhere), else the bonus token from p_{K-1}; the draw
// walks the chunk sums in order, then the chosen chunk's weights in token order.
template <typename L>
__global__ void __launch_bounds__(256) k_accept_sample(
    const L *__restrict__ logits, int V, int K, int k, int nch, const int32_t *__restrict__ path,
    const int32_t *__restrict__ ids, const float *__restrict__ pq,
    const float2 *__restrict__ part, const float *__restrict__ rsum,
    const float *__restrict__ psum, const float *__restrict__ uni,
    int32_t *__restrict__ accept_len, int32_t *__restrict__ tokens) {
  constexpr int NT = 256, PER = dflh::kArgmaxChunk / NT;  // 32 tokens per thread
  __shared__ int s_stop, s_chunk, s_usep, s_tok;
  __shared__ float s_target, s_pref[NT];
  __shared__ RowQ rq;
  pdl_launch();
  pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x;
  if (tid == 0) {
    int stop = K - 1;
    for (int i = 0; i < K - 1; ++i) {
      const size_t row = (size_t)b * K + i;
      const float2 MS = row_norm(part + row * nch, nch);
      const int x = path[(size_t)b * (K - 1) + i];
      float qx = 0.f;
      for (int j = 0; j < k; ++j)
        if (ids[((size_t)b * (K - 1) + i) * k + j] == x) qx += pq[((size_t)b * (K - 1) + i) * k + j];
      const float px = (x >= 0 && x < V && MS.y > 0.f)
                           ? expf(ldf(logits + row * V + x) - MS.x) / MS.y : 0.f;
      if (!(uni[row * 2] * qx < px)) {
        stop = i;
        break;
      }
    }
    const size_t row = (size_t)b * K + stop;
    rq.n = stop < K - 1 ? k : 0;
    for (int j = 0; j < rq.n; ++j) {
      rq.id[j] = ids[((size_t)b * (K - 1) + stop) * k + j];
      rq.q[j] = pq[((size_t)b * (K - 1) + stop) * k + j];
    }
    float tot = 0.f;
    for (int c = 0; c < nch; ++c) tot += rsum[row * nch + c];
    const bool usep = !(tot > 0.f);
    const float *cs = (usep ? psum : rsum) + row * nch;
    if (usep) {
      tot = 0.f;
      for (int c = 0; c < nch; ++c) tot += cs[c];
    }
    float target = uni[row * 2 + 1] * tot, run = 0.f;
    int ch = -1, lastpos = 0;
    for (int c = 0; c < nch; ++c) {
      if (cs[c] > 0.f) lastpos = c;
      if (ch < 0 && target < run + cs[c] && cs[c] > 0.f) ch = c;
      if (ch < 0) run += cs[c];
    }
    // rounding left the target past every chunk: the last positive weight
    if (ch < 0) ch = lastpos, run = 0.f, target = 3.0e38f;
    s_stop = stop;
    s_chunk = ch;
    s_usep = usep;
    s_target = target - run;  // position inside the chunk
    s_tok = -1;
  }
  __syncthreads();
  const int stop = s_stop;
  const size_t row = (size_t)b * K + stop;
  const float2 MS = row_norm(part + row * nch, nch);
  const L *z = logits + row * V;
  const int c0 = s_chunk * dflh::kArgmaxChunk;
  // this thread's run of PER consecutive tokens
  float w[PER], own = 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int v = c0 + tid * PER + e;
    float x = 0.f;
    if (v < V) {
      const float zv = ldf(z + v);
      x = s_usep ? (MS.y > 0.f ? expf(zv - MS.x) / MS.y : 0.f) : resid_w(zv, MS, v, rq);
    }
    w[e] = x;
    own += x;
  }
  s_pref[tid] = own;
  __syncthreads();
  if (tid == 0) {  // exclusive prefix over the threads, in order
    float run = 0.f;
    int hit = -1, lastpos = -1;
    for (int t = 0; t < NT; ++t) {
      const float o = s_pref[t];
      if (o > 0.f) lastpos = t;
      if (hit < 0 && s_target < run + o && o > 0.f) hit = t;
      s_pref[t] = run;
      run += o;
    }
    if (hit < 0) hit = lastpos < 0 ? 0 : lastpos, s_target = s_pref[hit] + 3.0e38f;
    s_tok = hit;  // the thread holding the draw
  }
  __syncthreads();
  if (tid == s_tok) {
    const float tgt = s_target - s_pref[tid];
    const int j = draw_inv_cdf(w, PER, 1.f, tgt > 0.f ? tgt : 0.f);
    // draw_inv_cdf(w, n, 1, T) walks the running sum against T directly
    int v = c0 + tid * PER + j;
    v = v >= V ? V - 1 : v;
    for (int i = 0; i < K; ++i)
      tokens[(size_t)b * K + i] = i < stop ? path[(size_t)b * (K - 1) + i] : i == stop ? v : -1;
    accept_len[b] = stop + 1;
  }
}

}  // namespace dfl

namespace dflh {

int launch_topk(const float *logits, const float2 *stats, int rows, int V, int k, int32_t *ids,
                float *logp, cudaStream_t st) {
  if (rows <= 0) return DFLASH_OK;
  const int nt = topk_tiles(V);
  if (nt > kTopkMaxTiles || k < 1 || k > DFLASH_MAX_TOPK || k > V) return DFLASH_ERR_DIMS;
  const size_t smem = (size_t)nt * 2 * sizeof(float);
  static int attr_done = 0;
  if (smem > 48 * 1024 && !attr_done) {
    if (cudaFuncSetAttribute(dfl::k_topk_rows, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTopkMaxTiles * 2 * (int)sizeof(float)) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    attr_done = 1;
  }
  DFL_CHECK_LAUNCH(
      launch(dfl::k_topk_rows, dim3(rows), dim3(256), smem, st, logits, stats, V, k, ids, logp));
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

int launch_viterbi(const float *U, const float *Vp, const int32_t *topk_ids,
                   const float *topk_logp, int B, int K, int k, int r, float *pair, int *tickets,
                   int32_t *path, float *score, const float *tab, int V, const int32_t *anchor,
                   int *err, cudaStream_t st) {
  const size_t smem = sizeof(float) * std::max(2 * (size_t)k * (r + 1),
                                               (size_t)(K - 1) * k * k + (size_t)(K - 1) * k);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(dfl::k_sel_pairs, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return DFLASH_ERR_CUDA;
  }
  DFL_CHECK_LAUNCH(launch(dfl::k_sel_pairs, dim3(K - 1, B), dim3(256), smem, st, U, Vp, K, k, r,
                          pair, tickets, topk_ids, topk_logp, path, score, tab, V, anchor, err));
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

int launch_sample_walk(const float *U, const float *Vp, const int32_t *topk_ids,
                       const float *topk_logp, int B, int K, int k, int r, const float *tab, int V,
                       const int32_t *anchor, const float *uniforms, int32_t *path, float *path_q,
                       int *err, cudaStream_t st) {
  const size_t smem = sizeof(float) * (size_t)r;
  DFL_CHECK_LAUNCH(launch(dfl::k_sample_walk, dim3(B), dim3(256), smem, st, U, Vp, topk_ids,
                          topk_logp, K, k, r, tab, V, anchor, uniforms, path, path_q,
                          (const float *)nullptr, (float *)nullptr, err));
  return DFLASH_OK;
}

int launch_greedy_walk(const float *U, const float *Vp, const int32_t *topk_ids,
                       const float *topk_logp, int B, int K, int k, int r, const float *tab, int V,
                       const int32_t *anchor, const float *gate, int32_t *path, float *score,
                       int *err, cudaStream_t st) {
  const size_t smem = sizeof(float) * (size_t)r;
  DFL_CHECK_LAUNCH(launch(dfl::k_sample_walk, dim3(B), dim3(256), smem, st, U, Vp, topk_ids,
                          topk_logp, K, k, r, tab, V, anchor, (const float *)nullptr, path,
                          (float *)nullptr, gate, score, err));
  return DFLASH_OK;
}

size_t accept_sample_floats(int B, int K, int V) {
  return (size_t)B * K * argmax_chunks(V) * 4;
}

int launch_accept_sample(const int32_t *path, const int32_t *topk_ids, const float *path_q,
                         const void *logits, int dtype, int B, int K, int V, int k,
                         const float *uniforms, float *scratch, int32_t *accept_len,
                         int32_t *tokens, cudaStream_t st) {
  const int nch = argmax_chunks(V);
  const size_t rows = (size_t)B * K;
  float2 *part = (float2 *)scratch;
  float *rsum = scratch + rows * nch * 2, *psum = rsum + rows * nch;
  if (dtype == DFLASH_F32) {
    const float *z = (const float *)logits;
    DFL_CHECK_LAUNCH(launch(dfl::k_row_chunk_stats<float>, dim3(nch, B * K), dim3(256), 0, st, z,
                            V, part));
    DFL_CHECK_LAUNCH(launch(dfl::k_resid_chunks<float>, dim3(nch, B * K), dim3(256), 0, st, z, V,
                            K, k, (const float2 *)part, topk_ids, path_q, rsum, psum));
    DFL_CHECK_LAUNCH(launch(dfl::k_accept_sample<float>, dim3(B), dim3(256), 0, st, z, V, K, k,
                            nch, path, topk_ids, path_q, (const float2 *)part, (const float *)rsum,
                            (const float *)psum, uniforms, accept_len, tokens));
  } else {
    const dfl::bf16 *z = (const dfl::bf16 *)logits;
    DFL_CHECK_LAUNCH(launch(dfl::k_row_chunk_stats<dfl::bf16>, dim3(nch, B * K), dim3(256), 0, st,
                            z, V, part));
    DFL_CHECK_LAUNCH(launch(dfl::k_resid_chunks<dfl::bf16>, dim3(nch, B * K), dim3(256), 0, st, z,
                            V, K, k, (const float2 *)part, topk_ids, path_q, rsum, psum));
    DFL_CHECK_LAUNCH(launch(dfl::k_accept_sample<dfl::bf16>, dim3(B), dim3(256), 0, st, z, V, K,
                            k, nch, path, topk_ids, path_q, (const float2 *)part,
                            (const float *)rsum, (const float *)psum, uniforms, accept_len,
                            tokens));
  }
  return DFLASH_OK;
}

}  // namespace dflh
