// Non-causal block attention (split over keys, then combined).
//
// Work item = (request b, kv head, query group, key split).  The K block
// queries of the group's q heads (K * Hq/Hkv rows) share every key/value tile
// staged in shared memory.  Keys: the last min(window, ctx_len) context
// positions from the paged cache, then the K block slots; no mask.  Each split
// keeps an online softmax (running max m, sum l, unnormalised output) and
// writes it out; the combine kernel merges the splits in order.
#include <math.h>

#include "attention.cuh"

namespace dfl {

constexpr int kQG = 64;   // query rows per CTA
constexpr int kCH = 64;   // keys per shared-memory tile

template <typename S, int DH>
__global__ void __launch_bounds__(256) k_attn_split(
    const S *__restrict__ qb, const S *__restrict__ kb, const S *__restrict__ vb,
    const S *__restrict__ kc, const S *__restrict__ vc, size_t layer_off,
    const int32_t *__restrict__ table, int max_pages, int num_pages, int P,
    const int32_t *__restrict__ ctx_len, int K, int Hq, int Hkv, int window, int kps, int nsplit,
    int nqg, float *__restrict__ part, int *err) {
  constexpr int LD = DH + 1;
  extern __shared__ float sm[];
  float *sQ = sm;                      // [kQG][LD]
  float *sK = sQ + kQG * LD;           // [kCH][LD]
  float *sV = sK + kCH * LD;           // [kCH][LD]
  float *sS = sV + kCH * LD;           // [kQG][kCH + 1]
  __shared__ int s_valid[kCH];
  pdl_launch();
  pdl_wait();

  const int split = blockIdx.x, kvh = blockIdx.y;
  const int b = blockIdx.z / nqg, qgi = blockIdx.z % nqg;
  const int grp = Hq / Hkv;
  const int QR = K * grp;
  const int ctx = ctx_len[b];
  const int n_ctx = ctx < window ? (ctx > 0 ? ctx : 0) : window;
  const int lo = ctx - n_ctx;
  const int n_keys = n_ctx + K;
  const int k_begin = split * kps;
  if (k_begin >= n_keys) return;
  const int k_end = min(n_keys, k_begin + kps);
  const float scale = rsqrtf((float)DH);

  // query rows of this group: qr = i*grp + g -> slot i, q head kvh*grp + g
  const int tid = threadIdx.x;
  for (int e = tid; e < kQG * DH; e += 256) {
    const int qr = e / DH, d = e % DH;
    const int qrg = qgi * kQG + qr;
    float v = 0.f;
    if (qrg < QR) {
      const int i = qrg / grp, g = qrg % grp;
      v = ldf(qb + ((size_t)(b * K + i) * Hq + kvh * grp + g) * DH + d);
    }
    sQ[qr * LD + d] = v;
  }

  constexpr int DPT = DH / 4;  // output columns per thread
  const int row = tid >> 2, part4 = tid & 3;
  float acc[DPT];
#pragma unroll
  for (int j = 0; j < DPT; ++j) acc[j] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;

  for (int t0 = k_begin; t0 < k_end; t0 += kCH) {
    const int nt = min(kCH, k_end - t0);
    __syncthreads();
    // stage keys/values of this tile
    for (int e = tid; e < kCH * DH; e += 256) {
      const int j = e / DH, d = e % DH;
      float kv = 0.f, vv = 0.f;
      int valid = 0;
      if (j < nt) {
        const int key = t0 + j;
        if (key < n_ctx) {
          const int p = lo + key;
          const int pi = p / P;
          int page = pi < max_pages ? table[(size_t)b * max_pages + pi] : -1;
          if (page >= 0 && page < num_pages) {
            const size_t off = layer_off + (((size_t)page * Hkv + kvh) * P + (p % P)) * DH + d;
            kv = ldf(kc + off);
            vv = ldf(vc + off);
            valid = 1;
          } else if (d == 0) {
            set_err(err, pi < max_pages ? DFLASH_DEV_PAGE_RANGE : DFLASH_DEV_POS_RANGE);
          }
        } else {
          const int i = key - n_ctx;
          const size_t off = ((size_t)(b * K + i) * Hkv + kvh) * DH + d;
          kv = ldf(kb + off);
          vv = ldf(vb + off);
          valid = 1;
        }
      }
      sK[j * LD + d] = kv;
      sV[j * LD + d] = vv;
      if (d == 0) s_valid[j] = valid;
    }
    __syncthreads();
    // scores: thread (row, part4) takes keys part4*16 .. +16
    float smax = -INFINITY;
#pragma unroll 4
    for (int jj = 0; jj < kCH / 4; ++jj) {
      const int j = part4 * (kCH / 4) + jj;
      float s = -INFINITY;
      if (j < nt && s_valid[j]) {
        float dot = 0.f;
#pragma unroll 8
        for (int d = 0; d < DH; ++d) dot = fmaf(sQ[row * LD + d], sK[j * LD + d], dot);
        s = dot * scale;
      }
      sS[row * (kCH + 1) + j] = s;
      smax = fmaxf(smax, s);
    }
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 1));
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 2));
    const float m_new = fmaxf(m_run, smax);
    const float alpha = (m_run == -INFINITY) ? 0.f : expf(m_run - m_new);
    __syncwarp();
    // probabilities (each thread its 16 keys), row sum
    float psum = 0.f;
    for (int jj = 0; jj < kCH / 4; ++jj) {
      const int j = part4 * (kCH / 4) + jj;
      const float s = sS[row * (kCH + 1) + j];
      const float pj = (s == -INFINITY) ? 0.f : expf(s - m_new);
      sS[row * (kCH + 1) + j] = pj;
      psum += pj;
    }
    psum += __shfl_xor_sync(0xffffffffu, psum, 1);
    psum += __shfl_xor_sync(0xffffffffu, psum, 2);
    l_run = l_run * alpha + psum;
    m_run = m_new;
    __syncwarp();
#pragma unroll
    for (int c = 0; c < DPT; ++c) acc[c] *= alpha;
    for (int j = 0; j < nt; ++j) {
      const float pj = sS[row * (kCH + 1) + j];
#pragma unroll
      for (int c = 0; c < DPT; ++c) acc[c] = fmaf(pj, sV[j * LD + part4 * DPT + c], acc[c]);
    }
  }
  // write this split's partial state
  const size_t base = ((((size_t)b * nqg + qgi) * Hkv + kvh) * nsplit + split) * kQG + row;
  float *po = part + base * (DH + 2);
#pragma unroll
  for (int c = 0; c < DPT; ++c) po[2 + part4 * DPT + c] = acc[c];
  if (part4 == 0) {
    po[0] = m_run;
    po[1] = l_run;
  }
}

// ---------------------------------------------------------------------------
// bf16 path: tensor-core tiles (mma.sync m16n8k16, fp32 accumulate).
// 4 warps x 16 query rows; key/value tiles of 64 rows staged by cp.async into
// a double-buffered, XOR-swizzled shared layout that ldmatrix reads without
// bank conflicts.  Online softmax in base 2; partial state in natural units.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t swz(int row, int chunk, int row_bytes) {
  return (uint32_t)(row * row_bytes + ((chunk ^ (row & 7)) << 4));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float *d, const uint32_t *a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *(uint32_t *)&h;
}

template <int DH>
__global__ void __launch_bounds__(128) k_attn_mma(
    const bf16 *__restrict__ qb, const bf16 *__restrict__ kb, const bf16 *__restrict__ vb,
    const bf16 *__restrict__ kc, const bf16 *__restrict__ vc, size_t layer_off,
    const int32_t *__restrict__ table, int max_pages, int num_pages, int P,
    const int32_t *__restrict__ ctx_len, int K, int Hq, int Hkv, int window, int kps, int nsplit,
    int nqg, float *__restrict__ part, int *err) {
  constexpr int CH = kCH;          // keys per tile
  constexpr int CHUNKS = DH / 8;   // 16-byte chunks per row
  constexpr int RB = DH * 2;       // bytes per row
  constexpr int TILE = CH * RB;    // bytes per K (or V) tile
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_valid[2][CH];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + kQG * RB;
  const uint32_t sV0 = sK0 + 2 * TILE;
  pdl_launch();
  pdl_wait();

  const int split = blockIdx.x, kvh = blockIdx.y;
  const int b = blockIdx.z / nqg, qgi = blockIdx.z % nqg;
  const int grp = Hq / Hkv, QR = K * grp;
  const int ctx = ctx_len[b];
  const int n_ctx = ctx < window ? (ctx > 0 ? ctx : 0) : window;
  const int lo = ctx - n_ctx, n_keys = n_ctx + K;
  const int k_begin = split * kps;
  if (k_begin >= n_keys) return;
  const int k_end = min(n_keys, k_begin + kps);
  const int ntiles = (k_end - k_begin + CH - 1) / CH;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // query rows qr = i*grp + g of this group
  for (int e = tid; e < kQG * CHUNKS; e += 128) {
    const int qr = e / CHUNKS, c = e % CHUNKS;
    const int qrg = qgi * kQG + qr;
    const bf16 *src = qb;
    int bytes = 0;
    if (qrg < QR) {
      const int i = qrg / grp, g = qrg % grp;
      src = qb + ((size_t)(b * K + i) * Hq + kvh * grp + g) * DH + c * 8;
      bytes = 16;
    }
    cp_async16(sQ + swz(qr, c, RB), src, bytes);
  }
  auto load_tile = [&](int t, int stage) {
    const int t0 = k_begin + t * CH;
    for (int e = tid; e < CH * CHUNKS; e += 128) {
      const int j = e / CHUNKS, c = e % CHUNKS;
      const int key = t0 + j;
      const bf16 *srck = kc, *srcv = vc;
      int ok = 0;
      if (key < k_end) {
        if (key < n_ctx) {
          const int p = lo + key, pi = p / P;
          const int page = pi < max_pages ? table[(size_t)b * max_pages + pi] : -1;
          if (page >= 0 && page < num_pages) {
            const size_t off = layer_off + (((size_t)page * Hkv + kvh) * P + (p % P)) * DH + c * 8;
            srck = kc + off;
            srcv = vc + off;
            ok = 1;
          } else if (c == 0) {
            set_err(err, pi < max_pages ? DFLASH_DEV_PAGE_RANGE : DFLASH_DEV_POS_RANGE);
          }
        } else {
          const size_t off = ((size_t)(b * K + key - n_ctx) * Hkv + kvh) * DH + c * 8;
          srck = kb + off;
          srcv = vb + off;
          ok = 1;
        }
      }
      cp_async16(sK0 + stage * TILE + swz(j, c, RB), srck, ok ? 16 : 0);
      cp_async16(sV0 + stage * TILE + swz(j, c, RB), srcv, ok ? 16 : 0);
      if (c == 0) s_valid[stage][j] = ok;
    }
  };
  load_tile(0, 0);
  cp_async_commit();

  const bool active = qgi * kQG + warp * 16 < QR;
  const int g8 = lane >> 2, t4 = lane & 3, r8 = lane & 7, mi = lane >> 3;
  const float sl2 = rsqrtf((float)DH) * 1.4426950408889634f;
  uint32_t qf[DH / 16][4];
  float o[DH / 8][4];
#pragma unroll
  for (int n = 0; n < DH / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  for (int t = 0; t < ntiles; ++t) {
    const int stage = t & 1;
    if (t + 1 < ntiles) {
      load_tile(t + 1, stage ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (t == 0 && active) {
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk)
        ldsm_x4(sQ + swz(warp * 16 + (mi & 1) * 8 + r8, 2 * kk + (mi >> 1), RB), qf[kk][0],
                qf[kk][1], qf[kk][2], qf[kk][3]);
    }
    if (active) {
      const uint32_t sK = sK0 + stage * TILE, sV = sV0 + stage * TILE;
      float sc[CH / 8][4];
#pragma unroll
      for (int j = 0; j < CH / 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
      for (int jp = 0; jp < CH / 16; ++jp) {
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sK + swz(16 * jp + (mi >> 1) * 8 + r8, 2 * kk + (mi & 1), RB), b0, b1, b2, b3);
          mma_bf16_16816(sc[2 * jp], qf[kk], b0, b1);
          mma_bf16_16816(sc[2 * jp + 1], qf[kk], b2, b3);
        }
      }
      // mask, scale, running max
      const int t0 = k_begin + t * CH;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < CH / 8; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = 8 * j + 2 * t4 + (e & 1);
          const bool ok = (t0 + col < k_end) && s_valid[stage][col];
          const float v = ok ? sc[j][e] * sl2 : -INFINITY;
          sc[j][e] = v;
          mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
      }
      float alpha[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float mnew = fmaxf(m_run[h], mx[h]);
        alpha[h] = (mnew == -INFINITY) ? 1.f : exp2f(m_run[h] - mnew);
        m_run[h] = mnew;
      }
      float ls[2] = {0.f, 0.f};
      uint32_t pa[CH / 16][4];
#pragma unroll
      for (int j = 0; j < CH / 8; ++j) {
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mm = m_run[e >> 1];
          p[e] = (sc[j][e] == -INFINITY) ? 0.f : exp2f(sc[j][e] - mm);
          ls[e >> 1] += p[e];
        }
        // scores of n-tile j become the A operand of P.V (keys 16*(j/2) ..)
        pa[j >> 1][(j & 1) * 2 + 0] = pack_bf16(p[0], p[1]);
        pa[j >> 1][(j & 1) * 2 + 1] = pack_bf16(p[2], p[3]);
      }
      l_run[0] = l_run[0] * alpha[0] + ls[0];
      l_run[1] = l_run[1] * alpha[1] + ls[1];
#pragma unroll
      for (int n = 0; n < DH / 8; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
#pragma unroll
      for (int kk = 0; kk < CH / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < DH / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sV + swz(16 * kk + (mi & 1) * 8 + r8, 2 * np + (mi >> 1), RB), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * np], pa[kk], b0, b1);
          mma_bf16_16816(o[2 * np + 1], pa[kk], b2, b3);
        }
      }
    }
    __syncthreads();
  }
  if (!active) return;
  // quad-reduce the row sums and write this split's state
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  const float ln2 = 0.6931471805599453f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = warp * 16 + g8 + 8 * h;
    const size_t base = ((((size_t)b * nqg + qgi) * Hkv + kvh) * nsplit + split) * kQG + row;
    float *po = part + base * (DH + 2);
    if (t4 == 0) {
      po[0] = m_run[h] == -INFINITY ? -INFINITY : m_run[h] * ln2;
      po[1] = l_run[h];
    }
#pragma unroll
    for (int n = 0; n < DH / 8; ++n) {
      po[2 + 8 * n + 2 * t4] = o[n][2 * h];
      po[2 + 8 * n + 2 * t4 + 1] = o[n][2 * h + 1];
    }
  }
}

// o[r][h*dh + d] = sum_s e^{m_s - M} O_s / sum_s e^{m_s - M} l_s.  grid (B*K, Hq), block dh.
template <typename S>
__global__ void k_attn_combine(const float *__restrict__ part, const int32_t *__restrict__ ctx_len,
                               int K, int Hq, int Hkv, int dh, int window, int kps, int nsplit,
                               int nqg, S *__restrict__ ob) {
  pdl_launch();
  pdl_wait();
  const int r = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const int b = r / K, i = r % K;
  const int grp = Hq / Hkv, kvh = h / grp, g = h % grp;
  const int qr = i * grp + g, qgi = qr / kQG, row = qr % kQG;
  const int ctx = ctx_len[b];
  const int n_ctx = ctx < window ? (ctx > 0 ? ctx : 0) : window;
  const int ns = (n_ctx + K + kps - 1) / kps;
  const size_t base0 = (((size_t)b * nqg + qgi) * Hkv + kvh) * nsplit;
  float M = -INFINITY;
#pragma unroll 4
  for (int s = 0; s < ns; ++s) M = fmaxf(M, part[((base0 + s) * kQG + row) * (dh + 2)]);
  float L = 0.f, O = 0.f;
#pragma unroll 4
  for (int s = 0; s < ns; ++s) {
    const float *po = part + ((base0 + s) * kQG + row) * (dh + 2);
    const float w = po[0] == -INFINITY ? 0.f : expf(po[0] - M);
    L += w * po[1];
    O += w * po[2 + d];
  }
  stf(ob + (size_t)r * Hq * dh + (size_t)h * dh + d, O / L);
}

}  // namespace dfl

namespace dflh {

AttnPlan attn_plan(int B, int K, int Hq, int Hkv, int dh, int window, int num_sms) {
  AttnPlan pl;
  pl.qg = dfl::kQG;
  const int QR = K * (Hq / Hkv);
  pl.nqg = (QR + dfl::kQG - 1) / dfl::kQG;
  const int n_keys = window + K;
  const long items = (long)B * Hkv * pl.nqg;
  // smallest key split (multiple of 64) that still gives ~2 CTAs per SM
  int kps = dfl::kCH;
  while ((long)items * ((n_keys + kps - 1) / kps) > 2L * num_sms && kps < n_keys) kps += dfl::kCH;
  pl.kps = kps;
  pl.nsplit = (n_keys + kps - 1) / kps;
  pl.part_floats = (size_t)B * pl.nqg * Hkv * pl.nsplit * dfl::kQG * (dh + 2);
  return pl;
}

template <typename S, int DH>
static int launch_attn_dh(const AttnPlan &pl, const S *qb, const S *kb, const S *vb, const S *kc,
                          const S *vc, int layer, const int32_t *table, int max_pages,
                          int num_pages, int P, const int32_t *ctx_len, int B, int K, int Hq,
                          int Hkv, int window, float *part, S *ob, int *err, cudaStream_t st) {
  const size_t layer_off = (size_t)layer * num_pages * Hkv * P * DH;
  if constexpr (sizeof(S) == 2) {
    const size_t smem = (size_t)dfl::kQG * DH * 2 + 4 * (size_t)dfl::kCH * DH * 2;
    static int attr_done = 0;
    if (!attr_done) {
      if (cudaFuncSetAttribute(dfl::k_attn_mma<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem) != cudaSuccess)
        return DFLASH_ERR_CUDA;
      attr_done = 1;
    }
    DFL_CHECK_LAUNCH(launch(dfl::k_attn_mma<DH>, dim3(pl.nsplit, Hkv, B * pl.nqg), dim3(128), smem,
                            st, qb, kb, vb, kc, vc, layer_off, table, max_pages, num_pages, P,
                            ctx_len, K, Hq, Hkv, window, pl.kps, pl.nsplit, pl.nqg, part, err));
  } else {
    constexpr int LD = DH + 1;
    const size_t smem = sizeof(float) * ((size_t)dfl::kQG * LD + 2 * (size_t)dfl::kCH * LD +
                                         (size_t)dfl::kQG * (dfl::kCH + 1));
    static int attr_done = 0;
    if (!attr_done) {
      if (cudaFuncSetAttribute(dfl::k_attn_split<S, DH>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DFLASH_ERR_CUDA;
      attr_done = 1;
    }
    DFL_CHECK_LAUNCH(launch(dfl::k_attn_split<S, DH>, dim3(pl.nsplit, Hkv, B * pl.nqg), dim3(256),
                            smem, st, qb, kb, vb, kc, vc, layer_off, table, max_pages, num_pages, P,
                            ctx_len, K, Hq, Hkv, window, pl.kps, pl.nsplit, pl.nqg, part, err));
  }
  DFL_CHECK_LAUNCH(launch(dfl::k_attn_combine<S>, dim3(B * K, Hq), dim3(DH), 0, st,
                          (const float *)part, ctx_len, K, Hq, Hkv, DH, window, pl.kps, pl.nsplit,
                          pl.nqg, ob));
  return DFLASH_OK;
}

template <typename S>
int launch_block_attention(const AttnPlan &pl, const S *qb, const S *kb, const S *vb,
                           const S *kc, const S *vc, int layer, const int32_t *page_table,
                           int max_pages, int num_pages, int page_size, const int32_t *ctx_len,
                           int B, int K, int Hq, int Hkv, int dh, int window, float *part, S *ob,
                           int *err, cudaStream_t st) {
  if (dh == 128)
    return launch_attn_dh<S, 128>(pl, qb, kb, vb, kc, vc, layer, page_table, max_pages, num_pages,
                                  page_size, ctx_len, B, K, Hq, Hkv, window, part, ob, err, st);
  if (dh == 64)
    return launch_attn_dh<S, 64>(pl, qb, kb, vb, kc, vc, layer, page_table, max_pages, num_pages,
                                 page_size, ctx_len, B, K, Hq, Hkv, window, part, ob, err, st);
  return DFLASH_ERR_DIMS;
}

template int launch_block_attention<float>(const AttnPlan &, const float *, const float *,
                                           const float *, const float *, const float *, int,
                                           const int32_t *, int, int, int, const int32_t *, int,
                                           int, int, int, int, int, float *, float *, int *,
                                           cudaStream_t);
template int launch_block_attention<dfl::bf16>(const AttnPlan &, const dfl::bf16 *,
                                               const dfl::bf16 *, const dfl::bf16 *,
                                               const dfl::bf16 *, const dfl::bf16 *, int,
                                               const int32_t *, int, int, int, const int32_t *,
                                               int, int, int, int, int, int, float *,
                                               dfl::bf16 *, int *, cudaStream_t);

}  // namespace dflh
