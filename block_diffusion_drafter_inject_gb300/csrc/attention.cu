// Non-causal block attention (split over keys, then combined).
//
// Work item = (request b, kv head, query group, key split).  The K block
// queries of the group's q heads (K * Hq/Hkv rows) share every key/value tile
// staged in shared memory.  Keys: the last min(window, ctx_len) context
// positions from the paged cache, then the K block slots; no mask.  Each split
// keeps an online softmax (running max m, sum l, unnormalised output) and
// writes it out; the combine kernel merges the splits in order.
#include <math.h>
#include <string.h>

#include <algorithm>

#include "attention.cuh"
#include "gemm.cuh"
#include "pointwise.cuh"

namespace dfl {

constexpr int kQG = 64;   // query rows per CTA
constexpr int kCH = 64;   // keys per shared-memory tile
constexpr int kAttnStages = 3;  // K/V tile stages of the tensor-core kernel (one split)
constexpr int kAttnPrePages = 32;  // context tiles per CTA whose pages are looked up early
constexpr int kPageAhead = 3;   // tiles whose pages a loader thread holds ahead

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
  const int k_begin = split * kps;  // the last split takes every key after it
  if (k_begin >= n_keys) return;
  const int k_end = split == nsplit - 1 ? n_keys : min(n_keys, k_begin + kps);
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
// K/V tile layout of the TMA loader: the tile's 64-column halves are separate
// [64 rows][128 B] boxes, each with the 128-byte swizzle (16-byte chunk index
// xor row % 8); chunk c of row r sits in half c / 8.
__device__ __forceinline__ uint32_t swzt(int row, int chunk) {
  return (uint32_t)((chunk >> 3) * 8192 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

struct AttnArgs {
  const bf16 *qkvb;  // [B*K, (Hq + 2Hkv) * DH]: q, k normed and rotated, v
  const bf16 *kc, *vc;
  size_t layer_off;
  int layer;
  const int32_t *table;
  int max_pages, num_pages, P;
  const int32_t *ctx_len;
  int K, Hq, Hkv, window, kps, nsplit, nqg;
  bf16 *ob;  // [B*K, Hq*DH]
  int *err;
  // context rows the pass itself injects (request row, position), written into
  // this layer's cache by the projection before it: no tile holding one of them
  // is read before the grid-dependency wait
  const int32_t *inj_req, *inj_pos;
  int inj_n;
};

// Injected rows scanned per CTA for the lowest position of its request; above
// this many, no context tile is loaded before the wait.
constexpr int kAttnScanMax = 1024;

// grid (nsplit, Hkv, B*nqg), cluster (nsplit, 1, 1); block 128 = 4 warps.
// KP warps share each 16-row query block and split every key tile KP ways
// (KP = 1, 2, 4 for groups of <= 64, 32, 16 query rows); their softmax states
// are merged in shared memory after the tile loop.
// TK (page size 64): the key tiles are the window's cache pages, each brought
// in by TMA (two 64x64 boxes for K and for V per 128-wide head) by one thread
// with an mbarrier per stage, then one tile of the block slots; rows outside
// the window are masked and their V rows zeroed.  Otherwise every thread copies
// 16-byte chunks of the tile's key rows with cp.async.
template <int DH, int KP, bool TK, int NST>
__global__ void __launch_bounds__(128)
    k_attn_mma(const AttnArgs A, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV) {
  constexpr int CH = kCH;          // keys per tile
  constexpr int CHUNKS = DH / 8;   // 16-byte chunks per row
  constexpr int RB = DH * 2;       // bytes per row
  constexpr int TILE = CH * RB;    // bytes per K (or V) tile
  constexpr int QROWS = 64 / KP;   // query rows staged (row blocks x 16)
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ int s_valid[NST][CH];
  __shared__ __align__(8) uint64_t kvbar[NST];
  __shared__ int s_tbase[NST], s_tok[NST];
  __shared__ int s_abort;
  __shared__ int s_pg[kAttnPrePages];
  __shared__ __align__(8) uint64_t cmbar;  // the peers' rows of this CTA have landed
  uint8_t *pQ = smem;
  uint8_t *pK0 = smem + QROWS * RB;
  // receive buffer of the cluster combine, [nsplit][per][DH + 4] fp32 rows (m, l,
  // two floats of padding, o) copied in by the peers, then the combine weights
  // [per][nsplit]
  uint8_t *pRecv = pK0 + 2 * NST * TILE;
  const uint32_t sQ = smem_u32(pQ), sK0 = smem_u32(pK0), sV0 = sK0 + NST * TILE;
  pdl_launch();
  // rows of this CTA's query group and the share that this CTA finishes
  const int QR0 = A.K * (A.Hq / A.Hkv), qg0 = blockIdx.z % A.nqg;
  const int nrows = min(kQG, QR0 - qg0 * kQG);
  const int per = (nrows + A.nsplit - 1) / A.nsplit;
  const int r0 = blockIdx.x * per, r1 = min(nrows, r0 + per);
  const bool clus = A.nsplit > 1;
  if (threadIdx.x == 0) {
    s_abort = 0;
    if (TK) {
      for (int st = 0; st < NST; ++st) mbar_init(&kvbar[st], 1);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    if (clus) {
      mbar_init(&cmbar, 1);
      mbar_expect_tx(&cmbar, (uint32_t)(A.nsplit * max(0, r1 - r0) * (DH + 4) * 4));
    }
    if (TK || clus) mbar_fence_init();
  }

  const int split = blockIdx.x, kvh = blockIdx.y;
  const int b = blockIdx.z / A.nqg, qgi = blockIdx.z % A.nqg;
  const int grp = A.Hq / A.Hkv, QR = A.K * grp;
  const int QKVW = (A.Hq + 2 * A.Hkv) * DH;
  const int ctx = A.ctx_len[b];
  const int n_ctx = ctx < A.window ? (ctx > 0 ? ctx : 0) : A.window;
  const int lo = ctx - n_ctx, n_keys = n_ctx + A.K;
  const int k_begin = split * A.kps;  // the last split takes every key after it
  const int k_end = split == A.nsplit - 1 ? n_keys : min(n_keys, k_begin + A.kps);
  // TK: window pages [pgf, pgf + nct) then the block tile, kps / 64 tiles a split
  const int pgf = lo / CH, nct = n_ctx > 0 ? (ctx - 1) / CH - pgf + 1 : 0;
  const int t_begin = split * (A.kps / CH);
  const int t_end = split == A.nsplit - 1 ? nct + 1 : min(nct + 1, t_begin + A.kps / CH);
  const int ntiles = TK ? max(0, t_end - t_begin)
                        : (k_begin < n_keys ? (k_end - k_begin + CH - 1) / CH : 0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // TK: the context lengths and the page table are inputs of the pass (no
  // kernel of the pass writes them), so the pages of the first context tiles
  // are looked up, one thread per tile, before waiting for the projection; the
  // first NST - 1 context tiles are loaded right away (the caches are complete:
  // the pass's first kernel lets no later kernel start before all earlier work
  // has completed) and the next two are prefetched into L2
  const int npre = TK ? min(max(0, min(t_end, nct) - t_begin), kAttnPrePages) : 0;
  // the lowest position of this request that the pass injects (rows written by
  // this layer's projection): tiles loaded before the wait must end below it
  __shared__ int s_fresh[4];
  if (TK) {
    int f = INT_MAX;
    if (A.inj_n > kAttnScanMax) {
      f = INT_MIN;
    } else {
      for (int i = tid; i < A.inj_n; i += 128)
        if (__ldg(A.inj_req + i) == b) f = min(f, __ldg(A.inj_pos + i));
    }
    f = __reduce_min_sync(0xffffffffu, f);
    if (lane == 0) s_fresh[warp] = f;
  }
  if (TK && tid < npre) {
    const int pi = pgf + t_begin + tid;
    int page = -1;
    if (pi < A.max_pages) {
      page = A.table[(size_t)b * A.max_pages + pi];
      if (page < 0 || page >= A.num_pages) {
        set_err(A.err, DFLASH_DEV_PAGE_RANGE);
        page = -1;
      }
    } else {
      set_err(A.err, DFLASH_DEV_POS_RANGE);
    }
    s_pg[tid] = page;
    if (page >= 0 && tid >= NST - 1 && tid < NST + 1) {  // the tiles after the first ones
      const int y = (int)((((size_t)A.layer * A.num_pages + page) * A.Hkv + kvh) * CH);
#pragma unroll
      for (int hh = 0; hh < DH / 64; ++hh) {
        tma_prefetch_l2_2d(&tmK, 64 * hh, y);
        tma_prefetch_l2_2d(&tmV, 64 * hh, y);
      }
    }
  }
  __syncthreads();  // barrier init and the looked-up pages visible to every thread
  if (clus) cluster_arrive_relaxed();  // this CTA's receive mbarrier is initialised
  const bf16 *blk = A.qkvb + (size_t)b * A.K * QKVW;  // this request's block rows
  const int fresh = TK ? min(min(s_fresh[0], s_fresh[1]), min(s_fresh[2], s_fresh[3])) : INT_MAX;
  // context tile t of this split may start before the wait: its cache rows are
  // complete when the pass began (it ends below every position injected now)
  auto early = [&](int t) {
    return TK && t < ntiles && t_begin + t < nct &&
           (long long)(pgf + t_begin + t + 1) * CH <= (long long)fresh;
  };
  uint64_t pol_kv = 0;
  if (TK) pol_kv = l2_policy_evict_first();

  // Loader: thread tid copies key row jrow = tid / 2 of every tile, chunks
  // [ch0, ch0 + CHUNKS/2) of its K and V rows: a context key from the paged
  // cache, a block slot from the projection rows, nothing (zeros) past the end.
  // The page of a context key is looked up kPageAhead tiles before the tile is
  // loaded (a register pipeline), so table reads never sit in front of copies.
  const int jrow = tid >> 1, ch0 = (tid & 1) * (CHUNKS / 2);
  auto key_page = [&](int t) -> int {  // >= 0 page; -1 not a context key; < -1 error bit
    const int key = k_begin + t * CH + jrow;
    if (t >= ntiles || key >= k_end || key >= n_ctx) return -1;
    const int pi = (lo + key) / A.P;
    if (pi >= A.max_pages) return -DFLASH_DEV_POS_RANGE;
    const int page = A.table[(size_t)b * A.max_pages + pi];
    return (page >= 0 && page < A.num_pages) ? page : -DFLASH_DEV_PAGE_RANGE;
  };
  // TK loader: one thread looks the page up and starts the boxes; the block
  // tile's rows come from the projection rows by cp.async (zeros past K)
  auto load_tile_tk = [&](int t, int stage) {
    const int gt = t_begin + t;
    if (gt < nct) {
      if (tid == 0) {
        const int pi = pgf + gt;
        int page = -1;
        if (t < npre) {
          page = s_pg[t];  // looked up (and checked) before the wait
        } else if (pi < A.max_pages) {
          page = A.table[(size_t)b * A.max_pages + pi];
          if (page < 0 || page >= A.num_pages) {
            set_err(A.err, DFLASH_DEV_PAGE_RANGE);
            page = -1;
          }
        } else {
          set_err(A.err, DFLASH_DEV_POS_RANGE);
        }
        s_tbase[stage] = pi * CH;
        s_tok[stage] = page >= 0;
        if (page >= 0) {
          mbar_expect_tx(&kvbar[stage], 2 * TILE);
          const int y = (int)((((size_t)A.layer * A.num_pages + page) * A.Hkv + kvh) * CH);
#pragma unroll
          for (int hh = 0; hh < DH / 64; ++hh) {
            tma_load_2d(pK0 + stage * TILE + hh * 8192, &tmK, &kvbar[stage], 64 * hh, y, pol_kv);
            tma_load_2d(pK0 + NST * TILE + stage * TILE + hh * 8192, &tmV, &kvbar[stage], 64 * hh,
                        y, pol_kv);
          }
        } else {
          mbar_arrive(&kvbar[stage]);
        }
      }
    } else {
      const bool ok = jrow < A.K;
      const bf16 *row = blk + (size_t)(ok ? jrow : 0) * QKVW;
      const bf16 *srck = row + (size_t)(A.Hq + kvh) * DH, *srcv = row + (size_t)(A.Hq + A.Hkv + kvh) * DH;
#pragma unroll
      for (int c = ch0; c < ch0 + CHUNKS / 2; ++c) {
        cp_async16(sK0 + stage * TILE + swzt(jrow, c), srck + c * 8, ok ? 16 : 0);
        cp_async16(sV0 + stage * TILE + swzt(jrow, c), srcv + c * 8, ok ? 16 : 0);
      }
      if (tid == 0) {
        s_tbase[stage] = -1;
        s_tok[stage] = 1;
        mbar_arrive(&kvbar[stage]);
      }
    }
  };
  auto load_tile = [&](int t, int stage, int page) {
    if constexpr (TK) {
      load_tile_tk(t, stage);
      return;
    }
    const int key = k_begin + t * CH + jrow;
    const bf16 *srck = A.kc, *srcv = A.vc;
    int ok = 0;
    if (key < k_end && key < n_ctx) {
      if (page >= 0) {
        const size_t off =
            A.layer_off + (((size_t)page * A.Hkv + kvh) * A.P + ((lo + key) % A.P)) * DH;
        srck = A.kc + off;
        srcv = A.vc + off;
        ok = 1;
      } else if (ch0 == 0) {
        set_err(A.err, -page);
      }
    } else if (key < k_end) {  // block slot i
      const bf16 *row = blk + (size_t)(key - n_ctx) * QKVW;
      srck = row + (size_t)(A.Hq + kvh) * DH;
      srcv = row + (size_t)(A.Hq + A.Hkv + kvh) * DH;
      ok = 1;
    }
#pragma unroll
    for (int c = ch0; c < ch0 + CHUNKS / 2; ++c) {
      cp_async16(sK0 + stage * TILE + swz(jrow, c, RB), srck + c * 8, ok ? 16 : 0);
      cp_async16(sV0 + stage * TILE + swz(jrow, c, RB), srcv + c * 8, ok ? 16 : 0);
    }
    if (ch0 == 0) s_valid[stage][jrow] = ok;
  };
  static_assert(TK || (kPageAhead == 3 && NST == 3), "page pipeline below holds three tiles");
  static_assert(DFLASH_DEV_PAGE_RANGE > 1 && DFLASH_DEV_POS_RANGE > 1, "error codes vs -1");
  int pg0 = TK ? 0 : key_page(0), pg1 = TK ? 0 : key_page(1), pg2 = TK ? 0 : key_page(2);
  // TK: the context tiles among the first NST - 1 start loading now
  if (TK)
#pragma unroll
    for (int t = 0; t < NST - 1; ++t)
      if (early(t)) load_tile_tk(t, t);
  pdl_wait();  // the projection rows (queries, block keys and values) are ready

  // queries qr = i*grp + g of this group: projection rows, copied (zeros past QR)
  for (int e = tid; e < QROWS * CHUNKS; e += 128) {
    const int row = e / CHUNKS, c = e % CHUNKS, qrg = qgi * kQG + row;
    const bool ok = qrg < QR;
    const bf16 *src = ok ? blk + (size_t)(qrg / grp) * QKVW + (size_t)(kvh * grp + qrg % grp) * DH
                         : A.qkvb;
    cp_async16(sQ + swz(row, c, RB), src + c * 8, ok ? 16 : 0);
  }
  // the first NST-1 tiles in flight; one commit group per tile (empty past the end)
#pragma unroll
  for (int t = 0; t < NST - 1; ++t) {
    if (t < ntiles && !early(t)) load_tile(t, t, t == 0 ? pg0 : pg1);
    cp_async_commit();
  }
  pg0 = pg2;  // page of tile NST-1 = 2
  pg1 = TK ? 0 : key_page(3);
  pg2 = TK ? 0 : key_page(4);

  constexpr int RW = 4 / KP;            // query row blocks per CTA
  constexpr int KW = CH / KP;           // keys of a tile per warp
  const int rb = warp % RW, kpart = warp / RW;
  const bool active = qgi * kQG + rb * 16 < QR;
  const int g8 = lane >> 2, t4 = lane & 3, r8 = lane & 7, mi = lane >> 3;
  const float sl2 = rsqrtf((float)DH) * 1.4426950408889634f;
  uint32_t qf[DH / 16][4];
  float o[DH / 8][4];
#pragma unroll
  for (int n = 0; n < DH / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  int stage = 0;
  for (int t = 0; t < ntiles; ++t) {
    // tile t + NST - 1 into the stage tile t - 1 used (free since the loop's end barrier)
    {
      const int tn = t + NST - 1;
      int sn = stage + NST - 1;
      if (sn >= NST) sn -= NST;
      if (tn < ntiles) load_tile(tn, sn, pg0);
      cp_async_commit();
      pg0 = pg1;
      pg1 = pg2;
      pg2 = TK ? 0 : key_page(t + NST + 2);
    }
    cp_async_wait<NST - 1>();  // tile t has landed (cp.async part)
    if constexpr (TK) {
      // the TMA part; then zero the V rows outside the window (a page's other
      // rows may hold anything, and 0 * NaN would reach the output)
      if (!mbar_wait(&kvbar[stage], (uint32_t)((t / NST) & 1), &s_abort) && tid == 0)
        set_err(A.err, DFLASH_DEV_TIMEOUT);
      const int base = s_tbase[stage];
      if (base >= 0 && tid < CH) {
        const int pos = base + tid;
        if (!(s_tok[stage] && pos >= lo && pos < ctx)) {
#pragma unroll
          for (int c = 0; c < CHUNKS; ++c)
            *(uint4 *)(pK0 + NST * TILE + stage * TILE + swzt(tid, c)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    __syncthreads();
    if (t == 0 && active) {
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk)
        ldsm_x4(sQ + swz(rb * 16 + (mi & 1) * 8 + r8, 2 * kk + (mi >> 1), RB), qf[kk][0],
                qf[kk][1], qf[kk][2], qf[kk][3]);
    }
    if (active) {
      const uint32_t sK = sK0 + stage * TILE, sV = sV0 + stage * TILE;
      const int kw0 = kpart * KW;  // this warp's keys within the tile
      float sc[KW / 8][4];
#pragma unroll
      for (int j = 0; j < KW / 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
      for (int jp = 0; jp < KW / 16; ++jp) {
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          uint32_t b0, b1, b2, b3;
          const int kr = kw0 + 16 * jp + (mi >> 1) * 8 + r8, kc = 2 * kk + (mi & 1);
          ldsm_x4(sK + (TK ? swzt(kr, kc) : swz(kr, kc, RB)), b0, b1, b2, b3);
          mma_bf16_16816(sc[2 * jp], qf[kk], b0, b1);
          mma_bf16_16816(sc[2 * jp + 1], qf[kk], b2, b3);
        }
      }
      const int t0 = k_begin + t * CH;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < KW / 8; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = kw0 + 8 * j + 2 * t4 + (e & 1);
          bool ok;
          if constexpr (TK) {
            const int base = s_tbase[stage];
            ok = base >= 0 ? (s_tok[stage] && base + col >= lo && base + col < ctx) : col < A.K;
          } else {
            ok = (t0 + col < k_end) && s_valid[stage][col];
          }
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
      // probabilities as a bf16 pair hi + lo (hi = bf16(p), lo = bf16(p - hi)):
      // two products with V keep P at ~16 significant bits
      uint32_t pa[KW / 16][4], pl[KW / 16][4];
#pragma unroll
      for (int j = 0; j < KW / 8; ++j) {
        float p[4], r[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mm = m_run[e >> 1];
          p[e] = (sc[j][e] == -INFINITY) ? 0.f : exp2f(sc[j][e] - mm);
          ls[e >> 1] += p[e];
          r[e] = p[e] - __bfloat162float(__float2bfloat16_rn(p[e]));
        }
        pa[j >> 1][(j & 1) * 2 + 0] = pack_bf16(p[0], p[1]);
        pa[j >> 1][(j & 1) * 2 + 1] = pack_bf16(p[2], p[3]);
        pl[j >> 1][(j & 1) * 2 + 0] = pack_bf16(r[0], r[1]);
        pl[j >> 1][(j & 1) * 2 + 1] = pack_bf16(r[2], r[3]);
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
      for (int kk = 0; kk < KW / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < DH / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          const int vr = kw0 + 16 * kk + (mi & 1) * 8 + r8, vc = 2 * np + (mi >> 1);
          ldsm_x4_t(sV + (TK ? swzt(vr, vc) : swz(vr, vc, RB)), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * np], pa[kk], b0, b1);
          mma_bf16_16816(o[2 * np + 1], pa[kk], b2, b3);
          mma_bf16_16816(o[2 * np], pl[kk], b0, b1);
          mma_bf16_16816(o[2 * np + 1], pl[kk], b2, b3);
        }
      }
    }
    if (TK) fence_proxy_async();  // this stage's generic writes before its next TMA fill
    __syncthreads();
    if (++stage == NST) stage = 0;
  }
  cp_async_wait<0>();
  __syncthreads();

  // merge the KP key parts of each row block (fragment layout, per thread)
  if (KP > 1) {
    constexpr int FS = 4 + DH / 2;  // floats per thread: m[2], l[2], o[DH/8][4]
    float *xs = (float *)pK0;        // [KP-1][RW][32 lanes][FS]
    if (kpart > 0) {
      float *d = xs + (((size_t)(kpart - 1) * RW + rb) * 32 + lane) * FS;
      d[0] = m_run[0], d[1] = m_run[1], d[2] = l_run[0], d[3] = l_run[1];
#pragma unroll
      for (int n = 0; n < DH / 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) d[4 + 4 * n + e] = o[n][e];
    }
    __syncthreads();
    if (kpart == 0) {
#pragma unroll
      for (int q = 0; q < KP - 1; ++q) {
        const float *d = xs + (((size_t)q * RW + rb) * 32 + lane) * FS;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float mo = d[h];
          const float M = fmaxf(m_run[h], mo);
          const float a = M == -INFINITY ? 0.f : exp2f(m_run[h] - M);
          const float c = M == -INFINITY ? 0.f : exp2f(mo - M);
          l_run[h] = l_run[h] * a + d[2 + h] * c;
#pragma unroll
          for (int n = 0; n < DH / 8; ++n) {
            o[n][2 * h] = o[n][2 * h] * a + d[4 + 4 * n + 2 * h] * c;
            o[n][2 * h + 1] = o[n][2 * h + 1] * a + d[4 + 4 * n + 2 * h + 1] * c;
          }
          m_run[h] = M;
        }
      }
    }
    __syncthreads();
  }

  // Combine through the cluster: query row `row` is finished by CTA
  // owner = row / per.  Every CTA stages its (m, l, o) rows in shared memory
  // (m, l, 2 floats of padding, o: DH + 4 floats, a multiple of 16 bytes) and
  // copies row `row` with one bulk copy into the owner's receive buffer
  // recv[split][row - owner*per], counted in bytes on the owner's mbarrier;
  // each owner waits for its bytes, then merges its rows from local shared
  // memory.  The cluster barrier arrived at the start makes every receive
  // mbarrier initialised before the first copy; the one arrived once a CTA's
  // rows have landed keeps every CTA (and its staged rows) alive until all
  // copies of the cluster have landed.
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  if (A.nsplit == 1) {  // one split: the rows are final here, o / l straight to bf16
    if (active && kpart == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = rb * 16 + g8 + 8 * h;
        if (row < nrows) {
          const int qrg = qgi * kQG + row, i = qrg / grp, g = qrg % grp;
          bf16 *dst = A.ob + ((size_t)(b * A.K + i) * A.Hq + kvh * grp + g) * DH + 2 * t4;
          const float il = 1.f / l_run[h];
#pragma unroll
          for (int n = 0; n < DH / 8; ++n)
            *(uint32_t *)(dst + 8 * n) = pack_bf16(o[n][2 * h] * il, o[n][2 * h + 1] * il);
        }
      }
    }
    return;
  }
  const uint32_t recv = smem_u32(pRecv);
  constexpr int RS = DH + 4;  // floats per staged / received row
  float *stg = (float *)pK0;  // staged rows [row][RS] (the tile buffers are free now)
  if (active && kpart == 0) {
    const float ln2 = 0.6931471805599453f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = rb * 16 + g8 + 8 * h;
      if (row < nrows) {
        float *d = stg + row * RS;
        if (t4 == 0) {
          d[0] = m_run[h] == -INFINITY ? -INFINITY : m_run[h] * ln2;
          d[1] = l_run[h];
        }
#pragma unroll
        for (int n = 0; n < DH / 8; ++n)
          *(float2 *)(d + 4 + 8 * n + 2 * t4) = make_float2(o[n][2 * h], o[n][2 * h + 1]);
      }
    }
  }
  fence_proxy_async();  // the staged rows, written by this thread, before the bulk copies
  __syncthreads();
  cluster_wait();  // every receive mbarrier of the cluster is initialised
  if (tid < nrows) {
    const int owner = tid / per, lr = tid - owner * per;
    bulk_copy_to_peer(cluster_addr(recv + (uint32_t)((split * per + lr) * RS) * 4u, owner),
                      smem_u32(stg + tid * RS), RS * 4, cluster_addr(smem_u32(&cmbar), owner));
  }
  if (!mbar_wait<true>(&cmbar, 0, &s_abort) && tid == 0) set_err(A.err, DFLASH_DEV_TIMEOUT);
  cluster_arrive();  // this CTA's rows have landed
  const float *rv = (const float *)pRecv;
  // weights of the splits of each owned row: w_q = e^(m_q - M) / sum_q e^(m_q - M) l_q
  float *wts = (float *)(pRecv + (size_t)A.nsplit * per * RS * 4);  // [per][nsplit]
  // one warp per owned row, lane q on split q (at most 16 splits); M and L
  // over the lanes by a fixed shuffle tree
  for (int lr = warp; lr < r1 - r0; lr += 4) {
    const bool has = lane < A.nsplit;
    const float m = has ? rv[(lane * per + lr) * RS] : -INFINITY;
    float M = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = m == -INFINITY ? 0.f : expf(m - M);
    float L = has ? w * rv[(lane * per + lr) * RS + 1] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (has) wts[lr * A.nsplit + lane] = w * (1.f / L);
  }
  __syncthreads();
  for (int e = tid; e < (r1 - r0) * DH; e += 128) {
    const int lr = e / DH, d = e % DH;
    float O = 0.f;
    for (int q = 0; q < A.nsplit; ++q) O += wts[lr * A.nsplit + q] * rv[(q * per + lr) * RS + 4 + d];
    const int qrg = qgi * kQG + r0 + lr, i = qrg / grp, g = qrg % grp;
    A.ob[((size_t)(b * A.K + i) * A.Hq + kvh * grp + g) * DH + d] = __float2bfloat16_rn(O);
  }
  cluster_wait();  // every CTA's rows have landed: no push is in flight into any of them
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
  const int ns = min(nsplit, (n_ctx + K + kps - 1) / kps);  // the last split holds the rest
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
  // smallest key split (multiple of 64) that still gives ~2 CTAs per SM; at
  // most 16 splits (the splits of one item form a thread-block cluster), the
  // last one also taking the keys left over, at most another split's worth
  int kps = dfl::kCH;
  while (kps < n_keys && ((long)items * std::min(16, (n_keys + kps - 1) / kps) > 2L * num_sms ||
                          n_keys - 16 * kps > kps))
    kps += dfl::kCH;
  pl.kps = kps;
  pl.nsplit = std::min(16, (n_keys + kps - 1) / kps);
  pl.part_floats = (size_t)B * pl.nqg * Hkv * pl.nsplit * dfl::kQG * (dh + 2);
  return pl;
}

template <typename S, int DH>
static int launch_attn_dh(const AttnPlan &pl, const S *qb, const S *kb, const S *vb, const S *kc,
                          const S *vc, int layer, const int32_t *table, int max_pages,
                          int num_pages, int P, const int32_t *ctx_len, int B, int K, int Hq,
                          int Hkv, int window, float *part, S *ob, int *err, cudaStream_t st) {
  // float32 storage: CUDA-core split kernel + combine
  const size_t layer_off = (size_t)layer * num_pages * Hkv * P * DH;
  constexpr int LD = DH + 1;
  const size_t smem = sizeof(float) * ((size_t)dfl::kQG * LD + 2 * (size_t)dfl::kCH * LD +
                                       (size_t)dfl::kQG * (dfl::kCH + 1));
  static int attr_done = 0;
  if (!attr_done) {
    if (cudaFuncSetAttribute(dfl::k_attn_split<S, DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    attr_done = 1;
  }
  DFL_CHECK_LAUNCH(launch(dfl::k_attn_split<S, DH>, dim3(pl.nsplit, Hkv, B * pl.nqg), dim3(256),
                          smem, st, qb, kb, vb, kc, vc, layer_off, table, max_pages, num_pages, P,
                          ctx_len, K, Hq, Hkv, window, pl.kps, pl.nsplit, pl.nqg, part, err));
  DFL_CHECK_LAUNCH(launch(dfl::k_attn_combine<S>, dim3(B * K, Hq), dim3(DH), 0, st,
                          (const float *)part, ctx_len, K, Hq, Hkv, DH, window, pl.kps, pl.nsplit,
                          pl.nqg, ob));
  return DFLASH_OK;
}

template <int DH, int KP, bool TK, int NST>
static int launch_attn_fused(const AttnPlan &pl, const dfl::AttnArgs &a, int B,
                             const CUtensorMap &mk, const CUtensorMap &mv, cudaStream_t st) {
  // Q, NST K and V tiles (1 KB of alignment slack; the key-part merge reuses
  // the tile buffers), then, with several splits, the receive buffer
  // [nsplit][per][DH + 4] and the combine weights [per][nsplit]
  const int QR = a.K * (a.Hq / a.Hkv);
  const size_t per = (std::min(dfl::kQG, QR) + pl.nsplit - 1) / pl.nsplit;
  const size_t recv = pl.nsplit > 1 ? pl.nsplit * per * (DH + 4) * 4 + pl.nsplit * per * 4 : 0;
  const size_t smem = 1024 + (size_t)(64 / KP) * DH * 2 + 2 * (size_t)NST * dfl::kCH * DH * 2 +
                      ((recv + 15) & ~(size_t)15);
  static size_t attr_smem = 0;
  static int attr_cluster = 0;
  if (smem > attr_smem) {
    if (cudaFuncSetAttribute(dfl::k_attn_mma<DH, KP, TK, NST>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    attr_smem = smem;
  }
  if (!attr_cluster) {
    if (cudaFuncSetAttribute(dfl::k_attn_mma<DH, KP, TK, NST>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    attr_cluster = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.nsplit, a.Hkv, B * pl.nqg);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  count_launch();
  DFL_CHECK_LAUNCH(cudaLaunchKernelEx(&cfg, dfl::k_attn_mma<DH, KP, TK, NST>, a, mk, mv));
  return DFLASH_OK;
}

int launch_attention_fused(const AttnPlan &pl, const dfl::bf16 *qkvb, const dfl::bf16 *kc,
                           const dfl::bf16 *vc, int layer, int n_layers, const int32_t *table,
                           int max_pages, int num_pages, int P, const int32_t *ctx_len, int B,
                           int K, int Hq, int Hkv, int dh, int window, dfl::bf16 *ob, int *err,
                           cudaStream_t st, const int32_t *inj_req, const int32_t *inj_pos,
                           int inj_n) {
  const Dev *d = device();
  if (!d) return DFLASH_ERR_DEVICE;
  dfl::AttnArgs a;
  a.qkvb = qkvb;
  a.kc = kc;
  a.vc = vc;
  a.layer_off = (size_t)layer * num_pages * Hkv * P * dh;
  a.layer = layer;
  a.table = table;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.P = P;
  a.ctx_len = ctx_len;
  a.K = K;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.window = window;
  a.kps = pl.kps;
  a.nsplit = pl.nsplit;
  a.nqg = pl.nqg;
  a.ob = ob;
  a.err = err;
  a.inj_req = inj_req;
  a.inj_pos = inj_pos;
  a.inj_n = inj_req && inj_pos ? inj_n : 0;
  // pages of 64 positions: whole pages are loaded by TMA from the caches viewed
  // as [n_layers * num_pages * Hkv * 64, dh] matrices
  CUtensorMap mk, mv;
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  const uint64_t rows = (uint64_t)n_layers * num_pages * Hkv * 64;
  const bool tk = P == dfl::kCH && rows < (1ull << 31) && (uintptr_t)kc % 16 == 0 &&
                  (uintptr_t)vc % 16 == 0 && bf16_map(&mk, kc, rows, dh, 64, d->id) &&
                  bf16_map(&mv, vc, rows, dh, 64, d->id);
  const int QR = K * (Hq / Hkv);
  const int kp = QR <= 16 ? 4 : QR <= 32 ? 2 : 1;
  // split launches (a cluster per item, a few tiles per CTA, plus the receive
  // buffer) keep two tile stages so that two CTAs fit on an SM
#define DFL_ATTN(D, KPV)                                                                   \
  return tk ? (pl.nsplit > 1 ? launch_attn_fused<D, KPV, true, 2>(pl, a, B, mk, mv, st)    \
                             : launch_attn_fused<D, KPV, true, 3>(pl, a, B, mk, mv, st))   \
            : launch_attn_fused<D, KPV, false, dfl::kAttnStages>(pl, a, B, mk, mv, st)
  if (dh == 128) {
    if (kp == 4) DFL_ATTN(128, 4);
    if (kp == 2) DFL_ATTN(128, 2);
    DFL_ATTN(128, 1);
  }
  if (dh == 64) {
    if (kp == 4) DFL_ATTN(64, 4);
    if (kp == 2) DFL_ATTN(64, 2);
    DFL_ATTN(64, 1);
  }
#undef DFL_ATTN
  return DFLASH_ERR_DIMS;
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
