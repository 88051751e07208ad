// Projection GEMMs.
//
// bf16 path: one persistent, warp-specialised kernel per shape class.
//   warp 0     TMA producer: weight tile [128 rows x 64] and activation tile
//              [BN rows x 64] per stage, 128-byte swizzle, into a ring of stages
//   warp 1     tensor-memory allocator and tcgen05.mma issuer (M=128, N=BN, K=16
//              per instruction), fp32 accumulators in tensor memory, double
//              buffered so the epilogue of one work unit overlaps the next unit
//   warps 2-9  epilogue, two groups of four (one warp per tensor-memory lane
//              quarter each) on alternate 16-column chunks: tcgen05.ld of the
//              accumulator, coalesced stores
// The weight matrix is the M operand ("swap AB"): at draft batch sizes the token
// count is 8..256, so weights stream through the M dimension and tokens fill N.
// A work unit is (weight tile, token tile, K slice); the CTA's pipeline runs on
// across units without draining.  Weight tiles are loaded with an evict-first
// L2 hint (each is read once per pass); activation tiles with evict-last.
//
// Split-K reduction happens inside the kernel: each unit of a split tile writes
// its slice to scratch, then takes a ticket on the tile (one atomic, no
// waiting); the CTA that takes the last ticket sums the S slices in slice
// order (so the result does not depend on timing), resets the ticket and runs
// the fused epilogue: fp32 and/or storage-dtype output, or SwiGLU, where each
// weight tile holds 64 gate rows and the matching 64 up rows.
//
// fp32 path (the float32 configuration): a shared-memory tiled CUDA-core GEMM.
#include <string.h>

#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "gemm.cuh"

namespace dfl {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kEpiGroups = 2;                         // epilogue warp groups
constexpr int kGemmThreads = 64 + kEpiGroups * 128;   // producer, MMA, epilogue warps

struct GemmParams {
  float *out;  // GEMM_PARTIAL output / slice scratch
  int ld;
  int N_out, T;
  int kb_per_split;
  int S, m_tiles, t_tiles, num_units;
  int mode;
  float *out_f32;
  bf16 *out_bf16;
  int ldb;
  int F;  // GEMM_SWIGLU: gate rows before the up rows
  int *counters;
  int *err;
  // balanced schedule (chunk > 0, reduce modes): the k-block iterations of all
  // tiles, tile after tile, are cut into equal chunks of `chunk`, one per CTA
  int chunk, kb_total, total;
  int nmax;  // slice slots per tile in the scratch
  // grouped weights (GEMM_REDUCE): weight tile m belongs to group m / mtg; group g's
  // outputs start at out_f32 + g * ostride; N_out is the rows of one group
  int mtg;
  size_t ostride;
  // GEMM_REDUCE: optional per-(token, weight tile) (max, sum e^(y - max)) [T][m_tiles]
  float2 *stats;
  // GEMM_QKV: head RMSNorm (q and k heads) + rotate-half RoPE, bf16 out
  const bf16 *q_norm, *k_norm;
  const float2 *rope_cs;  // [T][dh/2] (cos, sin)
  int Hq, Hkv, dh;
  float eps;
  // tokens [T0, T) are injected context rows: k/v heads to the paged cache
  int T0;
  // token tiles from tb on hold context rows only: they skip the first mq weight
  // tiles (q heads only), tiles enumerated as [m_tiles x tb] then [m_tiles - mq
  // x t_tiles - tb]; tb = t_tiles when nothing is skipped
  int tb, mq;
  const long long *ctx_slot;  // per context row: offset in a layer's cache, or -1
  bf16 *kc, *vc;  // this layer's caches
  int P;
  // tile order: weight tile fastest (activations too large to re-read per
  // weight tile) instead of token tile fastest
  int m_fastest;
  // limit of the pipeline's bounded waits; stall (failure-path test only): the
  // MMA issuer first waits on a barrier that nothing arrives on
  uint64_t wait_ns;
  int stall;
  // two-SM tiles (k_gemm_tc2): work units are over pairs of weight tiles
  int pair;
  // 4-bit weights (k_gemm_q4): records of 64 rows x 64 inputs, row block major
  const uint8_t *qdata;
};

// One CTA's share of one tile: k-blocks [kb0, kb0 + nkb), slice `seg` of the
// tile's `nseg` slices.
struct Seg {
  int m_tile, t_tile, kb0, nkb, seg, nseg;
};

// named barriers: 1 + eg for epilogue group eg, 3 for all epilogue warps
__device__ __forceinline__ void epi_bar(int eg) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + eg) : "memory");
}
template <int NEG = kEpiGroups>
__device__ __forceinline__ void epi_all_bar() {
  asm volatile("bar.sync 3, %0;" ::"n"(NEG * 128) : "memory");
}

template <int BN>
struct GemmShape {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int KB_BYTES = A_BYTES + B_BYTES;  // one k-block: weight tile, token tile
  // a stage carries KPS consecutive k-blocks of a segment (fewer at its end), so the
  // MMA issuer's barrier wait, fence and commit are paid once per KPS k-blocks
  static constexpr int KPS = BN <= 128 ? 2 : 1;
  static constexpr int STAGE_BYTES = KPS * KB_BYTES;
  // static shared memory of the epilogue: 18 KB, 27 KB with the staged RoPE rows
  // of a 16-token tile
  static constexpr int STATIC_BYTES = (BN <= 16 ? 27 : 18) * 1024;
  static constexpr int STAGES = (232448 - STATIC_BYTES - 1024 - 256) / STAGE_BYTES;
  static constexpr int TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  static_assert(STAGES >= 3 && 2 * STAGES + 6 <= 256 / 8 - 1, "ring and barriers");
};

// Tile index -> (weight tile, token tile).  Token tile fastest, so that the CTAs
// holding the token tiles of one weight tile run together and the weight tile
// is read from HBM once (the others hit L2) while the activations stay in L2
// throughout; or, when the activations are too large for that (bulk
// injection), weight tile fastest, so that every activation tile is read from
// HBM once and the weights, re-read once per wave of token tiles, come from L2.
__device__ __forceinline__ void tile_coords(int tile, const GemmParams &p, int &m_tile,
                                            int &t_tile) {
  if (p.tb < p.t_tiles) {
    const int a = p.m_tiles * p.tb;
    if (tile < a) {
      t_tile = tile % p.tb;
      m_tile = tile / p.tb;
    } else {
      const int r = tile - a, nt = p.t_tiles - p.tb;
      t_tile = p.tb + r % nt;
      m_tile = p.mq + r / nt;
    }
    return;
  }
  if (p.m_fastest) {
    m_tile = tile % p.m_tiles;
    t_tile = tile / p.m_tiles;
  } else {
    t_tile = tile % p.t_tiles;
    m_tile = tile / p.t_tiles;
  }
}
__device__ __forceinline__ void unit_coords(int u, const GemmParams &p, int &m_tile, int &t_tile,
                                            int &split) {
  split = u % p.S;  // the slices of one tile are adjacent units
  tile_coords(u / p.S, p, m_tile, t_tile);
}

// The i-th segment of this CTA; false when there is none.  Uniform schedule:
// units blockIdx.x + i * gridDim.x, each one K slice of one tile.  Balanced
// schedule: the CTA's chunk [blockIdx.x * chunk, + chunk) of the iteration
// space cut at tile boundaries; a tile's slices come from consecutive CTAs.
__device__ __forceinline__ bool get_seg(const GemmParams &p, int i, Seg &s) {
  if (p.chunk == 0) {
    const int u = blockIdx.x + i * gridDim.x;
    if (u >= p.num_units) return false;
    int split;
    unit_coords(u, p, s.m_tile, s.t_tile, split);
    s.kb0 = split * p.kb_per_split;
    s.nkb = p.kb_per_split;
    s.seg = split;
    s.nseg = p.S;
    return true;
  }
  const int pos0 = blockIdx.x * p.chunk;
  const int end = min(pos0 + p.chunk, p.total);
  const int tile = pos0 / p.kb_total + i;
  const int start = i == 0 ? pos0 : tile * p.kb_total;
  if (start >= end) return false;
  const int stop = min(end, (tile + 1) * p.kb_total);
  tile_coords(tile, p, s.m_tile, s.t_tile);
  s.kb0 = start - tile * p.kb_total;
  s.nkb = stop - start;
  const int first = tile * p.kb_total / p.chunk;
  const int last = ((tile + 1) * p.kb_total - 1) / p.chunk;
  s.seg = blockIdx.x - first;
  s.nseg = last - first + 1;
  return true;
}

constexpr int kMaxGroups = 8;
struct WMaps {
  CUtensorMap m[kMaxGroups];
};

// Weight tile of unit m_tile: 128 consecutive rows of its group's matrix, or for
// GEMM_SWIGLU the 64 gate rows [64m, 64m+64) followed by the 64 up rows
// [F+64m, F+64m+64).
__device__ __forceinline__ void load_w(uint8_t *dst, const WMaps &maps, uint64_t *bar, int kx,
                                       int m_tile, const GemmParams &p, uint64_t pol) {
  if (p.mode == 2) {
    tma_load_2d(dst, &maps.m[0], bar, kx, m_tile * 64, pol);
    tma_load_2d(dst + 64 * BK * 2, &maps.m[0], bar, kx, p.F + m_tile * 64, pol);
  } else {
    const int g = m_tile / p.mtg;
    tma_load_2d(dst, &maps.m[g], bar, kx, (m_tile - g * p.mtg) * BM, pol);
  }
}

// Final values v[16] of row `row` (0..127) of tile m_tile, columns c0..c0+15.
// The four warps of epilogue group eg call this in step (SwiGLU and the head
// norm exchange through the group's xbuf [128][17] and xss [4][16]).
// srope / sslot / sgain (GEMM_QKV, 16-token tiles): the chunk's RoPE rows
// [16][dh/2], cache slots [16] and the q / k norm gains [2][dh] staged in shared
// memory, else nullptr (read from global).
__device__ __forceinline__ void epi_store(const GemmParams &p, int m_tile, int row, int c0,
                                          float *v, float *xbuf, float *xss, int eg,
                                          const float2 *srope = nullptr,
                                          const long long *sslot = nullptr,
                                          const float *sgain = nullptr) {
  if (p.mode == 3) {
    // row n of the QKV projection: head h = n / dh, feature d = n % dh; a tile
    // holds 128 / dh whole heads.  q and k heads: y = RMSNorm(x) * gain, then
    // RoPE on the pairs (d, d + dh/2) with the token's (cos, sin); v heads as is.
    const int lane = row & 31, quarter = row >> 5;
    const int n = m_tile * BM + row, dh = p.dh, half = dh >> 1;
    const int h = n / dh, d = n - h * dh;
    const bool is_q = h < p.Hq, normed = h < p.Hq + p.Hkv;
    float ss[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) ss[j] = v[j] * v[j];
    warp_reduce_scatter<16>(ss, lane);  // lane L: token L >> 1 over this warp's 32 rows
    if ((lane & 1) == 0) xss[quarter * 16 + (lane >> 1)] = ss[0];
#pragma unroll
    for (int j = 0; j < 16; ++j) xbuf[row * 17 + j] = v[j];
    epi_bar(eg);
    if (normed && n < p.N_out) {
      const bf16 *gain = is_q ? p.q_norm : p.k_norm;
      const int w0 = (row - d) >> 5, nw = dh >> 5;  // the head's warps
      const int pr = d < half ? row + half : row - half, di = d < half ? d : d - half;
      const int dp = d < half ? d + half : d - half;
      const float g = sgain ? sgain[(is_q ? 0 : dh) + d] : __bfloat162float(gain[d]);
      const float gp = sgain ? sgain[(is_q ? 0 : dh) + dp] : __bfloat162float(gain[dp]);
      // every load of the chunk before its first store (stores may alias the table)
      float2 cs[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        cs[j] = c0 + j >= p.T ? make_float2(1.f, 0.f)
                : srope      ? srope[j * half + di]
                             : __ldg(&p.rope_cs[(size_t)(c0 + j) * half + di]);
      // the head's sum of squares per token: nw = 2 or 4 warp partials
      const float *s0 = xss + w0 * 16;
      float o[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float sq = s0[j] + s0[16 + j];
        if (nw == 4) sq += s0[32 + j] + s0[48 + j];
        const float inv = rsqrtf(sq / dh + p.eps);
        const float x = v[j] * inv * g, y = xbuf[pr * 17 + j] * inv * gp;
        o[j] = d < half ? x * cs[j].x - y * cs[j].y : x * cs[j].x + y * cs[j].y;
      }
      if (c0 + 16 <= p.T0) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          p.out_bf16[(size_t)(c0 + j) * p.ldb + n] = __float2bfloat16_rn(o[j]);
      } else {
        // injected context rows: k heads to this layer's cache, q heads dropped
        const size_t hoff = (size_t)(h - p.Hq) * p.P * dh + d;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = c0 + j;
          if (t < p.T0) {
            p.out_bf16[(size_t)t * p.ldb + n] = __float2bfloat16_rn(o[j]);
          } else if (t < p.T && !is_q) {
            const long long s = sslot ? sslot[j] : __ldg(p.ctx_slot + (t - p.T0));
            if (s >= 0) p.kc[s + hoff] = __float2bfloat16_rn(o[j]);
          }
        }
      }
    } else if (n < p.N_out) {
      const size_t hoff = (size_t)(h - p.Hq - p.Hkv) * p.P * dh + d;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = c0 + j;
        if (t < p.T0) {
          p.out_bf16[(size_t)t * p.ldb + n] = __float2bfloat16_rn(v[j]);
        } else if (t < p.T) {
          const long long s = sslot ? sslot[j] : __ldg(p.ctx_slot + (t - p.T0));
          if (s >= 0) p.vc[s + hoff] = __float2bfloat16_rn(v[j]);
        }
      }
    }
    epi_bar(eg);
  } else if (p.mode == 1) {
    const int grp = m_tile / p.mtg;
    const int n = (m_tile - grp * p.mtg) * BM + row;  // row within the group
    if (n < p.N_out) {
      float *of = p.out_f32 ? p.out_f32 + grp * p.ostride : nullptr;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = c0 + j;
        if (t < p.T) {
          if (of) of[(size_t)t * p.ld + n] = v[j];
          if (p.out_bf16) p.out_bf16[(size_t)t * p.ldb + n] = __float2bfloat16_rn(v[j]);
        }
      }
    }
    if (p.stats) {
      // per token of the chunk, over the tile's rows: m = max, s = sum e^(y - m)
      const int lane = row & 31, quarter = row >> 5;
      const bool valid = n < p.N_out;
      float w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) w[j] = valid ? v[j] : -INFINITY;
      warp_reduce_scatter_max<16>(w, lane);  // lane L: token L >> 1, this warp's rows
      if ((lane & 1) == 0) xss[quarter * 16 + (lane >> 1)] = w[0];
      epi_bar(eg);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float m = fmaxf(fmaxf(xss[j], xss[16 + j]), fmaxf(xss[32 + j], xss[48 + j]));
        w[j] = valid ? expf(v[j] - m) : 0.f;
      }
      warp_reduce_scatter<16>(w, lane);
      if ((lane & 1) == 0) xbuf[quarter * 16 + (lane >> 1)] = w[0];
      epi_bar(eg);
      if (row < 16 && c0 + row < p.T) {
        const float m = fmaxf(fmaxf(xss[row], xss[16 + row]), fmaxf(xss[32 + row], xss[48 + row]));
        const float sum = (xbuf[row] + xbuf[16 + row]) + (xbuf[32 + row] + xbuf[48 + row]);
        p.stats[(size_t)(c0 + row) * p.m_tiles + m_tile] = make_float2(m, sum);
      }
      epi_bar(eg);  // xss / xbuf are rewritten by the next chunk
    }
  } else {
    // rows 64..127 hold the up projections of the features of rows 0..63
    if (row >= 64) {
#pragma unroll
      for (int j = 0; j < 16; ++j) xbuf[(row - 64) * 17 + j] = v[j];
    }
    epi_bar(eg);
    if (row < 64) {
      const int f = m_tile * 64 + row;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = c0 + j;
        if (t < p.T) {
          const float g = v[j], u = xbuf[row * 17 + j];
          p.out_bf16[(size_t)t * p.ldb + f] = __float2bfloat16_rn(g / (1.f + expf(-g)) * u);
        }
      }
    }
    epi_bar(eg);
  }
}

// Epilogue role (warps 2..2+4*NEG-1): NEG groups of four warps (each group
// covers the four tensor-memory lane quarters); group eg takes the 16-column
// chunks c = 16*eg + 16*NEG*i of each accumulator the MMA issuer hands over.
template <int BN, int NEG = kEpiGroups>
__device__ __forceinline__ void gemm_epilogue(const GemmParams &p, uint32_t tmem_base,
                                              uint64_t *tfull, uint64_t *tempty,
                                              volatile int *abort_flag, int warp, int lane) {
  pdl_wait();
  __shared__ float xbuf[NEG][128 * 17];
  __shared__ float xss[NEG][4 * 16];
  __shared__ int s_last;
  // GEMM_QKV with 16-token tiles: the tile's RoPE rows and cache slots (and,
  // once, the head-norm gains) are staged in shared memory while its MMAs run
  // (the epilogue reads them without a trip to global memory)
  constexpr bool kStage = BN <= 16;
  __shared__ float2 s_rope[kStage ? 16 * 64 : 1];
  __shared__ long long s_slot[kStage ? 16 : 1];
  __shared__ float s_gain[kStage ? 2 * 128 : 1];  // q then k norm gains
  const bool stage_rope = kStage && p.mode == 3 && p.dh <= 128;
  const float2 *srope = stage_rope ? s_rope : nullptr;
  const long long *sslot = stage_rope && p.ctx_slot ? s_slot : nullptr;
  const float *sgain = stage_rope ? s_gain : nullptr;
  if (stage_rope)
    for (int i = threadIdx.x - 64; i < 2 * p.dh; i += 128 * NEG)
      s_gain[i] = __bfloat162float(i < p.dh ? p.q_norm[i] : p.k_norm[i - p.dh]);
  int staged = -1;
  const int quarter = warp & 3;  // tensor-memory lanes this warp may read
  const int eg = (warp - 2) >> 2;
  const int row = quarter * 32 + lane;
  float *gx = xbuf[eg], *gs = xss[eg];
  int acc = 0;
  uint32_t acc_phase = 0;
  Seg sg;
  for (int i = 0; get_seg(p, i, sg); ++i) {
    const int m_tile = sg.m_tile, t_tile = sg.t_tile, split = sg.seg;
    if (stage_rope && t_tile != staged) {
      epi_all_bar<NEG>();  // the previous tile's rows are no longer read
      const int et = threadIdx.x - 64, half = p.dh >> 1, tb = t_tile * BN;
      for (int i = et; i < 16 * half; i += 128 * NEG) {
        const int tok = tb + i / half;
        s_rope[i] =
            tok < p.T ? __ldg(&p.rope_cs[(size_t)tok * half + i % half]) : make_float2(1.f, 0.f);
      }
      if (p.ctx_slot && et < 16) {
        const int tok = tb + et;
        s_slot[et] = tok >= p.T0 && tok < p.T ? __ldg(p.ctx_slot + (tok - p.T0)) : -1;
      }
      epi_all_bar<NEG>();
      staged = t_tile;
    }
    if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, p.wait_ns)) break;
    tc_fence_after();
    const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
    const int tcol0 = t_tile * BN;
    if (p.mode == 0) {
      const int n = m_tile * BM + row;
      float *outp = p.out + (size_t)split * p.T * p.ld + n;
#pragma unroll 1
      for (int c = 16 * eg; c < BN; c += 16 * NEG) {
        float v[16];
        tc_ld16(taddr + c, v);
        const int t0 = tcol0 + c;
        if (n < p.N_out) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (t0 + j < p.T) outp[(size_t)(t0 + j) * p.ld] = v[j];
        }
      }
    } else if (sg.nseg == 1) {
#pragma unroll 1
      for (int c = 16 * eg; c < BN; c += 16 * NEG) {
        if (tcol0 + c >= p.T) break;  // uniform across the group
        float v[16];
        tc_ld16(taddr + c, v);
        epi_store(p, m_tile, row, tcol0 + c, v, gx, gs, eg, srope, sslot, sgain);
      }
    } else {
      // slice -> scratch slot (tile, slice) ([column][row] inside: every
      // store of a warp writes 128 consecutive bytes), then a ticket
      const size_t tile = (size_t)t_tile * p.m_tiles + m_tile;
      const size_t tile_sz = (size_t)BM * BN;
      float *mine = p.out + (tile * p.nmax + split) * tile_sz + row;
#pragma unroll 1
      for (int c = 16 * eg; c < BN; c += 16 * NEG) {
        if (tcol0 + c >= p.T) break;
        float v[16];
        tc_ld16(taddr + c, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) mine[(size_t)(c + j) * BM] = v[j];
      }
      // the accumulator can go back to the MMA warp now
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      // the ticket: the barrier orders every epilogue thread's slice stores
      // before one thread's acquire-release atomic (cumulative at GPU scope);
      // in the last CTA the second barrier orders the slice loads after it
      epi_all_bar<NEG>();
      if (threadIdx.x == 64) {
        const int old = atomic_add_acq_rel_gpu(&p.counters[tile], 1);
        s_last = old == sg.nseg - 1;
        if (s_last) p.counters[tile] = 0;
      }
      epi_all_bar<NEG>();
      if (s_last) {
        // sum the slices in slice order, CPI of the group's chunks per pass and
        // four slices (two for wider tiles) per round, so that their loads
        // are in flight together
        constexpr int CPI = BN >= 128 ? 4 : BN >= 64 ? 2 : 1;
        const float *base = p.out + tile * p.nmax * tile_sz + row;
#pragma unroll 1
        for (int c = 16 * eg; c < BN; c += 16 * NEG * CPI) {
          if (tcol0 + c >= p.T) break;
          float v[CPI][16];
#pragma unroll
          for (int k = 0; k < CPI; ++k)
#pragma unroll
            for (int j = 0; j < 16; ++j) v[k][j] = 0.f;
#pragma unroll(CPI == 1 ? 4 : 2)
          for (int q = 0; q < sg.nseg; ++q) {
#pragma unroll
            for (int k = 0; k < CPI; ++k) {
              const int cc = c + 16 * NEG * k;
              if (cc < BN && tcol0 + cc < p.T) {
                const float *src = base + (size_t)q * tile_sz + (size_t)cc * BM;
#pragma unroll
                for (int j = 0; j < 16; ++j) v[k][j] += __ldcg(src + (size_t)j * BM);
              }
            }
          }
#pragma unroll
          for (int k = 0; k < CPI; ++k) {
            const int cc = c + 16 * NEG * k;
            if (cc < BN && tcol0 + cc < p.T)  // uniform across the group
              epi_store(p, m_tile, row, tcol0 + cc, v[k], gx, gs, eg, srope, sslot, sgain);
          }
        }
      }
      if (++acc == 2) acc = 0, acc_phase ^= 1;
      continue;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&tempty[acc]);
    if (++acc == 2) acc = 0, acc_phase ^= 1;
  }
}
template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm_tc(const __grid_constant__ WMaps tmW, const __grid_constant__ CUtensorMap tmX,
              GemmParams p) {
  using SH = GemmShape<BN>;
  constexpr int STAGES = SH::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *full = (uint64_t *)(smem + STAGES * SH::STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint64_t *stallbar = drain + 1;
  uint32_t *tmem_slot = (uint32_t *)(stallbar + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4 * kEpiGroups);
    }
    mbar_init(drain, 1);
    mbar_init(stallbar, 1);
    *abort_flag = 0;
    mbar_fence_init();
    for (int g = 0; g * p.mtg < p.m_tiles && g < kMaxGroups; ++g) tma_prefetch_desc(&tmW.m[g]);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tc_alloc(tmem_slot, SH::TMEM_COLS);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t last_phase[STAGES];
      bool issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = false, last_phase[s] = 0;
      // Weights do not depend on the previous kernel: prefetch the first
      // stages' weight tiles before waiting for it, then add activations.
      int pre = 0;
      {
        Seg sg;
        for (int i = 0; pre < STAGES && get_seg(p, i, sg); ++i) {
          for (int kb = 0; kb < sg.nkb && pre < STAGES; kb += SH::KPS, ++pre) {
            const int nk = min(SH::KPS, sg.nkb - kb);
            mbar_expect_tx(&full[pre], nk * SH::KB_BYTES);
            for (int k = 0; k < nk; ++k)
              load_w(smem + pre * SH::STAGE_BYTES + k * SH::KB_BYTES, tmW, &full[pre],
                     (sg.kb0 + kb + k) * BK, sg.m_tile, p, pol_w);
          }
        }
      }
      pdl_wait();
      bool ok = true;
      int n = 0;  // fill counter across segments
      Seg sg;
      for (int i = 0; ok && get_seg(p, i, sg); ++i) {
        for (int kb = 0; kb < sg.nkb; kb += SH::KPS, ++n) {
          uint8_t *sa = smem + stage * SH::STAGE_BYTES;
          const int nk = min(SH::KPS, sg.nkb - kb);
          if (n >= pre) {
            if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&full[stage], nk * SH::KB_BYTES);
            for (int k = 0; k < nk; ++k)
              load_w(sa + k * SH::KB_BYTES, tmW, &full[stage], (sg.kb0 + kb + k) * BK, sg.m_tile,
                     p, pol_w);
          }
          for (int k = 0; k < nk; ++k)
            tma_load_2d(sa + k * SH::KB_BYTES + SH::A_BYTES, &tmX, &full[stage],
                        (sg.kb0 + kb + k) * BK, sg.t_tile * BN, pol_x);
          issued[stage] = true;
          last_phase[stage] = phase;
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
      }
      // every copy this warp issued has landed before shared memory is released
      // (already so when the MMA issuer consumed them; not when a wait gave up)
      {
        volatile int dummy = 0;
        for (int s = 0; s < STAGES; ++s)
          if (issued[s]) mbar_wait(&full[s], last_phase[s], (volatile int *)&dummy);
      }
    }
    __syncwarp();  // lane 0 rejoins its warp before the block-wide barrier below
  } else if (warp == 1) {
    pdl_wait();
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      if (p.stall && !mbar_wait(stallbar, 0, abort_flag, p.wait_ns)) ok = false;
      Seg sg;
      for (int i = 0; ok && get_seg(p, i, sg); ++i) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < sg.nkb; kb += SH::KPS) {
          const int nk = min(SH::KPS, sg.nkb - kb);
          if (!mbar_wait(&full[stage], phase, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int k = 0; k < nk; ++k) {
            const uint32_t sa = smem_u32(smem + stage * SH::STAGE_BYTES + k * SH::KB_BYTES);
            const uint64_t adesc = sdesc_k_sw128(sa);
            const uint64_t bdesc = sdesc_k_sw128(sa + SH::A_BYTES);
#pragma unroll
            for (int j = 0; j < BK / 16; ++j) {
              // advance 16 bf16 = 32 bytes along K inside the swizzled row
              tc_mma_bf16(d_tmem, adesc + (uint64_t)(j * 2), bdesc + (uint64_t)(j * 2), idesc,
                          (kb | k | j) != 0);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
        if (++acc == 2) acc = 0, acc_phase ^= 1;
      }
      if (!ok) {
        // drain: wait (bounded) until the MMAs issued so far have finished
        volatile int dummy = 0;
        tc_commit(drain);
        (void)mbar_wait(drain, 0, (volatile int *)&dummy);
      }
    }
    __syncwarp();  // lane 0 rejoins its warp before the block-wide barrier below
  } else {
    gemm_epilogue<BN>(p, tmem_base, tfull, tempty, abort_flag, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) set_err(p.err, DFLASH_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem_base, SH::TMEM_COLS);
  }
}


// ---------------------------------------------------------------------------
// 4-bit weights
// ---------------------------------------------------------------------------
// Weights kept as 4-bit codes q with one (scale s, bias b) pair per row and
// group of 64 input features (one k-block); the MMA multiplies w = bf16(s*q + b).
// Storage (the C ABI's dflash_q4): records of 2304 bytes, one per 64-row block
// and k-block, row block major: the 64 rows' codes (32 bytes a row; the 32-bit
// word of features 8j..8j+7 holds their codes, from the least significant
// nibble up, in the order 8j, 8j+2, 8j+4, 8j+6, 8j+1, 8j+3, 8j+5, 8j+7, so that
// (word >> 4i) & 0x000F000F is the pair (8j+2i, 8j+2i+1) in the two halves of
// a bf16x2), then the rows' (scale, bias) words (bf16 scale low, bias high).
// A k-block of a 128-row tile is two contiguous records, brought in by two bulk
// copies.
// Roles (448 threads): warp 0 bulk-copy producer (records, activation tiles),
// warp 1 MMA issuer, warps 2-5 one epilogue group (the epilogue of k_gemm_tc),
// warps 6-13 dequantize: the thread on tensor-memory lane r (warp w covers
// lanes 32*(w%4)..) of half h = (w - 6) / 4 turns inputs 32h..32h+31 of row r
// of a k-block into bf16 weights and stores them as columns 16h..16h+15 of an
// A buffer in tensor memory, from which the MMA reads its A operand; each warp
// overlaps one k-block's store with the next k-block's loads and arithmetic.
// Shared memory holds only the code stages (activation tile | codes | pairs),
// released by the dequantizers and the MMA together; tensor memory holds the
// two accumulators and a ring of A buffers released by the MMA's commits.
constexpr int kQ4Record = 64 * 32 + 64 * 4;  // codes and pairs of 64 rows x 64 inputs
// A stage carries KPS consecutive k-blocks of a segment (fewer at a segment's
// end): the MMA issuer's barrier waits, fence and commits, which cost more than
// its four MMAs per k-block, are paid once per stage.
template <int BN>
struct QShape {
  static_assert(BN <= 128, "4-bit tiles keep A buffers beside the accumulators");
  static constexpr int KPS = BN <= 64 ? 4 : 2;
  static constexpr int X_BYTES = BN * BK * 2;
  static constexpr int KB_TX = X_BYTES + 2 * kQ4Record;  // bytes one k-block brings in
  // KPS activation tiles (1024-byte aligned), then KPS pairs of records
  static constexpr int STAGE_BYTES = (KPS * KB_TX + 1023) / 1024 * 1024;
  static constexpr int NQ = (232448 - 18 * 1024 - 1024 - 768) / STAGE_BYTES;
  static constexpr int TMEM_COLS = 512;
  static constexpr int A_COL0 = 2 * BN < 32 ? 32 : 2 * BN;  // after the accumulators
  static constexpr int A_COLS = 32 * KPS;                    // one stage's A buffer
  static constexpr int NA = (TMEM_COLS - A_COL0) / A_COLS;
  static constexpr int SMEM_BYTES = NQ * STAGE_BYTES + 1024 + 768;
  static_assert(NA >= 2 && NQ >= 2, "rings");
  static_assert(SMEM_BYTES + 18 * 1024 <= 232448, "dynamic + the epilogue's static shared memory");
  static_assert(2 * NQ + 2 * NA + 5 <= 768 / 8 - 1, "barriers");
};
constexpr int kQ4Epi = 1;  // epilogue groups
constexpr int kQ4Dq = 8;   // dequantizing warps
constexpr int kQ4Threads = 64 + kQ4Epi * 128 + kQ4Dq * 32;

// the two records of weight tile m_tile, k-block kb, into dst; GEMM_SWIGLU: the
// gate rows' block m_tile, then the up rows' block F/64 + m_tile
__device__ __forceinline__ void load_wq(uint8_t *dst, uint64_t *bar, int kb, int m_tile,
                                        const GemmParams &p, uint64_t pol) {
  const int rb0 = p.mode == 2 ? m_tile : 2 * m_tile;
  const int rb1 = p.mode == 2 ? p.F / 64 + m_tile : 2 * m_tile + 1;
  const size_t per_block = (size_t)p.kb_total * kQ4Record;
  bulk_load(dst, p.qdata + rb0 * per_block + (size_t)kb * kQ4Record, kQ4Record, bar, pol);
  bulk_load(dst + kQ4Record, p.qdata + rb1 * per_block + (size_t)kb * kQ4Record, kQ4Record, bar,
            pol);
}

// bf16x2 (s*q_lo + b, s*q_hi + b), each rounded once, for the code pair at
// nibbles `shift` and 16 + shift of w; s2 / b2 hold the scale / bias twice
__device__ __forceinline__ uint32_t dq_pair(uint32_t w, int shift, uint32_t s2, uint32_t b2) {
  const uint32_t m = ((w >> shift) & 0x000F000Fu) | 0x43004300u;  // (128 + q_lo, 128 + q_hi)
  uint32_t q, r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(q) : "r"(m), "r"(0x43004300u));
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(q), "r"(s2), "r"(b2));
  return r;
}

template <int BN>
__global__ void __launch_bounds__(kQ4Threads, 1)
    k_gemm_q4(const __grid_constant__ CUtensorMap tmX, GemmParams p) {
  using QS = QShape<BN>;
  constexpr int NQ = QS::NQ, NA = QS::NA, KPS = QS::KPS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *qfull = (uint64_t *)(smem + NQ * QS::STAGE_BYTES);
  uint64_t *qempty = qfull + NQ;
  uint64_t *afull = qempty + NQ;
  uint64_t *aempty = afull + NA;
  uint64_t *tfull = aempty + NA;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = (uint32_t *)(drain + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // stage layout: activation tile k at k * X_BYTES, records of k-block k after the tiles
  auto xtile = [&](int st, int k) { return smem + st * QS::STAGE_BYTES + k * QS::X_BYTES; };
  auto recs = [&](int st, int k) {
    return smem + st * QS::STAGE_BYTES + KPS * QS::X_BYTES + k * 2 * kQ4Record;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NQ; ++s) {
      mbar_init(&qfull[s], 1);
      mbar_init(&qempty[s], 1 + kQ4Dq);  // the MMA's commit and the dequantizing warps
    }
    for (int a = 0; a < NA; ++a) {
      mbar_init(&afull[a], kQ4Dq);
      mbar_init(&aempty[a], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4 * kQ4Epi);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tc_alloc(tmem_slot, QS::TMEM_COLS);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- bulk-copy producer ----------------
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t last_phase[NQ];
      bool issued[NQ];
      for (int s = 0; s < NQ; ++s) issued[s] = false, last_phase[s] = 0;
      // records do not depend on the previous kernel: the first stages' start
      // before waiting for it, the activation tiles after
      int pre = 0;
      {
        Seg sg;
        for (int i = 0; pre < NQ && get_seg(p, i, sg); ++i) {
          for (int kb = 0; kb < sg.nkb && pre < NQ; kb += KPS, ++pre) {
            const int nk = min(KPS, sg.nkb - kb);
            mbar_expect_tx(&qfull[pre], nk * QS::KB_TX);
            for (int k = 0; k < nk; ++k)
              load_wq(recs(pre, k), &qfull[pre], sg.kb0 + kb + k, sg.m_tile, p, pol_w);
          }
        }
      }
      pdl_wait();
      bool ok = true;
      int n = 0;
      Seg sg;
      for (int i = 0; ok && get_seg(p, i, sg); ++i) {
        for (int kb = 0; kb < sg.nkb; kb += KPS, ++n) {
          const int nk = min(KPS, sg.nkb - kb);
          if (n >= pre) {
            if (!mbar_wait(&qempty[stage], phase ^ 1, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&qfull[stage], nk * QS::KB_TX);
            for (int k = 0; k < nk; ++k)
              load_wq(recs(stage, k), &qfull[stage], sg.kb0 + kb + k, sg.m_tile, p, pol_w);
          }
          for (int k = 0; k < nk; ++k)
            tma_load_2d(xtile(stage, k), &tmX, &qfull[stage], (sg.kb0 + kb + k) * BK,
                        sg.t_tile * BN, pol_x);
          issued[stage] = true;
          last_phase[stage] = phase;
          if (++stage == NQ) stage = 0, phase ^= 1;
        }
      }
      // every copy this warp issued has landed before shared memory is released
      {
        volatile int dummy = 0;
        for (int s = 0; s < NQ; ++s)
          if (issued[s]) mbar_wait(&qfull[s], last_phase[s], (volatile int *)&dummy);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    pdl_wait();
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      int qs = 0, as = 0;
      uint32_t qph = 0, aph = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      Seg sg;
      for (int i = 0; ok && get_seg(p, i, sg); ++i) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < sg.nkb; kb += KPS) {
          const int nk = min(KPS, sg.nkb - kb);
          if (!mbar_wait(&afull[as], aph, abort_flag, p.wait_ns) ||
              !mbar_wait(&qfull[qs], qph, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem_base + (uint32_t)(QS::A_COL0 + as * QS::A_COLS);
          for (int k = 0; k < nk; ++k) {
            const uint64_t bdesc = sdesc_k_sw128(smem_u32(xtile(qs, k)));
#pragma unroll
            for (int j = 0; j < BK / 16; ++j)  // 16 bf16 of K = 8 tensor-memory columns
              tc_mma_bf16_ta(d_tmem, a_tmem + (uint32_t)(k * 32 + j * 8),
                             bdesc + (uint64_t)(j * 2), idesc, (kb | k | j) != 0);
          }
          tc_commit(&qempty[qs]);
          tc_commit(&aempty[as]);
          if (++qs == NQ) qs = 0, qph ^= 1;
          if (++as == NA) as = 0, aph ^= 1;
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
        if (++acc == 2) acc = 0, acc_phase ^= 1;
      }
      if (!ok) {
        volatile int dummy = 0;
        tc_commit(drain);
        (void)mbar_wait(drain, 0, (volatile int *)&dummy);
      }
    }
    __syncwarp();
  } else if (warp < 2 + 4 * kQ4Epi) {
    gemm_epilogue<BN, kQ4Epi>(p, tmem_base, tfull, tempty, abort_flag, warp, lane);
  } else {
    // ---------------- dequantize: warps 6..13 ----------------
    // (records are weights: no wait for the previous kernel)
    const int quarter = warp & 3, h = (warp - 2 - 4 * kQ4Epi) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_addr =
        tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(QS::A_COL0 + 16 * h);
    const int roff = (r >> 6) * kQ4Record, rrow = r & 63;
    int qs = 0, as = 0, pq = 0, pa = 0;
    uint32_t qph = 0, aph = 0;
    bool ok = true, pending = false;
    // hand stage (pq, pa) over once its tensor-memory stores have completed
    auto release = [&]() {
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&afull[pa]);
        mbar_arrive(&qempty[pq]);
      }
    };
    Seg sg;
    for (int i = 0; ok && get_seg(p, i, sg); ++i) {
      for (int kb = 0; kb < sg.nkb; kb += KPS) {
        const int nk = min(KPS, sg.nkb - kb);
        const bool got = mbar_wait(&qfull[qs], qph, abort_flag, p.wait_ns) &&
                         mbar_wait(&aempty[as], aph ^ 1, abort_flag, p.wait_ns);
        if (!__all_sync(0xffffffffu, got)) {  // the warp gives up together
          ok = false;
          break;
        }
        tc_fence_after();
        for (int k = 0; k < nk; ++k) {
          const uint8_t *rec = recs(qs, k) + roff;
          const uint4 w = *(const uint4 *)(rec + rrow * 32 + 16 * h);
          const uint32_t sb = *(const uint32_t *)(rec + 64 * 32 + rrow * 4);
          const uint32_t s2 = (sb & 0xFFFFu) * 0x10001u, b2 = (sb >> 16) * 0x10001u;
          const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
          uint32_t a[16];  // column 16h + j: weights (32h + 2j, 32h + 2j + 1) of the row
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            a[4 * c + 0] = dq_pair(wd[c], 0, s2, b2);
            a[4 * c + 1] = dq_pair(wd[c], 4, s2, b2);
            a[4 * c + 2] = dq_pair(wd[c], 8, s2, b2);
            a[4 * c + 3] = dq_pair(wd[c], 12, s2, b2);
          }
          if (k == 0 && pending) release();  // the previous stage's stores had this long
          tc_st16(lane_addr + (uint32_t)(as * QS::A_COLS + k * 32), a);
        }
        pending = true;
        pq = qs;
        pa = as;
        if (++qs == NQ) qs = 0, qph ^= 1;
        if (++as == NA) as = 0, aph ^= 1;
      }
    }
    if (pending) {
      if (ok) {
        release();
      } else {
        tc_wait_st();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) set_err(p.err, DFLASH_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem_base, QS::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Two-SM tiles for wide token tiles
// ---------------------------------------------------------------------------
// A cluster of two CTAs on two SMs computes a 256-row x 256-token tile with
// tcgen05.mma.cta_group::2: CTA rank r holds weight tile 2*mp + r (its 128
// rows) and the r-th 128 tokens of the token tile in shared memory, each MMA
// reads A and B halves from both CTAs, and each CTA's tensor memory receives
// its 128 rows x 256 tokens.  Per SM a k-block then moves 32 KB for 4.2 MFLOP
// (a one-SM 128 x 256 tile moves 48 KB), so six stages fit where four did.
//   warp 0     TMA producer of this CTA's halves; both CTAs' loads of a stage
//              complete on the even CTA's full barrier (TMA with cta_group::2),
//              which the even producer arms for both CTAs' bytes
//   warp 1     even CTA: waits for full stages, issues the pair MMAs and commits
//              them to both CTAs' empty / tfull barriers (odd CTA: idle)
//   warps 2-9  epilogue of this CTA's rows, as in k_gemm_tc; they release an
//              accumulator on the even CTA's tempty barrier
// The two CTAs walk the same units (pair tile, token tile, K slice) in lockstep.
// Before leaving, the even CTA waits (bounded) on its full barriers for the
// last stage each CTA issued, so that no copy into either CTA is in flight.
constexpr int kPairBN = 256;
struct PairShape {
  static constexpr int A_BYTES = BM * BK * 2;             // this CTA's 128 weight rows
  static constexpr int B_BYTES = (kPairBN / 2) * BK * 2;  // this CTA's 128 tokens
  static constexpr int KB_BYTES = A_BYTES + B_BYTES;      // one k-block
  static constexpr int KPS = 2;                            // k-blocks a stage
  static constexpr int STAGE_BYTES = KPS * KB_BYTES;
  static constexpr int STAGES = 3;
  static constexpr int TMEM_COLS = 2 * kPairBN;  // two accumulators of 256 columns
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 512 /*barriers*/;
};

// The i-th unit of this CTA's pair (uniform schedule over pair tiles).
__device__ __forceinline__ bool get_seg_pair(const GemmParams &p, int i, uint32_t rank, Seg &s) {
  const int u = (int)(blockIdx.x >> 1) + i * (int)(gridDim.x >> 1);
  if (u >= p.num_units) return false;
  // an odd tile count: the last pair's odd CTA holds a phantom tile (rows past
  // the weights: zero-filled loads, nothing stored)
  const int split = u % p.S, tile = u / p.S, mpairs = (p.m_tiles + 1) >> 1;
  int mp, t;
  if (p.m_fastest) {
    mp = tile % mpairs;
    t = tile / mpairs;
  } else {
    t = tile % p.t_tiles;
    mp = tile / p.t_tiles;
  }
  s.m_tile = 2 * mp + (int)rank;
  s.t_tile = t;
  s.kb0 = split * p.kb_per_split;
  s.nkb = p.kb_per_split;
  s.seg = split;
  s.nseg = p.S;
  return true;
}

// load_w with the completion counted on the even CTA's barrier (cluster address)
__device__ __forceinline__ void load_w_pair(uint8_t *dst, const WMaps &maps, uint32_t bar_cl,
                                            int kx, int m_tile, const GemmParams &p,
                                            uint64_t pol) {
  if (p.mode == 2) {
    tma_load_2d_pair(dst, &maps.m[0], bar_cl, kx, m_tile * 64, pol);
    tma_load_2d_pair(dst + 64 * BK * 2, &maps.m[0], bar_cl, kx, p.F + m_tile * 64, pol);
  } else {
    // a phantom tile (m_tile == m_tiles, one weight group) reads past the
    // group's rows: the load fills zeros
    const int g = min(m_tile / p.mtg, p.m_tiles / p.mtg - 1);
    tma_load_2d_pair(dst, &maps.m[g], bar_cl, kx, (m_tile - g * p.mtg) * BM, pol);
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm_tc2(const __grid_constant__ WMaps tmW, const __grid_constant__ CUtensorMap tmX,
               GemmParams p) {
  using SH = PairShape;
  constexpr int STAGES = SH::STAGES, BN = kPairBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *full = (uint64_t *)(smem + STAGES * SH::STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = (uint32_t *)(drain + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool even = rank == 0;
  // the producer's issue record (per stage: issued, last phase), read by the even
  // CTA before the pair leaves
  __shared__ uint32_t s_issued[STAGES], s_lphase[STAGES];

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);  // the even CTA's: armed by its producer for both CTAs' bytes
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * 4 * kEpiGroups);  // the epilogue warps of both CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
    for (int g = 0; g * p.mtg < p.m_tiles && g < kMaxGroups; ++g) tma_prefetch_desc(&tmW.m[g]);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tc2_alloc(tmem_slot, SH::TMEM_COLS);
    tc2_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers and tensor memory exist before any traffic between them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (this CTA's halves) ----------------
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      const int xrow = (int)rank * (BN / 2);
      const uint32_t full0 = cluster_addr(smem_u32(&full[0]), 0);  // the even CTA's
      int stage = 0;
      uint32_t phase = 0;
      uint32_t last_phase[STAGES];
      bool issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = false, last_phase[s] = 0;
      int pre = 0;
      {
        Seg sg;
        for (int i = 0; pre < STAGES && get_seg_pair(p, i, rank, sg); ++i) {
          for (int kb = 0; kb < sg.nkb && pre < STAGES; kb += SH::KPS, ++pre) {
            const int nk = min(SH::KPS, sg.nkb - kb);
            if (even) mbar_expect_tx(&full[pre], 2 * nk * SH::KB_BYTES);
            for (int k = 0; k < nk; ++k)
              load_w_pair(smem + pre * SH::STAGE_BYTES + k * SH::KB_BYTES, tmW,
                          full0 + (uint32_t)(pre * 8), (sg.kb0 + kb + k) * BK, sg.m_tile, p,
                          pol_w);
          }
        }
      }
      pdl_wait();
      bool ok = true;
      int n = 0;
      Seg sg;
      for (int i = 0; ok && get_seg_pair(p, i, rank, sg); ++i) {
        for (int kb = 0; kb < sg.nkb; kb += SH::KPS, ++n) {
          uint8_t *sa = smem + stage * SH::STAGE_BYTES;
          const int nk = min(SH::KPS, sg.nkb - kb);
          const uint32_t fb = full0 + (uint32_t)(stage * 8);
          if (n >= pre) {
            if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            if (even) mbar_expect_tx(&full[stage], 2 * nk * SH::KB_BYTES);
            for (int k = 0; k < nk; ++k)
              load_w_pair(sa + k * SH::KB_BYTES, tmW, fb, (sg.kb0 + kb + k) * BK, sg.m_tile, p,
                          pol_w);
          }
          for (int k = 0; k < nk; ++k)
            tma_load_2d_pair(sa + k * SH::KB_BYTES + SH::A_BYTES, &tmX, fb, (sg.kb0 + kb + k) * BK,
                             sg.t_tile * BN + xrow, pol_x);
          issued[stage] = true;
          last_phase[stage] = phase;
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
      }
      for (int s = 0; s < STAGES; ++s) s_issued[s] = issued[s] ? 1u : 0u, s_lphase[s] = last_phase[s];
    }
    __syncwarp();
  } else if (warp == 1) {
    pdl_wait();
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Seg sg;
      if (even) {
        // ---------------- pair MMA issuer ----------------
        constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN);
        int acc = 0;
        uint32_t acc_phase = 0;
        bool any = false;
        for (int i = 0; ok && get_seg_pair(p, i, rank, sg); ++i) {
          if (!mbar_wait<true>(&tempty[acc], acc_phase ^ 1, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
          for (int kb = 0; kb < sg.nkb; kb += SH::KPS) {
            const int nk = min(SH::KPS, sg.nkb - kb);
            if (!mbar_wait<true>(&full[stage], phase, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int k = 0; k < nk; ++k) {
              const uint32_t sa = smem_u32(smem + stage * SH::STAGE_BYTES + k * SH::KB_BYTES);
              const uint64_t adesc = sdesc_k_sw128(sa);
              const uint64_t bdesc = sdesc_k_sw128(sa + SH::A_BYTES);
#pragma unroll
              for (int j = 0; j < BK / 16; ++j)
                tc2_mma_bf16(d_tmem, adesc + (uint64_t)(j * 2), bdesc + (uint64_t)(j * 2), idesc,
                             (kb | k | j) != 0);
            }
            any = true;
            tc2_commit_mc(&empty[stage], 0x3);
            if (++stage == STAGES) stage = 0, phase ^= 1;
          }
          if (!ok) break;
          tc2_commit_mc(&tfull[acc], 0x3);
          if (++acc == 2) acc = 0, acc_phase ^= 1;
        }
        if (!ok && any) {
          // drain: wait (bounded) until the pair MMAs issued so far have finished
          volatile int dummy = 0;
          tc2_commit_mc(drain, 0x1);
          (void)mbar_wait(drain, 0, (volatile int *)&dummy);
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: warps 2..9 (this CTA's 128 rows) ----------------
    pdl_wait();
    __shared__ float xbuf[kEpiGroups][128 * 17];
    __shared__ float xss[kEpiGroups][4 * 16];
    __shared__ int s_last;
    const int quarter = warp & 3;
    const int eg = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    float *gx = xbuf[eg], *gs = xss[eg];
    // where this CTA's warps release an accumulator: the even CTA's tempty
    const uint32_t te0 = cluster_addr(smem_u32(&tempty[0]), 0);
    auto release = [&](int a) {
      if (even)
        mbar_arrive(&tempty[a]);
      else
        mbar_arrive_cluster(te0 + (uint32_t)(a * sizeof(uint64_t)));
    };
    int acc = 0;
    uint32_t acc_phase = 0;
    Seg sg;
    for (int i = 0; get_seg_pair(p, i, rank, sg); ++i) {
      const int m_tile = sg.m_tile, t_tile = sg.t_tile, split = sg.seg;
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, p.wait_ns)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      const int tcol0 = t_tile * BN;
      if (m_tile >= p.m_tiles) {
        // a phantom tile: nothing to store (every CTA of it skips, tickets too)
      } else if (p.mode == 0) {
        const int n = m_tile * BM + row;
        float *outp = p.out + (size_t)split * p.T * p.ld + n;
#pragma unroll 1
        for (int c = 16 * eg; c < BN; c += 32) {
          float v[16];
          tc_ld16(taddr + c, v);
          const int t0 = tcol0 + c;
          if (n < p.N_out) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (t0 + j < p.T) outp[(size_t)(t0 + j) * p.ld] = v[j];
          }
        }
      } else if (sg.nseg == 1) {
#pragma unroll 1
        for (int c = 16 * eg; c < BN; c += 32) {
          if (tcol0 + c >= p.T) break;
          float v[16];
          tc_ld16(taddr + c, v);
          epi_store(p, m_tile, row, tcol0 + c, v, gx, gs, eg);
        }
      } else {
        const size_t tile = (size_t)t_tile * p.m_tiles + m_tile;
        const size_t tile_sz = (size_t)BM * BN;
        float *mine = p.out + (tile * p.nmax + split) * tile_sz + row;
#pragma unroll 1
        for (int c = 16 * eg; c < BN; c += 32) {
          if (tcol0 + c >= p.T) break;
          float v[16];
          tc_ld16(taddr + c, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) mine[(size_t)(c + j) * BM] = v[j];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release(acc);
        epi_all_bar();
        if (threadIdx.x == 64) {
          const int old = atomic_add_acq_rel_gpu(&p.counters[tile], 1);
          s_last = old == sg.nseg - 1;
          if (s_last) p.counters[tile] = 0;
        }
        epi_all_bar();
        if (s_last) {
          constexpr int CPI = 4;
          const float *base = p.out + tile * p.nmax * tile_sz + row;
#pragma unroll 1
          for (int c = 16 * eg; c < BN; c += 32 * CPI) {
            if (tcol0 + c >= p.T) break;
            float v[CPI][16];
#pragma unroll
            for (int k = 0; k < CPI; ++k)
#pragma unroll
              for (int j = 0; j < 16; ++j) v[k][j] = 0.f;
#pragma unroll 2
            for (int q = 0; q < sg.nseg; ++q) {
#pragma unroll
              for (int k = 0; k < CPI; ++k) {
                const int cc = c + 32 * k;
                if (cc < BN && tcol0 + cc < p.T) {
                  const float *src = base + (size_t)q * tile_sz + (size_t)cc * BM;
#pragma unroll
                  for (int j = 0; j < 16; ++j) v[k][j] += __ldcg(src + (size_t)j * BM);
                }
              }
            }
#pragma unroll
            for (int k = 0; k < CPI; ++k) {
              const int cc = c + 32 * k;
              if (cc < BN && tcol0 + cc < p.T) epi_store(p, m_tile, row, tcol0 + cc, v[k], gx, gs, eg);
            }
          }
        }
        if (++acc == 2) acc = 0, acc_phase ^= 1;
        continue;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release(acc);
      if (++acc == 2) acc = 0, acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs have stopped issuing; their issue records are visible
  if (even && threadIdx.x == 0) {
    // every copy either CTA issued has landed (already so unless a wait gave up)
    volatile int dummy = 0;
    for (int c = 0; c < 2; ++c)
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t iss = c == 0 ? s_issued[s] : ld_dsmem_u32(smem_u32(&s_issued[s]), 1);
        const uint32_t ph = c == 0 ? s_lphase[s] : ld_dsmem_u32(smem_u32(&s_lphase[s]), 1);
        if (iss) (void)mbar_wait<true>(&full[s], ph, (volatile int *)&dummy);
      }
  }
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair may still use its memory or barriers
  if (threadIdx.x == 0 && *abort_flag) set_err(p.err, DFLASH_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tc2_dealloc(tmem_base, SH::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// fp32 CUDA-core GEMM (float32 configuration)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_gemm_f32(const float *__restrict__ W,
                                                  const float *__restrict__ X,
                                                  float *__restrict__ out, int ld, int N, int T,
                                                  int K, int kps) {
  __shared__ float Ws[64][33];
  __shared__ float Xs[32][33];
  pdl_launch();
  pdl_wait();
  const int n0 = blockIdx.x * 64, t0 = blockIdx.y * 32, s = blockIdx.z;
  const int tn = threadIdx.x & 15, tt = threadIdx.x >> 4;  // 16 x 16 threads
  float acc[4][2] = {};
  const int kbeg = s * kps, kend = kbeg + kps;
  for (int k0 = kbeg; k0 < kend; k0 += 32) {
    for (int i = threadIdx.x; i < 64 * 32; i += 256) {
      int r = i >> 5, c = i & 31;
      Ws[r][c] = (n0 + r < N) ? W[(size_t)(n0 + r) * K + k0 + c] : 0.f;
    }
    for (int i = threadIdx.x; i < 32 * 32; i += 256) {
      int r = i >> 5, c = i & 31;
      Xs[r][c] = (t0 + r < T) ? X[(size_t)(t0 + r) * K + k0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < 32; ++c) {
      float x0 = Xs[tt * 2][c], x1 = Xs[tt * 2 + 1][c];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float w = Ws[tn * 4 + i][c];
        acc[i][0] = fmaf(w, x0, acc[i][0]);
        acc[i][1] = fmaf(w, x1, acc[i][1]);
      }
    }
    __syncthreads();
  }
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 2; ++j) {
      int n = n0 + tn * 4 + i, t = t0 + tt * 2 + j;
      if (n < N && t < T) out[((size_t)s * T + t) * ld + n] = acc[i][j];
    }
}

// fp32 configuration: reduce the slices of k_gemm_f32 and apply the epilogue.
// part: [S][T][ld_part]; mode 1 -> out_f32 / out (float storage); mode 2 -> SwiGLU.
__global__ void __launch_bounds__(256) k_gemm_f32_finish(const float *__restrict__ part, int S,
                                                         int T, int N_out, int ld_part, int mode,
                                                         int F, float *__restrict__ out_f32,
                                                         int ld, float *__restrict__ out_s,
                                                         int ldb) {
  pdl_launch();
  pdl_wait();
  const size_t n = (size_t)T * N_out;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / N_out), c = (int)(i % N_out);
    if (mode == 1) {
      float v = 0.f;
      for (int k = 0; k < S; ++k) v += part[((size_t)k * T + t) * ld_part + c];
      if (out_f32) out_f32[(size_t)t * ld + c] = v;
      if (out_s) out_s[(size_t)t * ldb + c] = v;
    } else {
      float g = 0.f, u = 0.f;
      for (int k = 0; k < S; ++k) {
        g += part[((size_t)k * T + t) * ld_part + c];
        u += part[((size_t)k * T + t) * ld_part + F + c];
      }
      out_s[(size_t)t * ldb + c] = g / (1.f + expf(-g)) * u;
    }
  }
}

}  // namespace dfl

// ===========================================================================
// host
// ===========================================================================
namespace dflh {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

struct MapKey {
  uintptr_t ptr;
  uint64_t rows, cols;
  uint32_t box_rows;
  int dev;
  bool operator==(const MapKey &o) const {
    return ptr == o.ptr && rows == o.rows && cols == o.cols && box_rows == o.box_rows &&
           dev == o.dev;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey &k) const {
    size_t h = (size_t)k.ptr * 0x9E3779B97F4A7C15ull;
    h ^= (k.rows * 1315423911ull) ^ (k.cols << 20) ^ ((size_t)k.box_rows << 40) ^ (size_t)k.dev;
    return h;
  }
};

// Tensor map of a row-major bf16 matrix [rows, cols]; box = 64 columns x box_rows rows.
bool bf16_map(CUtensorMap *out, const void *ptr, uint64_t rows, uint64_t cols,
              uint32_t box_rows, int dev) {
  static std::mutex mu;
  static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
  MapKey key{(uintptr_t)ptr, rows, cols, box_rows, dev};
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return true;
    }
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> g(mu);
  if (cache.size() > 8192) cache.clear();
  cache[key] = *out;
  return true;
}


static int token_tile(int T) { return T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : T <= 128 ? 128 : 256; }

// One k-block of one CTA (microseconds): the slowest of the weight tile from
// HBM (~46 GB/s per CTA, measured with per-CTA timestamps; a weight tile shared
// by several token tiles is streamed by the CTAs of those tiles together, mostly
// from L2), both tiles through TMA (~110 GB/s per CTA, the activation tile mostly
// from L2) and the MMA issuer: ~0.25 us of barrier wait, fence and commit per
// pipeline stage, shared by the stage's k-blocks, plus the tensor pipe's time
// (~11 TFLOP/s per CTA).
static double stage_us(int bn, bool shared_w) {
  const double a = 128.0 * 64 * 2, b = (double)bn * 64 * 2;
  const int kps = bn <= 128 ? 2 : 1;  // k-blocks a stage (GemmShape::KPS)
  const double issue = 0.25 / kps + 2.0 * 128 * bn * 64 / 11e6;
  return std::max(std::max(shared_w ? 0.0 : a / 46e3, (a + b) / 110e3), issue);
}

// Epilogue of one tile (microseconds): per 16-column chunk a tensor-memory
// load and the stores, plus the exchange of the SwiGLU / head-norm modes.
static double epilogue_us(int bn, int T, int mode) {
  const int chunks = (std::min(bn, T) + 15) / 16;
  const int per_group = (chunks + dfl::kEpiGroups - 1) / dfl::kEpiGroups;
  return per_group * (mode == GEMM_REDUCE ? 0.6 : 1.8);
}
// Tail of a split tile: the slice stores, the ticket, then the last CTA reads
// the S slices (per epilogue group four 16-column chunks of all slices per
// round trip) and runs the epilogue.  Fitted to per-CTA timestamps on GB300.
static double reduce_tail_us(int bn, int T, int S, int mode) {
  const int rounds = (std::min(bn, T) + 127) / 128;  // 4 chunks per group per round
  return 1.5 + 0.5 * S + rounds * (1.0 + 0.15 * S) + epilogue_us(bn, T, mode);
}

// Cost model (microseconds) of one launch with token tile bn split S ways,
// fitted to sweeps and per-CTA timestamps on GB300: stage_us per k-block, the
// GPU about 6.5 TB/s from HBM.  Each wave
// of units costs the slower of one unit's own time and the wave's share of HBM
// bandwidth (weights are read from HBM once per token tile when they do not
// fit in L2); split slices add their write + read traffic, and in the reduce
// modes the last CTA of a tile reads the S slices of its 128 x bn block.
static double gemm_cost(int N_out, int T, int K_in, int S, int bn, int mode, int num_sms) {
  const int kb = K_in / dfl::BK;
  const int t_tiles = (T + bn - 1) / bn;
  const int m_tiles = (N_out + dfl::BM - 1) / dfl::BM;
  const double kbps = kb / S;
  const double uA = 128.0 * 64 * 2 * kbps;
  const double t_unit = kbps * stage_us(bn, t_tiles > 1) + 0.15;
  const long U = (long)m_tiles * t_tiles * S;
  const double wbytes = 2.0 * N_out * K_in;
  const double hbm_share = wbytes > 48e6 ? 1.0 : 1.0 / t_tiles;  // re-read per token tile?
  double tot = 0.0;
  for (long w = 0; w * num_sms < U; ++w) {
    const long n = std::min<long>(num_sms, U - w * num_sms);
    tot += std::max(t_unit, n * uA * hbm_share / 6.5e6);
  }
  if (S > 1) {
    tot += (double)S * T * N_out * 8.0 / 8e6;
    if (mode != GEMM_PARTIAL) tot += reduce_tail_us(bn, T, S, mode);
  } else if (mode != GEMM_PARTIAL) {
    tot += epilogue_us(bn, T, mode);  // the last tile's epilogue is not overlapped
  }
  return tot;
}

int gemm_balanced_slots(int K_in, int chunk) {
  const int kb = K_in / dfl::BK;
  return chunk > 0 ? (kb + chunk - 1) / chunk + 1 : 1;
}

// Balanced schedule: every CTA streams `chunk` k-blocks (the iterations of all
// tiles cut evenly over the SMs), so no wave is partly empty; tiles cut across
// CTAs are reduced by their last CTA as in the split schedule.
static double gemm_cost_balanced(int N_out, int T, int K_in, int bn, int mode, int num_sms,
                                 int *chunk_out) {
  const int kb = K_in / dfl::BK;
  const int t_tiles = (T + bn - 1) / bn;
  const int m_tiles = (N_out + dfl::BM - 1) / dfl::BM;
  const long total = (long)m_tiles * t_tiles * kb;
  const long chunk = (total + num_sms - 1) / num_sms;
  *chunk_out = (int)chunk;
  if (chunk < 2 || total > (1L << 30)) return 1e300;
  const int segs = (int)((chunk + kb - 1) / kb) + 1;
  const double t_cta = chunk * stage_us(bn, t_tiles > 1) + 0.15 * segs;
  const double wbytes = 2.0 * N_out * K_in;
  const double hbm = wbytes * (wbytes > 48e6 ? t_tiles : 1) / 6.5e6;
  double tot = std::max(t_cta, hbm);
  if (chunk < kb || total % chunk) {  // cut tiles: slices written, then read by the last CTA
    // a cut tile's contributors finish at different points of their chunks: the
    // last one's reduction starts late and overlaps nothing; with the SwiGLU and
    // head-norm epilogues over several column chunks this measured about twice
    // the reduction itself
    const int slots = gemm_balanced_slots(K_in, (int)chunk);
    const bool heavy = mode != GEMM_REDUCE && std::min(bn, T) > 16;  // several epilogue chunks
    tot += (heavy ? 2.0 : 1.0) * reduce_tail_us(bn, T, slots, mode);
    tot += 2.0 * std::min<long>(num_sms, (long)m_tiles * t_tiles * slots) * 128 * std::min(bn, T) *
           4 / 8e6;
  } else {
    tot += epilogue_us(bn, T, mode);
  }
  return tot;
}

static GemmPlan plan_for(int N_out, int T, int K_in, int mode, int num_sms, int max_S,
                         bool choose_bn) {
  const int kb = K_in / dfl::BK;
  GemmPlan best{token_tile(T), 1};
  double best_cost = 1e300;
  const int bns[5] = {16, 32, 64, 128, 256};
  for (int bi = 0; bi < 5; ++bi) {
    const int bn = bns[bi];
    if (!choose_bn && bn != token_tile(T)) continue;
    if (bn > token_tile(T)) break;
    for (int S = 1; S <= kb && S <= max_S; ++S) {
      if (kb % S) continue;
      if (S > 1 && kb / S < 2) break;
      if (S > 1 && (size_t)S * T * N_out > kMaxPartialFloats) break;
      const double c = gemm_cost(N_out, T, K_in, S, bn, mode, num_sms);
      if (c < best_cost * 0.985) best_cost = c, best = GemmPlan{bn, S};
    }
    if (mode != GEMM_PARTIAL) {
      int chunk = 0;
      const double c = gemm_cost_balanced(N_out, T, K_in, bn, mode, num_sms, &chunk);
      const size_t fl = gemm_scratch_floats(mode == GEMM_SWIGLU ? N_out / 2 : N_out, T, 1, mode,
                                            bn, chunk, K_in);
      if (c < best_cost * 0.985 && fl <= kMaxPartialFloats) {
        best_cost = c;
        best = GemmPlan{bn, 1, chunk};
      }
    }
  }
  return best;
}

int gemm_splits(int N_out, int T, int K_in, int num_sms, int max_S) {
  return plan_for(N_out, T, K_in, GEMM_PARTIAL, num_sms, max_S, false).S;
}

GemmPlan gemm_plan(int N_out, int T, int K_in, int mode, int num_sms, int max_S) {
  const int rows = mode == GEMM_SWIGLU ? 2 * N_out : N_out;
  const int mt = mode == GEMM_SWIGLU ? N_out / 64 : (N_out + dfl::BM - 1) / dfl::BM;
  // many tokens: two-SM tiles (a call whose weight groups do not pair up falls
  // back to one-SM 256-token tiles with the same single slice)
  if (mode != GEMM_PARTIAL && T >= kPairMinTokens && mt % 2 == 0) return GemmPlan{256, 1, 0, 1};
  return plan_for(rows, T, K_in, mode, num_sms, max_S, true);
}

size_t gemm_tiles(int N_out, int T, int mode, int bn) {
  if (bn <= 0) bn = token_tile(T);
  const int rows = mode == GEMM_SWIGLU ? 64 : dfl::BM;
  return (size_t)((N_out + rows - 1) / rows) * ((T + bn - 1) / bn);
}

size_t gemm_scratch_floats(int N_out, int T, int S, int mode, int bn, int chunk, int K_in) {
  if (mode == GEMM_PARTIAL) return (size_t)S * T * N_out;
  if (bn <= 0) bn = token_tile(T);
  const size_t slots = chunk > 0 ? (size_t)gemm_balanced_slots(K_in, chunk) : (size_t)S;
  if (slots <= 1) return 0;
  return slots * gemm_tiles(N_out, T, mode, bn) * dfl::BM * bn;
}

// Activation bytes above which tiles are walked weight tile fastest.
constexpr double kMFastestActBytes = 64e6;

// Kernel parameters and grid of one launch with token tile BN.
static int make_params(const GemmCall &g, int BN, int num_sms, dfl::GemmParams &p) {
  const bool swiglu = g.mode == GEMM_SWIGLU;
  p.out = g.out;
  p.ld = g.ld;
  p.N_out = g.N_out;
  p.T = g.T;
  p.S = g.S;
  p.kb_per_split = g.K_in / dfl::BK / g.S;
  p.mtg = swiglu ? g.N_out / 64 : (g.N_out + dfl::BM - 1) / dfl::BM;
  p.m_tiles = p.mtg * g.groups;
  p.ostride = g.ostride;
  p.t_tiles = (g.T + BN - 1) / BN;
  p.tb = p.t_tiles;
  p.mq = 0;
  if (g.mode == GEMM_QKV && g.T0 > 0 && g.T0 < g.T && !g.pair) {
    // token tiles of injected context rows alone need only the k and v weight tiles
    p.tb = (g.T0 + BN - 1) / BN;
    p.mq = g.Hq * g.dh / dfl::BM;
  }
  const int tiles = p.m_tiles * p.tb + (p.m_tiles - p.mq) * (p.t_tiles - p.tb);
  p.num_units = tiles * g.S;
  p.mode = g.mode;
  p.out_f32 = g.out_f32;
  p.out_bf16 = (dfl::bf16 *)g.out_bf16;
  p.ldb = g.ldb;
  p.F = swiglu ? g.N_out : 0;
  p.counters = g.counters;
  p.err = g.err;
  p.stats = g.stats;
  p.q_norm = (const dfl::bf16 *)g.q_norm;
  p.k_norm = (const dfl::bf16 *)g.k_norm;
  p.rope_cs = g.rope_cs;
  p.Hq = g.Hq;
  p.Hkv = g.Hkv;
  p.dh = g.dh;
  p.eps = g.eps;
  p.T0 = g.T0 > 0 ? g.T0 : g.T;
  p.ctx_slot = g.ctx_slot;
  p.P = g.page_size;
  p.kc = g.kc ? (dfl::bf16 *)g.kc + (size_t)g.layer * g.layer_elems : nullptr;
  p.vc = g.vc ? (dfl::bf16 *)g.vc + (size_t)g.layer * g.layer_elems : nullptr;
  p.chunk = 0;
  p.kb_total = g.K_in / dfl::BK;
  p.total = 0;
  p.nmax = g.S;
  p.m_fastest = (double)g.T * g.K_in * 2 > kMFastestActBytes ? 1 : 0;
  p.wait_ns = g.wait_ns > 0 ? g.wait_ns : dfl::kWaitLimitNs;
  p.stall = g.stall;
  p.pair = 0;
  p.qdata = nullptr;
  int grid = p.num_units < num_sms ? p.num_units : num_sms;
  if (g.chunk > 0) {
    const long total = (long)tiles * p.kb_total;
    if (total >= (1L << 30)) return -1;
    p.chunk = g.chunk;
    p.total = (int)total;
    p.nmax = gemm_balanced_slots(g.K_in, g.chunk);
    p.S = 1;
    p.kb_per_split = p.kb_total;
    p.num_units = tiles;
    grid = (int)((total + g.chunk - 1) / g.chunk);
  }
  return grid;
}

template <int BN>
static int launch_tc(const GemmCall &g, cudaStream_t st, const Dev *d) {
  using SH = dfl::GemmShape<BN>;
  static int attr_set_dev[64] = {0};
  if (d->id < 64 && !attr_set_dev[d->id]) {
    if (cudaFuncSetAttribute(dfl::k_gemm_tc<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SH::SMEM_BYTES) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    attr_set_dev[d->id] = 1;
  }
  const bool swiglu = g.mode == GEMM_SWIGLU;
  const int w_rows = swiglu ? 2 * g.N_out : g.N_out;
  dfl::WMaps mw;
  CUtensorMap mx;
  memset(&mw, 0, sizeof(mw));
  for (int gi = 0; gi < g.groups; ++gi)
    if (!bf16_map(&mw.m[gi], gi == 0 ? g.W : g.Wg[gi], (uint64_t)w_rows, (uint64_t)g.K_in,
                  swiglu ? 64 : dfl::BM, d->id))
      return DFLASH_ERR_CUDA;
  if (!bf16_map(&mx, g.X, (uint64_t)g.T, (uint64_t)g.K_in, BN, d->id)) return DFLASH_ERR_CUDA;
  dfl::GemmParams p;
  const int grid = make_params(g, BN, d->num_sms, p);
  if (grid < 0) return DFLASH_ERR_DIMS;
  DFL_CHECK_LAUNCH(launch(dfl::k_gemm_tc<BN>, dim3(grid), dim3(dfl::kGemmThreads),
                          (size_t)SH::SMEM_BYTES, st, mw, mx, p));
  return DFLASH_OK;
}

template <int BN>
static int launch_q4(const GemmCall &g, cudaStream_t st, const Dev *d) {
  using QS = dfl::QShape<BN>;
  static int attr_set_dev[64] = {0};
  if (d->id < 64 && !attr_set_dev[d->id]) {
    if (cudaFuncSetAttribute(dfl::k_gemm_q4<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             QS::SMEM_BYTES) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    attr_set_dev[d->id] = 1;
  }
  CUtensorMap mx;
  if (!bf16_map(&mx, g.X, (uint64_t)g.T, (uint64_t)g.K_in, BN, d->id)) return DFLASH_ERR_CUDA;
  dfl::GemmParams p;
  const int grid = make_params(g, BN, d->num_sms, p);
  if (grid < 0) return DFLASH_ERR_DIMS;
  p.qdata = (const uint8_t *)g.Wq;
  DFL_CHECK_LAUNCH(launch(dfl::k_gemm_q4<BN>, dim3(grid), dim3(dfl::kQ4Threads),
                          (size_t)QS::SMEM_BYTES, st, mx, p));
  return DFLASH_OK;
}

// Two-SM tiles: a uniform schedule over pairs of weight tiles, 256-token tiles,
// launched as clusters of two CTAs.
static int launch_tc2(const GemmCall &g, cudaStream_t st, const Dev *d) {
  using SH = dfl::PairShape;
  static int attr_set_dev[64] = {0};
  if (d->id < 64 && !attr_set_dev[d->id]) {
    if (cudaFuncSetAttribute(dfl::k_gemm_tc2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SH::SMEM_BYTES) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    attr_set_dev[d->id] = 1;
  }
  const bool swiglu = g.mode == GEMM_SWIGLU;
  const int w_rows = swiglu ? 2 * g.N_out : g.N_out;
  dfl::WMaps mw;
  CUtensorMap mx;
  memset(&mw, 0, sizeof(mw));
  for (int gi = 0; gi < g.groups; ++gi)
    if (!bf16_map(&mw.m[gi], gi == 0 ? g.W : g.Wg[gi], (uint64_t)w_rows, (uint64_t)g.K_in,
                  swiglu ? 64 : dfl::BM, d->id))
      return DFLASH_ERR_CUDA;
  if (!bf16_map(&mx, g.X, (uint64_t)g.T, (uint64_t)g.K_in, dfl::kPairBN / 2, d->id))
    return DFLASH_ERR_CUDA;
  dfl::GemmParams p;
  if (make_params(g, dfl::kPairBN, d->num_sms, p) < 0) return DFLASH_ERR_DIMS;
  p.pair = 1;
  p.num_units = ((p.m_tiles + 1) / 2) * p.t_tiles * p.S;
  const int clusters = std::min(p.num_units, d->num_sms / 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(dfl::kGemmThreads);
  cfg.dynamicSmemBytes = SH::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  count_launch();
  DFL_CHECK_LAUNCH(cudaLaunchKernelEx(&cfg, dfl::k_gemm_tc2, mw, mx, p));
  return DFLASH_OK;
}

// Whether a call can run on two-SM tiles: bf16, uniform schedule, and weight
// tiles that pair up inside every weight group (an odd count only with one
// group in reduce mode: the last pair's second tile is a phantom).
static bool pair_ok(const GemmCall &g) {
  if (g.dtype != DFLASH_BF16 || g.chunk != 0 || g.stall) return false;
  const int mtg = g.mode == GEMM_SWIGLU ? g.N_out / 64 : (g.N_out + dfl::BM - 1) / dfl::BM;
  return mtg % 2 == 0 || (g.groups == 1 && g.mode == GEMM_REDUCE);
}

int gemm_run(const GemmCall &g, cudaStream_t st) {
  if (g.T <= 0 || g.N_out <= 0) return DFLASH_OK;
  const Dev *d = device();
  if (!d) return DFLASH_ERR_DEVICE;
  if (g.K_in % 64 || g.S < 1 || (g.K_in / 64) % g.S) return DFLASH_ERR_DIMS;
  if (g.chunk < 0 || (g.chunk > 0 && g.mode == GEMM_PARTIAL)) return DFLASH_ERR_DIMS;
  if (g.stats && (g.mode != GEMM_REDUCE || g.dtype != DFLASH_BF16)) return DFLASH_ERR_DIMS;
  if (g.groups < 1 || g.groups > dfl::kMaxGroups) return DFLASH_ERR_DIMS;
  if (g.groups > 1) {
    if (g.mode != GEMM_REDUCE || g.dtype != DFLASH_BF16 || g.N_out % dfl::BM || g.out_bf16 ||
        g.stats || !g.out_f32)
      return DFLASH_ERR_DIMS;
    for (int gi = 1; gi < g.groups; ++gi)
      if (!g.Wg[gi] || (uintptr_t)g.Wg[gi] % 16) return DFLASH_ERR_ALIGN;
  }
  if (g.chunk > 0 && (!g.counters || !g.out)) return DFLASH_ERR_NULL;
  if (g.mode == GEMM_SWIGLU && g.N_out % 64) return DFLASH_ERR_DIMS;
  if (g.mode == GEMM_QKV &&
      (g.dtype != DFLASH_BF16 || (g.dh != 64 && g.dh != 128) ||
       g.N_out != (g.Hq + 2 * g.Hkv) * g.dh || !g.q_norm || !g.k_norm || !g.rope_cs ||
       !g.out_bf16))
    return DFLASH_ERR_DIMS;
  if (g.T0 < 0 || g.T0 > g.T) return DFLASH_ERR_DIMS;
  if (g.T0 > 0 && g.T0 < g.T &&
      (g.mode != GEMM_QKV || !g.ctx_slot || !g.kc || !g.vc || g.page_size < 1 || g.layer < 0))
    return DFLASH_ERR_DIMS;
  if (g.mode != GEMM_PARTIAL && g.S > 1 && (!g.counters || !g.out)) return DFLASH_ERR_NULL;
  if (g.dtype == DFLASH_F32) {
    // CUDA-core path: slices to scratch (or the output itself), then the epilogue
    const int n_rows = g.mode == GEMM_SWIGLU ? 2 * g.N_out : g.N_out;
    float *part = g.out;
    const int ldp = g.mode == GEMM_PARTIAL ? g.ld : n_rows;
    dim3 grid((n_rows + 63) / 64, (g.T + 31) / 32, g.S);
    DFL_CHECK_LAUNCH(launch(dfl::k_gemm_f32, grid, dim3(256), 0, st, (const float *)g.W,
                            (const float *)g.X, part, ldp, n_rows, g.T, g.K_in, g.K_in / g.S));
    if (g.mode != GEMM_PARTIAL) {
      const size_t n = (size_t)g.T * g.N_out;
      const int blocks = (int)std::min<size_t>((n + 255) / 256, (size_t)d->num_sms * 8);
      DFL_CHECK_LAUNCH(launch(dfl::k_gemm_f32_finish, dim3(blocks), dim3(256), 0, st,
                              (const float *)part, g.S, g.T, g.N_out, ldp, g.mode, g.N_out,
                              g.out_f32, g.ld, (float *)g.out_bf16, g.ldb));
    }
    return DFLASH_OK;
  }
  if (g.Wq) {
    // 4-bit weights: one weight group, one-SM tiles
    if (g.dtype != DFLASH_BF16 || g.groups != 1 || g.stall) return DFLASH_ERR_DIMS;
    if (g.mode == GEMM_SWIGLU && g.N_out % 64) return DFLASH_ERR_DIMS;
    if ((uintptr_t)g.Wq % 16 || (uintptr_t)g.X % 16) return DFLASH_ERR_ALIGN;
    int qbn = g.bn > 0 && !g.pair ? g.bn : g.pair ? 256 : token_tile(g.T);
    if (qbn > 128) qbn = 128;  // the A buffers share tensor memory with the accumulators
    GemmCall gq = g;
    gq.pair = 0;
    switch (qbn) {
      case 16: return launch_q4<16>(gq, st, d);
      case 32: return launch_q4<32>(gq, st, d);
      case 64: return launch_q4<64>(gq, st, d);
      case 128: return launch_q4<128>(gq, st, d);
      default: return DFLASH_ERR_DIMS;
    }
  }
  if ((uintptr_t)g.W % 16 || (uintptr_t)g.X % 16) return DFLASH_ERR_ALIGN;
  if (g.pair && pair_ok(g)) return launch_tc2(g, st, d);
  const int bn = g.pair ? 256 : g.bn > 0 ? g.bn : token_tile(g.T);
  if (bn != 16 && bn != 32 && bn != 64 && bn != 128 && bn != 256) return DFLASH_ERR_DIMS;
  switch (bn) {
    case 16: return launch_tc<16>(g, st, d);
    case 32: return launch_tc<32>(g, st, d);
    case 64: return launch_tc<64>(g, st, d);
    case 128: return launch_tc<128>(g, st, d);
    default: return launch_tc<256>(g, st, d);
  }
}

int gemm_xwT(int dtype, const void *W, int N_out, int K_in, const void *X, int T, float *out,
             int ld, int S, int *err, cudaStream_t st) {
  GemmCall g;
  g.dtype = dtype;
  g.W = W;
  g.N_out = N_out;
  g.K_in = K_in;
  g.X = X;
  g.T = T;
  g.S = S;
  g.mode = GEMM_PARTIAL;
  g.out = out;
  g.ld = ld;
  g.err = err;
  return gemm_run(g, st);
}

}  // namespace dflh
