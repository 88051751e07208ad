// Projection GEMMs of the drafter: Y = X W^T with W [N_out, K_in] row-major
// (nn.Linear) and X [T, K_in] row-major, split over K into S slices whose
// fp32 partial sums are written to out[(s*T + t)*ld + n].  Consumers add the
// S slices in order, so results are deterministic.
#pragma once
#include "common.cuh"

namespace dflh {

constexpr size_t kMaxPartialFloats = size_t(48) << 20;  // cap of one partial buffer

// Number of K slices for a GEMM of this shape on `num_sms` SMs (at most max_S),
// for the default token tile.
int gemm_splits(int N_out, int T, int K_in, int num_sms, int max_S = 1 << 20);

// Token tile and K split of one GEMM: picked by a cost model of the waves of
// work units, the memory traffic, and (reduce modes) the last CTA's reduction.
struct GemmPlan {
  int bn;         // token tile: 16, 32, 64, 128 or 256
  int S;          // K slices (uniform schedule)
  int chunk = 0;  // > 0: balanced schedule, k-block iterations per CTA (reduce modes)
  int pair = 0;   // two-SM 256 x 256 tiles (k_gemm_tc2), one K slice
};
// Token count from which the reduce modes run on two-SM tiles (bulk injection):
// there a one-SM CTA is bound by its operand bytes per flop, while at draft
// batch sizes the pair tiles gain nothing.
constexpr int kPairMinTokens = 2048;
GemmPlan gemm_plan(int N_out, int T, int K_in, int mode, int num_sms, int max_S);

enum GemmMode {
  GEMM_PARTIAL = 0,  // slice s -> out[(s*T + t)*ld + n]; the caller sums the slices
  GEMM_REDUCE = 1,   // final Y -> out_f32[t*ld + n] and/or out_bf16[t*ldb + n]
  GEMM_SWIGLU = 2,   // rows [Wg; Wu] of a 2F-row weight: out_bf16[t*ldb + f] = SiLU(g_f) u_f
  GEMM_QKV = 3,      // QKV projection -> bf16 q, k (head RMSNorm + RoPE) and v, out_bf16
};

struct GemmCall {
  int dtype = DFLASH_BF16;
  const void *W = nullptr;
  int N_out = 0;       // output features (F for GEMM_SWIGLU)
  int K_in = 0;
  const void *X = nullptr;
  int T = 0;
  int S = 1;
  int chunk = 0;       // > 0: balanced schedule (reduce modes; S is then ignored)
  int bn = 0;          // token tile; 0 = the smallest tile that holds T (at most 256)
  int mode = GEMM_PARTIAL;
  float *out = nullptr;       // GEMM_PARTIAL output, or the slice scratch of the other modes
  int ld = 0;
  float *out_f32 = nullptr;   // GEMM_REDUCE
  void *out_bf16 = nullptr;   // GEMM_REDUCE / GEMM_SWIGLU (storage dtype)
  int ldb = 0;
  int *counters = nullptr;    // tile tickets, zero on entry and on exit (S > 1)
  int *err = nullptr;
  // GEMM_REDUCE (bf16) with groups > 1: one launch over `groups` weight matrices of
  // N_out rows each (N_out a multiple of 128, W = group 0, Wg[g] the others, all with
  // the same X); group g writes out_f32 + g * ostride
  int groups = 1;
  const void *Wg[8] = {};
  size_t ostride = 0;
  // GEMM_REDUCE (bf16): per token t and 128-row weight tile i, (max, sum e^(y - max))
  // of the tile's outputs -> stats[t * ceil(N_out/128) + i]
  float2 *stats = nullptr;
  // GEMM_QKV: head norm gains (bf16 [dh]), per-token RoPE (cos, sin) [T][dh/2]
  const void *q_norm = nullptr, *k_norm = nullptr;
  const float2 *rope_cs = nullptr;
  int Hq = 0, Hkv = 0, dh = 0;
  float eps = 0.f;
  // GEMM_QKV with injected context rows: tokens t >= T0 (0: none) are context
  // rows whose k and v heads go to layer `layer` of the paged caches [L][page]
  // [Hkv][page_size][dh] (layer_elems elements a layer) at element offset
  // ctx_slot[t - T0] + head * page_size * dh + feature (rows with a negative
  // slot are skipped); their q heads are dropped.
  int T0 = 0;
  const long long *ctx_slot = nullptr;
  size_t layer_elems = 0;
  int page_size = 0, layer = 0;
  void *kc = nullptr, *vc = nullptr;
  // limit of the kernel's bounded waits (0: the default, kWaitLimitNs); stall
  // (failure-path test only, bf16): the MMA issuer first waits on a barrier
  // that nothing arrives on, so that the wait gives up
  uint64_t wait_ns = 0;
  int stall = 0;
  // two-SM tiles (bf16, uniform schedule, an even number of weight tiles per
  // group): clusters of two CTAs compute 256-row x 256-token tiles
  int pair = 0;
  // 4-bit weights (W unused): Wq = the 2304-byte records of this matrix, its
  // row block 0 first (dflash_q4); one group, no two-SM tiles
  const void *Wq = nullptr;
};

// Floats of slice scratch a reduce-mode GEMM needs (0 when S == 1 and chunk == 0).
size_t gemm_scratch_floats(int N_out, int T, int S, int mode, int bn = 0, int chunk = 0,
                           int K_in = 0);
// Slice slots per tile of the balanced schedule.
int gemm_balanced_slots(int K_in, int chunk);
// Tile tickets a reduce-mode GEMM needs.
size_t gemm_tiles(int N_out, int T, int mode, int bn = 0);

// Launch one GEMM.  DFLASH_BF16 operands run on tcgen05 tensor cores fed by
// TMA; DFLASH_F32 on fp32 CUDA cores.  W and X 16-byte aligned, K_in a
// multiple of 64, S dividing K_in/64.  Returns DFLASH_OK or an error.
int gemm_run(const GemmCall &g, cudaStream_t stream);

// Tensor map (cached) of a row-major bf16 matrix [rows, cols] (cols * 2 a multiple of
// 16 bytes): boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool bf16_map(CUtensorMap *out, const void *ptr, uint64_t rows, uint64_t cols,
              uint32_t box_rows, int dev);

// GEMM_PARTIAL convenience form
int gemm_xwT(int dtype, const void *W, int N_out, int K_in, const void *X, int T, float *out,
             int ld, int S, int *err, cudaStream_t stream);

}  // namespace dflh
