// C ABI of the DFlash 2 draft cycle: argument checks, workspace layout and the
// kernel sequence of each call.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "attention.cuh"
#include "gemm.cuh"
#include "head.cuh"
#include "pointwise.cuh"

namespace dflh {

// ---------------------------------------------------------------------------
// device, launch counter, PDL switch
// ---------------------------------------------------------------------------
static thread_local int64_t g_launches = 0;
void count_launch() { ++g_launches; }

bool pdl_enabled() {
  static int v = -1;
  if (v < 0) {
    const char *e = getenv("DFLASH_PDL");
    v = (e && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}

const Dev *device() {
  static Dev devs[64];
  static std::mutex mu;
  int id = -1;
  if (cudaGetDevice(&id) != cudaSuccess || id < 0 || id >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> g(mu);
  Dev &d = devs[id];
  if (d.id < 0) {
    cudaDeviceProp p;
    if (cudaGetDeviceProperties(&p, id) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    d.num_sms = p.multiProcessorCount;
    d.max_smem_optin = (int)p.sharedMemPerBlockOptin;
    d.cc_major = p.major;
    d.cc_minor = p.minor;
    d.id = id;
  }
  if (d.cc_major != 10 || d.cc_minor != 3) return nullptr;  // built for sm_103a only
  return &d;
}

static int sm_count_or_default() {
  int id = -1, n = 0;
  if (cudaGetDevice(&id) == cudaSuccess &&
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, id) == cudaSuccess && n > 0)
    return n;
  cudaGetLastError();
  return 152;
}

// ---------------------------------------------------------------------------
// argument checks
// ---------------------------------------------------------------------------
static int check_cfg(const dflash_config *c) {
  if (!c) return DFLASH_ERR_NULL;
  if (c->dtype != DFLASH_F32 && c->dtype != DFLASH_BF16) return DFLASH_ERR_DTYPE;
  const bool ok =
      c->d_model > 0 && c->d_model % 64 == 0 && c->n_layers >= 1 &&
      c->n_layers <= DFLASH_MAX_LAYERS && c->n_kv_heads >= 1 && c->n_q_heads >= c->n_kv_heads &&
      c->n_q_heads % c->n_kv_heads == 0 && (c->head_dim == 64 || c->head_dim == 128) &&
      (c->n_q_heads * c->head_dim) % 64 == 0 && c->d_ff > 0 && c->d_ff % 64 == 0 &&
      c->vocab >= 2 && c->n_taps >= 1 && c->d_target >= 1 &&
      ((long)c->n_taps * c->d_target) % 64 == 0 && c->window >= 1 && c->page_size >= 1 &&
      c->top_k >= 1 && c->top_k <= DFLASH_MAX_TOPK && c->top_k <= c->vocab &&
      topk_tiles(c->vocab) <= kTopkMaxTiles &&
      c->sel_rank >= 16 && c->sel_rank % 16 == 0 && c->sel_rank <= 1024 &&
      c->top_k * c->sel_rank <= 16384 && c->conv_group >= 1 && c->d_model % c->conv_group == 0 &&
      c->mask_token_id >= 0 && c->mask_token_id < c->vocab && c->rms_eps >= 0.f &&
      c->rope_theta >= 0.f;
  if (!ok) return DFLASH_ERR_DIMS;
  if (c->weight_bits != 0 && c->weight_bits != 4) return DFLASH_ERR_DTYPE;
  if (c->weight_bits == 4 && c->dtype != DFLASH_BF16) return DFLASH_ERR_DTYPE;
  return DFLASH_OK;
}

static bool a16(const void *p) { return ((uintptr_t)p & 15) == 0; }

// A projection: its storage-dtype matrix, or with 4-bit weights its codes and
// (scale, bias) words.
static int check_proj(const dflash_config *c, const void *w, const dflash_q4 &q) {
  if (c->weight_bits == 4) {
    if (!q.data) return DFLASH_ERR_NULL;
    return a16(q.data) ? DFLASH_OK : DFLASH_ERR_ALIGN;
  }
  if (!w) return DFLASH_ERR_NULL;
  return a16(w) ? DFLASH_OK : DFLASH_ERR_ALIGN;
}

static int check_weights(const dflash_config *c, const dflash_weights *w, bool draft) {
  if (!w) return DFLASH_ERR_NULL;
  if (!w->fc_norm) return DFLASH_ERR_NULL;
  int rc;
  if ((rc = check_proj(c, w->fc, w->fc_q4)) != DFLASH_OK) return rc;
  for (int l = 0; l < c->n_layers; ++l) {
    const dflash_layer_weights &L = w->layer[l];
    if (!L.k_norm) return DFLASH_ERR_NULL;
    if ((rc = check_proj(c, L.wqkv, L.wqkv_q4)) != DFLASH_OK) return rc;
    if (!draft) continue;
    if (!L.attn_norm || !L.mlp_norm || !L.q_norm) return DFLASH_ERR_NULL;
    if ((rc = check_proj(c, L.wo, L.wo_q4)) != DFLASH_OK ||
        (rc = check_proj(c, L.w_gate_up, L.w_gate_up_q4)) != DFLASH_OK ||
        (rc = check_proj(c, L.w_down, L.w_down_q4)) != DFLASH_OK)
      return rc;
    for (int i = 0; i < 4; ++i) {
      if (!L.conv_w[i] || !L.conv_base[i]) return DFLASH_ERR_NULL;
      if (!a16(L.conv_w[i]) || !a16(L.conv_base[i])) return DFLASH_ERR_ALIGN;
    }
    if (!a16(L.mlp_norm)) return DFLASH_ERR_ALIGN;
  }
  if (draft) {
    if (!w->embed || !w->final_norm) return DFLASH_ERR_NULL;
    if ((rc = check_proj(c, w->lm_head, w->lm_head_q4)) != DFLASH_OK) return rc;
    if (!a16(w->embed) || !a16(w->final_norm)) return DFLASH_ERR_ALIGN;
    for (int l = 0; l < c->n_layers; ++l)
      if (!a16(w->layer[l].attn_norm)) return DFLASH_ERR_ALIGN;
  }
  return DFLASH_OK;
}

static int check_kv(const dflash_config *c, const dflash_kv *kv) {
  (void)c;
  if (!kv || !kv->k || !kv->v || !kv->page_table) return DFLASH_ERR_NULL;
  if (kv->num_pages < 1 || kv->max_pages_per_req < 1 || kv->num_rows < 1) return DFLASH_ERR_DIMS;
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
constexpr int kMaxReduceSplits = 16;      // slices a reduce-mode GEMM may use
constexpr size_t kTicketInts = 1 << 14;   // tile tickets of one reduce-mode GEMM
constexpr size_t kTopkTicketInts = 1 << 14;  // selector tickets, one per request (B at most)
constexpr int kKvGroup = 8;  // layers per grouped K/V projection launch of injection
// Fixed header of every workspace: status word, GEMM tile tickets, top-k row
// tickets.  They must stay zero between calls; every other region is scratch
// that a call fully writes before reading (acceptance's partials start here).
constexpr size_t kHeaderBytes = 256 + kTicketInts * 4 + kTopkTicketInts * 4;

struct Layout {
  size_t status, tickets, scratch;
  size_t x, un, ub, rf, rb, gates, qkv, qb, kb, vb, ob, hb, zf, logits, attn, topk, topk_tickets;
  size_t selrows, U, Vp, pairs, argmax, gn, cb, kvf, rope, rope_inj, selgate, slots, ssq;
  size_t total, sc_floats;
  GemmPlan P_gate, P_qkv, P_o, P_gu, P_down, P_sel, P_sel2, P_hgate;
  AttnPlan ap;
};

// Token tile and K slices of a reduce-mode GEMM: the cost model's choice,
// capped so the slice scratch and the tile tickets stay bounded; float32
// storage runs on CUDA cores with one slice.
static GemmPlan reduce_plan(const dflash_config *c, int N_out, int T, int K_in, int mode,
                            int sms) {
  if (c->dtype == DFLASH_F32) return GemmPlan{0, 1};
  GemmPlan p = gemm_plan(N_out, T, K_in, mode, sms, kMaxReduceSplits);
  if (c->weight_bits == 4 && (p.bn > 128 || p.pair)) {
    // 4-bit tiles are at most 128 tokens wide
    p.bn = 128;
    p.pair = 0;
  }
  if (gemm_tiles(N_out, T, mode, p.bn) > kTicketInts) p.S = 1, p.chunk = 0;
  return p;
}
static size_t reduce_scratch(const dflash_config *c, int N_out, int T, int K_in, GemmPlan p,
                             int mode) {
  if (c->dtype == DFLASH_F32)
    return (size_t)p.S * T * (mode == GEMM_SWIGLU ? 2 * N_out : N_out);
  return gemm_scratch_floats(N_out, T, p.S, mode, p.bn, p.chunk, K_in);
}

// The QKV projection over T block rows and n injected rows: the token tiles of
// the injected rows alone skip the q weight tiles, so the plan for T + n tokens
// is kept only when its token tile is no larger than the block's own plan's
// (larger tiles give fewer, longer work units); else the block's plan.
static GemmPlan fused_qkv_plan(const dflash_config *c, int QKVW, int T, int n, int D, int sms) {
  const GemmPlan pt = reduce_plan(c, QKVW, T, D, GEMM_QKV, sms);
  const GemmPlan pn = reduce_plan(c, QKVW, T + n, D, GEMM_QKV, sms);
  return pn.bn <= pt.bn || pn.pair ? pn : pt;
}

static bool make_layout(const dflash_config *c, int B, int K, int Nmax, Layout *L) {
  const int sms = sm_count_or_default();
  const size_t es = c->dtype == DFLASH_BF16 ? 2 : 4;
  const int D = c->d_model, F = c->d_ff, V = c->vocab, dh = c->head_dim;
  const int Hq = c->n_q_heads, Hkv = c->n_kv_heads, k = c->top_k, r = c->sel_rank;
  const int GW = 2 * D / c->conv_group;
  const int QKVW = (Hq + 2 * Hkv) * dh;
  const int TIN = c->n_taps * c->d_target;
  const int T = B * K, TL = B * (K - 1), R = 1 + (K - 1) * k, TR = B * R;
  const int N = Nmax > 0 ? Nmax : 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 255) & ~(size_t)255;
    return o;
  };
  // the conv gate linears (row path): bf16 writes K slices that the conv sums
  // itself, so the GEMM has no reduction tail; float32 one slice
  L->P_gate = c->dtype == DFLASH_BF16 ? gemm_plan(GW, T, D, GEMM_PARTIAL, sms, kMaxReduceSplits)
                                     : reduce_plan(c, GW, T, D, GEMM_REDUCE, sms);
  L->P_qkv = reduce_plan(c, QKVW, T, D, c->dtype == DFLASH_BF16 ? GEMM_QKV : GEMM_REDUCE, sms);
  L->P_o = reduce_plan(c, D, T, Hq * dh, GEMM_REDUCE, sms);
  L->P_gu = reduce_plan(c, F, T, D, GEMM_SWIGLU, sms);
  L->P_down = reduce_plan(c, D, T, F, GEMM_REDUCE, sms);
  L->P_sel = reduce_plan(c, r, TR, D, GEMM_REDUCE, sms);
  L->P_sel2 = reduce_plan(c, 2 * r, TR, D, GEMM_REDUCE, sms);
  L->P_hgate = reduce_plan(c, r, TL, D, GEMM_REDUCE, sms);
  L->ap = attn_plan(B, K, Hq, Hkv, dh, c->window, sms);
  // slice scratch shared by every reduce-mode GEMM (they run one after another)
  size_t sc = 0;
  sc = std::max(sc, reduce_scratch(c, QKVW, T, D, L->P_qkv,
                                    c->dtype == DFLASH_BF16 ? GEMM_QKV : GEMM_REDUCE));
  sc = std::max(sc, reduce_scratch(c, D, T, Hq * dh, L->P_o, GEMM_REDUCE));
  sc = std::max(sc, reduce_scratch(c, F, T, D, L->P_gu, GEMM_SWIGLU));
  sc = std::max(sc, reduce_scratch(c, D, T, F, L->P_down, GEMM_REDUCE));
  sc = std::max(sc, reduce_scratch(c, r, TR, D, L->P_sel, GEMM_REDUCE));
  sc = std::max(sc, reduce_scratch(c, 2 * r, TR, D, L->P_sel2, GEMM_REDUCE));
  sc = std::max(sc, reduce_scratch(c, r, TL, D, L->P_hgate, GEMM_REDUCE));
  sc = std::max(sc, reduce_scratch(c, V, TL, D, GemmPlan{0, 1}, GEMM_REDUCE));
  // injection GEMMs: the split depends on the token count; take the largest
  auto inj = [&](int n_out, int k_in) {
    size_t best = 0;
    auto eval = [&](int n) {
      if (n < 1 || n > N) return;
      const GemmPlan p = reduce_plan(c, n_out, n, k_in, GEMM_REDUCE, sms);
      best = std::max(best, reduce_scratch(c, n_out, n, k_in, p, GEMM_REDUCE));
    };
    for (int n = 1; n <= 16; ++n) eval(n);
    for (int n = 32; n <= 256; n *= 2) eval(n);
    for (int n = 512; n <= N; n += 256) eval(n);
    eval(N);
    return best;
  };
  sc = std::max(sc, inj(D, TIN));
  sc = std::max(sc, inj(2 * Hkv * dh, D));
  sc = std::max(sc, inj(std::min(c->n_layers, kKvGroup) * 2 * Hkv * dh, D));
  if (Nmax > 0 && c->dtype == DFLASH_BF16) {
    // the pass with injected rows: each layer's QKV GEMM over the block rows and
    // up to Nmax context rows
    auto eval = [&](int n) {
      if (n < 1 || n > Nmax) return;
      const GemmPlan p = fused_qkv_plan(c, QKVW, T, n, D, sms);
      sc = std::max(sc, reduce_scratch(c, QKVW, T + n, D, p, GEMM_QKV));
    };
    for (int n = 1; n <= 16; ++n) eval(n);
    for (int n = 32; n <= 256; n *= 2) eval(n);
    for (int n = 512; n <= Nmax; n += 256) eval(n);
    eval(Nmax);
  }
  L->sc_floats = sc;
  // buffers whose place does not depend on the injection capacity first (a
  // draft pass and dflash_draft_hidden agree on them whatever Nmax was)
  L->status = take(256);
  L->tickets = take(kTicketInts * sizeof(int));
  L->topk_tickets = take(kTopkTicketInts * sizeof(int));
  L->x = take((size_t)T * D * 4);
  L->un = take((size_t)T * D * es);
  L->rf = take((size_t)T * D * 4);
  L->rb = take((size_t)T * D * es);
  L->gates = take((size_t)L->P_gate.S * T * GW * 4);
  L->qkv = take((size_t)T * QKVW * 4);
  L->qb = take((size_t)T * Hq * dh * es);
  L->kb = take((size_t)T * Hkv * dh * es);
  L->vb = take((size_t)T * Hkv * dh * es);
  L->ob = take((size_t)T * Hq * dh * es);
  L->hb = take((size_t)T * F * es);
  L->zf = take((size_t)TL * D * es);
  L->logits = take((size_t)TL * V * 4);
  L->attn = take(L->ap.part_floats * 4);
  L->topk = take((size_t)TL * topk_tiles(V) * sizeof(float2));
  L->selrows = take((size_t)TR * D * es);
  L->U = take((size_t)TR * r * 4 * 2);  // U then Vp, back to back
  L->Vp = L->U + (size_t)TR * r * 4;
  L->pairs = take((size_t)B * (K - 1) * k * k * 4);
  L->argmax = take((size_t)T * argmax_chunks(V) * 2 * 4);
  L->selgate = take((size_t)TL * r * 4);
  // the fused convs' row sums of squares, [slots][16]
  L->ssq = take((size_t)std::max(1, gconv_ssq_slots(T, D, c->conv_group, c->dtype)) * 16 * 4);
  // then the ones sized by it: the QKV operand and the RoPE table hold the block
  // rows followed by up to N injected rows
  L->rope = take((size_t)(T + N) * (dh / 2) * 8);
  L->ub = take((size_t)(T + N) * D * es);
  L->rope_inj = take((size_t)N * (dh / 2) * 8);
  L->slots = take((size_t)N * 8);
  L->gn = take((size_t)N * TIN * es);
  L->cb = take((size_t)N * D * es);
  L->kvf = take((size_t)N * 2 * Hkv * dh * c->n_layers * 4);
  L->scratch = take(sc * 4);
  L->total = off;
  // acceptance keeps its scratch right after the fixed header
  L->total = std::max(L->total, kHeaderBytes + accept_sample_floats(B, K, V) * 4);
  return true;
}

// The call reads rows row0.. (a multiple of 64) of a 4-bit matrix with K_in
// input features: its records from row block row0 / 64 on.
static GemmCall with_q4(GemmCall g, const dflash_q4 &q, int K_in, int row0 = 0) {
  g.Wq = (const uint8_t *)q.data + (size_t)(row0 / 64) * (K_in / 64) * 2304;
  return g;
}

// A plan chosen at call time for a token count the layout sampled around: one
// K slice when its slice scratch would not fit the workspace's.
static GemmPlan fit_plan(const dflash_config &c, const Layout &L, int N_out, int T, int K_in,
                         int mode, GemmPlan p) {
  if (c.dtype == DFLASH_BF16 && reduce_scratch(&c, N_out, T, K_in, p, mode) > L.sc_floats)
    p.S = 1, p.chunk = 0;
  return p;
}

// ---------------------------------------------------------------------------
// the calls
// ---------------------------------------------------------------------------
#define TRY(e)                           \
  do {                                   \
    int rc_ = (e);                       \
    if (rc_ != DFLASH_OK) return rc_;    \
  } while (0)

// One reduce-mode GEMM on the shared scratch and tickets of the workspace.
static GemmCall reduce_call(const dflash_config &c, uint8_t *ws, const Layout &L, const void *W,
                            int N_out, int K_in, const void *X, int T, GemmPlan plan, int mode,
                            float *out_f32, int ld, void *out_s, int ldb) {
  GemmCall g;
  g.bn = plan.bn;
  const int S = plan.S;
  g.dtype = c.dtype;
  g.W = W;
  g.N_out = N_out;
  g.K_in = K_in;
  g.X = X;
  g.T = T;
  g.S = S;
  g.chunk = plan.chunk;
  g.pair = plan.pair;
  g.mode = mode;
  g.out = (float *)(ws + L.scratch);
  g.out_f32 = out_f32;
  g.ld = ld;
  g.out_bf16 = out_s;
  g.ldb = ldb;
  g.counters = (int *)(ws + L.tickets);
  g.err = (int *)(ws + L.status);
  return g;
}

template <typename S>
static int run_inject(const dflash_config &c, const dflash_weights &w, const dflash_kv &kv,
                      const void *hidden, const int32_t *req, const int32_t *pos, int N,
                      uint8_t *ws, const Layout &L, cudaStream_t st) {
  const int sms = device()->num_sms;
  const int D = c.d_model, Hq = c.n_q_heads, Hkv = c.n_kv_heads, dh = c.head_dim;
  const int TIN = c.n_taps * c.d_target, W2 = 2 * Hkv * dh;
  int *err = (int *)(ws + L.status);
  S *gn = (S *)(ws + L.gn);
  S *cb = (S *)(ws + L.cb);
  float *kvf = (float *)(ws + L.kvf);
  const RopeTable rope = rope_table(c.rope_theta, dh);
  float2 *rope_cs = (float2 *)(ws + L.rope_inj);
  TRY(launch_rows_norm<S>((const S *)hidden, N, TIN, (const S *)w.fc_norm, c.rms_eps, gn, pos,
                          rope, dh / 2, rope_cs, st));
  const GemmPlan S_fc =
      fit_plan(c, L, D, N, TIN, GEMM_REDUCE, reduce_plan(&c, D, N, TIN, GEMM_REDUCE, sms));
  const bool q4 = c.weight_bits == 4;
  GemmCall gf = reduce_call(c, ws, L, w.fc, D, TIN, gn, N, S_fc, GEMM_REDUCE, nullptr, D, cb, D);
  if (q4) gf = with_q4(gf, w.fc_q4, TIN);
  TRY(gemm_run(gf, st));
  // the [Wk; Wv] rows of every layer: one grouped launch per kKvGroup layers
  // (layer l's projection -> kvf [l][N][W2])
  LayerPtrs kn;
  memset(&kn, 0, sizeof(kn));
  const bool grouped = c.dtype == DFLASH_BF16 && W2 % 128 == 0 && !q4;
  const int per = grouped ? kKvGroup : 1;
  for (int l0 = 0; l0 < c.n_layers; l0 += per) {
    const int ng = std::min(per, c.n_layers - l0);
    const GemmPlan S_kv = fit_plan(c, L, ng * W2, N, D, GEMM_REDUCE,
                                   reduce_plan(&c, ng * W2, N, D, GEMM_REDUCE, sms));
    GemmCall g = reduce_call(c, ws, L, (const S *)w.layer[l0].wqkv + (size_t)Hq * dh * D, W2, D,
                             cb, N, S_kv, GEMM_REDUCE, kvf + (size_t)l0 * N * W2, W2, nullptr, 0);
    g.groups = ng;
    g.ostride = (size_t)N * W2;
    for (int j = 1; j < ng; ++j) g.Wg[j] = (const S *)w.layer[l0 + j].wqkv + (size_t)Hq * dh * D;
    if (q4) g = with_q4(g, w.layer[l0].wqkv_q4, D, Hq * dh);
    TRY(gemm_run(g, st));
  }
  for (int l = 0; l < c.n_layers; ++l) kn.p[l] = w.layer[l].k_norm;
  TRY(launch_inject_store<S>(kvf, N, c.n_layers, Hkv, dh, kn, req, pos, kv.page_table,
                             kv.num_rows, kv.max_pages_per_req, kv.num_pages, c.page_size, rope_cs,
                             c.rms_eps, (S *)kv.k, (S *)kv.v, err, st));
  return DFLASH_OK;
}

// Injected context rows carried by one draft pass (N = 0: none).
struct InjectRows {
  const void *hidden = nullptr;
  const int32_t *req = nullptr, *pos = nullptr;
  int N = 0;
};

template <typename S>
static int run_draft(const dflash_config &c, const dflash_weights &w, const dflash_kv &kv,
                     const int32_t *anchor, const int32_t *ctx_len, int B, int K, int32_t *ids,
                     float *logp, float *logits_opt, uint8_t *ws, const Layout &L,
                     cudaStream_t st, const InjectRows &inj = InjectRows()) {
  const int D = c.d_model, F = c.d_ff, V = c.vocab, dh = c.head_dim;
  const int Hq = c.n_q_heads, Hkv = c.n_kv_heads, g = c.conv_group;
  const int GW = 2 * D / g, QKVW = (Hq + 2 * Hkv) * dh;
  const int T = B * K;
  const float eps = c.rms_eps;
  int *err = (int *)(ws + L.status);
  float *x = (float *)(ws + L.x), *rf = (float *)(ws + L.rf);
  float *gates = (float *)(ws + L.gates), *qkv = (float *)(ws + L.qkv);
  S *un = (S *)(ws + L.un), *ub = (S *)(ws + L.ub), *rb = (S *)(ws + L.rb);
  S *qb = (S *)(ws + L.qb), *kb = (S *)(ws + L.kb), *vb = (S *)(ws + L.vb);
  S *ob = (S *)(ws + L.ob), *hb = (S *)(ws + L.hb), *zf = (S *)(ws + L.zf);
  float *logits = logits_opt ? logits_opt : (float *)(ws + L.logits);
  float *attnp = (float *)(ws + L.attn), *topkp = (float *)(ws + L.topk);
  const RopeTable rope = rope_table(c.rope_theta, dh);
  // the conv gate linear of the row path -> gates: nsl_gate K slices (bf16) or
  // the reduced rows (float32)
  const int nsl_gate = c.dtype == DFLASH_BF16 ? L.P_gate.S : 1;
  auto gate_gemm = [&](const void *Wg, const S *X) {
    if (c.dtype == DFLASH_BF16) {
      GemmCall gc = reduce_call(c, ws, L, Wg, GW, D, X, T, L.P_gate, GEMM_PARTIAL, nullptr, GW,
                                nullptr, 0);
      gc.out = gates;
      return gemm_run(gc, st);
    }
    return gemm_run(
        reduce_call(c, ws, L, Wg, GW, D, X, T, L.P_gate, GEMM_REDUCE, gates, GW, nullptr, 0), st);
  };

  // the projection GEMMs of the pass
  const int TL = B * (K - 1);
  // the lm_head's epilogue also writes each 128-entry vocab tile's (max, sum e^(z - max))
  float2 *tstats = c.dtype == DFLASH_BF16 ? (float2 *)topkp : nullptr;
  float2 *rope_cs = (float2 *)(ws + L.rope);
  // injected context rows (bf16): their fc outputs follow the block rows in the
  // QKV operand, so each layer's QKV GEMM also forms their K/V and stores them
  const int N = c.dtype == DFLASH_BF16 ? inj.N : 0;
  const int Tq = T + N;
  const bool q4 = c.weight_bits == 4;
  // each injected row's place in a layer's cache, found (and checked) once
  CacheSlots slots;
  if (N > 0) {
    slots.req = inj.req;
    slots.table = kv.page_table;
    slots.max_pages = kv.max_pages_per_req;
    slots.num_rows = kv.num_rows;
    slots.num_pages = kv.num_pages;
    slots.P = c.page_size;
    slots.Hkv = Hkv;
    slots.dh = dh;
    slots.slot = (long long *)(ws + L.slots);
    slots.err = err;
  }
  const GemmPlan P_qkv =
      N > 0 ? fit_plan(c, L, QKVW, Tq, D, GEMM_QKV,
                       fused_qkv_plan(&c, QKVW, T, N, D, device()->num_sms))
            : L.P_qkv;
  auto qkv_call = [&](int l) {
    const dflash_layer_weights &lw = w.layer[l];
    if (c.dtype != DFLASH_BF16)
      return reduce_call(c, ws, L, lw.wqkv, QKVW, D, ub, T, L.P_qkv, GEMM_REDUCE, qkv, QKVW,
                         nullptr, 0);
    // the projection's epilogue applies the q/k head norms and RoPE: bf16 q, k, v rows
    GemmCall gq = reduce_call(c, ws, L, lw.wqkv, QKVW, D, ub, Tq, P_qkv, GEMM_QKV, nullptr, 0,
                              ws + L.qkv, QKVW);
    gq.q_norm = lw.q_norm;
    gq.k_norm = lw.k_norm;
    gq.rope_cs = rope_cs;
    gq.Hq = Hq;
    gq.Hkv = Hkv;
    gq.dh = dh;
    gq.eps = eps;
    if (q4) gq = with_q4(gq, lw.wqkv_q4, D);
    if (N > 0) {
      gq.T0 = T;
      gq.ctx_slot = slots.slot;
      gq.layer_elems = (size_t)kv.num_pages * Hkv * c.page_size * dh;
      gq.page_size = c.page_size;
      gq.layer = l;
      gq.kc = kv.k;
      gq.vc = kv.v;
    }
    return gq;
  };
  auto o_call = [&](int l) {
    GemmCall g = reduce_call(c, ws, L, w.layer[l].wo, D, Hq * dh, ob, T, L.P_o, GEMM_REDUCE, rf,
                             D, rb, D);
    return q4 ? with_q4(g, w.layer[l].wo_q4, Hq * dh) : g;
  };
  auto gu_call = [&](int l) {
    GemmCall g = reduce_call(c, ws, L, w.layer[l].w_gate_up, F, D, ub, T, L.P_gu, GEMM_SWIGLU,
                             nullptr, 0, hb, F);
    return q4 ? with_q4(g, w.layer[l].w_gate_up_q4, D) : g;
  };
  auto down_call = [&](int l) {
    GemmCall g = reduce_call(c, ws, L, w.layer[l].w_down, D, F, hb, T, L.P_down, GEMM_REDUCE, rf,
                             D, rb, D);
    return q4 ? with_q4(g, w.layer[l].w_down_q4, F) : g;
  };
  auto lm_call = [&]() {
    // more than 128 draft rows: two-SM tiles, each SM taking in half of the
    // 256-token tile per k-block (one-SM tiles are bound by those bytes)
    const GemmPlan pl =
        c.dtype == DFLASH_BF16 && !q4 && TL > 128 ? GemmPlan{256, 1, 0, 1} : GemmPlan{0, 1};
    GemmCall gl = reduce_call(c, ws, L, w.lm_head, V, D, zf, TL, pl, GEMM_REDUCE, logits, V,
                              nullptr, 0);
    gl.stats = tstats;
    return q4 ? with_q4(gl, w.lm_head_q4, D) : gl;
  };
  // A few block rows: each conv is one launch with its gate linear fused (the
  // pre-norm formed inside).  More rows: the gate linear is a tensor-core GEMM
  // and the conv a row kernel.
  const bool fused = gconv_fits(T, D, g, c.dtype);
  // The fused path hands each row's sum of squares from the kernel that
  // updates the residual stream (the embedding kernel, the post-sublayer conv)
  // to the next pre-sublayer conv: ssq_n partials a row wait in ssq (0: none,
  // the conv forms them itself).
  const int ssq_slots = fused ? gconv_ssq_slots(T, D, g, c.dtype) : 0;
  float *ssq = ssq_slots > 0 ? (float *)(ws + L.ssq) : nullptr;
  int ssq_n = 0;
  auto conv_pre = [&](int l, int i, const void *gain) -> int {
    const dflash_layer_weights &lw = w.layer[l];
    if (fused) {
      const int n = ssq_n;
      ssq_n = 0;
      return launch_gconv_pre<S>(x, T, K, D, g, (const S *)lw.conv_w[i],
                                 (const S *)lw.conv_base[i], (const S *)gain, eps, ub, st,
                                 n > 0 ? ssq : nullptr, n);
    }
    int rc = gate_gemm(lw.conv_w[i], un);
    if (rc != DFLASH_OK) return rc;
    return launch_conv_pre<S>(un, gates, nsl_gate, T, K, D, g, (const S *)lw.conv_base[i], ub,
                              st);
  };
  // conv after a sublayer + residual; then the next pre-norm (row path) or,
  // after the last layer, the final norm into zf
  auto conv_post = [&](int l, int i, const void *next_gain, bool last) -> int {
    const dflash_layer_weights &lw = w.layer[l];
    int rc;
    if (fused) {
      rc = launch_gconv_post<S>(rf, rb, T, K, D, g, (const S *)lw.conv_w[i],
                                (const S *)lw.conv_base[i], x, st, ssq);
      ssq_n = ssq ? ssq_slots : 0;
      if (rc != DFLASH_OK || !last) return rc;
      return launch_final_norm<S>(x, B, K, D, (const S *)next_gain, eps, zf, st);
    }
    rc = gate_gemm(lw.conv_w[i], rb);
    if (rc != DFLASH_OK) return rc;
    return launch_conv_post_norm<S>(rf, gates, nsl_gate, T, K, D, g, (const S *)lw.conv_base[i],
                                    x, (const S *)next_gain, eps, un, last ? zf : (S *)nullptr,
                                    st);
  };

  if (N > 0) {
    // the injection's RMSNorm over the taps and fc to width D, into rows T.. of
    // the QKV operand (their RoPE rows after the block's)
    const int TIN = c.n_taps * c.d_target;
    S *gn = (S *)(ws + L.gn);
    TRY(launch_rows_norm<S>((const S *)inj.hidden, N, TIN, (const S *)w.fc_norm, eps, gn, inj.pos,
                            rope, dh / 2, rope_cs + (size_t)T * (dh / 2), st, slots));
    const GemmPlan pf = fit_plan(c, L, D, N, TIN, GEMM_REDUCE,
                                 reduce_plan(&c, D, N, TIN, GEMM_REDUCE, device()->num_sms));
    GemmCall gf =
        reduce_call(c, ws, L, w.fc, D, TIN, gn, N, pf, GEMM_REDUCE, nullptr, D, ub + (size_t)T * D, D);
    if (q4) gf = with_q4(gf, w.fc_q4, TIN);
    TRY(gemm_run(gf, st));
  }
  TRY(launch_embed_norm<S>((const S *)w.embed, anchor, c.mask_token_id, V, B, K, D,
                           (const S *)w.layer[0].attn_norm, eps, x, fused ? (S *)nullptr : un, err,
                           ctx_len, rope, dh / 2, rope_cs, st, ssq));
  ssq_n = ssq ? 1 : 0;
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights &lw = w.layer[l];
    const bool last = l + 1 == c.n_layers;
    // attention sublayer: conv -> QKV -> norm/RoPE -> block attention -> O -> conv, residual
    TRY(conv_pre(l, 0, lw.attn_norm));
    TRY(gemm_run(qkv_call(l), st));
    if constexpr (sizeof(S) == 2) {
      TRY(launch_attention_fused(L.ap, (const dfl::bf16 *)(ws + L.qkv), (const dfl::bf16 *)kv.k,
                                 (const dfl::bf16 *)kv.v, l, c.n_layers, kv.page_table,
                                 kv.max_pages_per_req, kv.num_pages, c.page_size, ctx_len, B, K,
                                 Hq, Hkv, dh, c.window, (dfl::bf16 *)ob, err, st, inj.req,
                                 inj.pos, N));
    } else {
      TRY(launch_qkv_post<S>(qkv, T, K, Hq, Hkv, dh, (const S *)lw.q_norm, (const S *)lw.k_norm,
                             rope_cs, eps, qb, kb, vb, st));
      TRY(launch_block_attention<S>(L.ap, qb, kb, vb, (const S *)kv.k, (const S *)kv.v, l,
                                    kv.page_table, kv.max_pages_per_req, kv.num_pages,
                                    c.page_size, ctx_len, B, K, Hq, Hkv, dh, c.window, attnp, ob,
                                    err, st));
    }
    TRY(gemm_run(o_call(l), st));
    TRY(conv_post(l, 1, lw.mlp_norm, false));
    // MLP sublayer: conv -> gate/up + SwiGLU -> down -> conv, residual
    TRY(conv_pre(l, 2, lw.mlp_norm));
    TRY(gemm_run(gu_call(l), st));
    TRY(gemm_run(down_call(l), st));
    TRY(conv_post(l, 3, last ? w.final_norm : w.layer[l + 1].attn_norm, last));
  }
  TRY(gemm_run(lm_call(), st));
  TRY(launch_topk(logits, tstats, TL, V, c.top_k, ids, logp, st));
  return DFLASH_OK;
}

// Both low-rank projections of the anchor and candidate rows (U then Vp in the
// workspace) when the weights carry no prepared selector table.
template <typename S>
static int sel_project(const dflash_config &c, const dflash_weights &w, const int32_t *anchor,
                       const int32_t *ids, int B, int K, uint8_t *ws, const Layout &L,
                       cudaStream_t st) {
  const int D = c.d_model, k = c.top_k, r = c.sel_rank;
  const int TR = B * (1 + (K - 1) * k);
  int *err = (int *)(ws + L.status);
  S *rows = (S *)(ws + L.selrows);
  float *U = (float *)(ws + L.U), *Vp = (float *)(ws + L.Vp);
  TRY(launch_sel_gather<S>((const S *)w.embed, anchor, ids, B, K, k, c.vocab, D, rows, err, st));
  if (c.dtype == DFLASH_BF16 && r % 128 == 0) {
    // both projections in one grouped launch (Vp follows U in the workspace)
    GemmCall g = reduce_call(c, ws, L, w.sel_pu, r, D, rows, TR, L.P_sel2, GEMM_REDUCE, U, r,
                             nullptr, 0);
    g.groups = 2;
    g.Wg[1] = w.sel_pv;
    g.ostride = (size_t)TR * r;
    TRY(gemm_run(g, st));
  } else {
    TRY(gemm_run(reduce_call(c, ws, L, w.sel_pu, r, D, rows, TR, L.P_sel, GEMM_REDUCE, U, r,
                             nullptr, 0),
                 st));
    TRY(gemm_run(reduce_call(c, ws, L, w.sel_pv, r, D, rows, TR, L.P_sel, GEMM_REDUCE, Vp, r,
                             nullptr, 0),
                 st));
  }
  return DFLASH_OK;
}

template <typename S>
static int run_select(const dflash_config &c, const dflash_weights &w, const int32_t *anchor,
                      const int32_t *ids, const float *logp, int B, int K, int32_t *path,
                      float *score, uint8_t *ws, const Layout &L, cudaStream_t st) {
  const int k = c.top_k, r = c.sel_rank;
  int *err = (int *)(ws + L.status);
  float *U = (float *)(ws + L.U), *Vp = (float *)(ws + L.Vp);
  // with a table the projections of every vocabulary row are read by token
  if (!w.sel_table) TRY(sel_project<S>(c, w, anchor, ids, B, K, ws, L, st));
  TRY(launch_viterbi(U, Vp, ids, logp, B, K, k, r, (float *)(ws + L.pairs),
                     (int *)(ws + L.topk_tickets), path, score, w.sel_table, c.vocab, anchor, err,
                     st));
  return DFLASH_OK;
}

template <typename S>
static int run_sample(const dflash_config &c, const dflash_weights &w, const int32_t *anchor,
                      const int32_t *ids, const float *logp, int B, int K, const float *uniforms,
                      int32_t *path, float *path_q, uint8_t *ws, const Layout &L,
                      cudaStream_t st) {
  int *err = (int *)(ws + L.status);
  if (!w.sel_table) TRY(sel_project<S>(c, w, anchor, ids, B, K, ws, L, st));
  TRY(launch_sample_walk((float *)(ws + L.U), (float *)(ws + L.Vp), ids, logp, B, K, c.top_k,
                         c.sel_rank, w.sel_table, c.vocab, anchor, uniforms, path, path_q, err,
                         st));
  return DFLASH_OK;
}

template <typename S>
static int run_greedy(const dflash_config &c, const dflash_weights &w, const int32_t *anchor,
                      const int32_t *ids, const float *logp, const void *hidden, int B, int K,
                      int32_t *path, float *score, uint8_t *ws, const Layout &L,
                      cudaStream_t st) {
  const int D = c.d_model, r = c.sel_rank, TL = B * (K - 1);
  int *err = (int *)(ws + L.status);
  float *gate = (float *)(ws + L.selgate);
  if (!w.sel_table) TRY(sel_project<S>(c, w, anchor, ids, B, K, ws, L, st));
  // the context gate's pre-activations W_H h_t of every draft position
  TRY(gemm_run(reduce_call(c, ws, L, w.sel_gate, r, D, hidden, TL, L.P_hgate, GEMM_REDUCE, gate,
                           r, nullptr, 0),
               st));
  TRY(launch_greedy_walk((float *)(ws + L.U), (float *)(ws + L.Vp), ids, logp, B, K, c.top_k, r,
                         w.sel_table, c.vocab, anchor, gate, path, score, err, st));
  return DFLASH_OK;
}

}  // namespace dflh

using namespace dflh;

extern "C" {

size_t dflash_workspace_bytes(const dflash_config *cfg, int32_t B, int32_t K,
                              int32_t max_inject_tokens) {
  if (check_cfg(cfg) != DFLASH_OK) return 0;
  if (B < 1 || K < 2 || K > DFLASH_MAX_BLOCK || max_inject_tokens < 0) return 0;
  Layout L;
  if (!make_layout(cfg, B, K, max_inject_tokens, &L)) return 0;
  return L.total;
}

int dflash_inject_context(const dflash_config *cfg, const dflash_weights *w, const dflash_kv *kv,
                          const void *target_hidden, const int32_t *req, const int32_t *pos,
                          int32_t N, void *ws, size_t ws_bytes, void *stream) {
  int rc = check_cfg(cfg);
  if (rc != DFLASH_OK) return rc;
  if (N < 0) return DFLASH_ERR_DIMS;
  if (N == 0) return DFLASH_OK;
  if (!target_hidden || !req || !pos || !ws) return DFLASH_ERR_NULL;
  if (!a16(target_hidden) || !a16(w->fc_norm)) return DFLASH_ERR_ALIGN;
  if ((rc = check_weights(cfg, w, false)) != DFLASH_OK) return rc;
  if ((rc = check_kv(cfg, kv)) != DFLASH_OK) return rc;
  if (!a16(ws)) return DFLASH_ERR_ALIGN;
  Layout L;
  make_layout(cfg, 1, 2, N, &L);
  if (ws_bytes < L.total) return DFLASH_ERR_WORKSPACE;
  if (!device()) return DFLASH_ERR_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cfg->dtype == DFLASH_BF16)
    return run_inject<dfl::bf16>(*cfg, *w, *kv, target_hidden, req, pos, N, (uint8_t *)ws, L, st);
  return run_inject<float>(*cfg, *w, *kv, target_hidden, req, pos, N, (uint8_t *)ws, L, st);
}

int dflash_draft_block(const dflash_config *cfg, const dflash_weights *w, const dflash_kv *kv,
                       const int32_t *anchor, const int32_t *ctx_len, int32_t B, int32_t K,
                       int32_t *topk_ids, float *topk_logp, float *logits_opt, void *ws,
                       size_t ws_bytes, void *stream) {
  int rc = check_cfg(cfg);
  if (rc != DFLASH_OK) return rc;
  if (B < 0 || K < 2 || K > DFLASH_MAX_BLOCK) return DFLASH_ERR_BLOCK;
  if (B == 0) return DFLASH_OK;
  if ((size_t)B * (K - 1) > kTopkTicketInts) return DFLASH_ERR_DIMS;
  if (!anchor || !ctx_len || !topk_ids || !topk_logp || !ws) return DFLASH_ERR_NULL;
  if ((rc = check_weights(cfg, w, true)) != DFLASH_OK) return rc;
  if ((rc = check_kv(cfg, kv)) != DFLASH_OK) return rc;
  if (!a16(ws)) return DFLASH_ERR_ALIGN;
  Layout L;
  make_layout(cfg, B, K, 0, &L);
  if (ws_bytes < L.total) return DFLASH_ERR_WORKSPACE;
  if (!device()) return DFLASH_ERR_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cfg->dtype == DFLASH_BF16)
    return run_draft<dfl::bf16>(*cfg, *w, *kv, anchor, ctx_len, B, K, topk_ids, topk_logp,
                                logits_opt, (uint8_t *)ws, L, st);
  return run_draft<float>(*cfg, *w, *kv, anchor, ctx_len, B, K, topk_ids, topk_logp, logits_opt,
                          (uint8_t *)ws, L, st);
}

int dflash_draft_block_inject(const dflash_config *cfg, const dflash_weights *w,
                              const dflash_kv *kv, const void *target_hidden, const int32_t *req,
                              const int32_t *pos, int32_t N, const int32_t *anchor,
                              const int32_t *ctx_len, int32_t B, int32_t K, int32_t *topk_ids,
                              float *topk_logp, float *logits_opt, void *ws, size_t ws_bytes,
                              void *stream) {
  int rc = check_cfg(cfg);
  if (rc != DFLASH_OK) return rc;
  if (N < 0) return DFLASH_ERR_DIMS;
  if (B < 0 || K < 2 || K > DFLASH_MAX_BLOCK) return DFLASH_ERR_BLOCK;
  if (N > 0 && B == 0)
    return dflash_inject_context(cfg, w, kv, target_hidden, req, pos, N, ws, ws_bytes, stream);
  if (B == 0) return DFLASH_OK;
  if ((size_t)B * (K - 1) > kTopkTicketInts) return DFLASH_ERR_DIMS;
  if (!anchor || !ctx_len || !topk_ids || !topk_logp || !ws) return DFLASH_ERR_NULL;
  if (N > 0 && (!target_hidden || !req || !pos)) return DFLASH_ERR_NULL;
  if (N > 0 && (!a16(target_hidden) || !a16(w->fc_norm))) return DFLASH_ERR_ALIGN;
  if (N > 0 && (rc = check_weights(cfg, w, false)) != DFLASH_OK) return rc;
  if ((rc = check_weights(cfg, w, true)) != DFLASH_OK) return rc;
  if ((rc = check_kv(cfg, kv)) != DFLASH_OK) return rc;
  if (!a16(ws)) return DFLASH_ERR_ALIGN;
  Layout L;
  make_layout(cfg, B, K, N, &L);
  if (ws_bytes < L.total) return DFLASH_ERR_WORKSPACE;
  if (!device()) return DFLASH_ERR_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cfg->dtype == DFLASH_BF16) {
    InjectRows inj;
    inj.hidden = target_hidden;
    inj.req = req;
    inj.pos = pos;
    inj.N = N;
    return run_draft<dfl::bf16>(*cfg, *w, *kv, anchor, ctx_len, B, K, topk_ids, topk_logp,
                                logits_opt, (uint8_t *)ws, L, st, inj);
  }
  // float32 storage: the injection, then the pass
  if (N > 0) {
    Layout Li;
    make_layout(cfg, 1, 2, N, &Li);
    TRY(run_inject<float>(*cfg, *w, *kv, target_hidden, req, pos, N, (uint8_t *)ws, Li, st));
  }
  Layout Ld;
  make_layout(cfg, B, K, 0, &Ld);
  return run_draft<float>(*cfg, *w, *kv, anchor, ctx_len, B, K, topk_ids, topk_logp, logits_opt,
                          (uint8_t *)ws, Ld, st);
}

int dflash_select_path(const dflash_config *cfg, const dflash_weights *w, const int32_t *anchor,
                       const int32_t *topk_ids, const float *topk_logp, int32_t B, int32_t K,
                       int32_t *path, float *path_score, void *ws, size_t ws_bytes,
                       void *stream) {
  int rc = check_cfg(cfg);
  if (rc != DFLASH_OK) return rc;
  if (B < 0 || K < 2 || K > DFLASH_MAX_BLOCK) return DFLASH_ERR_BLOCK;
  if (B == 0) return DFLASH_OK;
  if ((size_t)B > kTopkTicketInts) return DFLASH_ERR_DIMS;
  if (!w || !anchor || !topk_ids || !topk_logp || !path || !path_score || !ws)
    return DFLASH_ERR_NULL;
  if (!w->sel_table && (!w->embed || !w->sel_pu || !w->sel_pv)) return DFLASH_ERR_NULL;
  if (w->sel_table ? !a16(w->sel_table)
                   : (!a16(w->sel_pu) || !a16(w->sel_pv) || !a16(w->embed)))
    return DFLASH_ERR_ALIGN;
  if (!a16(ws)) return DFLASH_ERR_ALIGN;
  Layout L;
  make_layout(cfg, B, K, 0, &L);
  if (ws_bytes < L.total) return DFLASH_ERR_WORKSPACE;
  if (!device()) return DFLASH_ERR_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cfg->dtype == DFLASH_BF16)
    return run_select<dfl::bf16>(*cfg, *w, anchor, topk_ids, topk_logp, B, K, path, path_score,
                                 (uint8_t *)ws, L, st);
  return run_select<float>(*cfg, *w, anchor, topk_ids, topk_logp, B, K, path, path_score,
                           (uint8_t *)ws, L, st);
}

int dflash_sample_path(const dflash_config *cfg, const dflash_weights *w, const int32_t *anchor,
                       const int32_t *topk_ids, const float *topk_logp, int32_t B, int32_t K,
                       const float *uniforms, int32_t *path, float *path_q, void *ws,
                       size_t ws_bytes, void *stream) {
  int rc = check_cfg(cfg);
  if (rc != DFLASH_OK) return rc;
  if (B < 0 || K < 2 || K > DFLASH_MAX_BLOCK) return DFLASH_ERR_BLOCK;
  if (B == 0) return DFLASH_OK;
  if ((size_t)B > kTopkTicketInts) return DFLASH_ERR_DIMS;
  if (!w || !anchor || !topk_ids || !topk_logp || !uniforms || !path || !path_q || !ws)
    return DFLASH_ERR_NULL;
  if (!w->sel_table && (!w->embed || !w->sel_pu || !w->sel_pv)) return DFLASH_ERR_NULL;
  if (w->sel_table ? !a16(w->sel_table)
                   : (!a16(w->sel_pu) || !a16(w->sel_pv) || !a16(w->embed)))
    return DFLASH_ERR_ALIGN;
  if (!a16(ws)) return DFLASH_ERR_ALIGN;
  Layout L;
  make_layout(cfg, B, K, 0, &L);
  if (ws_bytes < L.total) return DFLASH_ERR_WORKSPACE;
  if (!device()) return DFLASH_ERR_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cfg->dtype == DFLASH_BF16)
    return run_sample<dfl::bf16>(*cfg, *w, anchor, topk_ids, topk_logp, B, K, uniforms, path,
                                 path_q, (uint8_t *)ws, L, st);
  return run_sample<float>(*cfg, *w, anchor, topk_ids, topk_logp, B, K, uniforms, path, path_q,
                           (uint8_t *)ws, L, st);
}

int dflash_select_greedy(const dflash_config *cfg, const dflash_weights *w,
                         const int32_t *anchor, const int32_t *topk_ids, const float *topk_logp,
                         const void *hidden, int32_t B, int32_t K, int32_t *path,
                         float *path_score, void *ws, size_t ws_bytes, void *stream) {
  int rc = check_cfg(cfg);
  if (rc != DFLASH_OK) return rc;
  if (B < 0 || K < 2 || K > DFLASH_MAX_BLOCK) return DFLASH_ERR_BLOCK;
  if (B == 0) return DFLASH_OK;
  if ((size_t)B > kTopkTicketInts) return DFLASH_ERR_DIMS;
  if (!w || !anchor || !topk_ids || !topk_logp || !hidden || !path || !path_score || !ws ||
      !w->sel_gate)
    return DFLASH_ERR_NULL;
  if (!w->sel_table && (!w->embed || !w->sel_pu || !w->sel_pv)) return DFLASH_ERR_NULL;
  if (w->sel_table ? !a16(w->sel_table)
                   : (!a16(w->sel_pu) || !a16(w->sel_pv) || !a16(w->embed)))
    return DFLASH_ERR_ALIGN;
  if (!a16(w->sel_gate) || !a16(hidden) || !a16(ws)) return DFLASH_ERR_ALIGN;
  Layout L;
  make_layout(cfg, B, K, 0, &L);
  if (ws_bytes < L.total) return DFLASH_ERR_WORKSPACE;
  if (!device()) return DFLASH_ERR_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cfg->dtype == DFLASH_BF16)
    return run_greedy<dfl::bf16>(*cfg, *w, anchor, topk_ids, topk_logp, hidden, B, K, path,
                                 path_score, (uint8_t *)ws, L, st);
  return run_greedy<float>(*cfg, *w, anchor, topk_ids, topk_logp, hidden, B, K, path, path_score,
                           (uint8_t *)ws, L, st);
}

const void *dflash_draft_hidden(const dflash_config *cfg, int32_t B, int32_t K, const void *ws,
                                size_t ws_bytes) {
  if (check_cfg(cfg) != DFLASH_OK || !ws || B < 1 || K < 2 || K > DFLASH_MAX_BLOCK) return nullptr;
  Layout L;
  make_layout(cfg, B, K, 0, &L);
  if (ws_bytes < L.total) return nullptr;
  return (const uint8_t *)ws + L.zf;
}

int dflash_accept_sample(const int32_t *path, const int32_t *topk_ids, const float *path_q,
                         const void *target_logits, int32_t logits_dtype, int32_t B, int32_t K,
                         int32_t V, int32_t top_k, const float *uniforms, int32_t *accept_len,
                         int32_t *tokens, void *ws, size_t ws_bytes, void *stream) {
  if (logits_dtype != DFLASH_F32 && logits_dtype != DFLASH_BF16) return DFLASH_ERR_DTYPE;
  if (B < 0 || K < 2 || K > DFLASH_MAX_BLOCK) return DFLASH_ERR_BLOCK;
  if (V < 1 || top_k < 1 || top_k > DFLASH_MAX_TOPK) return DFLASH_ERR_DIMS;
  if ((long)B * K > 65535) return DFLASH_ERR_DIMS;  // one grid row per target row
  if (B == 0) return DFLASH_OK;
  if (!path || !topk_ids || !path_q || !target_logits || !uniforms || !accept_len || !tokens ||
      !ws)
    return DFLASH_ERR_NULL;
  if (!a16(ws)) return DFLASH_ERR_ALIGN;
  // chunk statistics after the fixed header (scratch shared with the other calls)
  const size_t need = kHeaderBytes + accept_sample_floats(B, K, V) * 4;
  if (ws_bytes < need) return DFLASH_ERR_WORKSPACE;
  if (!device()) return DFLASH_ERR_DEVICE;
  return launch_accept_sample(path, topk_ids, path_q, target_logits, logits_dtype, B, K, V, top_k,
                              uniforms, (float *)((uint8_t *)ws + kHeaderBytes), accept_len,
                              tokens, (cudaStream_t)stream);
}

int dflash_prepare_selector(const dflash_config *cfg, const dflash_weights *w, float *table,
                            void *ws, size_t ws_bytes, void *stream) {
  int rc = check_cfg(cfg);
  if (rc != DFLASH_OK) return rc;
  if (!w || !table || !ws || !w->embed || !w->sel_pu || !w->sel_pv) return DFLASH_ERR_NULL;
  if (!a16(table) || !a16(w->embed) || !a16(w->sel_pu) || !a16(w->sel_pv) || !a16(ws))
    return DFLASH_ERR_ALIGN;
  Layout L;
  make_layout(cfg, 1, 2, 0, &L);
  if (ws_bytes < L.status + 256) return DFLASH_ERR_WORKSPACE;
  if (!device()) return DFLASH_ERR_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  const int V = cfg->vocab, D = cfg->d_model, r = cfg->sel_rank;
  int *err = (int *)((uint8_t *)ws + L.status);
  // one K slice each: the projections land directly in the table rows
  TRY(gemm_xwT(cfg->dtype, w->sel_pu, r, D, w->embed, V, table, r, 1, err, st));
  TRY(gemm_xwT(cfg->dtype, w->sel_pv, r, D, w->embed, V, table + (size_t)V * r, r, 1, err, st));
  return DFLASH_OK;
}

int dflash_accept_greedy(const int32_t *path, const void *target_logits, int32_t logits_dtype,
                         int32_t B, int32_t K, int32_t V, int32_t *accept_len, int32_t *tokens,
                         void *ws, size_t ws_bytes, void *stream) {
  if (logits_dtype != DFLASH_F32 && logits_dtype != DFLASH_BF16) return DFLASH_ERR_DTYPE;
  if (B < 0 || K < 2 || K > DFLASH_MAX_BLOCK) return DFLASH_ERR_BLOCK;
  if (V < 1 || (long)B * K > 65535) return DFLASH_ERR_DIMS;  // one grid row per target row
  if (B == 0) return DFLASH_OK;
  if (!path || !target_logits || !accept_len || !tokens || !ws) return DFLASH_ERR_NULL;
  if (!a16(ws)) return DFLASH_ERR_ALIGN;
  // argmax partials after the fixed header (scratch shared with the other calls)
  const size_t need = kHeaderBytes + (size_t)B * K * argmax_chunks(V) * 2 * 4;
  if (ws_bytes < need) return DFLASH_ERR_WORKSPACE;
  if (!device()) return DFLASH_ERR_DEVICE;
  return launch_accept(path, target_logits, logits_dtype, B, K, V,
                       (float *)((uint8_t *)ws + kHeaderBytes), accept_len, tokens,
                       (cudaStream_t)stream);
}

int dflash_linear(int32_t dtype, const void *W, int32_t N_out, int32_t K_in, const void *X,
                  int32_t T, int32_t splits, float *out, void *stream) {
  if (dtype != DFLASH_F32 && dtype != DFLASH_BF16) return DFLASH_ERR_DTYPE;
  if (N_out < 1 || T < 0 || K_in < 64 || K_in % 64) return DFLASH_ERR_DIMS;
  if (splits < 1 || (K_in / 64) % splits) return DFLASH_ERR_DIMS;
  if (T == 0) return DFLASH_OK;
  if (!W || !X || !out) return DFLASH_ERR_NULL;
  if (!a16(W) || !a16(X)) return DFLASH_ERR_ALIGN;
  if (!device()) return DFLASH_ERR_DEVICE;
  return gemm_xwT(dtype, W, N_out, K_in, X, T, out, N_out, splits, nullptr, (cudaStream_t)stream);
}

int dflash_linear_q4(dflash_q4 W, int32_t N_out, int32_t K_in, const void *X, int32_t T,
                     int32_t splits, float *out, void *stream) {
  if (N_out < 1 || T < 0 || K_in < 64 || K_in % 64) return DFLASH_ERR_DIMS;
  if (splits < 1 || (K_in / 64) % splits) return DFLASH_ERR_DIMS;
  if (T == 0) return DFLASH_OK;
  if (!W.data || !X || !out) return DFLASH_ERR_NULL;
  if (!a16(W.data) || !a16(X)) return DFLASH_ERR_ALIGN;
  if (!device()) return DFLASH_ERR_DEVICE;
  GemmCall g;
  g.dtype = DFLASH_BF16;
  g.N_out = N_out;
  g.K_in = K_in;
  g.X = X;
  g.T = T;
  g.S = splits;
  g.mode = GEMM_PARTIAL;
  g.out = out;
  g.ld = N_out;
  g = with_q4(g, W, K_in);
  return gemm_run(g, (cudaStream_t)stream);
}

int dflash_test_linear_wait(const void *W, int32_t N_out, int32_t K_in, const void *X, int32_t T,
                            float *out, void *ws, size_t ws_bytes, uint32_t stall_wait_us,
                            void *stream) {
  if (N_out < 1 || T < 1 || K_in < 64 || K_in % 64) return DFLASH_ERR_DIMS;
  if (!W || !X || !out || !ws) return DFLASH_ERR_NULL;
  if (!a16(W) || !a16(X) || !a16(ws)) return DFLASH_ERR_ALIGN;
  if (ws_bytes < 256) return DFLASH_ERR_WORKSPACE;
  if (!device()) return DFLASH_ERR_DEVICE;
  GemmCall g;
  g.dtype = DFLASH_BF16;
  g.W = W;
  g.N_out = N_out;
  g.K_in = K_in;
  g.X = X;
  g.T = T;
  g.S = 1;
  g.mode = GEMM_PARTIAL;
  g.out = out;
  g.ld = N_out;
  g.err = (int *)ws;  // the workspace's status word
  if (stall_wait_us > 0) {
    g.stall = 1;
    g.wait_ns = (uint64_t)stall_wait_us * 1000ull;
  }
  return gemm_run(g, (cudaStream_t)stream);
}

int32_t dflash_linear_splits(int32_t N_out, int32_t T, int32_t K_in) {
  if (N_out < 1 || T < 1 || K_in < 64 || K_in % 64) return 0;
  return gemm_splits(N_out, T, K_in, sm_count_or_default());
}

int dflash_read_device_status(const void *ws, void *stream) {
  if (!ws) return DFLASH_ERR_NULL;
  int h = 0;
  if (cudaMemcpyAsync(&h, ws, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream) !=
          cudaSuccess ||
      cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  return h;
}

int dflash_clear_device_status(void *ws, void *stream) {
  if (!ws) return DFLASH_ERR_NULL;
  if (cudaMemsetAsync(ws, 0, sizeof(int), (cudaStream_t)stream) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  return DFLASH_OK;
}

const char *dflash_status_string(int code) {
  switch (code) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_NULL: return "a required pointer is NULL";
    case DFLASH_ERR_DIMS: return "a dimension breaks the shape rules";
    case DFLASH_ERR_BLOCK: return "block size K outside 2..32 or negative batch";
    case DFLASH_ERR_WORKSPACE: return "workspace smaller than dflash_workspace_bytes";
    case DFLASH_ERR_DTYPE: return "unsupported dtype";
    case DFLASH_ERR_CUDA: return "a CUDA call failed";
    case DFLASH_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case DFLASH_ERR_DEVICE: return "no usable sm_103 device";
    case DFLASH_DEV_TOKEN_RANGE: return "device: token id out of range";
    case DFLASH_DEV_PAGE_RANGE: return "device: page id out of range";
    case DFLASH_DEV_POS_RANGE: return "device: position beyond the page table";
    case DFLASH_DEV_TIMEOUT: return "device: bounded wait expired";
    case DFLASH_DEV_REQ_RANGE: return "device: request row out of range";
    default: return "unknown status";
  }
}

int64_t dflash_launch_count(int reset) {
  int64_t v = g_launches;
  if (reset) g_launches = 0;
  return v;
}

}  // extern "C"
