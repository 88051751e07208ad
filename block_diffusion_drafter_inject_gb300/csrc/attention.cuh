// Non-causal block attention over the paged context window plus the block.
#pragma once
#include "common.cuh"

namespace dflh {

struct AttnPlan {
  int qg;        // query rows per CTA (64)
  int nqg;       // query groups per (request, kv head)
  int kps;       // keys per split (multiple of 64)
  int nsplit;    // splits per (request, kv head, query group) at the largest key count
  size_t part_floats;  // partial O + (m, l) floats
};

AttnPlan attn_plan(int B, int K, int Hq, int Hkv, int dh, int window, int num_sms);

// o[r, h*dh + :] for r = b*K + i, from q [B*K, Hq, dh], block k/v [B*K, Hkv, dh]
// and layer `layer` of the paged caches.
template <typename S>
int launch_block_attention(const AttnPlan &pl, const S *qb, const S *kb, const S *vb,
                           const S *kc, const S *vc, int layer, const int32_t *page_table,
                           int max_pages, int num_pages, int page_size, const int32_t *ctx_len,
                           int B, int K, int Hq, int Hkv, int dh, int window, float *part, S *ob,
                           int *err, cudaStream_t st);

// bf16 storage: one kernel per layer reads the block's q, k (head-normed and
// rotated) and v rows from qkvb [B*K, (Hq+2Hkv)*dh] and the paged context
// window, attends, and merges its key splits through the cluster's distributed
// shared memory into o [B*K, Hq*dh].
// Page size 64: whole cache pages are loaded by TMA (caches [n_layers][num_pages]
// [Hkv][64][dh]); other page sizes copy 16-byte chunks per key row.  The first
// context pages are loaded before the wait on the projection unless they hold
// one of the inj_n rows (inj_req, inj_pos) that the pass itself injects.
int launch_attention_fused(const AttnPlan &pl, const dfl::bf16 *qkvb, const dfl::bf16 *kc,
                           const dfl::bf16 *vc, int layer, int n_layers, const int32_t *table,
                           int max_pages, int num_pages, int P, const int32_t *ctx_len, int B,
                           int K, int Hq, int Hkv, int dh, int window, dfl::bf16 *ob, int *err,
                           cudaStream_t st, const int32_t *inj_req = nullptr,
                           const int32_t *inj_pos = nullptr, int inj_n = 0);

}  // namespace dflh
