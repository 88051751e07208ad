// Greedy acceptance without a caller-provided workspace.
//
// dflash_accept_greedy needs scratch for its per-chunk argmax partials, which
// normally lives in the caller's workspace.  Some callers cannot provide one:
// a runtime whose device memory is planned once at start-up and may not grow
// afterwards, a host binding with no device allocator of its own, or code that
// must not call cudaMalloc at the point where acceptance runs.  This variant
// keeps its scratch in a fixed array in the library's own device memory, so
// the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ symbol: every GPU that loads the
// library holds it until the process exits.  Host code cannot use the symbol's
// name as a device address, so the first call on each device looks the address
// up (cudaGetSymbolAddress, with that device current) and caches it.
#include <mutex>

#include "head.cuh"

namespace {

// 64 Ki floats (256 KiB): argmax partials of up to 32768 (row, chunk) pairs,
// i.e. B * K * ceil(V / 8192) <= 32768 (for V = 151936: B * K <= 1724).
constexpr size_t kNoAllocScratchFloats = size_t(1) << 16;

__device__ __align__(256) float g_accept_scratch[kNoAllocScratchFloats];

float *scratch_address(int *rc) {
  static std::mutex mu;
  static float *addr[64] = {nullptr};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    *rc = DFLASH_ERR_DEVICE;
    return nullptr;
  }
  std::lock_guard<std::mutex> g(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      *rc = DFLASH_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = (float *)p;
  }
  *rc = DFLASH_OK;
  return addr[dev];
}

}  // namespace

extern "C" int dflash_accept_greedy_noalloc(const int32_t *path, const void *target_logits,
                                            int32_t logits_dtype, int32_t B, int32_t K,
                                            int32_t V, int32_t *accept_len, int32_t *tokens,
                                            void *stream) {
  if (logits_dtype != DFLASH_F32 && logits_dtype != DFLASH_BF16) return DFLASH_ERR_DTYPE;
  if (B < 0 || K < 2 || K > DFLASH_MAX_BLOCK) return DFLASH_ERR_BLOCK;
  if (V < 1) return DFLASH_ERR_DIMS;
  if (B == 0) return DFLASH_OK;
  if (!path || !target_logits || !accept_len || !tokens) return DFLASH_ERR_NULL;
  // every partial is written before it is read, so nothing needs clearing
  const size_t need = (size_t)B * K * dflh::argmax_chunks(V) * 2;
  if (need > kNoAllocScratchFloats) return DFLASH_ERR_WORKSPACE;
  if (!dflh::device()) return DFLASH_ERR_DEVICE;
  int rc = DFLASH_OK;
  float *scratch = scratch_address(&rc);
  if (rc != DFLASH_OK) return rc;
  return dflh::launch_accept(path, target_logits, logits_dtype, B, K, V, scratch, accept_len,
                             tokens, (cudaStream_t)stream);
}
