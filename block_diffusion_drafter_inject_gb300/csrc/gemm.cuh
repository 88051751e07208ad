// Projection GEMMs of the drafter: Y = X W^T with W [N_out, K_in] row-major
// (nn.Linear) and X [T, K_in] row-major, split over K into S slices whose
// fp32 partial sums are written to out[(s*T + t)*ld + n].  Consumers add the
// S slices in order, so results are deterministic.
#pragma once
#include "common.cuh"

namespace dflh {

constexpr size_t kMaxPartialFloats = size_t(48) << 20;  // cap of one partial buffer

// Number of K slices for a GEMM of this shape on `num_sms` SMs.
int gemm_splits(int N_out, int T, int K_in, int num_sms);

// Launch one GEMM.  dtype selects the operand storage (DFLASH_BF16: tcgen05
// tensor cores fed by TMA; DFLASH_F32: fp32 CUDA cores).  W and X must be
// 16-byte aligned and K_in a multiple of 64.  Returns DFLASH_OK or an error.
int gemm_xwT(int dtype, const void *W, int N_out, int K_in, const void *X, int T, float *out,
             int ld, int S, int *err, cudaStream_t stream);

}  // namespace dflh
