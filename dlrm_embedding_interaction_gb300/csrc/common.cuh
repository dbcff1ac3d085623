// Internal declarations shared by the CUDA translation units of
// libdlrm_gb300.so. Nothing here is part of the public C ABI (include/dlrm.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/dlrm.h"

namespace dlrm {

constexpr int kWarp = 32;

__host__ __device__ __forceinline__ int64_t round_up(int64_t x, int64_t m) {
  return (x + m - 1) / m * m;
}

__device__ __forceinline__ float apply_act(float a, int act) {
  if (act == DLRM_ACT_RELU) return fmaxf(a, 0.0f);
  if (act == DLRM_ACT_SIGMOID) return 1.0f / (1.0f + expf(-a));
  return a;
}

// Pair index p -> (i, j) of the strict lower triangle, i-major:
// p = i(i-1)/2 + j with 0 <= j < i. The closed form i = floor((1+sqrt(1+8p))/2)
// (Luminal PairwiseDotLowerTriStackedKernel) is evaluated in fp32, then fixed
// up with exact integer comparisons so the map is exact for every p.
__device__ __forceinline__ void pair_from_index(int p, int& i, int& j) {
  int ii = static_cast<int>(floorf((1.0f + sqrtf(1.0f + 8.0f * static_cast<float>(p))) * 0.5f));
  while (ii * (ii - 1) / 2 > p) --ii;
  while ((ii + 1) * ii / 2 <= p) ++ii;
  i = ii;
  j = p - ii * (ii - 1) / 2;
}

// Kernel-parameter table for the multi-table gather: K (pointer, rows) pairs
// passed by value so a launch needs no device-side staging buffer.
struct GatherTables {
  const float* ptr[DLRM_MAX_TABLES];
  int64_t rows[DLRM_MAX_TABLES];
};

// ---- launchers (each returns cudaGetLastError() of its launch) ----------

cudaError_t launch_gather(const GatherTables& tabs, int k, int d, const int64_t* indices,
                          const int64_t* offsets, int b, int l, float* out, int ld_out_row,
                          int32_t* err_flag, cudaStream_t stream);

cudaError_t launch_interaction(const float* dense, int ld_dense, const float* emb, int b,
                               int k, int d, float* out, int ld_out, int copy_dense,
                               cudaStream_t stream);

cudaError_t launch_pair_map(int f, int32_t* i_out, int32_t* j_out, cudaStream_t stream);

size_t interaction_smem_per_sample(int k, int d);

cudaError_t launch_linear_fp32(const float* x, int ld_x, const float* w, int ld_w,
                               const float* bias, float* y, int ld_y, int m, int n, int k,
                               int act, cudaStream_t stream);

// Tensor-core (tcgen05) Linear, mode DLRM_MATH_TF32 / BF16 / TF32X3, fp32
// accumulation; err (nullable) receives DLRM_ERRBIT_TIMEOUT on a stuck wait.
cudaError_t launch_linear_tc(const float* x, int ld_x, const float* w, int ld_w, const float* bias,
                             float* y, int ld_y, int m, int n, int k, int act, int mode,
                             int32_t* err, cudaStream_t stream);

int device_sm_count();
size_t device_max_smem_optin();

}  // namespace dlrm
