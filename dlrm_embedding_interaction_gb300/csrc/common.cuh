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

// Programmatic dependent launch. A kernel launched by launch_pdl may start
// while the kernel before it in the stream is still running: it must call
// pdl_wait() before its first global-memory access (the wait returns once
// the previous kernel has completed and its writes are visible; at once when
// there is none), then pdl_trigger() lets the next kernel start its own
// set-up early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

__device__ __forceinline__ float apply_act(float a, int act) {
  if (act == DLRM_ACT_RELU) return fmaxf(a, 0.0f);
  if (act == DLRM_ACT_SIGMOID) return 1.0f / (1.0f + expf(-a));
  return a;
}

// a / b for 0 <= a < 2^20 and 1 <= b < 2^14, given rb = __frcp_rn(b): the
// rounded product a rb is within one of the quotient (its relative error is
// below 2^-22), and one correction step each way makes it exact
// (tests/test_quot.py restates it in float32 and checks it next to every
// multiple in that range). Shorter than the integer division sequence on the
// fused kernels' latency-bound tile paths, where every divisor is a loop
// invariant whose reciprocal is taken once. The dividends there are element
// or task indices of one tile (at most 16 samples x 8,256 pairs, below 2^18),
// and the divisors widths of arrays that one tile keeps in 227 KB of shared
// memory (a sample's k x D/4 bag-row chunks, a row of activations) or the
// pair count (8,256 at the 128-table limit): all below 2^14.
__device__ __forceinline__ int quot(int a, int b, float rb) {
  int q = __float2int_rz(__fmul_rn(__int2float_rn(a), rb));
  const int r = a - q * b;
  q += r >= b ? 1 : 0;
  q -= r < 0 ? 1 : 0;
  return q;
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

// Pair dots in 4 x 4 register blocks. The F rows of one sample's Z (d4
// float4 each, in shared memory) are dealt into nb = ceil(F / 4) residue
// classes, class b holding rows b, b + nb, b + 2 nb, b + 3 nb; block (bi, bj),
// bi >= bj, is the 4 x 4 grid of dots between the rows of classes bi and bj,
// and the blocks are numbered i-major with the diagonal included (block q is
// the strict pair (bi + 1, bj) of the same closed form). Every unordered pair
// of distinct rows falls in exactly one block: the one of its two rows'
// classes (gram_block_pair names the pair of each entry). One thread computes
// the 16 dots of a block from 8 128-bit shared loads per 4-wide step (64
// FMA), against 2 loads per 4 FMA one pair at a time. Dealing rows by residue
// rather than in runs of four puts the threads of a warp, which take
// consecutive blocks, on consecutive rows: with a row stride of an odd number
// of 16-byte words those fall in distinct bank groups, where runs of four
// rows meet in two. Rows past F are clamped to F - 1 (computed, never stored).
__host__ __device__ __forceinline__ int gram_blocks(int f) {
  const int nb = (f + 3) / 4;
  return nb * (nb + 1) / 2;
}

// The strict-lower-triangle index of entry (a, c) of block (bi, bj): rows
// i = bi + a nb and j = bj + c nb, stored as (max, min); -1 when the entry has
// no pair of its own (a row past F, the diagonal, or, in a diagonal block,
// the upper copy of a pair).
__host__ __device__ __forceinline__ int gram_block_pair(int f, int bi, int bj, int a, int c) {
  const int nb = (f + 3) / 4;
  const int i = bi + a * nb, j = bj + c * nb;
  if (i >= f || j >= f || i == j || (bi == bj && a < c)) return -1;
  const int hi = i > j ? i : j;
  const int lo = i + j - hi;
  return hi * (hi - 1) / 2 + lo;
}

template <class RowFn>
__device__ __forceinline__ void gram_block(const RowFn& row, int f, int d4, int q, int& bi,
                                           int& bj, float acc[4][4]) {
  int ii, jj;
  pair_from_index(q, ii, jj);
  bi = ii - 1;
  bj = jj;
  const float* ri[4];
  const float* rj[4];
  const int nb = (f + 3) / 4;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    ri[a] = row(min(bi + a * nb, f - 1));
    rj[a] = row(min(bj + a * nb, f - 1));
  }
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
  for (int c4 = 0; c4 < d4; ++c4) {
    float4 u[4], v[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      u[a] = *reinterpret_cast<const float4*>(ri[a] + 4 * c4);
      v[a] = *reinterpret_cast<const float4*>(rj[a] + 4 * c4);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc[a][c] = fmaf(u[a].x, v[c].x, acc[a][c]);
        acc[a][c] = fmaf(u[a].y, v[c].y, acc[a][c]);
        acc[a][c] = fmaf(u[a].z, v[c].z, acc[a][c]);
        acc[a][c] = fmaf(u[a].w, v[c].w, acc[a][c]);
      }
  }
}

// Bounded waits of a launch. Every wait of a kernel on another party (a
// weight stage or tile landing, a ring slot being released, tensor-core work
// completing) gives up after limit_ns (0: the default of 2 s), sets
// DLRM_ERRBIT_TIMEOUT and lets the kernel finish without the data. For
// failure-detection tests, withhold_last makes the kernel skip the last copy
// (or tensor-core commit) of its stream, so that the wait on it runs out.
struct WaitCfg {
  uint64_t limit_ns = 0;
  int withhold_last = 0;
};
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
__host__ __device__ __forceinline__ uint64_t wait_limit_ns(const WaitCfg& w) {
  return w.limit_ns ? w.limit_ns : kDefaultWaitNs;
}

// Kernel-parameter table for the multi-table gather: K (pointer, rows) pairs
// passed by value so a launch needs no device-side staging buffer.
struct GatherTables {
  const float* ptr[DLRM_MAX_TABLES];
  int64_t rows[DLRM_MAX_TABLES];
};

// ---- launchers (each returns cudaGetLastError() of its launch) ----------

cudaError_t launch_gather(const GatherTables& tabs, int k, int d, const int64_t* indices,
                          const int64_t* offsets, int b, int l, float* out, int32_t* err_flag,
                          cudaStream_t stream);
cudaError_t launch_gather_general(const GatherTables& tabs, int k, int d, const void* indices,
                                  int64_t n_idx, const void* offsets, int index_bits, int b,
                                  int mode, const float* per_sample_weights, int64_t padding_idx,
                                  float* out, int32_t* err_flag, cudaStream_t stream);

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
                             int32_t* err, cudaStream_t stream, WaitCfg wait = WaitCfg{});

int device_sm_count();
size_t device_max_smem_optin();

// An element pointer's natural alignment (`bytes` = the element size). A null
// pointer passes: null checks are made separately.
inline bool aligned_to(const void* p, size_t bytes) {
  return reinterpret_cast<uintptr_t>(p) % bytes == 0;
}

}  // namespace dlrm
