// Multi-table EmbeddingBag sum, all K tables in one launch.
//
// Computes out[b][t][:] = sum_{l < L} W_t[indices[t][offsets[t][b] + l]][:]
// (Luminal compare modal_ci_ready...vanilla-pytorch, commit message:
// MultiTableEmbeddingBagSumKernel, (batch, num_tables, d) F32 in one launch;
// compare dlrm-fused-kernels...dlrm-pt2-megakernel, LessonsLearned
// "EmbeddingBag translator gap": output[b] = sum over indices[offsets[b]:
// offsets[b+1]], uniform bags).
//
// GB300 design: the gather is HBM-bound (one random D*4-byte row per index),
// so the kernel is built for bytes in flight, not arithmetic:
//  * a group of TPB lanes owns one (sample, table) bag; each lane moves
//    CHUNKS 16-byte vectors of every row (128-bit loads, a D=128 row is one
//    fully coalesced 512-byte warp load);
//  * bag indices are loaded once per group (one lane per index) and
//    broadcast by shuffle; rows are fetched U at a time before any add, so a
//    warp keeps U * 512 bytes outstanding per group;
//  * bags are numbered b * K + t so consecutive groups write consecutive
//    output rows (coalesced stores of the (B, K, D) result);
//  * no shared-memory staging: each row is read exactly once and consumed in
//    registers, so a TMA or cp.async copy would only add a round trip.
// Bounds: every index is checked against rows[t]; a bad index contributes
// zeros and sets DLRM_ERRBIT_INDEX_OOB. The bag start must equal b * L (the
// uniform stride), which also keeps every index read inside (K, B*L); a bag
// whose offset differs is written as zeros with DLRM_ERRBIT_OFFSETS.
#include "common.cuh"

namespace dlrm {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ void flag_error(int32_t* err, uint32_t bit) {
  if (err) atomicOr(reinterpret_cast<unsigned int*>(err), bit);
}

__device__ __forceinline__ void add4(float4& a, const float4& v) {
  a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
}

// Vector path: D % 4 == 0, tables and out 16-byte aligned.
// TPB lanes per bag (power of two <= 32); each lane owns CHUNKS float4 columns
// col4 = lane + c * TPB (< D/4).
template <int TPB, int CHUNKS>
__global__ void __launch_bounds__(kGatherThreads)
gather_vec_kernel(const __grid_constant__ GatherTables tabs, int k_tables, int d4,
                  const int64_t* __restrict__ indices, const int64_t* __restrict__ offsets,
                  int batch, int bag, float* __restrict__ out, int32_t* err) {
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t bag_id = gtid / TPB;
  const int lane = threadIdx.x & (TPB - 1);
  const unsigned lane_in_warp = threadIdx.x & (kWarp - 1);
  const unsigned gmask = (TPB == 32) ? 0xffffffffu
                                     : (((1u << TPB) - 1u) << (lane_in_warp & ~(TPB - 1u)));
  if (bag_id >= static_cast<int64_t>(batch) * k_tables) return;  // whole group leaves
  const int b = static_cast<int>(bag_id / k_tables);
  const int t = static_cast<int>(bag_id - static_cast<int64_t>(b) * k_tables);

  float4* dst = reinterpret_cast<float4*>(out) + bag_id * d4;
  float4 acc[CHUNKS];
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);

  const int64_t n_idx = static_cast<int64_t>(batch) * bag;
  const int64_t start = offsets[static_cast<int64_t>(t) * batch + b];
  if (start != static_cast<int64_t>(b) * bag) {
    if (lane == 0) flag_error(err, DLRM_ERRBIT_OFFSETS);
  } else {
    const int64_t* idx = indices + static_cast<int64_t>(t) * n_idx + start;
    const float4* table = reinterpret_cast<const float4*>(tabs.ptr[t]);
    const int64_t rows = tabs.rows[t];
    bool oob = false;
    for (int l0 = 0; l0 < bag; l0 += TPB) {
      const int cnt = min(TPB, bag - l0);
      const int64_t mine = (lane < cnt) ? __ldg(idx + l0 + lane) : 0;
      for (int u0 = 0; u0 < cnt; u0 += kUnroll) {
        float4 v[kUnroll][CHUNKS];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
          const int64_t r = __shfl_sync(gmask, mine, (u0 + q) & (TPB - 1), TPB);
          const bool live = (u0 + q) < cnt;
          const bool ok = live && r >= 0 && r < rows;
          oob |= live && !ok;
#pragma unroll
          for (int c = 0; c < CHUNKS; ++c) {
            const int col4 = lane + c * TPB;
            v[q][c] = (ok && col4 < d4) ? __ldg(table + r * d4 + col4)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int q = 0; q < kUnroll; ++q)
#pragma unroll
          for (int c = 0; c < CHUNKS; ++c) add4(acc[c], v[q][c]);
      }
    }
    if (oob && lane == 0) flag_error(err, DLRM_ERRBIT_INDEX_OOB);
  }
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    const int col4 = lane + c * TPB;
    if (col4 < d4) dst[col4] = acc[c];
  }
}

// Scalar path for any D and alignment: TPB = 32 lanes per bag, lane owns
// columns lane, lane + 32, ...; indices re-read per column from L1.
__global__ void __launch_bounds__(kGatherThreads)
gather_scalar_kernel(const __grid_constant__ GatherTables tabs, int k_tables, int d,
                     const int64_t* __restrict__ indices, const int64_t* __restrict__ offsets,
                     int batch, int bag, float* __restrict__ out, int32_t* err) {
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t bag_id = gtid / kWarp;
  const int lane = threadIdx.x & (kWarp - 1);
  if (bag_id >= static_cast<int64_t>(batch) * k_tables) return;
  const int b = static_cast<int>(bag_id / k_tables);
  const int t = static_cast<int>(bag_id - static_cast<int64_t>(b) * k_tables);
  float* dst = out + bag_id * d;
  const int64_t n_idx = static_cast<int64_t>(batch) * bag;
  const int64_t start = offsets[static_cast<int64_t>(t) * batch + b];
  if (start != static_cast<int64_t>(b) * bag) {
    if (lane == 0) flag_error(err, DLRM_ERRBIT_OFFSETS);
    for (int c = lane; c < d; c += kWarp) dst[c] = 0.f;
    return;
  }
  const int64_t* idx = indices + static_cast<int64_t>(t) * n_idx + start;
  const float* table = tabs.ptr[t];
  const int64_t rows = tabs.rows[t];
  bool oob = false;
  for (int c = lane; c < d; c += kWarp) {
    float acc = 0.f;
    for (int l = 0; l < bag; ++l) {
      const int64_t r = __ldg(idx + l);
      if (r >= 0 && r < rows) acc += __ldg(table + r * d + c);
      else oob = true;
    }
    dst[c] = acc;
  }
  if (d == 0) return;
  if (__any_sync(0xffffffffu, oob) && lane == 0) flag_error(err, DLRM_ERRBIT_INDEX_OOB);
}

template <int TPB, int CHUNKS>
cudaError_t launch_vec(const GatherTables& tabs, int k, int d, const int64_t* indices,
                       const int64_t* offsets, int b, int l, float* out, int32_t* err,
                       cudaStream_t stream) {
  const int64_t bags = static_cast<int64_t>(b) * k;
  const int64_t per_block = kGatherThreads / TPB;
  const int64_t grid = (bags + per_block - 1) / per_block;
  gather_vec_kernel<TPB, CHUNKS><<<static_cast<unsigned>(grid), kGatherThreads, 0, stream>>>(
      tabs, k, d / 4, indices, offsets, b, l, out, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather(const GatherTables& tabs, int k, int d, const int64_t* indices,
                          const int64_t* offsets, int b, int l, float* out, int /*unused*/,
                          int32_t* err, cudaStream_t stream) {
  if (b == 0) return cudaSuccess;
  bool vec = (d % 4 == 0) && (reinterpret_cast<uintptr_t>(out) % 16 == 0);
  for (int t = 0; t < k && vec; ++t) vec = reinterpret_cast<uintptr_t>(tabs.ptr[t]) % 16 == 0;
  const int d4 = d / 4;
  if (vec && d4 <= 256) {
    if (d4 <= 1) return launch_vec<1, 1>(tabs, k, d, indices, offsets, b, l, out, err, stream);
    if (d4 <= 2) return launch_vec<2, 1>(tabs, k, d, indices, offsets, b, l, out, err, stream);
    if (d4 <= 4) return launch_vec<4, 1>(tabs, k, d, indices, offsets, b, l, out, err, stream);
    if (d4 <= 8) return launch_vec<8, 1>(tabs, k, d, indices, offsets, b, l, out, err, stream);
    if (d4 <= 16) return launch_vec<16, 1>(tabs, k, d, indices, offsets, b, l, out, err, stream);
    if (d4 <= 32) return launch_vec<32, 1>(tabs, k, d, indices, offsets, b, l, out, err, stream);
    if (d4 <= 64) return launch_vec<32, 2>(tabs, k, d, indices, offsets, b, l, out, err, stream);
    if (d4 <= 128) return launch_vec<32, 4>(tabs, k, d, indices, offsets, b, l, out, err, stream);
    return launch_vec<32, 8>(tabs, k, d, indices, offsets, b, l, out, err, stream);
  }
  const int64_t bags = static_cast<int64_t>(b) * k;
  const int64_t per_block = kGatherThreads / kWarp;
  const int64_t grid = (bags + per_block - 1) / per_block;
  gather_scalar_kernel<<<static_cast<unsigned>(grid), kGatherThreads, 0, stream>>>(
      tabs, k, d, indices, offsets, b, l, out, err);
  return cudaGetLastError();
}

}  // namespace dlrm
