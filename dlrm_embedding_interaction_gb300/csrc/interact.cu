// Strict-lower-triangular pairwise-dot interaction with the concat fused.
//
// Per sample: Z = [x; e_0; ...; e_{K-1}] is (F, D), F = K + 1, and
// z[p] = <Z_i, Z_j> for p = i(i-1)/2 + j, j < i (i-major), R = [x, z]
// (Luminal compare dlrm-fused-kernels...dlrm-pt2-megakernel,
// dlrm_megakernel.rs steps 4-5; compare modal_ci_ready...vanilla-pytorch,
// commit message: PairwiseDotLowerTriStackedKernel, block-per-batch-row with
// all F*D features cached in shared memory and (i, j) from the closed form).
//
// GB300 design: a block takes S consecutive samples (S = 1 for wide F, more
// when F is small so the block has S * P >= blockDim pair tasks), stages
// their S*F*D features in shared memory with 128-bit coalesced loads (rows
// padded to D + 4 floats so the 16-byte reads of different rows fall in
// different banks), then thread w computes tasks w, w + T, ...: with D a
// multiple of 4 a task is a 4 x 4 block of pairs held in registers
// (gram_block), a quarter of the shared-memory reads of one pair per thread.
#include <atomic>

#include "common.cuh"

namespace dlrm {
namespace {

constexpr int kInteractThreads = 256;

// 16-byte global -> shared copy that does not hold the thread (cp.async), so
// every row of the block's samples is in flight at once.
__device__ __forceinline__ void copy16_async(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}

__host__ __device__ __forceinline__ int z_stride(int d) {
  return static_cast<int>(round_up(d, 4)) + 4;
}

template <bool VEC>
__global__ void __launch_bounds__(kInteractThreads)
interaction_kernel(const float* __restrict__ dense, int ld_dense, const float* __restrict__ emb,
                   int batch, int k_tables, int d, float* __restrict__ out, int ld_out,
                   int copy_dense, int samples_per_block, int use_blocks) {
  extern __shared__ float4 smem_f4[];
  float* zs = reinterpret_cast<float*>(smem_f4);
  const int f = k_tables + 1;
  const int p_count = f * (f - 1) / 2;
  const int ldz = z_stride(d);
  const int b0 = blockIdx.x * samples_per_block;
  const int ns = min(samples_per_block, batch - b0);
  const int tid = threadIdx.x;

  // Stage Z for ns samples: row 0 from dense, rows 1..K from emb.
  if (VEC) {
    const int d4 = d / 4;
    const int per_sample = f * d4;
    for (int e = tid; e < ns * per_sample; e += blockDim.x) {
      const int s = e / per_sample;
      const int r = e - s * per_sample;
      const int row = r / d4;
      const int c4 = r - row * d4;
      const float4* src =
          row == 0 ? reinterpret_cast<const float4*>(dense + static_cast<int64_t>(b0 + s) * ld_dense) + c4
                   : reinterpret_cast<const float4*>(emb) +
                         (static_cast<int64_t>(b0 + s) * k_tables + (row - 1)) * d4 + c4;
      copy16_async(zs + (s * f + row) * ldz + c4 * 4, src);
    }
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
  } else {
    const int per_sample = f * d;
    for (int e = tid; e < ns * per_sample; e += blockDim.x) {
      const int s = e / per_sample;
      const int r = e - s * per_sample;
      const int row = r / d;
      const int c = r - row * d;
      const float v = (row == 0)
          ? __ldg(dense + static_cast<int64_t>(b0 + s) * ld_dense + c)
          : __ldg(emb + (static_cast<int64_t>(b0 + s) * k_tables + (row - 1)) * d + c);
      zs[(s * f + row) * ldz + c] = v;
    }
  }
  __syncthreads();

  int col0 = 0;
  if (copy_dense) {
    for (int e = tid; e < ns * d; e += blockDim.x) {
      const int s = e / d;
      const int c = e - s * d;
      out[static_cast<int64_t>(b0 + s) * ld_out + c] = zs[(s * f) * ldz + c];
    }
    col0 = d;
  }
  const int nblk = gram_blocks(f);
  if (VEC && use_blocks) {
    // 4 x 4 register blocks of pairs (gram_block)
    const int d4 = d / 4;
    for (int w = tid; w < ns * nblk; w += blockDim.x) {
      const int s = w / nblk;
      const int q = w - s * nblk;
      const float* zsam = zs + s * f * ldz;
      float acc[4][4];
      int bi, bj;
      gram_block([&](int r) { return zsam + r * ldz; }, f, d4, q, bi, bj, acc);
      float* o = out + static_cast<int64_t>(b0 + s) * ld_out + col0;
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int i = 4 * bi + a;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int j = 4 * bj + c;
          if (i < f && j < i) o[i * (i - 1) / 2 + j] = acc[a][c];
        }
      }
    }
  } else if (VEC) {
    const int d4 = d / 4;
    for (int w = tid; w < ns * p_count; w += blockDim.x) {
      const int s = w / p_count;
      const int p = w - s * p_count;
      int i, j;
      pair_from_index(p, i, j);
      const float* zi = zs + (s * f + i) * ldz;
      const float* zj = zs + (s * f + j) * ldz;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c4 = 0; c4 < d4; ++c4) {
        const float4 u = *reinterpret_cast<const float4*>(zi + 4 * c4);
        const float4 v = *reinterpret_cast<const float4*>(zj + 4 * c4);
        a.x = fmaf(u.x, v.x, a.x);
        a.y = fmaf(u.y, v.y, a.y);
        a.z = fmaf(u.z, v.z, a.z);
        a.w = fmaf(u.w, v.w, a.w);
      }
      out[static_cast<int64_t>(b0 + s) * ld_out + col0 + p] = (a.x + a.y) + (a.z + a.w);
    }
  } else {
    for (int w = tid; w < ns * p_count; w += blockDim.x) {
      const int s = w / p_count;
      const int p = w - s * p_count;
      int i, j;
      pair_from_index(p, i, j);
      const float* zi = zs + (s * f + i) * ldz;
      const float* zj = zs + (s * f + j) * ldz;
      float acc = 0.f;
      for (int c = 0; c < d; ++c) acc = fmaf(zi[c], zj[c], acc);
      out[static_cast<int64_t>(b0 + s) * ld_out + col0 + p] = acc;
    }
  }
}

// Bag sums and the interaction in one launch (the layer-wise plan, bags of a
// uniform L): a block takes S samples, copies their bottom-MLP rows x into
// shared memory, sums their K bags there with lane groups of TPB lanes (each
// lane CHUNKS 16-byte vectors of a row, kGiUnroll rows in flight per group,
// as the standalone gather), then computes the pair dots from shared memory
// and writes R = [x, z]. The (B, K, D) bag sums never travel through HBM.
// Bounds: an index outside [0, rows) contributes zeros and sets
// DLRM_ERRBIT_INDEX_OOB; a bag start other than b * L zeroes the bag and sets
// DLRM_ERRBIT_OFFSETS.
constexpr int kGiUnroll = 8;

template <int TPB, int CHUNKS>
__global__ void __launch_bounds__(kInteractThreads)
gather_interact_kernel(const __grid_constant__ GatherTables tabs, int k_tables, int d,
                       const int64_t* __restrict__ indices, const int64_t* __restrict__ offsets,
                       int batch, int bag, const float* __restrict__ x, int ld_x,
                       float* __restrict__ out, int ld_out, int samples_per_block, int use_blocks,
                       int32_t* err) {
  extern __shared__ float4 smem_f4[];
  float* zs = reinterpret_cast<float*>(smem_f4);
  const int f = k_tables + 1;
  const int d4 = d / 4;
  const int ldz = z_stride(d);
  const int b0 = blockIdx.x * samples_per_block;
  const int ns = min(samples_per_block, batch - b0);
  const int tid = threadIdx.x;

  // row 0 of every sample: its x
  for (int e = tid; e < ns * d4; e += blockDim.x) {
    const int s = e / d4;
    const int c4 = e - s * d4;
    copy16_async(zs + (s * f) * ldz + 4 * c4, x + static_cast<int64_t>(b0 + s) * ld_x + 4 * c4);
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");

  // rows 1..K: the bag sums, one lane group per bag
  const int lane = tid & (TPB - 1);
  const unsigned lane_in_warp = tid & (kWarp - 1);
  const unsigned gmask = (TPB == 32) ? 0xffffffffu
                                     : (((1u << TPB) - 1u) << (lane_in_warp & ~(TPB - 1u)));
  const int groups = blockDim.x / TPB;
  const int64_t n_idx = static_cast<int64_t>(batch) * bag;
  bool oob = false, bad_off = false;
  for (int q = tid / TPB; q < ns * k_tables; q += groups) {
    const int s = q / k_tables;
    const int t = q - s * k_tables;
    const int b = b0 + s;
    float4 acc[CHUNKS];
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t start = offsets[static_cast<int64_t>(t) * batch + b];
    if (start != static_cast<int64_t>(b) * bag) {
      bad_off = true;
    } else {
      const int64_t* idx = indices + static_cast<int64_t>(t) * n_idx + start;
      const float4* table = reinterpret_cast<const float4*>(tabs.ptr[t]);
      const int64_t rows = tabs.rows[t];
      for (int l0 = 0; l0 < bag; l0 += TPB) {
        const int cnt = min(TPB, bag - l0);
        const int64_t mine = (lane < cnt) ? __ldg(idx + l0 + lane) : 0;
        for (int u0 = 0; u0 < cnt; u0 += kGiUnroll) {
          float4 v[kGiUnroll][CHUNKS];
#pragma unroll
          for (int u = 0; u < kGiUnroll; ++u) {
            const int64_t r = __shfl_sync(gmask, mine, (u0 + u) & (TPB - 1), TPB);
            const bool live = (u0 + u) < cnt;
            const bool ok = live && r >= 0 && r < rows;
            oob |= live && !ok;
#pragma unroll
            for (int c = 0; c < CHUNKS; ++c) {
              const int col4 = lane + c * TPB;
              v[u][c] = (ok && col4 < d4) ? __ldg(table + r * d4 + col4)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int u = 0; u < kGiUnroll; ++u)
#pragma unroll
            for (int c = 0; c < CHUNKS; ++c) {
              acc[c].x += v[u][c].x;
              acc[c].y += v[u][c].y;
              acc[c].z += v[u][c].z;
              acc[c].w += v[u][c].w;
            }
        }
      }
    }
    float* row = zs + (s * f + 1 + t) * ldz;
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
      const int col4 = lane + c * TPB;
      if (col4 < d4) *reinterpret_cast<float4*>(row + 4 * col4) = acc[c];
    }
  }
  if (err) {
    if (oob) atomicOr(reinterpret_cast<unsigned int*>(err), DLRM_ERRBIT_INDEX_OOB);
    if (bad_off) atomicOr(reinterpret_cast<unsigned int*>(err), DLRM_ERRBIT_OFFSETS);
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  __syncthreads();

  // R = [x, z]
  for (int e = tid; e < ns * d4; e += blockDim.x) {
    const int s = e / d4;
    const int c4 = e - s * d4;
    *reinterpret_cast<float4*>(out + static_cast<int64_t>(b0 + s) * ld_out + 4 * c4) =
        *reinterpret_cast<const float4*>(zs + (s * f) * ldz + 4 * c4);
  }
  const int p_count = f * (f - 1) / 2;
  if (use_blocks) {
    const int nblk = gram_blocks(f);
    for (int w = tid; w < ns * nblk; w += blockDim.x) {
      const int s = w / nblk;
      const int q = w - s * nblk;
      const float* zsam = zs + s * f * ldz;
      float acc[4][4];
      int bi, bj;
      gram_block([&](int r) { return zsam + r * ldz; }, f, d4, q, bi, bj, acc);
      float* o = out + static_cast<int64_t>(b0 + s) * ld_out + d;
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int i = 4 * bi + a;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int j = 4 * bj + c;
          if (i < f && j < i) o[i * (i - 1) / 2 + j] = acc[a][c];
        }
      }
    }
  } else {
    for (int w = tid; w < ns * p_count; w += blockDim.x) {
      const int s = w / p_count;
      const int p = w - s * p_count;
      int i, j;
      pair_from_index(p, i, j);
      const float* zi = zs + (s * f + i) * ldz;
      const float* zj = zs + (s * f + j) * ldz;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c4 = 0; c4 < d4; ++c4) {
        const float4 u = *reinterpret_cast<const float4*>(zi + 4 * c4);
        const float4 v = *reinterpret_cast<const float4*>(zj + 4 * c4);
        a.x = fmaf(u.x, v.x, a.x);
        a.y = fmaf(u.y, v.y, a.y);
        a.z = fmaf(u.z, v.z, a.z);
        a.w = fmaf(u.w, v.w, a.w);
      }
      out[static_cast<int64_t>(b0 + s) * ld_out + d + p] = (a.x + a.y) + (a.z + a.w);
    }
  }
}

__global__ void pair_map_kernel(int f, int32_t* i_out, int32_t* j_out) {
  const int p_count = f * (f - 1) / 2;
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < p_count; p += gridDim.x * blockDim.x) {
    int i, j;
    pair_from_index(p, i, j);
    i_out[p] = i;
    j_out[p] = j;
  }
}

// Raise a kernel's dynamic shared-memory limit to the device maximum, once per
// (kernel, device). Done on first use, outside any stream capture in practice
// (the first call of a shape), and never again on later launches.
template <class K>
cudaError_t enable_large_smem(K kernel, int slot) {
  static std::atomic<uint64_t> done[2];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit && (done[slot].load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(device_max_smem_optin()));
  if (e == cudaSuccess && bit) done[slot].fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace

size_t interaction_smem_per_sample(int k, int d) {
  return static_cast<size_t>(k + 1) * z_stride(d) * sizeof(float);
}

cudaError_t launch_interaction(const float* dense, int ld_dense, const float* emb, int b,
                               int k, int d, float* out, int ld_out, int copy_dense,
                               cudaStream_t stream) {
  if (b == 0) return cudaSuccess;
  const int f = k + 1;
  const int p_count = f * (f - 1) / 2;
  const size_t per = interaction_smem_per_sample(k, d);
  const size_t budget = 64 * 1024;
  const bool vec = (d % 4 == 0) && (ld_dense % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(dense) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(emb) % 16 == 0);
  // per-sample tasks: 4 x 4 pair blocks from F = 9 on (at least 6 blocks a
  // sample), single pairs below, where blocks would leave threads idle
  const int blocks4 = gram_blocks(f);
  const int use_blocks = (vec && f >= 9) ? 1 : 0;
  const int tasks = use_blocks ? blocks4 : p_count;
  int s = tasks > 0 ? (kInteractThreads + tasks - 1) / tasks : kInteractThreads;
  s = static_cast<int>(std::min<size_t>(static_cast<size_t>(s), std::max<size_t>(1, budget / per)));
  // keep at least two blocks per SM when the batch allows it
  const int sms = device_sm_count();
  const int cap = std::max(1, (b + 2 * sms - 1) / (2 * sms));
  s = std::max(1, std::min(s, cap));
  const size_t smem = per * s;
  const unsigned grid = static_cast<unsigned>((b + s - 1) / s);
  if (smem > 48 * 1024) {
    cudaError_t e = vec ? enable_large_smem(interaction_kernel<true>, 0)
                        : enable_large_smem(interaction_kernel<false>, 1);
    if (e != cudaSuccess) return e;
  }
  if (vec) {
    interaction_kernel<true><<<grid, kInteractThreads, smem, stream>>>(
        dense, ld_dense, emb, b, k, d, out, ld_out, copy_dense, s, use_blocks);
  } else {
    interaction_kernel<false><<<grid, kInteractThreads, smem, stream>>>(
        dense, ld_dense, emb, b, k, d, out, ld_out, copy_dense, s, 0);
  }
  return cudaGetLastError();
}

bool gather_interaction_fits(const GatherTables& tabs, int k, int d) {
  if (d % 4 != 0 || d / 4 > 4 * kWarp) return false;
  for (int t = 0; t < k; ++t)
    if (reinterpret_cast<uintptr_t>(tabs.ptr[t]) % 16 != 0) return false;
  return interaction_smem_per_sample(k, d) <= device_max_smem_optin();
}

namespace {

template <int TPB, int CHUNKS>
cudaError_t launch_gi(const GatherTables& tabs, int k, int d, const int64_t* indices,
                      const int64_t* offsets, int b, int l, const float* x, int ld_x, float* out,
                      int ld_out, int32_t* err, cudaStream_t stream) {
  // samples per block: about 72 KB of rows (three blocks per SM), at least one
  const size_t per = interaction_smem_per_sample(k, d);
  int s = static_cast<int>(std::max<size_t>(1, (72 * 1024) / per));
  const int sms = device_sm_count();
  s = std::max(1, std::min(s, (b + 2 * sms - 1) / (2 * sms)));
  const size_t smem = per * s;
  if (smem > 48 * 1024) {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (!bit || !(done.load(std::memory_order_acquire) & bit)) {
      e = cudaFuncSetAttribute(gather_interact_kernel<TPB, CHUNKS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(device_max_smem_optin()));
      if (e != cudaSuccess) return e;
      if (bit) done.fetch_or(bit, std::memory_order_acq_rel);
    }
  }
  const int use_blocks = (k + 1 >= 9) ? 1 : 0;
  const unsigned grid = static_cast<unsigned>((b + s - 1) / s);
  gather_interact_kernel<TPB, CHUNKS><<<grid, kInteractThreads, smem, stream>>>(
      tabs, k, d, indices, offsets, b, l, x, ld_x, out, ld_out, s, use_blocks, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_interaction(const GatherTables& tabs, int k, int d,
                                      const int64_t* indices, const int64_t* offsets, int b,
                                      int l, const float* x, int ld_x, float* out, int ld_out,
                                      int32_t* err, cudaStream_t stream) {
  if (b == 0) return cudaSuccess;
  const int d4 = d / 4;
#define DLRM_GI(TPB_, CH_) \
  launch_gi<TPB_, CH_>(tabs, k, d, indices, offsets, b, l, x, ld_x, out, ld_out, err, stream)
  if (d4 <= 1) return DLRM_GI(1, 1);
  if (d4 <= 2) return DLRM_GI(2, 1);
  if (d4 <= 4) return DLRM_GI(4, 1);
  if (d4 <= 8) return DLRM_GI(8, 1);
  if (d4 <= 16) return DLRM_GI(16, 1);
  if (d4 <= 32) return DLRM_GI(32, 1);
  if (d4 <= 64) return DLRM_GI(32, 2);
  return DLRM_GI(32, 4);
#undef DLRM_GI
}

cudaError_t launch_pair_map(int f, int32_t* i_out, int32_t* j_out, cudaStream_t stream) {
  const int p_count = f * (f - 1) / 2;
  if (p_count == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(std::min(1024, (p_count + 255) / 256));
  pair_map_kernel<<<grid, 256, 0, stream>>>(f, i_out, j_out);
  return cudaGetLastError();
}

}  // namespace dlrm
