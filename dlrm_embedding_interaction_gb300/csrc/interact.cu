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
// (gram_block), a quarter of the shared-memory reads of one pair per thread;
// when the block's samples have too few such blocks for its threads, each
// block is split over two adjacent lanes (alternate 16-byte chunks of D, one
// shuffle to add).
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
  pdl_wait();     // launched after the previous kernel may still run
  pdl_trigger();

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
  if (VEC && use_blocks == 2) {
    // 4 x 4 register blocks of pairs, each over half of D (alternate 16-byte
    // chunks) on two adjacent lanes (w = 2 task + half), added with one
    // shuffle per dot: twice the tasks when a block's samples have too few
    // blocks for its threads
    const int d4 = d / 4;
    const int total = ns * nblk * 2;
    for (int base = 0; base < total; base += blockDim.x) {   // uniform per warp
      const int w = base + tid;
      const bool active = w < total;
      const int task = active ? (w >> 1) : 0;
      const int half = w & 1;
      const int s = task / nblk;
      const int q = task - s * nblk;
      const float* zsam = zs + s * f * ldz;
      int ii, jj;
      pair_from_index(q, ii, jj);
      const int bi = ii - 1, bj = jj;
      const float* ri[4];
      const float* rj[4];
      const int nb = (f + 3) / 4;   // rows dealt by residue class (gram_block)
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        ri[a] = zsam + min(bi + a * nb, f - 1) * ldz;
        rj[a] = zsam + min(bj + a * nb, f - 1) * ldz;
      }
      float acc[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
      // the two halves take alternate 16-byte chunks of the rows: the pair's
      // loads fall in adjacent bank groups instead of colliding
      const int c_end = active ? d4 : 0;
      for (int c4 = half; c4 < c_end; c4 += 2) {
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
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] += __shfl_xor_sync(0xffffffffu, acc[a][c], 1);
      if (active && half == 0) {
        float* o = out + static_cast<int64_t>(b0 + s) * ld_out + col0;
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int q2 = gram_block_pair(f, bi, bj, a, c);
            if (q2 >= 0) o[q2] = acc[a][c];
          }
      }
    }
  } else if (VEC && use_blocks) {
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
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int q2 = gram_block_pair(f, bi, bj, a, c);
          if (q2 >= 0) o[q2] = acc[a][c];
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
  // half-D tasks on lane pairs when the block's pair blocks would leave more
  // than a third of its threads idle (wide D only: each half keeps >= 8 steps)
  int mode = use_blocks;
  if (use_blocks && s * blocks4 * 3 < 2 * kInteractThreads && d >= 64) mode = 2;
  const size_t smem = per * s;
  const unsigned grid = static_cast<unsigned>((b + s - 1) / s);
  if (smem > 48 * 1024) {
    cudaError_t e = vec ? enable_large_smem(interaction_kernel<true>, 0)
                        : enable_large_smem(interaction_kernel<false>, 1);
    if (e != cudaSuccess) return e;
  }
  if (vec)
    return launch_pdl(interaction_kernel<true>, dim3(grid), dim3(kInteractThreads), smem, stream,
                      dense, ld_dense, emb, b, k, d, out, ld_out, copy_dense, s, mode);
  return launch_pdl(interaction_kernel<false>, dim3(grid), dim3(kInteractThreads), smem, stream,
                    dense, ld_dense, emb, b, k, d, out, ld_out, copy_dense, s, 0);
}

cudaError_t launch_pair_map(int f, int32_t* i_out, int32_t* j_out, cudaStream_t stream) {
  const int p_count = f * (f - 1) / 2;
  if (p_count == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(std::min(1024, (p_count + 255) / 256));
  pair_map_kernel<<<grid, 256, 0, stream>>>(f, i_out, j_out);
  return cudaGetLastError();
}

}  // namespace dlrm
