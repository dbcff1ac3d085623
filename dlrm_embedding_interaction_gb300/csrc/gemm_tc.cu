// Opt-in tensor-core Linear + bias + activation (TF32 or BF16 operands, fp32
// accumulation in TMEM) on the 5th-generation tensor cores (tcgen05).
//
// y[m][n] = act(sum_k x[m][k] * W[n][k] + bias[n]) with x (M, K) and W (N, K)
// fp32 in global memory (Luminal compare modal_ci_ready...vanilla-pytorch,
// commit message: linear_bias_(relu|sigmoid); the tensor-core mode is this
// library's opt-in, outside the fp32 parity mode).
//
// Design (sm_103a):
//  * CTA tile 128 rows x 128 columns, one tcgen05.mma.cta_group::1 of shape
//    M=128, N=128 per K step (K = 8 for tf32, 16 for bf16); the accumulator
//    (128 lanes x 128 fp32 columns) lives in tensor memory allocated with
//    tcgen05.alloc;
//  * operands are staged per 128-byte K block (32 tf32 / 64 bf16 values per
//    row) in the canonical K-major 128B-swizzled layout: 8-row atoms of
//    1024 bytes, 16-byte chunk c of row r stored at chunk c ^ (r % 8). Both x
//    and W are K-contiguous in global memory, so no transpose is needed;
//    BF16 operands are rounded from fp32 while staging (cvt.rn.bf16x2.f32),
//    TF32 operands are the fp32 words as loaded;
//  * a 3-stage ring: all 128 threads stage block kb while the MMAs of the
//    previous blocks run; one elected thread issues the four MMAs of a block
//    and tcgen05.commit's them to the stage's mbarrier, which frees the stage;
//  * epilogue: each warp reads its 32 TMEM lanes (rows) with
//    tcgen05.ld.32x32b, adds the bias, applies ReLU/sigmoid and stores.
// Every mbarrier wait is bounded (%globaltimer); on expiry the kernel sets
// its error flag, finishes without further MMAs and frees its TMEM.
#include <atomic>

#include "common.cuh"

namespace dlrm {
namespace {

constexpr int kTcThreads = 128;
constexpr int kTcM = 128;
constexpr int kTcN = 128;
constexpr int kTcStages = 3;
constexpr int kTileBytes = 128 * 128;                 // 128 rows x 128 B
constexpr int kStageBytes = 2 * kTileBytes;           // A + B
constexpr uint64_t kTcWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; false on timeout (the caller sets the error flag).
__device__ bool wait_bar(uint32_t bar, uint32_t parity) {
  if (try_wait(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  while (!try_wait(bar, parity))
    if (now_ns() - t0 > kTcWaitNs) return false;
  return true;
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFF);          // start address
  d |= static_cast<uint64_t>(1) << 16;                         // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                 // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                         // version
  d |= static_cast<uint64_t>(2) << 61;                         // 128-byte swizzle
  return d;
}

// Instruction descriptor: D fp32, A/B format (bf16 = 1 under kind::f16,
// tf32 = 2 under kind::tf32), both K-major, N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t ab_format) {
  return (1u << 4) | (ab_format << 7) | (ab_format << 10) |
         (static_cast<uint32_t>(kTcN >> 3) << 17) | (static_cast<uint32_t>(kTcM >> 4) << 24);
}

template <bool BF16>
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                    uint32_t accumulate) {
  if (BF16) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Stage rows [row0, row0+128) x one 128-byte K block of a K-contiguous fp32
// matrix into the swizzled tile. Rows >= rows or k >= k_total read as zero.
template <bool BF16>
__device__ void stage_tile(unsigned char* tile, const float* __restrict__ src, int ld, int row0,
                           int rows, int k0, int k_total, bool vec) {
  constexpr int kElems = BF16 ? 64 : 32;                 // K values per 128-byte row
  // 128 rows x 8 chunks of 16 bytes; chunk = 8 bf16 (8 floats) or 4 tf32 (4 floats)
  for (int c = threadIdx.x; c < 128 * 8; c += kTcThreads) {
    const int r = c >> 3;
    const int ch = c & 7;
    const int gr = row0 + r;
    const int kk = k0 + ch * (kElems / 8);
    float v[8];
    constexpr int n = kElems / 8;                         // floats per chunk: 8 or 4
#pragma unroll
    for (int q = 0; q < n; ++q) v[q] = 0.f;
    if (gr < rows) {
      const float* p = src + static_cast<int64_t>(gr) * ld + kk;
      if (vec && kk + n <= k_total) {
#pragma unroll
        for (int q = 0; q < n; q += 4) {
          const float4 t = __ldg(reinterpret_cast<const float4*>(p + q));
          v[q] = t.x; v[q + 1] = t.y; v[q + 2] = t.z; v[q + 3] = t.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < n; ++q)
          if (kk + q < k_total) v[q] = __ldg(p + q);
      }
    }
    uint4 word;
    if (BF16) {
      word.x = pack_bf16x2(v[0], v[1]);
      word.y = pack_bf16x2(v[2], v[3]);
      word.z = pack_bf16x2(v[4], v[5]);
      word.w = pack_bf16x2(v[6], v[7]);
    } else {
      word.x = __float_as_uint(v[0]);
      word.y = __float_as_uint(v[1]);
      word.z = __float_as_uint(v[2]);
      word.w = __float_as_uint(v[3]);
    }
    const int dst = (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4);
    *reinterpret_cast<uint4*>(tile + dst) = word;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tc_kernel(const float* __restrict__ x, int ldx, const float* __restrict__ w, int ldw,
               const float* __restrict__ bias, float* __restrict__ y, int ldy, int m, int n, int k,
               int act, int vec_x, int vec_w, int32_t* err) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte alignment for the swizzle atoms
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* stages = base;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kTcStages * kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kTcStages + 1);
  const int warp = threadIdx.x / kWarp;
  const int lane = threadIdx.x % kWarp;
  const int m0 = blockIdx.x * kTcM;
  const int n0 = blockIdx.y * kTcN;
  constexpr int kBlockK = BF16 ? 64 : 32;
  constexpr int kStepK = BF16 ? 16 : 8;                   // K per MMA
  constexpr uint32_t kIdesc = instr_desc(BF16 ? 1u : 2u);
  const int kb_count = (k + kBlockK - 1) / kBlockK;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "n"(kTcN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s <= kTcStages; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bars[s])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  for (int kb = 0; kb < kb_count; ++kb) {
    const int s = kb % kTcStages;
    if (kb >= kTcStages && ok) {
      // the MMAs that read this stage kTcStages blocks ago must be done
      ok = wait_bar(smem_addr(&bars[s]), ((kb / kTcStages) - 1) & 1);
    }
    unsigned char* a_tile = stages + s * kStageBytes;
    unsigned char* b_tile = a_tile + kTileBytes;
    stage_tile<BF16>(a_tile, x, ldx, m0, m, kb * kBlockK, k, vec_x != 0);
    stage_tile<BF16>(b_tile, w, ldw, n0, n, kb * kBlockK, k, vec_w != 0);
    // generic-proxy writes -> visible to the tensor core's async proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0 && ok) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint64_t da = smem_desc(smem_addr(a_tile));
      const uint64_t db = smem_desc(smem_addr(b_tile));
#pragma unroll
      for (int j = 0; j < kBlockK / kStepK; ++j) {
        // advance the start address by 32 bytes per K step inside the atom
        const uint64_t off = static_cast<uint64_t>((j * 32) >> 4);
        mma<BF16>(tmem, da + off, db + off, kIdesc, (kb > 0 || j > 0) ? 1u : 0u);
      }
      mma_commit(smem_addr(&bars[s]));
    }
  }
  // all MMAs done: the last commit's stage barrier
  if (kb_count > 0 && ok) {
    const int last = kb_count - 1;
    ok = wait_bar(smem_addr(&bars[last % kTcStages]), (last / kTcStages) & 1);
  }
  if (!ok && threadIdx.x == 0 && err) atomicOr(reinterpret_cast<unsigned int*>(err), DLRM_ERRBIT_TIMEOUT);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  // Epilogue: warp w owns TMEM lanes (rows) 32w .. 32w+31.
  const int row = m0 + warp * 32 + lane;
  for (int c0 = 0; c0 < kTcN; c0 += 8) {
    uint32_t r[8];
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    if (row < m && ok) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int col = n0 + c0 + q;
        if (col < n) {
          const float bv = bias ? __ldg(bias + col) : 0.f;
          y[static_cast<int64_t>(row) * ldy + col] = apply_act(__uint_as_float(r[q]) + bv, act);
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTcN)
                 : "memory");
  }
}

template <bool BF16>
cudaError_t enable_tc_smem(size_t bytes) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(gemm_tc_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes));
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace

size_t gemm_tc_smem_bytes() {
  return 1024 + static_cast<size_t>(kTcStages) * kStageBytes + (kTcStages + 1) * 8 + 16;
}

cudaError_t launch_linear_tc(const float* x, int ld_x, const float* w, int ld_w, const float* bias,
                             float* y, int ld_y, int m, int n, int k, int act, bool bf16,
                             int32_t* err, cudaStream_t stream) {
  if (m == 0) return cudaSuccess;
  auto aligned = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
  const int vec_x = (ld_x % 4 == 0 && aligned(x)) ? 1 : 0;
  const int vec_w = (ld_w % 4 == 0 && aligned(w)) ? 1 : 0;
  const size_t smem = gemm_tc_smem_bytes();
  const dim3 grid((m + kTcM - 1) / kTcM, (n + kTcN - 1) / kTcN);
  cudaError_t e = bf16 ? enable_tc_smem<true>(smem) : enable_tc_smem<false>(smem);
  if (e != cudaSuccess) return e;
  if (bf16)
    gemm_tc_kernel<true><<<grid, kTcThreads, smem, stream>>>(x, ld_x, w, ld_w, bias, y, ld_y, m,
                                                             n, k, act, vec_x, vec_w, err);
  else
    gemm_tc_kernel<false><<<grid, kTcThreads, smem, stream>>>(x, ld_x, w, ld_w, bias, y, ld_y, m,
                                                              n, k, act, vec_x, vec_w, err);
  return cudaGetLastError();
}

}  // namespace dlrm
