// Opt-in tensor-core Linear + bias + activation on the 5th-generation tensor
// cores (tcgen05): TF32 or BF16 operands, or split TF32 (3xTF32), with fp32
// accumulation in tensor memory.
//
// y[m][n] = act(sum_k x[m][k] * W[n][k] + bias[n]) with x (M, K) and W (N, K)
// fp32 in global memory (Luminal compare modal_ci_ready...vanilla-pytorch,
// commit message: linear_bias_(relu|sigmoid); the tensor-core modes are this
// library's opt-in, outside the fp32 parity mode).
//
// Design (sm_103a):
//  * CTA tile 128 rows x NT columns (NT = 128, or 64 when 128 would leave
//    the GPU short of one wave of tiles); one tcgen05.mma.cta_group::1 of
//    shape M=128, N=NT per K step (K = 8 for tf32, 16 for bf16) into an
//    accumulator of 128 lanes x NT fp32 columns in tensor memory;
//  * operands are staged per 128-byte K block (32 tf32 / 64 bf16 values per
//    row) in the canonical K-major 128B-swizzled layout (8-row atoms of 1024
//    bytes, 16-byte chunk c of row r at chunk c ^ (r % 8)); x and W are both
//    K-contiguous, so no transpose is needed;
//  * TF32 with 16-byte aligned rows: a 4-stage cp.async ring lands blocks
//    kb+1 and kb+2 while the MMAs of block kb run; a stage is refilled only
//    after tcgen05.commit of the MMAs that read it (two blocks earlier) has
//    arrived on its mbarrier. BF16 (rounded from fp32 while staging) and unaligned TF32
//    stage through registers;
//  * 3xTF32: each staged fp32 value v is split into hi = v with the low 13
//    mantissa bits cleared (exact as tf32) and lo = v - hi (exact in fp32);
//    three MMAs hi*hi + hi*lo + lo*hi accumulate a product whose error is
//    about 2^-21 relative, inside the fp32 parity tolerance;
//  * epilogue: each warp reads its 32 TMEM lanes (rows) with tcgen05.ld
//    32x32b, adds the bias, applies ReLU/sigmoid and stores.
// Every mbarrier wait is bounded (%globaltimer; 2 s unless the launch sets
// another limit); on expiry the kernel sets its error flag, stops issuing
// MMAs, waits (bounded) for the MMAs it issued and still frees its TMEM.
#include <atomic>

#include "common.cuh"
#include "tc.cuh"

namespace dlrm {
namespace {

using namespace tc;

constexpr int kTcThreads = 128;
constexpr int kTcM = tc::kM;

enum TcMode { kTF32 = 0, kBF16 = 1, kTF32x3 = 2 };

// Bounded wait; false on timeout (the caller sets the error flag).
__device__ bool wait_bar(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (try_wait(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  while (!try_wait(bar, parity))
    if (now_ns() - t0 > limit_ns) return false;
  return true;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// Asynchronous staging of rows [row0, row0+rows_tile) x one 128-byte K block
// of fp32 (tf32) values; rows >= rows or k >= k_total are zero-filled.
__device__ void stage_async(unsigned char* tile, int rows_tile, const float* __restrict__ src,
                            int ld, int row0, int rows, int k0, int k_total) {
  for (int c = threadIdx.x; c < rows_tile * 8; c += kTcThreads) {
    const int r = c >> 3;
    const int ch = c & 7;
    const int gr = row0 + r;
    const int kk = k0 + ch * 4;
    int bytes = 0;
    const float* p = src;
    if (gr < rows && kk < k_total) {
      p = src + static_cast<int64_t>(gr) * ld + kk;
      bytes = (k_total - kk >= 4) ? 16 : 4 * (k_total - kk);
    }
    cp_async16(smem_addr(tile + swz_offset(r, ch)), p, bytes);
  }
}

// Register staging (BF16, or rows that are not 16-byte aligned).
template <bool BF16>
__device__ void stage_regs(unsigned char* tile, int rows_tile, const float* __restrict__ src,
                           int ld, int row0, int rows, int k0, int k_total, bool vec) {
  constexpr int n = BF16 ? 8 : 4;                         // values per 16-byte chunk
  for (int c = threadIdx.x; c < rows_tile * 8; c += kTcThreads) {
    const int r = c >> 3;
    const int ch = c & 7;
    const int gr = row0 + r;
    const int kk = k0 + ch * n;
    float v[8];
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
    *reinterpret_cast<uint4*>(tile + swz_offset(r, ch)) = word;
  }
}

// 3xTF32: split a staged fp32 tile in place into hi (low 13 mantissa bits
// cleared) and write lo = v - hi into `lo_tile` (same layout).
__device__ void split_tf32(unsigned char* tile, unsigned char* lo_tile, int bytes) {
  for (int off = threadIdx.x * 16; off < bytes; off += kTcThreads * 16) {
    uint4 v = *reinterpret_cast<uint4*>(tile + off);
    uint4 hi, lo;
    hi.x = v.x & 0xFFFFE000u; lo.x = __float_as_uint(__uint_as_float(v.x) - __uint_as_float(hi.x));
    hi.y = v.y & 0xFFFFE000u; lo.y = __float_as_uint(__uint_as_float(v.y) - __uint_as_float(hi.y));
    hi.z = v.z & 0xFFFFE000u; lo.z = __float_as_uint(__uint_as_float(v.z) - __uint_as_float(hi.z));
    hi.w = v.w & 0xFFFFE000u; lo.w = __float_as_uint(__uint_as_float(v.w) - __uint_as_float(hi.w));
    *reinterpret_cast<uint4*>(tile + off) = hi;
    *reinterpret_cast<uint4*>(lo_tile + off) = lo;
  }
}

template <int MODE, int NT>
struct TcLayout {
  static constexpr int kA = kTcM * 128;                  // A tile bytes
  static constexpr int kB = NT * 128;                    // B tile bytes
  static constexpr int kParts = MODE == kTF32x3 ? 2 : 1; // hi (+ lo)
  static constexpr int kStage = kParts * (kA + kB);
  // 4 stages (prefetch distance 2, refill waits on MMAs two blocks old);
  // 3 where four would not fit (3xTF32 with 128-column tiles)
  static constexpr int kStages = (4 * kStage + 2048 <= 227 * 1024) ? 4 : 3;
  static constexpr int kSmem = 1024 + kStages * kStage + (kStages + 1) * 8 + 16;
};

template <int MODE, int NT>
__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tc_kernel(const float* __restrict__ x, int ldx, const float* __restrict__ w, int ldw,
               const float* __restrict__ bias, float* __restrict__ y, int ldy, int m, int n, int k,
               int act, int vec_x, int vec_w, int32_t* err, WaitCfg wait) {
  using Lay = TcLayout<MODE, NT>;
  constexpr int kStages = Lay::kStages;
  constexpr bool BF16 = MODE == kBF16;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* stages = base;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kStages * Lay::kStage);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kStages + 1);
  const int warp = threadIdx.x / kWarp;
  const int lane = threadIdx.x % kWarp;
  const int m0 = blockIdx.x * kTcM;
  const int n0 = blockIdx.y * NT;
  constexpr int kBlockK = BF16 ? 64 : 32;
  constexpr int kStepK = BF16 ? 16 : 8;
  constexpr uint32_t kIdesc = instr_desc(BF16 ? 1u : 2u, NT);
  const int kb_count = (k + kBlockK - 1) / kBlockK;
  const bool async = !BF16 && vec_x && vec_w;
  const uint64_t limit = wait_limit_ns(wait);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "n"(NT)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s <= kStages; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bars[s])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  auto a_tile = [&](int s) { return stages + s * Lay::kStage; };
  auto b_tile = [&](int s) { return stages + s * Lay::kStage + Lay::kA; };
  auto stage_block = [&](int kb) {
    const int s = kb % kStages;
    if (async) {
      stage_async(a_tile(s), kTcM, x, ldx, m0, m, kb * kBlockK, k);
      stage_async(b_tile(s), NT, w, ldw, n0, n, kb * kBlockK, k);
    } else {
      stage_regs<BF16>(a_tile(s), kTcM, x, ldx, m0, m, kb * kBlockK, k, vec_x != 0);
      stage_regs<BF16>(b_tile(s), NT, w, ldw, n0, n, kb * kBlockK, k, vec_w != 0);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };

  bool ok = true;
  // prologue: blocks 0 and 1 in flight; exactly two commit groups either way,
  // so that "all but the 2 most recent groups" below always means block kb
  for (int kb = 0; kb < 2; ++kb) {
    if (kb < kb_count) stage_block(kb);
    else asm volatile("cp.async.commit_group;\n" ::: "memory");
  }
  for (int kb = 0; kb < kb_count; ++kb) {
    const int s = kb % kStages;
    // refill for block kb+2 the stage that block kb+2-kStages used: wait for
    // the MMAs of that older block (kStages - 2 iterations back)
    if (kb + 2 < kb_count) {
      const int old = kb + 2 - kStages;
      if (old >= 0 && ok)
        ok = wait_bar(smem_addr(&bars[old % kStages]), (old / kStages) & 1, limit);
      stage_block(kb + 2);
    } else {
      asm volatile("cp.async.commit_group;\n" ::: "memory");
    }
    asm volatile("cp.async.wait_group 2;\n" ::: "memory");   // block kb has landed
    if (MODE == kTF32x3) {
      __syncthreads();
      unsigned char* lo = stages + s * Lay::kStage + Lay::kA + Lay::kB;
      split_tf32(a_tile(s), lo, Lay::kA);
      split_tf32(b_tile(s), lo + Lay::kA, Lay::kB);
    }
    // generic-proxy writes -> visible to the tensor core's async proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0 && ok) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint64_t da = smem_desc(smem_addr(a_tile(s)));
      const uint64_t db = smem_desc(smem_addr(b_tile(s)));
#pragma unroll
      for (int j = 0; j < kBlockK / kStepK; ++j) {
        // advance the start address by 32 bytes per K step inside the atom
        const uint64_t off = static_cast<uint64_t>((j * 32) >> 4);
        const uint32_t acc0 = (kb > 0 || j > 0) ? 1u : 0u;
        mma<BF16>(tmem, da + off, db + off, kIdesc, acc0);
        if (MODE == kTF32x3) {
          const uint64_t la = smem_desc(smem_addr(stages + s * Lay::kStage + Lay::kA + Lay::kB));
          const uint64_t lb = smem_desc(smem_addr(stages + s * Lay::kStage + 2 * Lay::kA + Lay::kB));
          mma<false>(tmem, da + off, lb + off, kIdesc, 1u);   // hi * lo
          mma<false>(tmem, la + off, db + off, kIdesc, 1u);   // lo * hi
        }
      }
      // failure-detection tests: the last block's commit is withheld, so
      // the wait on it below runs out
      if (!(wait.withhold_last && kb + 1 == kb_count)) mma_commit(smem_addr(&bars[s]));
    }
  }
  // all MMAs done: the last commit's stage barrier
  if (kb_count > 0 && ok) {
    const int last = kb_count - 1;
    ok = wait_bar(smem_addr(&bars[last % kStages]), (last / kStages) & 1, limit);
  }
  if (!ok && threadIdx.x == 0 && err) atomicOr(reinterpret_cast<unsigned int*>(err), DLRM_ERRBIT_TIMEOUT);
  // After a wait gave up, MMAs may still be running: before the tensor memory
  // is read or freed, thread 0 commits once more on the spare barrier (one
  // phase: its parity is unambiguous), which tracks every MMA it issued, and
  // waits for it (bounded); the others meet it at the barrier below.
  if (!ok && threadIdx.x == 0) {
    mma_commit(smem_addr(&bars[kStages]));
    wait_bar(smem_addr(&bars[kStages]), 0, limit);
  }
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  // Epilogue: warp w owns TMEM lanes (rows) 32w .. 32w+31.
  const int row = m0 + warp * 32 + lane;
  for (int c0 = 0; c0 < NT; c0 += 8) {
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
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(NT)
                 : "memory");
  }
}

template <int MODE, int NT>
cudaError_t launch_mode(const float* x, int ld_x, const float* w, int ld_w, const float* bias,
                        float* y, int ld_y, int m, int n, int k, int act, int vec_x, int vec_w,
                        int32_t* err, cudaStream_t stream, WaitCfg wait) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  constexpr int kSmem = TcLayout<MODE, NT>::kSmem;
  if (!bit || !(done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_tc_kernel<MODE, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmem);
    if (e != cudaSuccess) return e;
    if (bit) done.fetch_or(bit, std::memory_order_acq_rel);
  }
  const dim3 grid((m + kTcM - 1) / kTcM, (n + NT - 1) / NT);
  gemm_tc_kernel<MODE, NT><<<grid, kTcThreads, kSmem, stream>>>(x, ld_x, w, ld_w, bias, y, ld_y,
                                                                m, n, k, act, vec_x, vec_w, err,
                                                                wait);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_tiles(const float* x, int ld_x, const float* w, int ld_w, const float* bias,
                         float* y, int ld_y, int m, int n, int k, int act, int vec_x, int vec_w,
                         int32_t* err, cudaStream_t stream, WaitCfg wait) {
  const int64_t tiles128 = static_cast<int64_t>((m + kTcM - 1) / kTcM) * ((n + 127) / 128);
  if (tiles128 >= device_sm_count() || n <= 64)
    return n <= 64 ? launch_mode<MODE, 64>(x, ld_x, w, ld_w, bias, y, ld_y, m, n, k, act, vec_x,
                                           vec_w, err, stream, wait)
                   : launch_mode<MODE, 128>(x, ld_x, w, ld_w, bias, y, ld_y, m, n, k, act, vec_x,
                                            vec_w, err, stream, wait);
  return launch_mode<MODE, 64>(x, ld_x, w, ld_w, bias, y, ld_y, m, n, k, act, vec_x, vec_w, err,
                               stream, wait);
}

}  // namespace

cudaError_t launch_linear_tc(const float* x, int ld_x, const float* w, int ld_w, const float* bias,
                             float* y, int ld_y, int m, int n, int k, int act, int mode,
                             int32_t* err, cudaStream_t stream, WaitCfg wait) {
  if (m == 0) return cudaSuccess;
  auto aligned = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
  const int vec_x = (ld_x % 4 == 0 && aligned(x)) ? 1 : 0;
  const int vec_w = (ld_w % 4 == 0 && aligned(w)) ? 1 : 0;
  switch (mode) {
    case DLRM_MATH_BF16:
      return launch_tiles<kBF16>(x, ld_x, w, ld_w, bias, y, ld_y, m, n, k, act, vec_x, vec_w, err,
                                 stream, wait);
    case DLRM_MATH_TF32X3:
      return launch_tiles<kTF32x3>(x, ld_x, w, ld_w, bias, y, ld_y, m, n, k, act, vec_x, vec_w,
                                   err, stream, wait);
    default:
      return launch_tiles<kTF32>(x, ld_x, w, ld_w, bias, y, ld_y, m, n, k, act, vec_x, vec_w, err,
                                 stream, wait);
  }
}

}  // namespace dlrm
