// 5th-generation tensor-core (tcgen05) and mbarrier helpers shared by the
// tensor-core GEMM (gemm_tc.cu) and the fused tensor-core forward
// (fused_tc.cu). Inline PTX for sm_103a.
#pragma once

#include "common.cuh"

namespace dlrm {
namespace tc {

constexpr int kM = 128;                     // MMA rows (cta_group::1)

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

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms
// 1024 bytes apart (stride byte offset), descriptor version 1. The K step
// inside a 128-byte row advances the start address (addr >> 4 units).
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
// tf32 = 2 under kind::tf32), both K-major, N >> 3, M >> 4 (M = 128).
__host__ __device__ constexpr uint32_t instr_desc(uint32_t ab_format, int n) {
  return (1u << 4) | (ab_format << 7) | (ab_format << 10) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(kM >> 4) << 24);
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

// The mbarrier completes one arrival when every tcgen05 operation this
// thread issued before it has completed.
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

// Byte offset of 16-byte chunk `ch` of row `r` in a K-major 128B-swizzled
// tile: 8-row atoms of 1024 bytes, chunk c of row r at chunk c ^ (r % 8).
__host__ __device__ __forceinline__ int swz_offset(int r, int ch) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4);
}

}  // namespace tc
}  // namespace dlrm
