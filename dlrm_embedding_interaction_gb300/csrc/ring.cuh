// Device helpers of the persistent kernels that stream packed weights
// through a ring of shared-memory stages (fused.cu, fused_cluster.cu):
// mbarrier operations, 1-D bulk async copies, cp.async, bounded waits, and
// the ring's producer. Everything is internal to the including translation
// unit (anonymous namespace).
#pragma once

#include "common.cuh"

namespace dlrm {
namespace {

// Floats of one ring stage (32 KB).
constexpr int kRingStageFloats = 8192;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// As mbar_try_wait, but the thread may be suspended (not issuing) for up to
// `ns` nanoseconds while the phase is incomplete; it resumes when the phase
// completes or the hint runs out.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src));
}

// 16 zero bytes (src-size 0: nothing is read from src).
__device__ __forceinline__ void cp_async16_zero(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 0;\n" ::"r"(smem_u32(dst)), "l"(src));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <int CW>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(CW * kWarp) : "memory");
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity. Returns false when this or
// another thread gave up (abort raised); the caller then carries on without
// the data so every named barrier is still reached. SPIN: poll without
// suspending (computing warps, whose next stage is usually moments away);
// otherwise the thread sleeps in the barrier between polls (the producer,
// which shares a sub-partition with computing warps).
constexpr uint32_t kSuspendNs = 20000;
template <bool SPIN>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int32_t* err, uint64_t limit_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  if (*abort_flag) return false;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (SPIN ? mbar_test_wait(bar, parity) : mbar_try_wait_suspend(bar, parity, kSuspendNs))
      return true;
    if (!SPIN || (i & 63) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        if (err) atomicOr(reinterpret_cast<unsigned int*>(err), DLRM_ERRBIT_TIMEOUT);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- weight ring

// The weight stream flows through a ring of s_count stages: stream stage j
// lands in slot j % s_count, full[slot] completes when its bytes have arrived
// and empty[slot] when all CW computing warps are done with it. The producer
// warp walks the stage table, waiting on empty before refilling a slot; it
// runs ahead across layer boundaries.
struct Ring {
  float* stages;
  uint64_t* full;
  uint64_t* empty;
  volatile int* abort_flag;
  uint32_t s_count;
  int32_t* err;
  uint64_t limit_ns;   // bound of every wait
};

// A consumer's place in the stream: the slot of its next stage (stage % S)
// and that stage's full-barrier parity ((stage / S) & 1), advanced in step
// rather than divided out per stage.
struct RingPos {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void advance(uint32_t s_count) {
    if (++slot == s_count) {
      slot = 0;
      phase ^= 1;
    }
  }
};

// The warp is done with the stage in `slot`.
__device__ __forceinline__ void ring_release(const Ring& r, uint32_t slot) {
  __syncwarp();
  if ((threadIdx.x % kWarp) == 0) mbar_arrive(smem_u32(&r.empty[slot]));
}

// Bring this CTA's 1/gridDim share of the weight stream (16-byte granules)
// into L2 at kernel start: every CTA then finds each stage in L2, and a
// stage consumed faster than HBM latency does not stall the ring.
__device__ void prefetch_stream_l2(const float* wstream, size_t floats) {
  const size_t granules = floats / 4;
  const size_t per = (granules + gridDim.x - 1) / gridDim.x;
  const size_t g0 = per * blockIdx.x;
  if (g0 >= granules) return;
  size_t left = (granules - g0 < per ? granules - g0 : per) * 16;
  const char* src = reinterpret_cast<const char*>(wstream) + g0 * 16;
  while (left > 0) {
    const uint32_t chunk = static_cast<uint32_t>(left < 65536 ? left : 65536);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(chunk) : "memory");
    src += chunk;
    left -= chunk;
  }
}

// Issuing lanes of the producer warp. One thread's bulk copies run one after
// another at about 45 GB/s, while several threads' copies overlap (four reach
// ~150 GB/s per SM). So every stage is cut into kIssuers pieces, one per
// lane, and lands about four times sooner than from a single thread. The
// lanes stay converged on one stage at a time: they wait on the same empty
// barrier, lane 0 posts the stage's byte count on its full barrier, then each
// lane copies its piece (complete_tx on that barrier).
constexpr uint32_t kIssuers = 4;
constexpr unsigned kIssuerMask = (1u << kIssuers) - 1;

// The stage table runs once per tile of the CTA (n_tiles passes). With
// withhold_last (failure-detection tests) the stream's last stage is never
// copied: the computing warps' wait on it runs out.
__device__ void produce(const Ring& r, const float* wstream, const uint2* tab, uint32_t n_tab,
                        uint32_t n_tiles, bool withhold_last) {
  const uint32_t lane = threadIdx.x % kWarp;
  if (lane >= kIssuers) return;
  const char* src0 = reinterpret_cast<const char*>(wstream);
  const uint32_t n_stages = n_tab * n_tiles;
  uint32_t j = 0, slot = 0, phase = 0;   // slot = j % S, phase = (j / S) & 1
  uint32_t jt = 0;                       // j % n_tab
  for (; j < n_stages; ++j) {
    const bool ok = j < r.s_count || wait_phase<false>(smem_u32(&r.empty[slot]), phase ^ 1,
                                                         r.abort_flag, r.err, r.limit_ns);
    if (!__all_sync(kIssuerMask, ok)) break;
    if (withhold_last && j + 1 == n_stages) break;   // not issued: not drained below
    const uint2 e = __ldg(tab + jt);
    if (++jt == n_tab) jt = 0;
    const uint32_t full = smem_u32(&r.full[slot]);
    if (lane == 0) mbar_arrive_expect_tx(full, e.y);
    __syncwarp(kIssuerMask);
    const uint32_t piece = (e.y / 16 + kIssuers - 1) / kIssuers * 16;
    const uint32_t off = lane * piece;
    if (off < e.y)
      bulk_g2s(smem_u32(r.stages + slot * kRingStageFloats) + off,
               src0 + static_cast<size_t>(e.x) * sizeof(float) + off, min(piece, e.y - off), full);
    if (++slot == r.s_count) {
      slot = 0;
      phase ^= 1;
    }
  }
  // Copies still in flight must land before the CTA's shared memory is
  // released: wait (bounded, regardless of abort) for the stages issued
  // within the last ring.
  const uint32_t first = j > r.s_count ? j - r.s_count : 0;
  for (uint32_t q = first; q < j; ++q) {
    const uint32_t bar = smem_u32(&r.full[q % r.s_count]);
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, (q / r.s_count) & 1)) {
      if (global_ns() - t0 > r.limit_ns) {
        if (r.err) atomicOr(reinterpret_cast<unsigned int*>(r.err), DLRM_ERRBIT_TIMEOUT);
        break;
      }
    }
  }
}

}  // namespace
}  // namespace dlrm
