// Fused single-launch DLRMv1 forward on the 5th-generation tensor cores:
// the opt-in TF32 and BF16 modes (fp32 accumulation in tensor memory).
//
// The forward is the fused fp32 forward's (Luminal compare
// dlrm-fused-kernels...dlrm-pt2-megakernel, dlrm_megakernel.rs steps 1-6:
// bottom Linear+ReLU on every layer, lookups, i-major pairwise dots with
// Vec[0] = x, R = [x, z], top Linear+ReLU then Linear+sigmoid); the MLP
// GEMMs run as tcgen05.mma with the layer's weights as the A operand.
//
// One CTA per tile of 16 samples:
//  * every GEMM layer computes C^T = W X^T: M = 128 output features per
//    M-tile, N = 16 samples, K in 128-byte blocks (32 tf32 / 64 bf16), four
//    MMAs of 32 bytes of K per block. Each (M-tile, K step) pair has its own
//    16 accumulator columns in tensor memory (lane = output feature) and the
//    tiles arrive K-block-major, so consecutive MMAs are independent; the
//    epilogue adds the four K-step partial sums of each M-tile.
//  * the weights of all layers form one stream of 16 KB tiles (128 rows x
//    128 bytes, K-major, 128-byte swizzle), pre-packed at create time and
//    streamed by a producer warp through a ring of bulk async copies; the
//    MMA warp releases a ring slot with tcgen05.commit once its MMAs ran.
//  * the activations (the B operand) stay in shared memory in the same
//    swizzled K-major layout, ping-ponging between two buffers.
//  * four epilogue warps (one per 32-lane quarter of tensor memory) read
//    the accumulators with tcgen05.ld, add the bias, apply ReLU and write the
//    next layer's operand; at kernel start they check the bags and write the
//    dense rows as layer 0's operand in one round of global loads, signal the
//    MMA warp, then fetch the bag rows (cp.async for bags of one row, sums in
//    registers for longer bags); they compute the pair dots into R (fp32,
//    from an fp32 copy of x) and the last layer's fp32 dot and sigmoid.
// Every wait is bounded (%globaltimer; 2 s unless the launch sets another
// limit): on expiry the kernel sets DLRM_ERRBIT_TIMEOUT, stops issuing and
// waiting, waits (bounded) for its copies in flight and for every MMA it
// issued, and still frees its tensor memory.
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "fused_tc.cuh"
#include "tc.cuh"

namespace dlrm {
namespace {

using namespace tc;

constexpr int kEpiWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * kWarp;
constexpr int kActBlock = kTcTile * 128;           // one K-block of the B operand (bytes)

// Phase stamps and wait timers exist only in the TRACE instances (launched
// while a trace buffer is set), so the plain instances carry no trace code.
template <bool TRACE>
__device__ __forceinline__ void stamp(const FusedTcParams& p, int slot) {
  if (TRACE && p.trace && threadIdx.x == 0)
    p.trace[static_cast<size_t>(blockIdx.x) * kTcTraceSlots + slot] = now_ns();
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

// Non-blocking probe of the phase (no suspension): the waits below spin on
// it, so a completed phase is seen within a few cycles.
__device__ __forceinline__ bool test_wait(uint32_t bar, uint32_t parity) {
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

// Like test_wait, but a thread whose phase is incomplete may be suspended in
// the barrier (up to the hint) instead of issuing: for waiters that share an
// SM sub-partition with the MMA-issuing thread.
__device__ __forceinline__ bool try_wait_suspend(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

// Bounded wait; false when this or another thread gave up (abort raised).
// SPIN: poll without suspending (the MMA thread's critical path); otherwise
// sleep in the barrier between polls.
template <bool SPIN>
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                             int32_t* err, uint64_t limit_ns) {
  if (test_wait(bar, parity)) return true;
  if (*abort_flag) return false;
  const uint64_t t0 = now_ns();
  for (uint32_t i = 1;; ++i) {
    if (SPIN ? test_wait(bar, parity) : try_wait_suspend(bar, parity)) return true;
    if (!SPIN || (i & 63) == 0) {
      if (*abort_flag) return false;
      if (now_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        if (err) atomicOr(reinterpret_cast<unsigned int*>(err), DLRM_ERRBIT_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_addr(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * kWarp) : "memory");
}

// Element (sample s, feature f) of a B-operand buffer: K-block f / KB, then
// the swizzled 16-byte chunk of row s.
template <bool BF16>
__device__ __forceinline__ void put_operand(unsigned char* buf, int s, int f, float v) {
  constexpr int KB = BF16 ? 64 : 32;
  constexpr int ESZ = BF16 ? 2 : 4;
  const int e = f % KB;
  unsigned char* q = buf + (f / KB) * kActBlock + swz_offset(s, (e * ESZ) >> 4) + ((e * ESZ) & 15);
  if (BF16) {
    *reinterpret_cast<uint16_t*>(q) = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
  } else {
    *reinterpret_cast<float*>(q) = v;
  }
}

// Zeros features [f0, f1) of every sample of a B-operand buffer: the 16-byte
// chunks wholly inside the range by one vector store each, the partial
// chunks at either end element by element.
template <bool BF16>
__device__ void zero_operand(unsigned char* buf, int f0, int f1, int tid, int nthreads) {
  constexpr int EPC = BF16 ? 8 : 4;             // elements per 16-byte chunk
  constexpr int KB = BF16 ? 64 : 32;
  const int c0 = (f0 + EPC - 1) / EPC, c1 = f1 / EPC;   // whole chunks [c0, c1)
  if (c0 >= c1) {
    const int w = f1 - f0;
    const float rw = __frcp_rn(static_cast<float>(max(w, 1)));
    for (int e = tid; e < kTcTile * w; e += nthreads) {
      const int s = quot(e, w, rw);
      put_operand<BF16>(buf, s, f0 + (e - s * w), 0.f);
    }
    return;
  }
  const int head = c0 * EPC - f0, tail = f1 - c1 * EPC;
  const int ht = head + tail;
  const float rht = __frcp_rn(static_cast<float>(max(ht, 1)));
  for (int e = tid; e < kTcTile * ht; e += nthreads) {
    const int s = quot(e, ht, rht), q = e - s * ht;
    put_operand<BF16>(buf, s, q < head ? f0 + q : c1 * EPC + (q - head), 0.f);
  }
  const int nch = c1 - c0;
  const float rnch = __frcp_rn(static_cast<float>(nch));
  for (int e = tid; e < kTcTile * nch; e += nthreads) {
    const int s = quot(e, nch, rnch), c = c0 + (e - s * nch);   // chunk c of the feature axis
    const int f = c * EPC;
    *reinterpret_cast<uint4*>(buf + (f / KB) * kActBlock + swz_offset(s, (f % KB) * (BF16 ? 2 : 4) >> 4)) =
        make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---------------------------------------------------------------- roles


// Lanes 0 .. kIssuers-1 of the producer warp copy every stream tile in
// kIssuers pieces: one thread's bulk copies run one after another at about
// 45 GB/s, while several threads' copies overlap (four reach ~150 GB/s per
// SM), so a tile lands about four times sooner than from one thread. The
// lanes stay converged on one tile at a time: they wait on the same empty
// barrier, lane 0 posts the tile's bytes on its full barrier, then each lane
// copies its quarter.
constexpr int kIssuers = 4;
constexpr unsigned kIssuerMask = (1u << kIssuers) - 1;

__device__ void produce(const FusedTcParams& p, unsigned char* ring, uint64_t* full,
                        uint64_t* empty, volatile int* abort_flag) {
  const int lane = threadIdx.x % kWarp;
  // this CTA's share of the stream into L2, from a lane that issues no copies
  // (a thread's bulk operations run one after another)
  if (lane == kWarp - 1) {
    const size_t bytes = static_cast<size_t>(p.n_tiles) * kTcTileBytes;
    const size_t per = ((bytes / 16 + gridDim.x - 1) / gridDim.x) * 16;
    const size_t b0 = per * blockIdx.x;
    if (b0 < bytes) {
      size_t left = bytes - b0 < per ? bytes - b0 : per;
      const unsigned char* src = p.wstream + b0;
      while (left > 0) {
        const uint32_t chunk = static_cast<uint32_t>(left < 65536 ? left : 65536);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(chunk)
                     : "memory");
        src += chunk;
        left -= chunk;
      }
    }
  }
  if (lane >= kIssuers) return;
  constexpr uint32_t kPiece = kTcTileBytes / kIssuers;
  const uint32_t s_count = static_cast<uint32_t>(p.stages);
  const uint32_t n = static_cast<uint32_t>(p.n_tiles);
  uint32_t j = 0, slot = 0, phase = 0;   // slot = j % S, phase = (j / S) & 1
  const uint64_t limit = wait_limit_ns(p.wait);
  for (; j < n; ++j) {
    const bool ok = j < s_count || wait_bounded<false>(smem_addr(&empty[slot]), phase ^ 1,
                                                       abort_flag, p.err, limit);
    if (!__all_sync(kIssuerMask, ok)) break;
    // failure-detection tests: the last tile is never copied, so the MMA
    // thread's wait on it runs out (not issued: not drained below)
    if (p.wait.withhold_last && j + 1 == n) break;
    const uint32_t bar = smem_addr(&full[slot]);
    if (lane == 0) mbar_arrive_expect_tx(bar, kTcTileBytes);
    __syncwarp(kIssuerMask);
    bulk_g2s(smem_addr(ring + slot * kTcTileBytes) + lane * kPiece,
             p.wstream + static_cast<size_t>(j) * kTcTileBytes + lane * kPiece, kPiece, bar);
    if (++slot == s_count) {
      slot = 0;
      phase ^= 1;
    }
  }
  // copies still in flight must land before the CTA's shared memory is
  // freed: the tiles issued within the last ring
  const uint32_t first = j > s_count ? j - s_count : 0;
  for (uint32_t q = first; q < j; ++q) {
    const uint32_t bar = smem_addr(&full[q % s_count]);
    const uint64_t t0 = now_ns();
    while (!try_wait(bar, (q / s_count) & 1)) {
      if (now_ns() - t0 > limit) {
        if (p.err) atomicOr(reinterpret_cast<unsigned int*>(p.err), DLRM_ERRBIT_TIMEOUT);
        break;
      }
    }
  }
}

template <bool BF16, bool TRACE>
__device__ void issue_mmas(const FusedTcParams& p, uint32_t tmem, unsigned char* ring,
                           unsigned char* const act[2], uint64_t* full, uint64_t* empty,
                           uint64_t* acc_ready, uint64_t* act_ready, uint64_t* drain,
                           volatile int* abort_flag) {
  constexpr uint32_t kIdesc = instr_desc(BF16 ? 1u : 2u, kTcTile);
  const uint32_t s_count = static_cast<uint32_t>(p.stages);
  const uint64_t limit = wait_limit_ns(p.wait);
  bool ok = true;
  uint32_t slot = 0, phase = 0;   // of stream tile j: j % S and (j / S) & 1
  for (int g = 0; g < p.n_gemm; ++g) {
    const TcGemm& L = p.gemm[g];
    const uint64_t ta = (TRACE && p.trace) ? now_ns() : 0;
    if (ok) ok = wait_bounded<true>(smem_addr(act_ready), g & 1, abort_flag, p.err, limit);
    uint64_t act_wait = (TRACE && p.trace) ? now_ns() - ta : 0, tile_wait = 0;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t b_base = smem_addr(act[g & 1]);
    // Tiles arrive K-block-major; each (M-tile, K step) pair accumulates into
    // its own 16 columns, so consecutive MMAs never wait on one another.
    for (int kb = 0; kb < L.kbs; ++kb) {
      for (int mt = 0; mt < L.mts; ++mt) {
        const uint64_t tw = (TRACE && p.trace) ? now_ns() : 0;
        if (ok) ok = wait_bounded<true>(smem_addr(&full[slot]), phase, abort_flag, p.err, limit);
        if (TRACE && p.trace) tile_wait += now_ns() - tw;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (ok) {
          const uint64_t da = smem_desc(smem_addr(ring + slot * kTcTileBytes));
          const uint64_t db = smem_desc(b_base + kb * kActBlock);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)   // 32 bytes of K per MMA
            mma<BF16>(tmem + static_cast<uint32_t>((mt * 4 + ks) * kTcTile), da + 2 * ks,
                      db + 2 * ks, kIdesc, kb > 0 ? 1u : 0u);
        }
        mma_commit(smem_addr(&empty[slot]));     // the slot is free once these ran
        if (++slot == s_count) {
          slot = 0;
          phase ^= 1;
        }
      }
    }
    mma_commit(smem_addr(acc_ready));             // the layer's accumulators are final
    // profiling: per layer, ns the MMA thread waited for its input
    // activations (slot 20 + 2g) and for landed weight tiles (21 + 2g)
    if (TRACE && p.trace && p.n_gemm + 3 < 20 && 21 + 2 * g < kTcTraceSlots) {
      unsigned long long* t = p.trace + static_cast<size_t>(blockIdx.x) * kTcTraceSlots;
      t[20 + 2 * g] = act_wait;
      t[21 + 2 * g] = tile_wait;
    }
  }
  // Every MMA must have run before the CTA frees its tensor memory, also when
  // a wait gave up and the epilogue skipped its own waits: one more commit on
  // a barrier of its own (a single phase, so its parity is unambiguous)
  // tracks them all; wait for it, bounded.
  mma_commit(smem_addr(drain));
  const uint64_t t0 = now_ns();
  while (!try_wait(smem_addr(drain), 0)) {
    if (now_ns() - t0 > limit) {
      if (p.err) atomicOr(reinterpret_cast<unsigned int*>(p.err), DLRM_ERRBIT_TIMEOUT);
      break;
    }
  }
}

template <bool BF16, bool TRACE>
__device__ void epilogue(const FusedTcParams& p, uint32_t tmem, unsigned char* const act[2],
                         float* xf, float* hf, float* zs, int* rowidx_s, float* bias_s,
                         float* wlast_s, uint64_t* acc_ready, uint64_t* act_ready,
                         volatile int* abort_flag) {
  constexpr int KB = BF16 ? 64 : 32;
  const int tid = threadIdx.x;                 // 0 .. 127
  const int warp = tid / kWarp;
  const int lane = tid % kWarp;
  const int m0 = blockIdx.x * kTcTile;
  const int rows = min(kTcTile, p.batch - m0);
  const int k = p.k_tables, d = p.d, d4 = d >> 2;
  const int f = k + 1;
  const int pairs = f * (f - 1) / 2;
  // quotients by these on the tile's paths come from quot (no divisions)
  const float r_k = __frcp_rn(static_cast<float>(k));
  const float r_d4 = __frcp_rn(static_cast<float>(d4));
  const float r_dn = __frcp_rn(static_cast<float>(max(p.n_dense, 1)));
  bool oob = false, bad_off = false;

  // ---- prologue. Biases and last-layer weights by cp.async. Then global
  // loads, two per thread in flight before either is used: every bag (size
  // 1) checked and its row (or -1) kept in shared memory, and the dense
  // features written as layer 0's operand (the padding is zeroed apart). The
  // MMA warp may start once the operand is complete; the bag rows follow by
  // cp.async and land while layer 0 runs.
  constexpr int kEpi = kEpiWarps * kWarp;
  for (int c = tid; c < p.bias_floats / 4; c += kEpi) cp_async16(bias_s + 4 * c, p.bias + 4 * c, 16);
  for (int c = tid; c < p.k_last / 4; c += kEpi) cp_async16(wlast_s + 4 * c, p.wlast + 4 * c, 16);
  {
    const int n_bag = p.bag == 1 ? kTcTile * k : 0;
    const int n_dn = kTcTile * p.n_dense;
    const int n_all = n_bag > n_dn ? n_bag : n_dn;
    for (int e0 = 0; e0 < n_all; e0 += 2 * kEpi) {
      int64_t start[2], row[2];
      float dv[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = e0 + h * kEpi + tid;
        start[h] = row[h] = 0;
        dv[h] = 0.f;
        if (e < n_bag) {
          const int s = quot(e, k, r_k), t = e - s * k;
          if (s < rows) {
            start[h] = __ldg(p.offsets + static_cast<int64_t>(t) * p.batch + m0 + s);
            row[h] = __ldg(p.indices + static_cast<int64_t>(t) * p.batch + m0 + s);
          }
        }
        if (e < n_dn) {
          const int s = quot(e, p.n_dense, r_dn);
          if (s < rows) dv[h] = __ldg(p.dense + static_cast<int64_t>(m0) * p.n_dense + e);
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = e0 + h * kEpi + tid;
        if (e < n_bag) {
          const int s = quot(e, k, r_k), t = e - s * k;
          int row32 = -1;
          if (s < rows) {
            if (start[h] != m0 + s) bad_off = true;
            else if (row[h] < 0 || row[h] >= p.tabs.rows[t]) oob = true;
            else row32 = static_cast<int>(row[h]);
          }
          rowidx_s[e] = row32;
        }
        if (e < n_dn) {
          const int s = quot(e, p.n_dense, r_dn);
          put_operand<BF16>(act[0], s, e - s * p.n_dense, dv[h]);
        }
      }
    }
    // layer 0 input, zero-padded to its K-blocks
    zero_operand<BF16>(act[0], p.n_dense, p.gemm[0].kbs * KB, tid, kEpi);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  epi_sync();
  if (tid == 0) mbar_arrive(smem_addr(act_ready));
  if (p.bag == 1) {
    for (int e = tid; e < kTcTile * k * d4; e += kEpi) {
      const int sk = quot(e, d4, r_d4);         // sample * k + table
      const int c4 = e - sk * d4;
      const float* table = p.tabs.ptr[sk - quot(sk, k, r_k) * k];
      const int row = rowidx_s[sk];
      cp_async16(zs + sk * p.ldz + 4 * c4,
                 row >= 0 ? table + static_cast<int64_t>(row) * d + 4 * c4 : table, row >= 0 ? 16 : 0);
    }
  } else {
    // bags of p.bag rows at offsets b * bag: summed in registers (an
    // out-of-range row adds nothing and raises the flag)
    for (int e = tid; e < kTcTile * k * d4; e += kEpi) {
      const int sk = quot(e, d4, r_d4);
      const int c4 = e - sk * d4;
      const int s = quot(sk, k, r_k), t = sk - s * k;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s < rows) {
        const int64_t b = m0 + s;
        const int64_t start = __ldg(p.offsets + static_cast<int64_t>(t) * p.batch + b);
        if (start != b * p.bag) {
          bad_off = true;
        } else {
          const int64_t* idx = p.indices + static_cast<int64_t>(t) * p.batch * p.bag + start;
          const float4* table = reinterpret_cast<const float4*>(p.tabs.ptr[t]);
          for (int l = 0; l < p.bag; ++l) {
            const int64_t row = __ldg(idx + l);
            if (row >= 0 && row < p.tabs.rows[t]) {
              const float4 u = __ldg(table + row * d4 + c4);
              v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
            } else {
              oob = true;
            }
          }
        }
      }
      *reinterpret_cast<float4*>(zs + sk * p.ldz + 4 * c4) = v;
    }
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  // biases, last-layer weights and bag rows land while layer 0 runs
  asm volatile("cp.async.wait_all;\n" ::: "memory");
  epi_sync();
  stamp<TRACE>(p, 1);

  // ---- layers
  for (int g = 0; g < p.n_gemm; ++g) {
    const TcGemm& L = p.gemm[g];
    const bool last_bottom = g == p.n_bot - 1;
    const bool last_hidden = g == p.n_gemm - 1;
    wait_bounded<false>(smem_addr(acc_ready), g & 1, abort_flag, p.err, wait_limit_ns(p.wait));
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    unsigned char* out = act[(g + 1) & 1];
    for (int mt = 0; mt < L.mts; ++mt) {
      // the four K-step partial sums of this M-tile: four loads, one wait
      uint32_t r[4][kTcTile];
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) +
                               static_cast<uint32_t>((mt * 4 + ks) * kTcTile);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
            "%10, %11, %12, %13, %14, %15}, [%16];"
            : "=r"(r[ks][0]), "=r"(r[ks][1]), "=r"(r[ks][2]), "=r"(r[ks][3]), "=r"(r[ks][4]),
              "=r"(r[ks][5]), "=r"(r[ks][6]), "=r"(r[ks][7]), "=r"(r[ks][8]), "=r"(r[ks][9]),
              "=r"(r[ks][10]), "=r"(r[ks][11]), "=r"(r[ks][12]), "=r"(r[ks][13]),
              "=r"(r[ks][14]), "=r"(r[ks][15])
            : "r"(taddr));
      }
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      float acc[kTcTile];
#pragma unroll
      for (int c = 0; c < kTcTile; ++c)
        acc[c] = (__uint_as_float(r[0][c]) + __uint_as_float(r[1][c])) +
                 (__uint_as_float(r[2][c]) + __uint_as_float(r[3][c]));
      const int feat = mt * 128 + warp * 32 + lane;
      const bool live = feat < L.n;
      const float bv = live ? bias_s[L.b_off + feat] : 0.f;
#pragma unroll
      for (int s = 0; s < kTcTile; ++s) {
        const float v = live ? fmaxf(acc[s] + bv, 0.f) : 0.f;
        if (last_hidden) {
          if (feat < p.k_last) hf[s * p.k_last + feat] = v;
        } else {
          put_operand<BF16>(out, s, feat, v);
          if (last_bottom && feat < d) xf[s * d + feat] = v;
        }
      }
    }
    if (last_bottom) {
      // R = [x, z]: pair dots in fp32 into features d .. d + pairs - 1 of the
      // top MLP's input, zeros up to its padded width
      asm volatile("cp.async.wait_all;\n" ::: "memory");
      epi_sync();
      stamp<TRACE>(p, 2 + g);
      // one (sample, pair) dot per thread, then zeros to the padded width
      const int kw = p.gemm[g + 1].kbs * KB;
      const float r_pairs = __frcp_rn(static_cast<float>(pairs));
      for (int e = tid; e < kTcTile * pairs; e += kEpiWarps * kWarp) {
        const int s = quot(e, pairs, r_pairs);
        const int q = e - s * pairs;
        int i, jj;
        pair_from_index(q, i, jj);
        const float* vi = (i == 0) ? xf + s * d : zs + (s * k + i - 1) * p.ldz;
        const float* vj = (jj == 0) ? xf + s * d : zs + (s * k + jj - 1) * p.ldz;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int c4 = 0; c4 < d4; ++c4) {
          const float4 u = *reinterpret_cast<const float4*>(vi + 4 * c4);
          const float4 w = *reinterpret_cast<const float4*>(vj + 4 * c4);
          a.x = fmaf(u.x, w.x, a.x);
          a.y = fmaf(u.y, w.y, a.y);
          a.z = fmaf(u.z, w.z, a.z);
          a.w = fmaf(u.w, w.w, a.w);
        }
        put_operand<BF16>(out, s, d + q, (a.x + a.y) + (a.z + a.w));
      }
      zero_operand<BF16>(out, d + pairs, kw, tid, kEpiWarps * kWarp);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    if (!last_hidden) {
      // generic-proxy writes of the operand -> visible to the tensor cores
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      epi_sync();
      if (tid == 0) mbar_arrive(smem_addr(act_ready));
      stamp<TRACE>(p, last_bottom ? 2 + p.n_bot : (g < p.n_bot ? 2 + g : 3 + g));
    } else {
      epi_sync();
      stamp<TRACE>(p, 3 + g);
    }
  }

  // ---- last layer: fp32 dot and sigmoid, a warp per sample
  // (warp w takes samples w, w + 4, w + 8, w + 12 together: four
  // independent sums per lane)
  const float bl = bias_s[p.b_last];
  {
    constexpr int kPer = kTcTile / kEpiWarps;
    static_assert(kTcTile % kEpiWarps == 0, "whole samples per warp");
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    for (int q = lane; q < p.k_last; q += kWarp) {
      const float wq = wlast_s[q];
#pragma unroll
      for (int i = 0; i < kPer; ++i) acc[i] = fmaf(hf[(warp + i * kEpiWarps) * p.k_last + q], wq, acc[i]);
    }
#pragma unroll
    for (int o = kWarp / 2; o > 0; o /= 2)
#pragma unroll
      for (int i = 0; i < kPer; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int s = warp + i * kEpiWarps;
      if (lane == 0 && s < rows) p.out[m0 + s] = 1.0f / (1.0f + expf(-(acc[i] + bl)));
    }
  }
  if (p.err) {
    if (oob) atomicOr(reinterpret_cast<unsigned int*>(p.err), DLRM_ERRBIT_INDEX_OOB);
    if (bad_off) atomicOr(reinterpret_cast<unsigned int*>(p.err), DLRM_ERRBIT_OFFSETS);
  }
  if (TRACE && p.trace) {
    epi_sync();
    stamp<TRACE>(p, 2 + p.n_gemm + 1);
  }
}

template <bool BF16, bool TRACE>
__global__ void __launch_bounds__(kThreads, 1)
fused_tc_kernel(const __grid_constant__ FusedTcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* ring = base;
  unsigned char* const act[2] = {base + p.off_act0, base + p.off_act1};
  float* xf = reinterpret_cast<float*>(base + p.off_xf);
  float* hf = reinterpret_cast<float*>(base + p.off_hf);
  float* zs = reinterpret_cast<float*>(base + p.off_z);
  int* rowidx_s = reinterpret_cast<int*>(base + p.off_rowidx);
  float* bias_s = reinterpret_cast<float*>(base + p.off_bias);
  float* wlast_s = reinterpret_cast<float*>(base + p.off_wlast);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + p.off_bar);
  uint64_t* empty = full + p.stages;
  uint64_t* acc_ready = empty + p.stages;
  uint64_t* act_ready = acc_ready + 1;
  uint64_t* drain = act_ready + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x / kWarp;
  stamp<TRACE>(p, 0);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(static_cast<uint32_t>(p.tmem_cols))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == kWarp) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), 1);
    }
    mbar_init(smem_addr(acc_ready), 1);
    mbar_init(smem_addr(act_ready), 1);
    mbar_init(smem_addr(drain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    produce(p, ring, full, empty, abort_flag);
  } else if (warp == kMmaWarp) {
    if (threadIdx.x % kWarp == 0)
      issue_mmas<BF16, TRACE>(p, tmem, ring, act, full, empty, acc_ready, act_ready, drain,
                       abort_flag);
  } else {
    epilogue<BF16, TRACE>(p, tmem, act, xf, hf, zs, rowidx_s, bias_s, wlast_s, acc_ready, act_ready,
                   abort_flag);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(static_cast<uint32_t>(p.tmem_cols))
                 : "memory");
  }
}

template <bool BF16, bool TRACE>
cudaError_t enable_smem() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(fused_tc_kernel<BF16, TRACE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(device_max_smem_optin()));
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Round-to-nearest-even fp32 -> bf16 bits (finite inputs; NaN kept quiet).
uint16_t bf16_bits(float v) {
  uint32_t u;
  std::memcpy(&u, &v, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return static_cast<uint16_t>((u >> 16) | 0x40);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

cudaError_t fused_tc_prepare(int bf16) {
  cudaError_t e = bf16 ? enable_smem<true, false>() : enable_smem<false, false>();
  if (e == cudaSuccess) e = bf16 ? enable_smem<true, true>() : enable_smem<false, true>();
  return e;
}

cudaError_t launch_fused_tc(const FusedTcParams& p, cudaStream_t stream) {
  if (p.batch == 0) return cudaSuccess;
  cudaError_t e = fused_tc_prepare(p.bf16);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>((p.batch + kTcTile - 1) / kTcTile);
  if (p.bf16) {
    if (p.trace) fused_tc_kernel<true, true><<<grid, kThreads, p.smem_bytes, stream>>>(p);
    else fused_tc_kernel<true, false><<<grid, kThreads, p.smem_bytes, stream>>>(p);
  } else {
    if (p.trace) fused_tc_kernel<false, true><<<grid, kThreads, p.smem_bytes, stream>>>(p);
    else fused_tc_kernel<false, false><<<grid, kThreads, p.smem_bytes, stream>>>(p);
  }
  return cudaGetLastError();
}

bool fused_tc_plan(int n_dense, int k_tables, int d, int bag, const std::vector<int>& ln_bot,
                   const std::vector<int>& ln_top, const std::vector<std::vector<float>>& w,
                   const std::vector<std::vector<float>>& b, const GatherTables& tabs, int math,
                   size_t smem_limit, FusedTcPlan* plan) {
  if (math != DLRM_MATH_TF32 && math != DLRM_MATH_BF16) return false;
  const bool bf16 = math == DLRM_MATH_BF16;
  const int kb_vals = bf16 ? 64 : 32;            // K values per 128-byte block
  const int n_bot = static_cast<int>(ln_bot.size()) - 1;
  const int n_top = static_cast<int>(ln_top.size()) - 1;
  const int n_gemm = n_bot + n_top - 1;
  if (bag < 1 || d % 4 != 0 || n_bot < 1 || n_top < 2 || ln_top.back() != 1 ||
      n_gemm > kTcMaxGemm)
    return false;
  for (int t = 0; t < k_tables; ++t)
    if (reinterpret_cast<uintptr_t>(tabs.ptr[t]) % 16 != 0) return false;
  FusedTcParams& p = plan->params;
  p = FusedTcParams{};
  p.n_dense = n_dense;
  p.k_tables = k_tables;
  p.d = d;
  p.bag = bag;
  p.n_bot = n_bot;
  p.n_top = n_top;
  p.n_gemm = n_gemm;
  p.bf16 = bf16 ? 1 : 0;
  const int f = k_tables + 1;
  const int pairs = f * (f - 1) / 2;

  std::vector<int> kin(n_gemm), nout(n_gemm);
  for (int g = 0; g < n_gemm; ++g) {
    kin[g] = g < n_bot ? ln_bot[g] : ln_top[g - n_bot];
    nout[g] = g < n_bot ? ln_bot[g + 1] : ln_top[g - n_bot + 1];
  }
  int tiles = 0, bias_floats = 0, act_blocks = 0, acc_cols = 0;
  for (int g = 0; g < n_gemm; ++g) {
    TcGemm& L = p.gemm[g];
    L.n = nout[g];
    L.k = kin[g];
    L.mts = (L.n + 127) / 128;
    L.kbs = (L.k + kb_vals - 1) / kb_vals;
    L.first = tiles;
    L.b_off = bias_floats;
    tiles += L.mts * L.kbs;
    bias_floats += L.mts * 128;
    act_blocks = std::max({act_blocks, L.kbs, (L.mts * 128 + kb_vals - 1) / kb_vals});
    acc_cols = std::max(acc_cols, L.mts * 4 * kTcTile);     // (M-tile, K step) accumulators
  }
  p.n_tiles = tiles;
  int tcols = 32;
  while (tcols < acc_cols) tcols *= 2;
  if (tcols > 512) return false;
  p.tmem_cols = tcols;
  p.k_last = static_cast<int>(round_up(ln_top[n_top - 1], 4));
  p.b_last = bias_floats;
  bias_floats += 4;
  p.bias_floats = bias_floats;
  p.ldz = static_cast<int>(round_up(d, 4)) + 4;
  p.act_bytes = act_blocks * kActBlock;
  if (nout[n_bot - 1] != d || kin[n_bot] != d + pairs) return false;

  // shared-memory carve from the 1024-aligned base
  const size_t fixed_tail =
      2 * static_cast<size_t>(p.act_bytes) + align_up(static_cast<size_t>(kTcTile) * d * 4, 128) +
      align_up(static_cast<size_t>(kTcTile) * p.k_last * 4, 128) +
      align_up(static_cast<size_t>(kTcTile) * k_tables * p.ldz * 4, 128) +
      align_up(static_cast<size_t>(kTcTile) * k_tables * 4, 128) +
      align_up(static_cast<size_t>(bias_floats) * 4, 128) + align_up(p.k_last * 4, 128);
  int stages = 0;
  for (int s = 12; s >= 2; --s) {         // the deepest ring that fits
    const size_t bars = align_up((2 * s + 3) * 8 + 16, 128);
    if (1024 + static_cast<size_t>(s) * kTcTileBytes + fixed_tail + bars <= smem_limit) {
      stages = s;
      break;
    }
  }
  if (stages == 0) return false;
  p.stages = stages;
  size_t off = static_cast<size_t>(stages) * kTcTileBytes;
  p.off_act0 = static_cast<int>(off);
  off += p.act_bytes;
  p.off_act1 = static_cast<int>(off);
  off += p.act_bytes;
  p.off_xf = static_cast<int>(off);
  off += align_up(static_cast<size_t>(kTcTile) * d * 4, 128);
  p.off_hf = static_cast<int>(off);
  off += align_up(static_cast<size_t>(kTcTile) * p.k_last * 4, 128);
  p.off_z = static_cast<int>(off);
  off += align_up(static_cast<size_t>(kTcTile) * k_tables * p.ldz * 4, 128);
  p.off_rowidx = static_cast<int>(off);
  off += align_up(static_cast<size_t>(kTcTile) * k_tables * 4, 128);
  p.off_bias = static_cast<int>(off);
  off += align_up(static_cast<size_t>(bias_floats) * 4, 128);
  p.off_wlast = static_cast<int>(off);
  off += align_up(p.k_last * 4, 128);
  p.off_bar = static_cast<int>(off);
  off += align_up((2 * stages + 3) * 8 + 16, 128);   // full, empty, acc/act ready, drain
  p.smem_bytes = static_cast<int>(off + 1024);
  if (static_cast<size_t>(p.smem_bytes) > smem_limit) return false;

  // weight tiles: (layer, M-tile, K-block), 128 rows x 128 bytes each,
  // K-major with the 128-byte swizzle; rows past n and k past kin are zero
  const int esz = bf16 ? 2 : 4;
  plan->wstream.assign(static_cast<size_t>(tiles) * kTcTileBytes, 0);
  for (int g = 0; g < n_gemm; ++g) {
    const TcGemm& L = p.gemm[g];
    const std::vector<float>& W = w[g];
    for (int mt = 0; mt < L.mts; ++mt)
      for (int kb = 0; kb < L.kbs; ++kb) {
        unsigned char* tile =
            plan->wstream.data() + static_cast<size_t>(L.first + kb * L.mts + mt) * kTcTileBytes;
        for (int r = 0; r < 128; ++r) {
          const int n = mt * 128 + r;
          if (n >= L.n) break;
          for (int e = 0; e < kb_vals; ++e) {
            const int kk = kb * kb_vals + e;
            if (kk >= L.k) break;
            const float v = W[static_cast<size_t>(n) * L.k + kk];
            unsigned char* q = tile + swz_offset(r, (e * esz) >> 4) + ((e * esz) & 15);
            if (bf16) {
              const uint16_t h = bf16_bits(v);
              std::memcpy(q, &h, 2);
            } else {
              std::memcpy(q, &v, 4);
            }
          }
        }
      }
  }
  plan->bias.assign(bias_floats, 0.f);
  for (int g = 0; g < n_gemm; ++g)
    for (int n = 0; n < nout[g]; ++n) plan->bias[p.gemm[g].b_off + n] = b[g][n];
  plan->bias[p.b_last] = b[n_gemm][0];
  plan->wlast.assign(p.k_last, 0.f);
  for (int c = 0; c < ln_top[n_top - 1]; ++c) plan->wlast[c] = w[n_gemm][c];
  p.tabs = tabs;
  return true;
}

}  // namespace dlrm
