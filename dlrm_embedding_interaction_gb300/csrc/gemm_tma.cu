// Linear layers of many rows on the tensor cores, warp-specialized, with TMA
// operand loads: the layer-wise plan's GEMM in the opt-in TF32 and TF32X3
// (split-TF32, fp32-accurate) modes for batches of several 128-row tiles.
//
//   Y[m][n] = act(sum_k X[m][k] W[n][k] + b[n])   (Luminal compare
//   modal_ci_ready...vanilla-pytorch, commit message: linear_bias_(relu|sigmoid))
//
// A persistent CTA (at most one per SM) walks output tiles of 128 rows x BN
// columns (BN = 128, or 64 when that still gives one tile per SM, or the
// layer has at most 64 outputs: with one tile per CTA a tile's time is its K
// loop, and halving BN halves the MMA work per block on twice the SMs),
// t = blockIdx.x, blockIdx.x + gridDim.x, ... with the column tile fastest,
// so the CTAs running at one time share their rows of X through L2.
// Per tile the K dimension flows in blocks of 32 values (128 bytes of fp32:
// one 128-byte swizzle atom row) through a ring of shared-memory stages:
//  * warp 0, one lane: loads each block's X tile (128 x 32) and weight tiles
//    with cp.async.bulk.tensor (TMA, 128-byte swizzle: the canonical K-major
//    layout the MMA descriptors read), completing on the stage's full
//    mbarrier;
//  * warps 2-3 and 8-15 (TF32X3): split the X tile in place into its tf32 head
//    (hi = x with the low 13 mantissa bits cleared, exact in tf32) and write
//    the remainder lo = x - hi (exact in fp32) beside it; the weights arrive
//    already split (head and remainder streams made at create time);
//  * warp 1, one lane: issues tcgen05.mma kind::tf32, M = 128, N = BN, four
//    K steps of 8 per block (hi*hi + hi*lo + lo*hi in TF32X3), into one of
//    two TMEM accumulators of BN columns, and releases the stage with
//    tcgen05.commit to its empty barrier;
//  * warps 4-7: read the finished accumulator (tcgen05.ld 32x32b, warp w
//    the TMEM lanes 32 (w % 4) ...), release it to the next tile but one,
//    add the bias, apply the activation and store through a shared-memory
//    transpose, so that every store instruction writes 128 bytes of a row.
// Every wait is bounded (WaitCfg); on expiry the kernel sets
// DLRM_ERRBIT_TIMEOUT, every role leaves its loop, the loads and MMAs in
// flight are waited for (bounded) and the tensor memory is freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "gemm_tma.cuh"
#include "tc.cuh"

namespace dlrm {

using namespace tc;

namespace {

constexpr int kThreads = 512;             // warps 8-15: more X split warps
constexpr int kSplitWarps = 10;          // warps 2-3 and 8-15
constexpr int kBM = 128;                 // rows of X per tile (the MMA M)
constexpr int kBK = 32;                  // k per block: 128 bytes of fp32
constexpr int kTile = kBM * kBK * 4;     // 16 KB: one 128 x 32 fp32 tile
constexpr int kWBox = 64;                // weight rows per TMA load (the maps' box)
constexpr int kWBoxBytes = kWBox * kBK * 4;

template <bool SPLIT, int BN>
struct Layout {
  // X, [X lo,] W (hi), [W lo]; BN weight rows of 128 bytes per W tile
  static constexpr int kWTile = BN * kBK * 4;
  static constexpr int kStage = (SPLIT ? 2 : 1) * (kTile + kWTile);
  static constexpr int kStages = SPLIT ? (BN == 128 ? 3 : 4) : (BN == 128 ? 6 : 8);
  static constexpr int kBars = 3 * kStages + 5;      // full, split, empty; acc full/empty x2; drain
  // epilogue: per epilogue warp a 32 x 32 staging block (stride 33 floats)
  static constexpr int kEpiFloats = 4 * 32 * 33;
  static constexpr int kSmem = 1024 + kStages * kStage + kBars * 8 + 16 + kEpiFloats * 4;
  static_assert(BN % kWBox == 0 && kWTile % 1024 == 0 && kStage % 1024 == 0, "swizzle atoms");
  static_assert(kSmem <= 232448, "shared memory of one CTA");
};

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Bounded wait; false on timeout (which raises the abort flag and the error
// bit) or when another thread has raised the abort flag.
__device__ bool wait_for(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                         uint64_t limit) {
  if (try_wait(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  for (uint32_t i = 1;; ++i) {
    if (try_wait(bar, parity)) return true;
    if ((i & 15) == 0) {
      if (*abort_flag) return false;
      if (now_ns() - t0 > limit) {
        *abort_flag = 1;
        if (err) atomicOr(reinterpret_cast<unsigned int*>(err), DLRM_ERRBIT_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait regardless of the abort flag (draining work in flight).
__device__ void drain_wait(uint32_t bar, uint32_t parity, int32_t* err, uint64_t limit) {
  const uint64_t t0 = now_ns();
  while (!try_wait(bar, parity)) {
    if (now_ns() - t0 > limit) {
      if (err) atomicOr(reinterpret_cast<unsigned int*>(err), DLRM_ERRBIT_TIMEOUT);
      return;
    }
  }
}

template <bool SPLIT, int BN>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tma_kernel(const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_w,
                const __grid_constant__ CUtensorMap tmap_wlo, const TmaGemmParams p) {
  using Lay = Layout<SPLIT, BN>;
  constexpr int kAccCols = BN;   // TMEM columns of one accumulator
  constexpr int S = Lay::kStages;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + S * Lay::kStage);
  uint64_t* full = bars;
  uint64_t* split_done = bars + S;
  uint64_t* empty = bars + 2 * S;
  uint64_t* acc_full = bars + 3 * S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* epi_s = reinterpret_cast<float*>(bars + Lay::kBars + 2);   // after the flag words
  // stage s: X at 0, [X lo at kTile,] W at (SPLIT ? 2 : 1) kTile, [W lo after it]
  auto x_tile = [&](int s) { return base + s * Lay::kStage; };
  auto xlo_tile = [&](int s) { return base + s * Lay::kStage + kTile; };
  auto w_tile = [&](int s) { return base + s * Lay::kStage + (SPLIT ? 2 : 1) * kTile; };
  auto wlo_tile = [&](int s) { return base + s * Lay::kStage + 2 * kTile + Lay::kWTile; };

  const int warp = threadIdx.x / kWarp;
  const int lane = threadIdx.x % kWarp;
  const uint64_t limit = wait_limit_ns(p.wait);
  const int tiles = p.m_tiles * p.n_tiles;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "n"(2 * kAccCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == kWarp) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&split_done[s]), kSplitWarps);   // the split warps
      mbar_init(smem_addr(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_addr(&acc_full[a]), 1);
      mbar_init(smem_addr(&acc_empty[a]), 4);           // the four epilogue warps
    }
    mbar_init(smem_addr(drain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  // launched while the previous kernel may still run: its outputs (this
  // layer's input) and its reads of this layer's output buffer are done
  // after the wait
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x))
                   : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w))
                   : "memory");
      if (SPLIT)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_wlo))
                     : "memory");
      constexpr uint32_t kBytes = kTile + (SPLIT ? 2 : 1) * Lay::kWTile;
      uint32_t stage = 0, phase = 0, it = 0;
      bool ok = true;
      const uint32_t total = static_cast<uint32_t>(
          ((tiles - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x) * p.kb_count);
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int mt = t / p.n_tiles, nt = t % p.n_tiles;
        for (int kb = 0; kb < p.kb_count; ++kb) {
          if (it >= static_cast<uint32_t>(S) &&
              !wait_for(smem_addr(&empty[stage]), phase ^ 1, abort_flag, p.err, limit)) {
            ok = false;
            break;
          }
          // failure-detection tests: the last block is never loaded, so the
          // wait on it runs out (not issued: not drained below)
          if (p.wait.withhold_last && it + 1 == total) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(&full[stage]);
          mbar_expect_tx(bar, kBytes);
          tma_load_2d(smem_addr(x_tile(stage)), &tmap_x, kb * kBK, mt * kBM, bar);
#pragma unroll
          for (int h = 0; h < BN / kWBox; ++h) {   // 64-row boxes, 8 swizzle atoms each
            tma_load_2d(smem_addr(w_tile(stage)) + h * kWBoxBytes, &tmap_w, kb * kBK,
                        nt * BN + h * kWBox, bar);
            if (SPLIT)
              tma_load_2d(smem_addr(wlo_tile(stage)) + h * kWBoxBytes, &tmap_wlo, kb * kBK,
                          nt * BN + h * kWBox, bar);
          }
          ++it;
          if (++stage == static_cast<uint32_t>(S)) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // loads in flight must land before the shared memory is released
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
      for (uint32_t q = first; q < it; ++q) drain_wait(smem_addr(&full[q % S]), (q / S) & 1, p.err, limit);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdesc = instr_desc(2u, BN);    // tf32 x tf32 -> fp32, N = BN
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      int i = 0;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++i) {
        const int abuf = i & 1;
        const uint32_t aphase = (i >> 1) & 1;
        if (i >= 2 && !wait_for(smem_addr(&acc_empty[abuf]), aphase ^ 1, abort_flag, p.err, limit))
          break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t acc = tmem + static_cast<uint32_t>(abuf * kAccCols);
        for (int kb = 0; kb < p.kb_count; ++kb) {
          const uint32_t ready = smem_addr(SPLIT ? &split_done[stage] : &full[stage]);
          if (!wait_for(ready, phase, abort_flag, p.err, limit)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint64_t dx = smem_desc(smem_addr(x_tile(stage)));
          const uint64_t dw = smem_desc(smem_addr(w_tile(stage)));
          const uint64_t dxl = smem_desc(smem_addr(xlo_tile(stage)));
          const uint64_t dwl = smem_desc(smem_addr(wlo_tile(stage)));
#pragma unroll
          for (int j = 0; j < kBK / 8; ++j) {
            const uint64_t off = static_cast<uint64_t>((j * 32) >> 4);   // 32 bytes per K step
            mma<false>(acc, dx + off, dw + off, kIdesc, (kb > 0 || j > 0) ? 1u : 0u);
            if (SPLIT) {
              mma<false>(acc, dx + off, dwl + off, kIdesc, 1u);   // hi * lo
              mma<false>(acc, dxl + off, dw + off, kIdesc, 1u);   // lo * hi
            }
          }
          mma_commit(smem_addr(&empty[stage]));     // the stage is free once these ran
          if (++stage == static_cast<uint32_t>(S)) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(smem_addr(&acc_full[abuf]));     // the tile's accumulator is final
      }
      // every MMA must have run before the tensor memory is freed: one more
      // commit on a barrier of its own (one phase) tracks them all
      mma_commit(smem_addr(drain));
      drain_wait(smem_addr(drain), 0, p.err, limit);
    }
  } else if (warp < 4 || warp >= 8) {
    // ---------------------------------------------------------------- X split (TF32X3)
    if (SPLIT) {
      const int st = (warp < 4 ? warp - 2 : warp - 6) * kWarp + lane;   // 0 .. 191
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        for (int kb = 0; kb < p.kb_count; ++kb) {
          if (!wait_for(smem_addr(&full[stage]), phase, abort_flag, p.err, limit)) {
            ok = false;
            break;
          }
          unsigned char* xs = x_tile(stage);
          unsigned char* xl = xlo_tile(stage);
#pragma unroll 4
          for (int off = st * 16; off < kTile; off += kSplitWarps * kWarp * 16) {
            const uint4 v = *reinterpret_cast<const uint4*>(xs + off);
            uint4 hi, lo;
            hi.x = v.x & 0xFFFFE000u;
            hi.y = v.y & 0xFFFFE000u;
            hi.z = v.z & 0xFFFFE000u;
            hi.w = v.w & 0xFFFFE000u;
            lo.x = __float_as_uint(__uint_as_float(v.x) - __uint_as_float(hi.x));
            lo.y = __float_as_uint(__uint_as_float(v.y) - __uint_as_float(hi.y));
            lo.z = __float_as_uint(__uint_as_float(v.z) - __uint_as_float(hi.z));
            lo.w = __float_as_uint(__uint_as_float(v.w) - __uint_as_float(hi.w));
            *reinterpret_cast<uint4*>(xs + off) = hi;
            *reinterpret_cast<uint4*>(xl + off) = lo;
          }
          // generic-proxy writes -> visible to the tensor core's async proxy
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&split_done[stage]));
          if (++stage == static_cast<uint32_t>(S)) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    // Warp q reads TMEM lanes 32 q .. 32 q + 31 (the tile's rows) 32 columns
    // at a time, stages the 32 x 32 block in shared memory and writes it back
    // row by row: each store instruction writes 32 consecutive floats (128
    // bytes) of one row.
    const int q = warp & 3;                              // TMEM lane quarter
    float* blk = epi_s + q * 32 * 33;
    int i = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
      const int abuf = i & 1;
      const uint32_t aphase = (i >> 1) & 1;
      const int mt = t / p.n_tiles, nt = t % p.n_tiles;
      // the bias of the lane's column in each 32-column chunk, loaded while
      // the accumulator is still being made
      float bv[BN / 32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        const int col = nt * BN + 32 * c + lane;
        bv[c] = (p.bias && col < p.n) ? __ldg(p.bias + col) : 0.f;
      }
      if (!wait_for(smem_addr(&acc_full[abuf]), aphase, abort_flag, p.err, limit)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int row0 = mt * kBM + q * 32;
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        const uint32_t taddr =
            tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(abuf * kAccCols + c0);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
            "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
            "%27, %28, %29, %30, %31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
              "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
              "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
              "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
              "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
              "=r"(r[30]), "=r"(r[31])
            : "r"(taddr));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (c0 + 32 == BN) {
          // every TMEM read of this accumulator is done: release it
          asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&acc_empty[abuf]));
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) blk[lane * 33 + j] = __uint_as_float(r[j]);
        __syncwarp();
        const int col = nt * BN + c0 + lane;
        const float b = bv[c0 / 32];
        const int rows = min(32, p.m - row0);
        if (col < p.n) {
          float* ycol = p.y + static_cast<int64_t>(row0) * p.ldy + col;
          for (int rr = 0; rr < rows; ++rr)
            ycol[static_cast<int64_t>(rr) * p.ldy] = apply_act(blk[rr * 33 + lane] + b, p.act);
        }
        __syncwarp();
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(2 * kAccCols)
                 : "memory");
  }
}

template <bool SPLIT, int BN>
cudaError_t prepare() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(gemm_tma_kernel<SPLIT, BN>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<SPLIT, BN>::kSmem);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<void*> fn{nullptr};
  void* f = fn.load(std::memory_order_acquire);
  if (!f) {
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn.store(f, std::memory_order_release);
  }
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

}  // namespace

bool tma_operand_ok(const void* base, int ld) {
  return base && reinterpret_cast<uintptr_t>(base) % 16 == 0 && ld > 0 && ld % 4 == 0;
}

bool encode_operand_map(void* map, const float* base, int inner, int rows, int ld, int box_rows) {
  static_assert(sizeof(CUtensorMap) == kTensorMapBytes, "tensor map size");
  if (!tma_operand_ok(base, ld) || inner < 1 || rows < 1 || inner > ld) return false;
  if (box_rows != kBM && box_rows != kWBox) return false;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * sizeof(float)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estrides[2] = {1, 1};
  const CUresult r = enc(reinterpret_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                         const_cast<float*>(base), dims, strides, box, estrides,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_linear_tma(const TmaLayer& L, int m, const float* bias, float* y, int ldy,
                              int act, int32_t* err, cudaStream_t stream, WaitCfg wait) {
  if (m == 0) return cudaSuccess;
  TmaGemmParams p{};
  p.m = m;
  p.n = L.n;
  p.ldy = ldy;
  p.y = y;
  p.bias = bias;
  p.act = act;
  p.err = err;
  p.wait = wait;
  p.m_tiles = (m + kBM - 1) / kBM;
  p.kb_count = (L.k + kBK - 1) / kBK;
  p.vec_y = (ldy % 4 == 0 && reinterpret_cast<uintptr_t>(y) % 16 == 0 &&
             (bias == nullptr || reinterpret_cast<uintptr_t>(bias) % 16 == 0))
                ? 1
                : 0;
  // 64-column tiles when they still fit one tile per SM (each CTA's K loop
  // then does half the MMA work), or when the layer has at most 64 outputs
  const int sms = device_sm_count();
  const int64_t tiles64 = static_cast<int64_t>(p.m_tiles) * ((L.n + 63) / 64);
  const bool narrow = L.n <= 64 || tiles64 <= sms;
  const int bn = narrow ? 64 : 128;
  p.n_tiles = (L.n + bn - 1) / bn;
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(tiles, sms));
  const CUtensorMap* mx = reinterpret_cast<const CUtensorMap*>(L.map_x);
  const CUtensorMap* mw = reinterpret_cast<const CUtensorMap*>(L.map_w);
  const CUtensorMap* mwl = reinterpret_cast<const CUtensorMap*>(L.split ? L.map_wlo : L.map_w);
  cudaError_t e;
  if (L.split) {
    if (narrow) {
      if ((e = prepare<true, 64>()) != cudaSuccess) return e;
      return launch_pdl(gemm_tma_kernel<true, 64>, dim3(grid), dim3(kThreads),
                        Layout<true, 64>::kSmem, stream, *mx, *mw, *mwl, p);
    }
    if ((e = prepare<true, 128>()) != cudaSuccess) return e;
    return launch_pdl(gemm_tma_kernel<true, 128>, dim3(grid), dim3(kThreads),
                      Layout<true, 128>::kSmem, stream, *mx, *mw, *mwl, p);
  }
  if (narrow) {
    if ((e = prepare<false, 64>()) != cudaSuccess) return e;
    return launch_pdl(gemm_tma_kernel<false, 64>, dim3(grid), dim3(kThreads),
                      Layout<false, 64>::kSmem, stream, *mx, *mw, *mwl, p);
  }
  if ((e = prepare<false, 128>()) != cudaSuccess) return e;
  return launch_pdl(gemm_tma_kernel<false, 128>, dim3(grid), dim3(kThreads),
                    Layout<false, 128>::kSmem, stream, *mx, *mw, *mwl, p);
}

}  // namespace dlrm
