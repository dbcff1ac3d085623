// fp32 Linear + bias + activation (the parity-mode MLP GEMM).
//
// y[m][n] = act(sum_k x[m][k] * W[n][k] + bias[n]), W in nn.Linear (N, K)
// layout (Luminal compare modal_ci_ready...vanilla-pytorch, commit message:
// linear_bias_(relu|sigmoid) over the fused Matmul2D kernel; compare
// dlrm-fused-kernels...dlrm-pt2-megakernel, dlrm_megakernel.rs steps 2 and 6).
//
// GB300 design (SIMT FFMA; the fp32 mode must stay fp32, so no tensor cores):
//  * block tile BM x BN, K-step 16, thread tile TM x TN in registers
//    (outer products from shared memory, 128-bit LDS, broadcast-friendly);
//  * both operands are K-contiguous in global memory; tiles are loaded with
//    128-bit loads and stored transposed (k-major) in shared memory, double
//    buffered with the next tile's loads in flight during the FFMA loop;
//  * the tile shape is chosen per call so the grid fills the 152 SMs (small
//    M x N DLRM layers would leave most SMs idle with 128 x 128 tiles);
//  * bias and ReLU/sigmoid are applied in registers before the single store.
// N < 16 (the final 256 -> 1 sigmoid layer) runs a warp-per-row GEMV instead.
#include <algorithm>
#include <atomic>

#include "common.cuh"

namespace dlrm {
namespace {

constexpr int kBK = 16;

// Load one (ROWS x kBK) tile of a K-contiguous matrix into registers.
// VEC: row stride % 4 == 0 and base 16-byte aligned, so a 16-byte load at any
// k < K stays inside the row's padded width; values at k >= K are zeroed.
template <int ROWS, int THREADS, bool VEC>
struct TileLoader {
  static constexpr int kVecs = ROWS * kBK / 4;
  static constexpr int kPer = (kVecs + THREADS - 1) / THREADS;
  float4 reg[kPer];

  __device__ __forceinline__ void load(const float* __restrict__ src, int ld, int row0,
                                       int rows, int k0, int k) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = threadIdx.x + i * THREADS;
      const int r = e / (kBK / 4);
      const int kq = (e % (kBK / 4)) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      const int gr = row0 + r;
      const int gk = k0 + kq;
      if (e < kVecs && gr < rows && gk < k) {
        const float* p = src + static_cast<int64_t>(gr) * ld + gk;
        if (VEC) {
          v = __ldg(reinterpret_cast<const float4*>(p));
          if (gk + 1 >= k) v.y = 0.f;
          if (gk + 2 >= k) v.z = 0.f;
          if (gk + 3 >= k) v.w = 0.f;
        } else {
          v.x = __ldg(p);
          if (gk + 1 < k) v.y = __ldg(p + 1);
          if (gk + 2 < k) v.z = __ldg(p + 2);
          if (gk + 3 < k) v.w = __ldg(p + 3);
        }
      }
      reg[i] = v;
    }
  }

  // Store transposed: dst[k][r], row stride LDS floats.
  template <int LDS>
  __device__ __forceinline__ void store(float* dst) const {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = threadIdx.x + i * THREADS;
      if (e < kVecs) {
        const int r = e / (kBK / 4);
        const int kq = (e % (kBK / 4)) * 4;
        dst[(kq + 0) * LDS + r] = reg[i].x;
        dst[(kq + 1) * LDS + r] = reg[i].y;
        dst[(kq + 2) * LDS + r] = reg[i].z;
        dst[(kq + 3) * LDS + r] = reg[i].w;
      }
    }
  }
};

// Thread-tile coordinate: TM/TN of 4 are contiguous; 8 is split in two
// 4-wide halves half a block tile apart (conflict-free 128-bit LDS).
template <int T, int B>
__device__ __forceinline__ int tile_coord(int t, int i) {
  if (T == 4) return t * 4 + i;
  return (i / 4) * (B / 2) + t * 4 + (i % 4);
}

template <int BM, int BN, int TM, int TN, int ACT, bool VA, bool VW>
__global__ void __launch_bounds__((BM / TM) * (BN / TN))
sgemm_bias_act_kernel(const float* __restrict__ x, int ldx, const float* __restrict__ w, int ldw,
                      const float* __restrict__ bias, float* __restrict__ y, int ldy, int m,
                      int n, int k, int vec_y) {
  pdl_wait();     // launched after the previous kernel may still run
  pdl_trigger();

  constexpr int kThreads = (BM / TM) * (BN / TN);
  constexpr int kLdA = BM + 4;
  constexpr int kLdB = BN + 4;
  __shared__ __align__(16) float as[2][kBK * kLdA];
  __shared__ __align__(16) float bs[2][kBK * kLdB];

  const int tx = threadIdx.x % (BN / TN);
  const int ty = threadIdx.x / (BN / TN);
  const int m0 = blockIdx.x * BM;   // M tiles on x: no 65535 limit for large batches
  const int n0 = blockIdx.y * BN;

  TileLoader<BM, kThreads, VA> la;
  TileLoader<BN, kThreads, VW> lb;
  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

  const int k_tiles = (k + kBK - 1) / kBK;
  la.load(x, ldx, m0, m, 0, k);
  lb.load(w, ldw, n0, n, 0, k);
  la.template store<kLdA>(as[0]);
  lb.template store<kLdB>(bs[0]);
  __syncthreads();

  for (int kt = 0; kt < k_tiles; ++kt) {
    const int cur = kt & 1;
    if (kt + 1 < k_tiles) {
      la.load(x, ldx, m0, m, (kt + 1) * kBK, k);
      lb.load(w, ldw, n0, n, (kt + 1) * kBK, k);
    }
    const float* a_s = as[cur];
    const float* b_s = bs[cur];
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float a[TM], b[TN];
#pragma unroll
      for (int i = 0; i < TM; i += 4) {
        const float4 v = *reinterpret_cast<const float4*>(a_s + kk * kLdA + tile_coord<TM, BM>(ty, i));
        a[i] = v.x; a[i + 1] = v.y; a[i + 2] = v.z; a[i + 3] = v.w;
      }
#pragma unroll
      for (int j = 0; j < TN; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(b_s + kk * kLdB + tile_coord<TN, BN>(tx, j));
        b[j] = v.x; b[j + 1] = v.y; b[j + 2] = v.z; b[j + 3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (kt + 1 < k_tiles) {
      la.template store<kLdA>(as[cur ^ 1]);
      lb.template store<kLdB>(bs[cur ^ 1]);
    }
    __syncthreads();
  }

  // Epilogue: bias + activation, 16-byte stores where the row allows.
#pragma unroll
  for (int j = 0; j < TN; j += 4) {
    const int gn = n0 + tile_coord<TN, BN>(tx, j);
    float bv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) bv[q] = (bias && gn + q < n) ? __ldg(bias + gn + q) : 0.f;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int gm = m0 + tile_coord<TM, BM>(ty, i);
      if (gm >= m) continue;
      float v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = apply_act(acc[i][j + q] + bv[q], ACT);
      float* dst = y + static_cast<int64_t>(gm) * ldy + gn;
      if (vec_y && gn + 3 < n) {
        *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (gn + q < n) dst[q] = v[q];
      }
    }
  }
}

// Large-M tile (M >= 64 rows per block for at least two blocks per SM): the
// broadcast-row register tile of the fused forward. Block 64 rows x 128
// columns, 8 warps; warp w owns rows 8w .. 8w+7 (every lane reads the same
// row values: broadcast shared loads) and lane l owns columns l + 32 j, j < 4,
// accumulating the even-k and odd-k partial sums of each output in one float2
// with fma.rn.f32x2. Per packed FMA the tile needs 2/8 + 1/4 shared
// wavefronts, in balance with the FMA pipe. Tiles of 32 k stream through a
// 3-stage cp.async ring (zero-filled past M, N and K); W rows are stored with
// their 16-byte chunks XOR-swizzled by row so 8 consecutive lanes' rows fall
// on 8 distinct bank groups.
constexpr int kLmBM = 64, kLmBN = 128, kLmBK = 32, kLmStages = 3, kLmThreads = 256;
constexpr int kLmStageFloats = (kLmBM + kLmBN) * kLmBK;

__device__ __forceinline__ void lm_cp_async16(float* dst, const float* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(static_cast<uint32_t>(
                   __cvta_generic_to_shared(dst))),
               "l"(src), "r"(bytes)
               : "memory");
}

template <int ACT>
__global__ void __launch_bounds__(kLmThreads, 2)
sgemm_large_m_kernel(const float* __restrict__ x, int ldx, const float* __restrict__ w, int ldw,
                     const float* __restrict__ bias, float* __restrict__ y, int ldy, int m, int n,
                     int k) {
  pdl_wait();     // launched after the previous kernel may still run
  pdl_trigger();

  extern __shared__ __align__(16) float lm_smem[];
  const int tid = threadIdx.x;
  const int warp = tid / kWarp;
  const int lane = tid % kWarp;
  const int m0 = blockIdx.x * kLmBM;
  const int n0 = blockIdx.y * kLmBN;
  const int k_tiles = (k + kLmBK - 1) / kLmBK;

  // stage loader: A 64 rows x 8 chunks, W 128 rows x 8 chunks of 16 bytes
  auto load_stage = [&](int kt, int s) {
    float* as = lm_smem + s * kLmStageFloats;
    float* ws = as + kLmBM * kLmBK;
    const int k0 = kt * kLmBK;
    for (int c = tid; c < (kLmBM + kLmBN) * 8; c += kLmThreads) {
      const bool is_a = c < kLmBM * 8;
      const int cc = is_a ? c : c - kLmBM * 8;
      const int r = cc >> 3;
      const int ch = cc & 7;
      const int kk = k0 + ch * 4;
      const int gr = (is_a ? m0 : n0) + r;
      const int rows = is_a ? m : n;
      const float* src = is_a ? x : w;
      int bytes = 0;
      if (gr < rows && kk < k) {
        src += static_cast<int64_t>(gr) * (is_a ? ldx : ldw) + kk;
        bytes = k - kk >= 4 ? 16 : 4 * (k - kk);
      }
      float* dst = is_a ? as + r * kLmBK + ch * 4 : ws + r * kLmBK + ((ch ^ (r & 7)) * 4);
      lm_cp_async16(dst, src, bytes);
    }
  };

  float2 acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);

#pragma unroll
  for (int s = 0; s < kLmStages - 1; ++s) {
    if (s < k_tiles) load_stage(s, s);
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  }
  const int sw = lane & 7;
  for (int kt = 0; kt < k_tiles; ++kt) {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(kLmStages - 2) : "memory");
    __syncthreads();
    // refill the stage read two tiles ago (every warp is past it)
    if (kt + kLmStages - 1 < k_tiles) load_stage(kt + kLmStages - 1, (kt + kLmStages - 1) % kLmStages);
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    const float* as = lm_smem + (kt % kLmStages) * kLmStageFloats + warp * 8 * kLmBK;
    const float* ws = lm_smem + (kt % kLmStages) * kLmStageFloats + kLmBM * kLmBK + lane * kLmBK;
#pragma unroll
    for (int step = 0; step < kLmBK / 4; ++step) {
      float4 wv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        wv[j] = *reinterpret_cast<const float4*>(ws + 32 * j * kLmBK + ((step ^ sw) * 4));
      float4 av[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) av[i] = *reinterpret_cast<const float4*>(as + i * kLmBK + step * 4);
      // component-outer: 32 independent accumulators between the even-k and
      // odd-k updates of each
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          acc[i][j] = __ffma2_rn(make_float2(av[i].x, av[i].y), make_float2(wv[j].x, wv[j].y),
                                 acc[i][j]);
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          acc[i][j] = __ffma2_rn(make_float2(av[i].z, av[i].w), make_float2(wv[j].z, wv[j].w),
                                 acc[i][j]);
    }
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");

#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int gn = n0 + lane + 32 * j;
    if (gn >= n) continue;
    const float bv = bias ? __ldg(bias + gn) : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int gm = m0 + warp * 8 + i;
      if (gm < m)
        y[static_cast<int64_t>(gm) * ldy + gn] = apply_act((acc[i][j].x + acc[i][j].y) + bv, ACT);
    }
  }
}

// Warp per row for N < 16: lanes stride K, butterfly reduction, lane 0 writes.
template <int ACT>
__global__ void __launch_bounds__(256)
gemv_rows_kernel(const float* __restrict__ x, int ldx, const float* __restrict__ w, int ldw,
                 const float* __restrict__ bias, float* __restrict__ y, int ldy, int m, int n,
                 int k, int vec) {
  pdl_wait();     // launched after the previous kernel may still run
  pdl_trigger();

  const int row = blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp;
  const int lane = threadIdx.x & (kWarp - 1);
  if (row >= m) return;
  const float* xr = x + static_cast<int64_t>(row) * ldx;
  for (int col = 0; col < n; ++col) {
    const float* wr = w + static_cast<int64_t>(col) * ldw;
    float acc = 0.f;
    if (vec) {
      const int k4 = k / 4;
      for (int q = lane; q < k4; q += kWarp) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(xr) + q);
        const float4 b = __ldg(reinterpret_cast<const float4*>(wr) + q);
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
        acc = fmaf(a.z, b.z, acc);
        acc = fmaf(a.w, b.w, acc);
      }
      for (int q = 4 * k4 + lane; q < k; q += kWarp) acc = fmaf(__ldg(xr + q), __ldg(wr + q), acc);
    } else {
      for (int q = lane; q < k; q += kWarp) acc = fmaf(__ldg(xr + q), __ldg(wr + q), acc);
    }
#pragma unroll
    for (int o = kWarp / 2; o > 0; o /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      const float bv = bias ? __ldg(bias + col) : 0.f;
      y[static_cast<int64_t>(row) * ldy + col] = apply_act(acc + bv, ACT);
    }
  }
}

template <int BM, int BN, int TM, int TN, int ACT>
cudaError_t launch_tile(const float* x, int ldx, const float* w, int ldw, const float* bias,
                        float* y, int ldy, int m, int n, int k, bool va, bool vw, bool vy,
                        cudaStream_t stream) {
  constexpr int kThreads = (BM / TM) * (BN / TN);
  const dim3 grid((m + BM - 1) / BM, (n + BN - 1) / BN);
  if (va && vw)
    return launch_pdl(sgemm_bias_act_kernel<BM, BN, TM, TN, ACT, true, true>, grid, dim3(kThreads), 0,
                      stream, x, ldx, w, ldw, bias, y, ldy, m, n, k, vy);
  else if (va)
    return launch_pdl(sgemm_bias_act_kernel<BM, BN, TM, TN, ACT, true, false>, grid, dim3(kThreads), 0,
                      stream, x, ldx, w, ldw, bias, y, ldy, m, n, k, vy);
  else if (vw)
    return launch_pdl(sgemm_bias_act_kernel<BM, BN, TM, TN, ACT, false, true>, grid, dim3(kThreads), 0,
                      stream, x, ldx, w, ldw, bias, y, ldy, m, n, k, vy);
  else
    return launch_pdl(sgemm_bias_act_kernel<BM, BN, TM, TN, ACT, false, false>, grid, dim3(kThreads), 0,
                      stream, x, ldx, w, ldw, bias, y, ldy, m, n, k, vy);
  return cudaGetLastError();
}

template <int ACT>
cudaError_t launch_act(const float* x, int ldx, const float* w, int ldw, const float* bias,
                       float* y, int ldy, int m, int n, int k, cudaStream_t stream) {
  auto aligned = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
  const bool va = (ldx % 4 == 0) && aligned(x);
  const bool vw = (ldw % 4 == 0) && aligned(w);
  const bool vy = (ldy % 4 == 0) && aligned(y);
  if (n < 16) {
    const bool vec = va && vw;
    const unsigned grid = static_cast<unsigned>((m + 7) / 8);
    return launch_pdl(gemv_rows_kernel<ACT>, dim3(grid), dim3(256), 0, stream, x, ldx, w, ldw, bias,
                      y, ldy, m, n, k, vec);
  }
  const int64_t sms = device_sm_count();
  auto blocks = [&](int bm, int bn) {
    return static_cast<int64_t>((m + bm - 1) / bm) * ((n + bn - 1) / bn);
  };
  if (va && vw && blocks(kLmBM, kLmBN) >= 2 * sms) {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    constexpr int kSmem = kLmStages * kLmStageFloats * static_cast<int>(sizeof(float));
    if (!bit || !(done.load(std::memory_order_acquire) & bit)) {
      e = cudaFuncSetAttribute(sgemm_large_m_kernel<ACT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      if (e != cudaSuccess) return e;
      if (bit) done.fetch_or(bit, std::memory_order_acq_rel);
    }
    const dim3 grid((m + kLmBM - 1) / kLmBM, (n + kLmBN - 1) / kLmBN);
    return launch_pdl(sgemm_large_m_kernel<ACT>, grid, dim3(kLmThreads), kSmem, stream, x, ldx, w,
                      ldw, bias, y, ldy, m, n, k);
  }
  if (blocks(128, 128) >= sms)
    return launch_tile<128, 128, 8, 8, ACT>(x, ldx, w, ldw, bias, y, ldy, m, n, k, va, vw, vy, stream);
  if (blocks(64, 64) >= sms)
    return launch_tile<64, 64, 4, 4, ACT>(x, ldx, w, ldw, bias, y, ldy, m, n, k, va, vw, vy, stream);
  if (blocks(32, 64) >= sms)
    return launch_tile<32, 64, 4, 4, ACT>(x, ldx, w, ldw, bias, y, ldy, m, n, k, va, vw, vy, stream);
  return launch_tile<32, 32, 4, 4, ACT>(x, ldx, w, ldw, bias, y, ldy, m, n, k, va, vw, vy, stream);
}

}  // namespace

cudaError_t launch_linear_fp32(const float* x, int ld_x, const float* w, int ld_w,
                               const float* bias, float* y, int ld_y, int m, int n, int k,
                               int act, cudaStream_t stream) {
  if (m == 0) return cudaSuccess;
  switch (act) {
    case DLRM_ACT_RELU:
      return launch_act<DLRM_ACT_RELU>(x, ld_x, w, ld_w, bias, y, ld_y, m, n, k, stream);
    case DLRM_ACT_SIGMOID:
      return launch_act<DLRM_ACT_SIGMOID>(x, ld_x, w, ld_w, bias, y, ld_y, m, n, k, stream);
    default:
      return launch_act<DLRM_ACT_NONE>(x, ld_x, w, ld_w, bias, y, ld_y, m, n, k, stream);
  }
}

}  // namespace dlrm
