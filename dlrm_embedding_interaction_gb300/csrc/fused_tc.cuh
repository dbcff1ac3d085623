// Parameter block and host planning of the fused single-launch forward on
// the tensor cores (fused_tc.cu): the opt-in TF32 and BF16 modes.
#pragma once

#include <vector>

#include "common.cuh"

namespace dlrm {

constexpr int kTcTile = 16;                 // samples per CTA (the MMA N)
constexpr int kTcTileBytes = 16384;         // one weight tile: 128 rows x 128 bytes
constexpr int kTcMaxGemm = 2 * DLRM_MAX_LAYERS;
constexpr int kTcTraceSlots = 40;

// One GEMM layer: output features n in M-tiles of 128, input k in K-blocks of
// 128 bytes (32 tf32 / 64 bf16 values). Its weight tiles follow each other
// in the stream, K-block-major: tile (mt, kb) = stream tile first + kb * mts + mt.
struct TcGemm {
  int n, k, mts, kbs, first, b_off;
};

struct FusedTcParams {
  int batch, n_dense, k_tables, d, bag, n_bot, n_top;
  int n_gemm;          // n_bot + n_top - 1 (the last top layer is an fp32 dot)
  int bf16;            // operand type: 0 tf32, 1 bf16
  int stages;          // weight ring depth
  int n_tiles;         // tiles in the weight stream
  int tmem_cols;       // accumulator columns allocated (power of two >= 32)
  int ldz;             // fp32 bag-row stride (floats)
  int k_last;          // padded input width of the last (N = 1) layer
  int b_last;          // its bias offset in the bias block
  int bias_floats;
  // shared-memory carve (bytes from the 1024-aligned base)
  int off_act0, off_act1, off_xf, off_hf, off_z, off_rowidx, off_bias, off_wlast, off_bar;
  int act_bytes;       // one activation buffer
  int smem_bytes;      // dynamic shared memory requested (base alignment included)
  TcGemm gemm[kTcMaxGemm];
  const unsigned char* wstream;   // packed weight tiles
  const float* bias;              // bias block
  const float* wlast;             // last layer weights, k_last floats
  const float* dense;
  const int64_t* indices;
  const int64_t* offsets;
  float* out;
  int32_t* err;
  unsigned long long* trace;      // optional phase stamps, kTcTraceSlots per tile
  WaitCfg wait;                   // wait limit; failure tests: the last tile withheld
  GatherTables tabs;
};

struct FusedTcPlan {
  FusedTcParams params{};
  std::vector<unsigned char> wstream;
  std::vector<float> bias, wlast;
};

// Builds the plan for math DLRM_MATH_TF32 or DLRM_MATH_BF16 from host copies
// of the (out, in) weights and biases; false when the model does not fit
// (tables not 16-byte aligned, shared memory, tensor memory).
bool fused_tc_plan(int n_dense, int k_tables, int d, int bag, const std::vector<int>& ln_bot,
                   const std::vector<int>& ln_top, const std::vector<std::vector<float>>& w,
                   const std::vector<std::vector<float>>& b, const GatherTables& tabs, int math,
                   size_t smem_limit, FusedTcPlan* plan);

cudaError_t fused_tc_prepare(int bf16);
cudaError_t launch_fused_tc(const FusedTcParams& p, cudaStream_t stream);

}  // namespace dlrm
