// Warp-specialized TMA + tcgen05 Linear (gemm_tma.cu): the layer-wise plan's
// GEMM for layers whose input is a 16-byte aligned buffer of the handle, in
// the opt-in TF32 and TF32X3 modes.
#pragma once

#include "common.cuh"

namespace dlrm {

constexpr int kTensorMapBytes = 128;   // sizeof(CUtensorMap)

// One layer's TMA plan, made at create time: tensor maps (opaque 128-byte
// CUtensorMap images) of its input buffer X (max_batch x k, row stride ld)
// and of its weights W (n x k) -- in TF32X3 the tf32 head of W in map_w and
// the remainder W - head in map_wlo (split once, at create time).
struct TmaLayer {
  alignas(64) unsigned char map_x[kTensorMapBytes];
  alignas(64) unsigned char map_w[kTensorMapBytes];
  alignas(64) unsigned char map_wlo[kTensorMapBytes];
  int n = 0, k = 0;
  int split = 0;     // 1: TF32X3 (three products per K step), 0: TF32
};

struct TmaGemmParams {
  int m, n, ldy, act, vec_y;
  int m_tiles, n_tiles, kb_count;
  float* y;
  const float* bias;
  int32_t* err;
  WaitCfg wait;
};

// A buffer TMA can read: 16-byte aligned base, row stride a multiple of 4
// floats.
bool tma_operand_ok(const void* base, int ld);

// Encodes a 2-D fp32 tensor map of `rows` rows of `inner` values, row stride
// `ld` floats, read in boxes of 32 values x box_rows rows (128 for an input
// X, 64 for weights: a 128-row weight tile is two loads) with the 128-byte
// swizzle; zeros past the inner width and the last row. `map` points to
// kTensorMapBytes, 64-byte aligned. false when the operand is not TMA-able,
// box_rows is neither 128 nor 64, or the driver's encoder is unavailable.
bool encode_operand_map(void* map, const float* base, int inner, int rows, int ld, int box_rows);

// Y (m x L.n, row stride ldy) = act(X W^T + bias) for the first m rows of the
// layer's input buffer.
cudaError_t launch_linear_tma(const TmaLayer& L, int m, const float* bias, float* y, int ldy,
                              int act, int32_t* err, cudaStream_t stream, WaitCfg wait);

}  // namespace dlrm
