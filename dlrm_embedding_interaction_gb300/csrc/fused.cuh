// Parameter block and host planning of the fused single-launch forward
// (fused.cu).
#pragma once

#include <vector>

#include "common.cuh"

namespace dlrm {

// Warps per CTA: 8 computing warps (two warpgroups) and a producer warpgroup
// whose first warp streams the weights (fused.cu, fused_forward_kernel).
constexpr int kFusedStageFloats = 8192;                        // 32 KB weight stage
constexpr int kFusedMaxGemm = 2 * DLRM_MAX_LAYERS;
// Bags of several rows prefetched whole: at most this many float4 bag sums
// per computing thread (tile samples x tables x D / 4 <= 8 x 256).
constexpr int kFusedBagRowSums = 8;

// One GEMM layer of the weight stream. Its weights occupy `passes * n_kst`
// consecutive stages of the packed stream: pass p covers output columns
// [P p, P p + rows), P = (2 / ksplit) * 32 * tn, stage s covers k in
// [s*KS, (s+1)*KS), KS = 16*ksplit, stored row-major (rows x KS) with 16-byte
// chunk c of row r at position c ^ swz(r) (swz = (r >> 1) & 3 when KS = 16,
// else r & 7).
//   n      output width; wider than 256: n_pad = round_up(n, 256), tn = 8,
//          ksplit = 1; else n_pad = 32 * tn (tn a power of two), ksplit = 2
//   tn     the stage's columns per pass / 32 (each computing warp takes 64
//          of them, or all 32 when tn = 1, for one k-slice)
//   k_pad  input width padded to a multiple of KS (zero weights)
//   b_off  offset of the layer's zero-padded bias in the bias block
struct FusedGemm {
  int n, n_pad, tn, k_pad, ksplit, passes, n_kst, b_off;
};

struct FusedParams {
  int batch, n_dense, k_tables, d, bag, n_bot, n_top;
  int n_gemm;        // n_bot + n_top - 1 (the last top layer is the N = 1 dot)
  int cw;            // computing warps (8)
  int lda;           // activation row stride (floats), >= 528, = 16 mod 32
  int ldz;           // bag-sum row stride, round_up(d, 4) + 4
  int sg;            // samples per gather/interaction group
  int prefetch_z;    // 1: all BM samples' rows are fetched at kernel start (bag 1, or
                     //    every row of every bag when bag_rows is set)
  int bag_rows;      // 1: bags of bag > 1 rows, all rows prefetched, summed at the interaction
  int zbuf;          // bag 1 without prefetch: 2 group buffers, rows streamed with cp.async
  int stages;        // weight ring depth
  int n_stages;      // stages of the whole weight stream
  int k_last;        // padded input width of the last (N = 1) layer
  int b_last;        // its bias offset in the bias block
  int bias_floats;   // bias block length (multiple of 4)
  // shared-memory carve (bytes from the dynamic base)
  int off_act0, off_act1, off_z, off_bias, off_wlast, off_bar, off_rowidx;
  // barriers block: full[stages], empty[stages] (u64), abort flag
  int smem_bytes;
  FusedGemm gemm[kFusedMaxGemm];
  const float* wstream;    // packed weight stream
  const uint2* stage_tab;  // per stream stage: (offset in floats, bytes)
  size_t stream_floats;    // length of the weight stream (a multiple of 4)
  const float* bias;       // bias block
  const float* wlast;      // last layer weights, k_last floats (zero-padded)
  const float* dense;
  const int64_t* indices;
  const int64_t* offsets;
  float* out;
  int32_t* err;
  unsigned long long* trace;   // optional phase stamps, kFusedTraceSlots per tile
  WaitCfg wait;                // wait limit; failure tests: the last stage withheld
  GatherTables tabs;
};

constexpr int kFusedTraceSlots = 40;

// Host plan: shapes, smem carve and the packed weight/bias images.
struct FusedPlan {
  FusedParams params{};
  int bm = 0;
  std::vector<float> wstream, bias, wlast;
  std::vector<uint2> stage_tab;
};

// Builds the plan from host copies of the (out, in) weights and biases;
// false when the model does not fit the fused kernel.
// The tile height is the one of 4, 8, 12, 14, 16 rows with the least
// rounds x (rows + 12), rounds = ceil(tiles of max_batch / sms) (the launch is
// persistent, and a tile costs about 12 rows' worth more than its rows),
// falling back to smaller tiles when the shared-memory carve does not fit.
bool fused_plan(int n_dense, int k_tables, int d, int bag, const std::vector<int>& ln_bot,
                const std::vector<int>& ln_top, const std::vector<std::vector<float>>& w,
                const std::vector<std::vector<float>>& b, const GatherTables& tabs,
                int max_batch, int sms, size_t smem_limit, int consumer_warps, FusedPlan* plan);

// The activation stride of the kernel instance a plan runs on: 528 or 624
// (compile-time strides, one bag-row mode each) when the plan's stride and
// mode match those instances, else 0 (the run-time-stride instances).
inline int fused_instance_lda(const FusedParams& p) {
  if (p.lda == 528 && p.prefetch_z && !p.bag_rows) return 528;
  if (p.lda == 624 && p.zbuf == 2) return 624;
  return 0;
}
// lda: fused_instance_lda of the plan.
cudaError_t fused_prepare(int bm, int consumer_warps, int lda);
cudaError_t launch_fused(const FusedParams& p, int bm, cudaStream_t stream);
// The instances with phase-trace stamps (fused_trace.cu): launch_fused takes
// them while p.trace is set.
cudaError_t fused_prepare_traced(int bm, int consumer_warps, int lda);
cudaError_t launch_fused_traced(const FusedParams& p, int bm, cudaStream_t stream);

}  // namespace dlrm
