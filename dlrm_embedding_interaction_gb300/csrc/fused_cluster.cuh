// Parameter block and host planning of the cluster-split fused forward
// (fused_cluster.cu): the whole forward of a tile of samples in one launch,
// every layer's output columns split over the CTAs of a thread-block cluster.
#pragma once

#include <vector>

#include "common.cuh"

namespace dlrm {

constexpr int kClusterWarps = 8;                         // computing warps (+1 producer warp)
constexpr int kClusterThreads = kClusterWarps * kWarp;   // computing threads
constexpr int kClusterMaxGemm = 2 * DLRM_MAX_LAYERS;
constexpr int kClusterTileRows[3] = {4, 8, 16};          // tile heights with a kernel instance

// One GEMM layer. CTA q of a cluster of C computes output columns
// [q s, (q + 1) s) of every sample of the tile (n_pad = s C columns in all,
// zero beyond n). Its 256 computing threads each take a column pair and a
// k-slice: thread t has pair t % (s / 2) and k-slice t / (s / 2) of
// kslices = 512 / s, the float4 k-steps ks4 + kslices i. The rank's weights
// stream in n_kst stages of up to kst_k inputs (the last one shorter), each
// packed so that step i of thread t reads two consecutive-in-t float4s.
struct ClusterGemm {
  int n, k;      // output and input width
  int s;         // columns per CTA: a power of two, 4..512
  int kslices;   // 512 / s
  int k_pad;     // k rounded up to 4 * kslices
  int kst_k;     // inputs per full stage (a multiple of 4 * kslices)
  int n_kst;     // stages of the layer
  int b_off;     // the rank's bias slice in its bias block
};

struct ClusterParams {
  int batch, n_dense, k_tables, d, bag, n_bot, n_top, n_gemm;
  int csize;          // CTAs per cluster
  int bm;             // samples per tile (one tile per cluster)
  int lda;            // activation row stride (floats)
  int ldz;            // bag-sum row stride (floats)
  int ld_r;           // interaction row width pushed to the cluster: round_up(d + pairs, 4)
  int zrows;          // interaction rows per CTA: ceil(bm / csize)
  int stages;         // ring depth
  int rank_stages;    // stages of one rank's weight stream
  int k_last;         // padded width of the last (N = 1) layer's input
  int bias_floats;    // one rank's bias block (floats, a multiple of 4)
  float b_last;       // the last layer's bias
  // shared-memory carve (bytes from the dynamic base)
  int off_act0, off_act1, off_scratch, off_z, off_rowidx, off_bias, off_wlast, off_bar;
  int smem_bytes;
  ClusterGemm gemm[kClusterMaxGemm];
  const float* wstream;     // the ranks' weight streams, one after another
  const uint2* stage_tab;   // (offset in floats, bytes) per stage; rank r's at r * rank_stages
  const float* bias;        // rank r's bias block at r * bias_floats
  const float* wlast;       // k_last floats (zero-padded)
  const float* dense;
  const int64_t* indices;
  const int64_t* offsets;
  float* out;
  int32_t* err;
  WaitCfg wait;
  GatherTables tabs;
};

// Host plan for one cluster size: the weight stream, bias blocks and the
// parameter blocks of every tile height that fits shared memory.
struct ClusterPlan {
  int csize = 0;
  bool fits[3] = {false, false, false};
  ClusterParams params[3]{};
  std::vector<float> wstream, bias, wlast;
  std::vector<uint2> stage_tab;
};

// Builds the plan from host copies of the (out, in) weights and biases; false
// when no tile height fits (a layer wider than 512 * csize, or shared memory).
bool fused_cluster_plan(int n_dense, int k_tables, int d, int bag, const std::vector<int>& ln_bot,
                        const std::vector<int>& ln_top, const std::vector<std::vector<float>>& w,
                        const std::vector<std::vector<float>>& b, const GatherTables& tabs,
                        int csize, size_t smem_limit, ClusterPlan* plan);

// Clusters of the tile height's instance that one wave holds on this device
// (0 when the instance cannot launch with these shared-memory bytes).
int fused_cluster_max_active(int bm, int csize, int smem_bytes);

cudaError_t launch_fused_cluster(const ClusterParams& p, cudaStream_t stream);

}  // namespace dlrm
