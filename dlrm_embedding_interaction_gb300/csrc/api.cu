// C ABI of libdlrm_gb300.so (declared in include/dlrm.h): argument checks,
// the forward plan (handle), its workspace, and the launch sequence.
//
// The forward follows Luminal compare dlrm-fused-kernels...dlrm-pt2-megakernel,
// dlrm_megakernel.rs steps 1-6 (bottom MLP with ReLU after every layer,
// lookups, i-major pairwise dots with Vec[0] = x, R = [x, z], top MLP with ReLU
// then a final sigmoid), with the shape checks of its validate(). All device
// memory of a handle is one arena allocated in dlrm_create; forward calls
// allocate nothing and never synchronise.
#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "common.cuh"
#include "fused.cuh"
#include "fused_cluster.cuh"
#include "fused_tc.cuh"
#include "gemm_tma.cuh"

namespace dlrm {

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_smem_optin[kMaxDevices];

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  return dev;
}

}  // namespace

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 148;
  int v = g_sm_count[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    g_sm_count[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

size_t device_max_smem_optin() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 48 * 1024;
  int v = g_smem_optin[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        v <= 0)
      v = 48 * 1024;
    g_smem_optin[dev].store(v, std::memory_order_relaxed);
  }
  return static_cast<size_t>(v);
}

}  // namespace dlrm

using dlrm::round_up;

struct dlrm_handle_s {
  int device = 0;
  int n_bot = 0, n_top = 0, k = 0, d = 0, bag = 0, max_batch = 0, n_dense = 0;
  dlrm_math_t math = DLRM_MATH_FP32;
  std::vector<int> ln_bot, ln_top;
  dlrm::GatherTables tabs{};
  // packed parameters: W as (N, ldw = round_up(K, 4)) zero-padded, bias (N)
  std::vector<float*> bot_w, bot_b, top_w, top_b;
  std::vector<int> bot_ldw, top_ldw;
  // workspace
  float* emb = nullptr;          // (max_batch, K, D)
  float* act[2] = {nullptr, nullptr};
  int ld_act = 0;                // widest hidden width, rounded to 4
  float* r = nullptr;            // (max_batch, ld_r), R = [x, z]
  int ld_r = 0;
  int32_t* err = nullptr;        // device error word
  // staging for dlrm_forward_host
  float* dense_stage = nullptr;
  int64_t* idx_stage = nullptr;
  int64_t* off_stage = nullptr;
  float* out_stage = nullptr;
  void* arena = nullptr;
  size_t arena_bytes = 0;
  // kernel plan
  int path = DLRM_PATH_LAYERWISE;
  int fused_bm = 0;
  dlrm::FusedParams fused{};     // per-call fields filled by run_forward
  bool fused_tc = false;         // the fused plan runs on the tensor cores (TF32 / BF16)
  dlrm::FusedTcParams tcp{};
  // fp32 fused plan, small batches: the cluster-split kernel (fused_cluster.cu)
  bool cluster_on = false;
  // per cluster size (kClusterSizes) and tile height (4, 8, 16 samples): the
  // parameter block, and the clusters one wave holds (0: unavailable)
  dlrm::ClusterParams cparams[2][3]{};
  int cmax[2][3] = {{0, 0, 0}, {0, 0, 0}};
  int cluster_limit = 0;              // batches up to this run on the cluster kernel
  int cluster_default = 0;
  // AUTO fp32 fused handles: forwards of at least this many samples take the
  // layer-wise plan with split-TF32 GEMMs (0: never)
  int64_t layerwise_from = 0;
  unsigned long long* trace = nullptr;
  dlrm::WaitCfg wait{};          // dlrm_test_stall: wait limit, withheld last copy
  // layer-wise TF32 / TF32X3: per layer (bottom, then top), the TMA plan of
  // the warp-specialized tensor-core GEMM, or off (tma_on 0)
  std::vector<dlrm::TmaLayer> tma;
  std::vector<char> tma_on;
  // per-stage profiling (dlrm_set_profiling)
  std::vector<std::string> stage_names;
  std::vector<cudaEvent_t> events;      // stage boundaries, empty when off
  std::vector<double> stage_ms;
  int64_t profiled_calls = 0;
  bool report_on_destroy = false;   // DLRM_PROFILE=1 at dlrm_create
};

namespace {

dlrm_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA; }

// Bump allocator over one cudaMalloc'd arena; 256-byte aligned slices.
struct ArenaPlan {
  size_t bytes = 0;
  template <class T>
  size_t take(size_t count) {
    const size_t off = bytes;
    bytes = static_cast<size_t>(round_up(static_cast<int64_t>(off + count * sizeof(T)), 256));
    return off;
  }
};

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// The cluster-split kernel for small batches of the fp32 fused plan: CTAs per
// cluster, and the largest batch it takes by default (one wave of clusters
// at most). Measured on the 13-512-256-64 / 512-256-1 models (flushed L2):
// it wins at any table count up to 256 samples (128 samples: 22.3-29.9
// against 26.4-43.2 us for one CTA per tile; 256 samples: 25.8-35.2 against
// 26.5-43.1) and loses from 384 on (32.5-47.3 against 26.5-43.1), where the
// tiles of 16 samples make the per-layer k-loops long.
constexpr int kClusterSizes[2] = {8, 4};
int cluster_max_batch(int n_tables) { (void)n_tables; return 256; }
// Clusters of 8 CTAs up to this batch (the fewest weights per CTA: 20 us at
// 1-32 samples against 22.5 with 4), clusters of 4 above it (128 samples, 3
// tables: 22.6 us against 28.8 with 8 and 26.7 on one CTA per tile).
constexpr int kWideClusterMaxBatch = 32;
// It pays only for models whose weights the one-CTA tile streams for long:
// a stream of 1 MiB (32 stages; 1.3 MB on those models) or more. The 20 KB
// weights of a 64-wide model ran in 14 us on one CTA per tile against 18.6
// on the cluster kernel, whose per-layer exchanges cost more than the
// stream they save (12.3 us on one CTA per tile now).
constexpr size_t kClusterMinStreamBytes = size_t(1) << 20;

bool tensor_core_math(int math) { return math == DLRM_MATH_TF32 || math == DLRM_MATH_BF16; }
bool fp32_math(int math) { return math == DLRM_MATH_FP32 || math == DLRM_MATH_FP32_FFMA; }

// Layer-wise plan, GEMM layer g (bottom layers, then top) of n outputs and k
// inputs: on the TMA tensor-core GEMM (its input a buffer of the handle, so
// not the first bottom layer; split-TF32 in FP32 and TF32X3, where it needs
// 64 or more inputs to pay), ...
bool tma_layer(int math, int g, int n, int k) {
  if (g == 0 || n < 16) return false;
  // BF16 takes the TMA GEMM with tf32 operands: that kernel has no bf16 form,
  // tf32 keeps more precision than bf16, and the staged bf16 GEMM it replaces
  // ran the 32-table 2048-sample forward in 298 us against 107 in TF32
  if (math == DLRM_MATH_TF32 || math == DLRM_MATH_BF16) return true;
  return (math == DLRM_MATH_FP32 || math == DLRM_MATH_TF32X3) && k >= 64;
}
bool split_tf32_math(int math) { return math == DLRM_MATH_FP32 || math == DLRM_MATH_TF32X3; }
// ... else on the staged tcgen05 GEMM (opt-in modes only), else on FFMA.
bool staged_tc_layer(int math, int n, int k) {
  if (n < 16) return false;
  if (tensor_core_math(math)) return true;
  return math == DLRM_MATH_TF32X3 && k >= 64;
}

// The kernels one forward of `batch` samples runs (dlrm_forward_kernels).
// Per-stage timing and the phase trace keep the handle's own plan and kernel.
int forward_kind(const dlrm_handle_s* h, int batch) {
  if (h->path != DLRM_PATH_FUSED) return DLRM_KERNELS_LAYERWISE;
  const bool plain = h->events.empty() && !h->trace;
  if (h->layerwise_from > 0 && batch >= h->layerwise_from && plain) return DLRM_KERNELS_LAYERWISE;
  if (h->fused_tc) return DLRM_KERNELS_FUSED_TC;
  if (h->cluster_on && batch <= h->cluster_limit && !h->trace) return DLRM_KERNELS_FUSED_CLUSTER;
  return DLRM_KERNELS_FUSED;
}

dlrm_status_t run_forward(dlrm_handle_t h, const float* dense, const int64_t* indices,
                          const int64_t* offsets, float* out, int batch, cudaStream_t s) {
  cudaError_t e;
  const bool prof = !h->events.empty();
  int stage = 0;
  auto mark = [&]() -> bool {
    return !prof || cudaEventRecord(h->events[stage++], s) == cudaSuccess;
  };
  if (!mark()) return DLRM_ERR_CUDA;
  const int kind = forward_kind(h, batch);
  if (kind != DLRM_KERNELS_LAYERWISE) {
    // the whole forward in one launch
    dlrm::FusedParams p = h->fused;
    p.batch = batch;
    p.dense = dense;
    p.indices = indices;
    p.offsets = offsets;
    p.out = out;
    p.err = h->err;
    p.trace = h->trace;
    p.wait = h->wait;
    if (kind == DLRM_KERNELS_FUSED_TC) {
      dlrm::FusedTcParams q = h->tcp;
      q.batch = batch;
      q.dense = dense;
      q.indices = indices;
      q.offsets = offsets;
      q.out = out;
      q.err = h->err;
      q.trace = h->trace;
      q.wait = h->wait;
      e = dlrm::launch_fused_tc(q, s);
    } else if (kind == DLRM_KERNELS_FUSED_CLUSTER) {
      // clusters of 8 for the smallest batches, else of 4 (when planned);
      // then the smallest tile height whose tiles fit one wave of clusters,
      // else the tallest available
      const bool have8 = h->cmax[0][0] + h->cmax[0][1] + h->cmax[0][2] > 0;
      const bool have4 = h->cmax[1][0] + h->cmax[1][1] + h->cmax[1][2] > 0;
      const int ci = (have4 && (batch > kWideClusterMaxBatch || !have8)) ? 1 : 0;
      int hi = -1;
      for (int i = 0; i < 3 && hi < 0; ++i) {
        const int bm = dlrm::kClusterTileRows[i];
        if (h->cmax[ci][i] > 0 && (batch + bm - 1) / bm <= h->cmax[ci][i]) hi = i;
      }
      for (int i = 2; i >= 0 && hi < 0; --i)
        if (h->cmax[ci][i] > 0) hi = i;
      dlrm::ClusterParams q = h->cparams[ci][hi];
      q.batch = batch;
      q.dense = dense;
      q.indices = indices;
      q.offsets = offsets;
      q.out = out;
      q.err = h->err;
      q.wait = h->wait;
      e = dlrm::launch_fused_cluster(q, s);
    } else {
      e = dlrm::launch_fused(p, h->fused_bm, s);
    }
    if (e != cudaSuccess || !mark()) return DLRM_ERR_CUDA;
  } else {
    // [G] bag sums, all tables in one launch
    e = dlrm::launch_gather(h->tabs, h->k, h->d, indices, offsets, batch, h->bag, h->emb,
                            h->err, s);
    if (e != cudaSuccess || !mark()) return DLRM_ERR_CUDA;
    // [M1] bottom MLP, ReLU after every layer
    const float* in = dense;
    int ld_in = h->n_dense;
    // GEMMs on the tensor cores: the warp-specialized TMA GEMM where the
    // layer has a TMA plan (TF32, and split-TF32 in FP32 / TF32X3; input in a
    // buffer of the handle), else the staged tcgen05 GEMM in the opt-in
    // modes. Everything else, among it the N = 1 sigmoid layer (a dot product
    // per row), runs on the FFMA pipe.
    auto linear = [&](int layer, const float* x, int ldx, const float* w, int ldw,
                      const float* b, float* y, int ldy, int n, int k, int act) {
      if (!h->tma_on.empty() && h->tma_on[layer])
        return dlrm::launch_linear_tma(h->tma[layer], batch, b, y, ldy, act, h->err, s, h->wait);
      if (staged_tc_layer(h->math, n, k))
        return dlrm::launch_linear_tc(x, ldx, w, ldw, b, y, ldy, batch, n, k, act,
                                      static_cast<int>(h->math), h->err, s, h->wait);
      return dlrm::launch_linear_fp32(x, ldx, w, ldw, b, y, ldy, batch, n, k, act, s);
    };
    for (int l = 0; l < h->n_bot; ++l) {
      float* o = h->act[l & 1];
      e = linear(l, in, ld_in, h->bot_w[l], h->bot_ldw[l], h->bot_b[l], o, h->ld_act,
                 h->ln_bot[l + 1], h->ln_bot[l], DLRM_ACT_RELU);
      if (e != cudaSuccess || !mark()) return DLRM_ERR_CUDA;
      in = o;
      ld_in = h->ld_act;
    }
    // [I] interaction; R = [x, z]
    e = dlrm::launch_interaction(in, ld_in, h->emb, batch, h->k, h->d, h->r, h->ld_r, 1, s);
    if (e != cudaSuccess || !mark()) return DLRM_ERR_CUDA;
    // [M2] top MLP: ReLU, ..., sigmoid into out
    in = h->r;
    ld_in = h->ld_r;
    for (int l = 0; l < h->n_top; ++l) {
      const bool last = (l == h->n_top - 1);
      float* o = last ? out : h->act[l & 1];
      const int ld_o = last ? 1 : h->ld_act;
      e = linear(h->n_bot + l, in, ld_in, h->top_w[l], h->top_ldw[l], h->top_b[l], o, ld_o,
                 h->ln_top[l + 1], h->ln_top[l], last ? DLRM_ACT_SIGMOID : DLRM_ACT_RELU);
      if (e != cudaSuccess || !mark()) return DLRM_ERR_CUDA;
      in = o;
      ld_in = ld_o;
    }
  }  // layer-wise
  if (prof) {
    if (cudaEventSynchronize(h->events.back()) != cudaSuccess) return DLRM_ERR_CUDA;
    for (size_t i = 0; i + 1 < h->events.size(); ++i) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, h->events[i], h->events[i + 1]) != cudaSuccess)
        return DLRM_ERR_CUDA;
      h->stage_ms[i] += ms;
    }
    ++h->profiled_calls;
  }
  return DLRM_OK;
}

void destroy_events(dlrm_handle_t h) {
  for (cudaEvent_t ev : h->events) cudaEventDestroy(ev);
  h->events.clear();
}

// Host copies of the (out, in) weights and biases (host or device pointers,
// read with cudaMemcpyDefault), bottom layers then top, for the fused planner.
bool host_params(dlrm_handle_t h, const float* const* bot_w, const float* const* bot_b,
                 const float* const* top_w, const float* const* top_b,
                 std::vector<std::vector<float>>* w, std::vector<std::vector<float>>* b) {
  w->clear();
  b->clear();
  for (int side = 0; side < 2; ++side) {
    const std::vector<int>& ln = side == 0 ? h->ln_bot : h->ln_top;
    const float* const* ws = side == 0 ? bot_w : top_w;
    const float* const* bs = side == 0 ? bot_b : top_b;
    for (size_t l = 0; l + 1 < ln.size(); ++l) {
      w->emplace_back(static_cast<size_t>(ln[l]) * ln[l + 1]);
      b->emplace_back(ln[l + 1]);
      if (cudaMemcpy(w->back().data(), ws[l], w->back().size() * sizeof(float),
                     cudaMemcpyDefault) != cudaSuccess ||
          cudaMemcpy(b->back().data(), bs[l], b->back().size() * sizeof(float),
                     cudaMemcpyDefault) != cudaSuccess)
        return false;
    }
  }
  return true;
}

// validate() shape rules ([P4] dlrm_megakernel.rs) and the library's own
// limits, on the config alone: at least one layer each side, widths chain,
// ln_bot.last() = m_spa, ln_top[0] = m_spa + n_pairs, ln_top.last() = 1.
dlrm_status_t check_config(const dlrm_config_t* cfg, size_t smem_limit) {
  if (!cfg->ln_bot || !cfg->ln_top || !cfg->rows) return DLRM_ERR_INVALID_ARG;
  if (cfg->n_bot < 1 || cfg->n_top < 1) return DLRM_ERR_INVALID_ARG;
  if (cfg->n_bot > DLRM_MAX_LAYERS || cfg->n_top > DLRM_MAX_LAYERS) return DLRM_ERR_UNSUPPORTED;
  if (cfg->n_tables < 1 || cfg->emb_dim < 1 || cfg->bag_size < 1 || cfg->max_batch < 1)
    return DLRM_ERR_INVALID_ARG;
  if (cfg->n_tables > DLRM_MAX_TABLES) return DLRM_ERR_UNSUPPORTED;
  for (int l = 0; l <= cfg->n_bot; ++l) if (cfg->ln_bot[l] < 1) return DLRM_ERR_INVALID_ARG;
  for (int l = 0; l <= cfg->n_top; ++l) if (cfg->ln_top[l] < 1) return DLRM_ERR_INVALID_ARG;
  const int64_t f = cfg->n_tables + 1;
  const int64_t p = f * (f - 1) / 2;
  if (cfg->ln_bot[cfg->n_bot] != cfg->emb_dim) return DLRM_ERR_INVALID_ARG;
  if (cfg->ln_top[0] != cfg->emb_dim + p) return DLRM_ERR_INVALID_ARG;
  if (cfg->ln_top[cfg->n_top] != 1) return DLRM_ERR_INVALID_ARG;
  for (int t = 0; t < cfg->n_tables; ++t) if (cfg->rows[t] < 1) return DLRM_ERR_INVALID_ARG;
  if (static_cast<int64_t>(cfg->max_batch) * cfg->bag_size > (int64_t(1) << 31))
    return DLRM_ERR_UNSUPPORTED;
  if (cfg->math != DLRM_MATH_FP32 && cfg->math != DLRM_MATH_TF32 &&
      cfg->math != DLRM_MATH_BF16 && cfg->math != DLRM_MATH_TF32X3 &&
      cfg->math != DLRM_MATH_FP32_FFMA)
    return DLRM_ERR_INVALID_ARG;
  if (cfg->path != DLRM_PATH_AUTO && cfg->path != DLRM_PATH_LAYERWISE &&
      cfg->path != DLRM_PATH_FUSED)
    return DLRM_ERR_INVALID_ARG;
  // fused plans: fp32 (SIMT) and the TF32 / BF16 tensor-core modes; TF32X3 is
  // layer-wise only
  if (cfg->math == DLRM_MATH_TF32X3 && cfg->path == DLRM_PATH_FUSED) return DLRM_ERR_UNSUPPORTED;
  if (dlrm::interaction_smem_per_sample(cfg->n_tables, cfg->emb_dim) > smem_limit)
    return DLRM_ERR_UNSUPPORTED;
  return DLRM_OK;
}

// The fused planner is consulted unless the layer-wise plan was asked for or
// the math has no fused kernel (TF32X3).
bool wants_fused_plan(const dlrm_config_t* cfg) {
  return cfg->path != DLRM_PATH_LAYERWISE && (fp32_math(cfg->math) || tensor_core_math(cfg->math));
}

// The batch from which the layer-wise plan (its large GEMMs as split-TF32 on
// the tensor cores, launches overlapped) replaces the fp32 fused kernel. The
// fused kernel is persistent: one wave of `sms` tiles of `bm` samples runs in
// the time of one tile, and the next sample starts a second round. Measured
// on the 13-512-256-64 / (64 + P)-512-256-1 models (L2 flushed), the
// layer-wise plan takes ~70-90 us from 1024 to 4096 samples, while the fused
// kernel's round takes ~3.13e-8 us per MLP flop plus ~2.04e-7 us per pair-dot
// flop per sample of the wave (41.5 us at 3 tables, 104 at 32). So the switch
// is at the first sample of the second round, when the estimated layer-wise
// time (70 us plus a third of the fused per-sample cost per sample) is below
// two fused rounds there; never for models whose fused round is short (the
// 64-wide model) or that have no split-TF32 layer. Measured crossovers: ~3000
// samples with 3 tables (2200: layer-wise 74 against fused ~75), ~2800 with 16,
// ~2100 with 32.
int64_t layerwise_crossover(const dlrm_config_t* cfg, int bm, int sms) {
  double mlp = 0.0;
  bool split_layer = false;
  for (int g = 0; g < cfg->n_bot + cfg->n_top; ++g) {
    const bool top = g >= cfg->n_bot;
    const int l = top ? g - cfg->n_bot : g;
    const int n = top ? cfg->ln_top[l + 1] : cfg->ln_bot[l + 1];
    const int k = top ? cfg->ln_top[l] : cfg->ln_bot[l];
    mlp += 2.0 * n * k;
    split_layer = split_layer || tma_layer(DLRM_MATH_FP32, g, n, k);
  }
  if (!split_layer || bm < 1 || sms < 1) return 0;
  const double f = cfg->n_tables + 1.0;
  const double pair_flops = f * (f - 1.0) * cfg->emb_dim;
  const double per_sample_us = 3.13e-8 * mlp + 2.04e-7 * pair_flops;
  const int64_t wave = static_cast<int64_t>(sms) * bm;
  const double fused_two_rounds = 4.5 + 2.0 * static_cast<double>(wave) * per_sample_us;
  const double layerwise = 70.0 + per_sample_us / 3.0 * static_cast<double>(wave + 1);
  return layerwise < fused_two_rounds ? wave + 1 : 0;
}

struct PlanChoice {
  int path = DLRM_PATH_LAYERWISE;
  bool fused_fits = false;
  bool fused_tc = false;    // the fused plan runs on the tensor cores
  int fused_bm = 0;         // samples per fused tile
  int64_t tiles = 0;        // fused tiles of max_batch
  int64_t layerwise_from = 0;   // AUTO fp32 fused plan: the layer-wise plan from this batch
};

// The kernel plan of a checked config, from host copies of the weights and
// biases (bottom layers then top; their values only fill the packed images)
// and the device's SM count and opt-in shared memory per block. The same
// call serves dlrm_create and dlrm_plan_query.
dlrm_status_t choose_plan(const dlrm_config_t* cfg, const std::vector<std::vector<float>>& hw,
                          const std::vector<std::vector<float>>& hb,
                          const dlrm::GatherTables& tabs, int sms, size_t smem_limit,
                          dlrm::FusedPlan* fplan, dlrm::FusedTcPlan* tplan, PlanChoice* c) {
  *c = PlanChoice{};
  const std::vector<int> ln_bot(cfg->ln_bot, cfg->ln_bot + cfg->n_bot + 1);
  const std::vector<int> ln_top(cfg->ln_top, cfg->ln_top + cfg->n_top + 1);
  const bool tc_math = tensor_core_math(cfg->math);
  if (wants_fused_plan(cfg)) {
    if (tc_math) {
      c->fused_fits = dlrm::fused_tc_plan(ln_bot[0], cfg->n_tables, cfg->emb_dim, cfg->bag_size,
                                          ln_bot, ln_top, hw, hb, tabs,
                                          static_cast<int>(cfg->math), smem_limit, tplan);
      c->fused_tc = c->fused_fits;
      c->fused_bm = dlrm::kTcTile;
    } else {
      const int cw = 8;   // computing warps of the fused kernel
      c->fused_fits = dlrm::fused_plan(ln_bot[0], cfg->n_tables, cfg->emb_dim, cfg->bag_size,
                                       ln_bot, ln_top, hw, hb, tabs, cfg->max_batch, sms,
                                       smem_limit, cw, fplan);
      c->fused_bm = fplan->bm;
    }
  }
  c->tiles = c->fused_fits ? (cfg->max_batch + c->fused_bm - 1) / c->fused_bm : 0;
  if (cfg->path == DLRM_PATH_FUSED) {
    if (!c->fused_fits) return DLRM_ERR_UNSUPPORTED;
    c->path = DLRM_PATH_FUSED;
  } else if (cfg->path == DLRM_PATH_AUTO) {
    // The fp32 fused kernel is persistent and beats the layer-wise launches at
    // every batch when bags hold one row (8192 samples: 171 vs 238 us); with
    // longer bags, gathered one row at a time inside the kernel, and for the
    // tensor-core kernel (one CTA per tile), it is kept to two waves of tiles.
    const bool persistent = !tc_math && cfg->bag_size == 1;
    c->path = (c->fused_fits && (persistent || c->tiles <= 2 * static_cast<int64_t>(sms)))
                  ? DLRM_PATH_FUSED
                  : DLRM_PATH_LAYERWISE;
    // large batches of the fp32 fused plan: the layer-wise split-TF32 plan
    if (c->path == DLRM_PATH_FUSED && cfg->math == DLRM_MATH_FP32) {
      const int64_t from = layerwise_crossover(cfg, c->fused_bm, sms);
      if (from > 0 && cfg->max_batch >= from) c->layerwise_from = from;
    }
  } else {
    c->path = DLRM_PATH_LAYERWISE;
  }
  if (c->path != DLRM_PATH_FUSED) c->fused_tc = false;
  return DLRM_OK;
}

// Inputs and output of a forward at their elements' natural alignment.
bool forward_args_aligned(const void* dense, const void* indices, const void* offsets,
                          const void* out) {
  return dlrm::aligned_to(dense, sizeof(float)) && dlrm::aligned_to(indices, sizeof(int64_t)) &&
         dlrm::aligned_to(offsets, sizeof(int64_t)) && dlrm::aligned_to(out, sizeof(float));
}

}  // namespace

extern "C" {

int32_t dlrm_version(void) { return 100; }

const char* dlrm_status_string(int32_t status) {
  switch (status) {
    case DLRM_OK: return "ok";
    case DLRM_ERR_INVALID_ARG: return "invalid argument";
    case DLRM_ERR_UNSUPPORTED: return "unsupported";
    case DLRM_ERR_CUDA: return "CUDA error";
    case DLRM_ERR_OOM: return "out of device memory";
    case DLRM_ERR_INDEX_OOB: return "index out of range";
    case DLRM_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

dlrm_status_t dlrm_create(const dlrm_config_t* cfg, const float* const* tables,
                          const float* const* bot_w, const float* const* bot_b,
                          const float* const* top_w, const float* const* top_b,
                          dlrm_handle_t* out) {
  if (!out) return DLRM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !tables || !bot_w || !bot_b || !top_w || !top_b) return DLRM_ERR_INVALID_ARG;
  const dlrm_status_t checked = check_config(cfg, dlrm::device_max_smem_optin());
  if (checked != DLRM_OK) return checked;
  for (int t = 0; t < cfg->n_tables; ++t)
    if (!tables[t] || !dlrm::aligned_to(tables[t], sizeof(float))) return DLRM_ERR_INVALID_ARG;
  for (int l = 0; l < cfg->n_bot; ++l) if (!bot_w[l] || !bot_b[l]) return DLRM_ERR_INVALID_ARG;
  for (int l = 0; l < cfg->n_top; ++l) if (!top_w[l] || !top_b[l]) return DLRM_ERR_INVALID_ARG;

  dlrm_handle_t h = new (std::nothrow) dlrm_handle_s();
  if (!h) return DLRM_ERR_OOM;
  cudaGetDevice(&h->device);
  h->n_bot = cfg->n_bot;
  h->n_top = cfg->n_top;
  h->k = cfg->n_tables;
  h->d = cfg->emb_dim;
  h->bag = cfg->bag_size;
  h->max_batch = cfg->max_batch;
  h->n_dense = cfg->ln_bot[0];
  h->math = cfg->math;
  h->ln_bot.assign(cfg->ln_bot, cfg->ln_bot + cfg->n_bot + 1);
  h->ln_top.assign(cfg->ln_top, cfg->ln_top + cfg->n_top + 1);
  for (int t = 0; t < h->k; ++t) {
    h->tabs.ptr[t] = tables[t];
    h->tabs.rows[t] = cfg->rows[t];
  }
  // Kernel plan.
  dlrm::FusedPlan fplan;
  dlrm::FusedTcPlan tplan;
  std::vector<std::vector<float>> hw, hb;
  if (wants_fused_plan(cfg) && !host_params(h, bot_w, bot_b, top_w, top_b, &hw, &hb)) {
    cudaGetLastError();
    delete h;
    return DLRM_ERR_CUDA;
  }
  PlanChoice choice;
  const dlrm_status_t planned =
      choose_plan(cfg, hw, hb, h->tabs, dlrm::device_sm_count(), dlrm::device_max_smem_optin(),
                  &fplan, &tplan, &choice);
  if (planned != DLRM_OK) {
    delete h;
    return planned;
  }
  h->path = choice.path;
  h->fused_tc = choice.fused_tc;
  h->fused_bm = choice.fused_bm;
  h->layerwise_from = choice.layerwise_from;
  if (h->path == DLRM_PATH_FUSED) {
    h->stage_names.push_back("fused");
  } else {
    h->stage_names.push_back("gather");
    for (int l = 0; l < h->n_bot; ++l) h->stage_names.push_back("bottom" + std::to_string(l));
    h->stage_names.push_back("interaction");
    for (int l = 0; l < h->n_top; ++l) h->stage_names.push_back("top" + std::to_string(l));
  }
  h->stage_ms.assign(h->stage_names.size(), 0.0);

  // Layout of the arena.
  int widest = 4;
  for (int l = 1; l <= h->n_bot; ++l) widest = std::max(widest, h->ln_bot[l]);
  for (int l = 1; l < h->n_top; ++l) widest = std::max(widest, h->ln_top[l]);
  h->ld_act = static_cast<int>(round_up(widest, 4));
  h->ld_r = static_cast<int>(round_up(h->ln_top[0], 4));
  const size_t mb = static_cast<size_t>(h->max_batch);
  ArenaPlan plan;
  std::vector<size_t> off_bw(h->n_bot), off_bb(h->n_bot), off_tw(h->n_top), off_tb(h->n_top);
  h->bot_ldw.resize(h->n_bot);
  h->top_ldw.resize(h->n_top);
  for (int l = 0; l < h->n_bot; ++l) {
    h->bot_ldw[l] = static_cast<int>(round_up(h->ln_bot[l], 4));
    off_bw[l] = plan.take<float>(static_cast<size_t>(h->ln_bot[l + 1]) * h->bot_ldw[l]);
    off_bb[l] = plan.take<float>(h->ln_bot[l + 1]);
  }
  for (int l = 0; l < h->n_top; ++l) {
    h->top_ldw[l] = static_cast<int>(round_up(h->ln_top[l], 4));
    off_tw[l] = plan.take<float>(static_cast<size_t>(h->ln_top[l + 1]) * h->top_ldw[l]);
    off_tb[l] = plan.take<float>(h->ln_top[l + 1]);
  }
  const size_t off_emb = plan.take<float>(mb * h->k * h->d);
  const size_t off_a0 = plan.take<float>(mb * h->ld_act);
  const size_t off_a1 = plan.take<float>(mb * h->ld_act);
  const size_t off_r = plan.take<float>(mb * h->ld_r);
  const size_t off_err = plan.take<int32_t>(4);
  const size_t off_dense = plan.take<float>(mb * h->n_dense);
  const size_t off_idx = plan.take<int64_t>(mb * h->k * h->bag);
  const size_t off_off = plan.take<int64_t>(mb * h->k);
  const size_t off_out = plan.take<float>(mb);
  // Layer-wise plan: the warp-specialized TMA GEMM for the layers tma_layer
  // picks; in split-TF32 (FP32, TF32X3) their weights get two more copies:
  // their tf32 head and the remainder.
  const bool tma_math = (h->path == DLRM_PATH_LAYERWISE || h->layerwise_from > 0) &&
                        (tensor_core_math(h->math) || split_tf32_math(h->math));
  const bool split = split_tf32_math(h->math);
  const int n_layers = h->n_bot + h->n_top;
  std::vector<size_t> off_whi(n_layers, 0), off_wlo(n_layers, 0);
  std::vector<char> want_tma(n_layers, 0);
  auto layer_shape = [&](int g, int* n, int* k, int* ldw) {
    const bool top = g >= h->n_bot;
    const int l = top ? g - h->n_bot : g;
    *n = top ? h->ln_top[l + 1] : h->ln_bot[l + 1];
    *k = top ? h->ln_top[l] : h->ln_bot[l];
    *ldw = top ? h->top_ldw[l] : h->bot_ldw[l];
  };
  if (tma_math) {
    for (int g = 1; g < n_layers; ++g) {
      int n, k, ldw;
      layer_shape(g, &n, &k, &ldw);
      if (!tma_layer(h->math, g, n, k)) continue;
      want_tma[g] = 1;
      if (split) {
        off_whi[g] = plan.take<float>(static_cast<size_t>(n) * ldw);
        off_wlo[g] = plan.take<float>(static_cast<size_t>(n) * ldw);
      }
    }
  }
  // fused weight stream, its stage table, biases, last layer
  size_t off_fw = 0, off_ft = 0, off_fb = 0, off_fl = 0;
  if (h->path == DLRM_PATH_FUSED && h->fused_tc) {
    off_fw = plan.take<unsigned char>(tplan.wstream.size());
    off_fb = plan.take<float>(tplan.bias.size());
    off_fl = plan.take<float>(tplan.wlast.size());
  } else if (h->path == DLRM_PATH_FUSED) {
    off_fw = plan.take<float>(fplan.wstream.size());
    off_ft = plan.take<uint2>(fplan.stage_tab.size());
    off_fb = plan.take<float>(fplan.bias.size());
    off_fl = plan.take<float>(fplan.wlast.size());
  }
  // the cluster-split kernel's weight streams, stage table, bias blocks
  dlrm::ClusterPlan cplan[2];
  bool cluster_planned[2] = {false, false};
  size_t off_cw[2] = {0, 0}, off_ct[2] = {0, 0}, off_cb[2] = {0, 0}, off_cl[2] = {0, 0};
  if (h->path == DLRM_PATH_FUSED && !h->fused_tc &&
      fplan.wstream.size() * sizeof(float) >= kClusterMinStreamBytes) {
    for (int ci = 0; ci < 2; ++ci) {
      cluster_planned[ci] = dlrm::fused_cluster_plan(
          h->n_dense, h->k, h->d, h->bag, h->ln_bot, h->ln_top, hw, hb, h->tabs,
          kClusterSizes[ci], dlrm::device_max_smem_optin(), &cplan[ci]);
      if (cluster_planned[ci]) {
        off_cw[ci] = plan.take<float>(cplan[ci].wstream.size());
        off_ct[ci] = plan.take<uint2>(cplan[ci].stage_tab.size());
        off_cb[ci] = plan.take<float>(cplan[ci].bias.size());
        off_cl[ci] = plan.take<float>(cplan[ci].wlast.size());
      }
    }
  }

  if (cudaMalloc(&h->arena, plan.bytes) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return DLRM_ERR_OOM;
  }
  h->arena_bytes = plan.bytes;
  char* base = static_cast<char*>(h->arena);
  auto at = [&](size_t off) { return reinterpret_cast<float*>(base + off); };
  dlrm_status_t st = cuda_status(cudaMemset(h->arena, 0, plan.bytes));
  for (int l = 0; l < h->n_bot && st == DLRM_OK; ++l) {
    h->bot_w.push_back(at(off_bw[l]));
    h->bot_b.push_back(at(off_bb[l]));
    st = cuda_status(cudaMemcpy2D(at(off_bw[l]), h->bot_ldw[l] * sizeof(float), bot_w[l],
                                  h->ln_bot[l] * sizeof(float), h->ln_bot[l] * sizeof(float),
                                  h->ln_bot[l + 1], cudaMemcpyDefault));
    if (st == DLRM_OK)
      st = cuda_status(cudaMemcpy(at(off_bb[l]), bot_b[l], h->ln_bot[l + 1] * sizeof(float),
                                  cudaMemcpyDefault));
  }
  for (int l = 0; l < h->n_top && st == DLRM_OK; ++l) {
    h->top_w.push_back(at(off_tw[l]));
    h->top_b.push_back(at(off_tb[l]));
    st = cuda_status(cudaMemcpy2D(at(off_tw[l]), h->top_ldw[l] * sizeof(float), top_w[l],
                                  h->ln_top[l] * sizeof(float), h->ln_top[l] * sizeof(float),
                                  h->ln_top[l + 1], cudaMemcpyDefault));
    if (st == DLRM_OK)
      st = cuda_status(cudaMemcpy(at(off_tb[l]), top_b[l], h->ln_top[l + 1] * sizeof(float),
                                  cudaMemcpyDefault));
  }
  if (h->path == DLRM_PATH_FUSED && h->fused_tc && st == DLRM_OK) {
    st = cuda_status(cudaMemcpy(at(off_fw), tplan.wstream.data(), tplan.wstream.size(),
                                cudaMemcpyHostToDevice));
    if (st == DLRM_OK)
      st = cuda_status(cudaMemcpy(at(off_fb), tplan.bias.data(), tplan.bias.size() * sizeof(float),
                                  cudaMemcpyHostToDevice));
    if (st == DLRM_OK)
      st = cuda_status(cudaMemcpy(at(off_fl), tplan.wlast.data(),
                                  tplan.wlast.size() * sizeof(float), cudaMemcpyHostToDevice));
    h->tcp = tplan.params;
    h->tcp.wstream = reinterpret_cast<const unsigned char*>(at(off_fw));
    h->tcp.bias = at(off_fb);
    h->tcp.wlast = at(off_fl);
    if (st == DLRM_OK) st = cuda_status(dlrm::fused_tc_prepare(h->tcp.bf16));
  } else if (h->path == DLRM_PATH_FUSED && st == DLRM_OK) {
    st = cuda_status(cudaMemcpy(at(off_fw), fplan.wstream.data(),
                                fplan.wstream.size() * sizeof(float), cudaMemcpyHostToDevice));
    if (st == DLRM_OK)
      st = cuda_status(cudaMemcpy(at(off_ft), fplan.stage_tab.data(),
                                  fplan.stage_tab.size() * sizeof(uint2), cudaMemcpyHostToDevice));
    if (st == DLRM_OK)
      st = cuda_status(cudaMemcpy(at(off_fb), fplan.bias.data(), fplan.bias.size() * sizeof(float),
                                  cudaMemcpyHostToDevice));
    if (st == DLRM_OK)
      st = cuda_status(cudaMemcpy(at(off_fl), fplan.wlast.data(),
                                  fplan.wlast.size() * sizeof(float), cudaMemcpyHostToDevice));
    h->fused = fplan.params;
    h->fused.wstream = at(off_fw);
    h->fused.stage_tab = reinterpret_cast<const uint2*>(at(off_ft));
    h->fused.bias = at(off_fb);
    h->fused.wlast = at(off_fl);
    if (st == DLRM_OK) st = cuda_status(dlrm::fused_prepare(h->fused_bm, h->fused.cw, dlrm::fused_instance_lda(h->fused)));
  }
  int cluster_limit = 0;
  for (int ci = 0; ci < 2 && st == DLRM_OK; ++ci) {
    if (!cluster_planned[ci]) continue;
    const dlrm::ClusterPlan& cp = cplan[ci];
    st = cuda_status(cudaMemcpy(at(off_cw[ci]), cp.wstream.data(),
                                cp.wstream.size() * sizeof(float), cudaMemcpyHostToDevice));
    if (st == DLRM_OK)
      st = cuda_status(cudaMemcpy(at(off_ct[ci]), cp.stage_tab.data(),
                                  cp.stage_tab.size() * sizeof(uint2), cudaMemcpyHostToDevice));
    if (st == DLRM_OK)
      st = cuda_status(cudaMemcpy(at(off_cb[ci]), cp.bias.data(), cp.bias.size() * sizeof(float),
                                  cudaMemcpyHostToDevice));
    if (st == DLRM_OK)
      st = cuda_status(cudaMemcpy(at(off_cl[ci]), cp.wlast.data(),
                                  cp.wlast.size() * sizeof(float), cudaMemcpyHostToDevice));
    for (int i = 0; i < 3 && st == DLRM_OK; ++i) {
      if (!cp.fits[i]) continue;
      dlrm::ClusterParams& q = h->cparams[ci][i];
      q = cp.params[i];
      q.wstream = at(off_cw[ci]);
      q.stage_tab = reinterpret_cast<const uint2*>(at(off_ct[ci]));
      q.bias = at(off_cb[ci]);
      q.wlast = at(off_cl[ci]);
      h->cmax[ci][i] = dlrm::fused_cluster_max_active(q.bm, q.csize, q.smem_bytes);
      cluster_limit = std::max(cluster_limit, h->cmax[ci][i] * q.bm);
    }
  }
  h->cluster_default = std::min(cluster_limit, cluster_max_batch(h->k));
  h->cluster_limit = h->cluster_default;
  h->cluster_on = h->cluster_limit > 0;
  if (st == DLRM_OK) st = cuda_status(cudaDeviceSynchronize());
  if (st != DLRM_OK) {
    cudaGetLastError();
    cudaFree(h->arena);
    delete h;
    return st;
  }
  h->emb = at(off_emb);
  h->act[0] = at(off_a0);
  h->act[1] = at(off_a1);
  h->r = at(off_r);
  h->err = reinterpret_cast<int32_t*>(base + off_err);
  h->dense_stage = at(off_dense);
  h->idx_stage = reinterpret_cast<int64_t*>(base + off_idx);
  h->off_stage = reinterpret_cast<int64_t*>(base + off_off);
  h->out_stage = at(off_out);
  if (tma_math) {
    // tensor maps of each TMA layer's input buffer (max_batch rows) and of
    // its weights; a layer whose maps cannot be made keeps the staged GEMM
    h->tma.resize(n_layers);
    h->tma_on.assign(n_layers, 0);
    for (int g = 1; g < n_layers && st == DLRM_OK; ++g) {
      if (!want_tma[g]) continue;
      int n, k, ldw;
      layer_shape(g, &n, &k, &ldw);
      const bool top = g >= h->n_bot;
      const int l = top ? g - h->n_bot : g;
      const float* in = (top && l == 0) ? h->r : h->act[(l - 1) & 1];
      const int ld_in = (top && l == 0) ? h->ld_r : h->ld_act;
      const float* w = top ? h->top_w[l] : h->bot_w[l];
      dlrm::TmaLayer& T = h->tma[g];
      T.n = n;
      T.k = k;
      T.split = split ? 1 : 0;
      const float* w_head = w;
      if (T.split) {
        // w = head + rest: head keeps the top 10 mantissa bits (exact in
        // tf32), rest = w - head is exact in fp32
        const size_t count = static_cast<size_t>(n) * ldw;
        std::vector<float> hw(count), hi(count), lo(count);
        st = cuda_status(cudaMemcpy(hw.data(), w, count * sizeof(float), cudaMemcpyDeviceToHost));
        if (st != DLRM_OK) break;
        for (size_t i = 0; i < count; ++i) {
          uint32_t bits;
          std::memcpy(&bits, &hw[i], sizeof(bits));
          bits &= 0xFFFFE000u;
          std::memcpy(&hi[i], &bits, sizeof(bits));
          lo[i] = hw[i] - hi[i];
        }
        st = cuda_status(cudaMemcpy(at(off_whi[g]), hi.data(), count * sizeof(float),
                                    cudaMemcpyHostToDevice));
        if (st == DLRM_OK)
          st = cuda_status(cudaMemcpy(at(off_wlo[g]), lo.data(), count * sizeof(float),
                                      cudaMemcpyHostToDevice));
        if (st != DLRM_OK) break;
        w_head = at(off_whi[g]);
      }
      const bool ok =
          dlrm::encode_operand_map(T.map_x, in, k, h->max_batch, ld_in, 128) &&
          dlrm::encode_operand_map(T.map_w, w_head, k, n, ldw, 64) &&
          (!T.split || dlrm::encode_operand_map(T.map_wlo, at(off_wlo[g]), k, n, ldw, 64));
      h->tma_on[g] = ok ? 1 : 0;
    }
    if (st != DLRM_OK) {
      cudaGetLastError();
      cudaFree(h->arena);
      delete h;
      return st;
    }
  }
  // DLRM_PROFILE=1: per-stage timing from the first forward on, reported on
  // stderr by dlrm_destroy (the same counters dlrm_stage_times returns)
  const char* prof = std::getenv("DLRM_PROFILE");
  if (prof && prof[0] == '1' && prof[1] == '\0') {
    if (dlrm_set_profiling(h, 1) != DLRM_OK) {
      dlrm_destroy(h);
      return DLRM_ERR_CUDA;
    }
    h->report_on_destroy = true;
  }
  *out = h;
  return DLRM_OK;
}

dlrm_status_t dlrm_plan_query(const dlrm_config_t* cfg, int32_t sm_count, int64_t smem_per_block,
                              dlrm_plan_info_t* info) {
  if (!cfg || !info || sm_count < 1 || smem_per_block < 1) return DLRM_ERR_INVALID_ARG;
  const size_t smem = static_cast<size_t>(smem_per_block);
  const dlrm_status_t checked = check_config(cfg, smem);
  if (checked != DLRM_OK) return checked;
  // zero weights of the model's shapes: the plan depends on shapes alone
  std::vector<std::vector<float>> hw, hb;
  if (wants_fused_plan(cfg)) {
    for (int side = 0; side < 2; ++side) {
      const int32_t* ln = side == 0 ? cfg->ln_bot : cfg->ln_top;
      const int n = side == 0 ? cfg->n_bot : cfg->n_top;
      for (int l = 0; l < n; ++l) {
        hw.emplace_back(static_cast<size_t>(ln[l]) * ln[l + 1], 0.f);
        hb.emplace_back(ln[l + 1], 0.f);
      }
    }
  }
  dlrm::GatherTables tabs{};   // null table pointers pass the 16-byte alignment test
  dlrm::FusedPlan fplan;
  dlrm::FusedTcPlan tplan;
  PlanChoice c;
  const dlrm_status_t planned = choose_plan(cfg, hw, hb, tabs, sm_count, smem, &fplan, &tplan, &c);
  if (planned != DLRM_OK) return planned;
  dlrm_plan_info_t r{};
  r.path = c.path;
  r.fused_fits = c.fused_fits ? 1 : 0;
  if (c.fused_fits) {
    const bool tc = tensor_core_math(cfg->math);
    r.tensor_core = tc ? 1 : 0;
    r.tile_samples = c.fused_bm;
    r.tiles = c.tiles;
    r.grid = static_cast<int32_t>(tc ? c.tiles : std::min<int64_t>(c.tiles, sm_count));
    r.smem_bytes = tc ? tplan.params.smem_bytes : fplan.params.smem_bytes;
    r.ring_stages = tc ? tplan.params.stages : fplan.params.stages;
    r.stream_copies = tc ? tplan.params.n_tiles : fplan.params.n_stages;
    r.stream_bytes = tc ? static_cast<int64_t>(tplan.wstream.size())
                        : static_cast<int64_t>(fplan.wstream.size() * sizeof(float));
  }
  r.layerwise_from = c.layerwise_from;
  if (c.path == DLRM_PATH_LAYERWISE || c.layerwise_from > 0) {
    for (int g = 0; g < cfg->n_bot + cfg->n_top; ++g) {
      const bool top = g >= cfg->n_bot;
      const int l = top ? g - cfg->n_bot : g;
      const int n = top ? cfg->ln_top[l + 1] : cfg->ln_bot[l + 1];
      const int k = top ? cfg->ln_top[l] : cfg->ln_bot[l];
      if (tma_layer(cfg->math, g, n, k) || staged_tc_layer(cfg->math, n, k))
        r.tensor_core_layers |= 1 << g;
    }
    r.split_tf32 = (r.tensor_core_layers && split_tf32_math(cfg->math)) ? 1 : 0;
  }
  *info = r;
  return DLRM_OK;
}

dlrm_status_t dlrm_forward(dlrm_handle_t h, const float* dense, const int64_t* indices,
                           const int64_t* offsets, float* out, int32_t batch, void* stream) {
  if (!h || !dense || !indices || !offsets || !out) return DLRM_ERR_INVALID_ARG;
  if (!forward_args_aligned(dense, indices, offsets, out)) return DLRM_ERR_INVALID_ARG;
  if (batch < 1 || batch > h->max_batch) return DLRM_ERR_INVALID_ARG;
  return run_forward(h, dense, indices, offsets, out, batch, static_cast<cudaStream_t>(stream));
}

namespace {

// Device address of a host buffer the GPU can reach directly (pinned and
// mapped: on GB300 host memory is coherent over NVLink-C2C), else null.
const void* device_view(const void* host) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return (a.type == cudaMemoryTypeHost && a.devicePointer) ? a.devicePointer : nullptr;
}

}  // namespace

dlrm_status_t dlrm_forward_host(dlrm_handle_t h, const float* dense_host,
                                const int64_t* indices_host, const int64_t* offsets_host,
                                float* out_host, int32_t batch, void* stream) {
  if (!h || !dense_host || !indices_host || !offsets_host || !out_host)
    return DLRM_ERR_INVALID_ARG;
  if (!forward_args_aligned(dense_host, indices_host, offsets_host, out_host))
    return DLRM_ERR_INVALID_ARG;
  if (batch < 1 || batch > h->max_batch) return DLRM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t nb = static_cast<size_t>(batch);
  // Pinned buffers are read and written in place by the kernels; any other
  // buffer goes through the handle's staging area with one copy each way.
  const float* dense = static_cast<const float*>(device_view(dense_host));
  const int64_t* idx = static_cast<const int64_t*>(device_view(indices_host));
  const int64_t* off = static_cast<const int64_t*>(device_view(offsets_host));
  float* out = static_cast<float*>(const_cast<void*>(device_view(out_host)));
  if (!dense) {
    if (cudaMemcpyAsync(h->dense_stage, dense_host, nb * h->n_dense * sizeof(float),
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
      return DLRM_ERR_CUDA;
    dense = h->dense_stage;
  }
  if (!idx) {
    if (cudaMemcpyAsync(h->idx_stage, indices_host, nb * h->k * h->bag * sizeof(int64_t),
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
      return DLRM_ERR_CUDA;
    idx = h->idx_stage;
  }
  if (!off) {
    if (cudaMemcpyAsync(h->off_stage, offsets_host, nb * h->k * sizeof(int64_t),
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
      return DLRM_ERR_CUDA;
    off = h->off_stage;
  }
  dlrm_status_t st = run_forward(h, dense, idx, off, out ? out : h->out_stage, batch, s);
  if (st != DLRM_OK || out) return st;
  return cuda_status(cudaMemcpyAsync(out_host, h->out_stage, nb * sizeof(float),
                                     cudaMemcpyDeviceToHost, s));
}

dlrm_status_t dlrm_get_error(dlrm_handle_t h, void* stream) {
  if (!h) return DLRM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DLRM_ERR_CUDA;
  int32_t word = 0;
  if (cudaMemcpy(&word, h->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DLRM_ERR_CUDA;
  if (word != 0 && cudaMemset(h->err, 0, sizeof(int32_t)) != cudaSuccess) return DLRM_ERR_CUDA;
  const uint32_t bits = static_cast<uint32_t>(word);
  if (bits & DLRM_ERRBIT_INDEX_OOB) return DLRM_ERR_INDEX_OOB;
  if (bits & DLRM_ERRBIT_OFFSETS) return DLRM_ERR_UNSUPPORTED;
  if (bits & DLRM_ERRBIT_TIMEOUT) return DLRM_ERR_TIMEOUT;
  return DLRM_OK;
}

dlrm_status_t dlrm_test_stall(dlrm_handle_t h, int64_t wait_limit_ns, int32_t withhold_last) {
  if (!h || wait_limit_ns < 0) return DLRM_ERR_INVALID_ARG;
  h->wait.limit_ns = static_cast<uint64_t>(wait_limit_ns);
  h->wait.withhold_last = withhold_last ? 1 : 0;
  return DLRM_OK;
}

int32_t dlrm_forward_kernels(dlrm_handle_t h, int32_t batch) {
  if (!h || batch < 1 || batch > h->max_batch) return -1;
  return forward_kind(h, batch);
}

dlrm_status_t dlrm_set_cluster_batch_limit(dlrm_handle_t h, int32_t limit) {
  if (!h || limit < -1) return DLRM_ERR_INVALID_ARG;
  const bool planned = h->cluster_default > 0;
  if (limit == -1) {
    h->cluster_limit = h->cluster_default;
  } else {
    if (limit > 0 && !planned) return DLRM_ERR_UNSUPPORTED;
    h->cluster_limit = limit;
  }
  h->cluster_on = planned && h->cluster_limit > 0;
  return DLRM_OK;
}

dlrm_status_t dlrm_get_cluster_batch_limit(dlrm_handle_t h, int32_t* limit) {
  if (!h || !limit) return DLRM_ERR_INVALID_ARG;
  *limit = h->cluster_on ? h->cluster_limit : 0;
  return DLRM_OK;
}

int64_t dlrm_workspace_bytes(dlrm_handle_t h) {
  return h ? static_cast<int64_t>(h->arena_bytes) : 0;
}

int32_t dlrm_path(dlrm_handle_t h) { return h ? h->path : -1; }

dlrm_status_t dlrm_set_phase_trace(dlrm_handle_t h, uint64_t* buf, int64_t capacity,
                                   int32_t* tile_rows) {
  static_assert(DLRM_TRACE_SLOTS == dlrm::kFusedTraceSlots, "trace slot count");
  if (!h) return DLRM_ERR_INVALID_ARG;
  if (h->path != DLRM_PATH_FUSED) return DLRM_ERR_UNSUPPORTED;
  if (tile_rows) *tile_rows = h->fused_bm;
  if (!buf) {
    h->trace = nullptr;
    return DLRM_OK;
  }
  if (!dlrm::aligned_to(buf, sizeof(uint64_t))) return DLRM_ERR_INVALID_ARG;
  const int64_t tiles = (h->max_batch + h->fused_bm - 1) / h->fused_bm;
  if (capacity < tiles * DLRM_TRACE_SLOTS) return DLRM_ERR_INVALID_ARG;
  h->trace = reinterpret_cast<unsigned long long*>(buf);
  return DLRM_OK;
}

int32_t dlrm_num_stages(dlrm_handle_t h) {
  return h ? static_cast<int32_t>(h->stage_names.size()) : 0;
}

const char* dlrm_stage_name(dlrm_handle_t h, int32_t i) {
  if (!h || i < 0 || i >= static_cast<int32_t>(h->stage_names.size())) return nullptr;
  return h->stage_names[i].c_str();
}

dlrm_status_t dlrm_set_profiling(dlrm_handle_t h, int32_t enable) {
  if (!h) return DLRM_ERR_INVALID_ARG;
  destroy_events(h);
  h->stage_ms.assign(h->stage_names.size(), 0.0);
  h->profiled_calls = 0;
  if (!enable) return DLRM_OK;
  for (size_t i = 0; i <= h->stage_names.size(); ++i) {
    cudaEvent_t ev;
    if (cudaEventCreate(&ev) != cudaSuccess) {
      destroy_events(h);
      return DLRM_ERR_CUDA;
    }
    h->events.push_back(ev);
  }
  return DLRM_OK;
}

int32_t dlrm_stage_times(dlrm_handle_t h, double* total_ms, int32_t capacity, int64_t* calls) {
  if (!h) return -1;
  const int32_t n = static_cast<int32_t>(h->stage_names.size());
  for (int32_t i = 0; i < n && i < capacity && total_ms; ++i) total_ms[i] = h->stage_ms[i];
  if (calls) *calls = h->profiled_calls;
  return n;
}

void dlrm_destroy(dlrm_handle_t h) {
  if (!h) return;
  cudaDeviceSynchronize();
  if (h->report_on_destroy && h->profiled_calls > 0) {
    std::fprintf(stderr, "dlrm profile: %lld forward calls, %s plan; mean ms per call:\n",
                 static_cast<long long>(h->profiled_calls),
                 h->path == DLRM_PATH_FUSED ? "fused" : "layer-wise");
    for (size_t i = 0; i < h->stage_names.size(); ++i)
      std::fprintf(stderr, "  %-14s %10.4f\n", h->stage_names[i].c_str(),
                   h->stage_ms[i] / static_cast<double>(h->profiled_calls));
  }
  destroy_events(h);
  if (h->arena) cudaFree(h->arena);
  delete h;
}

dlrm_status_t embedding_bag_sum_multi(const float* const* tables, const int64_t* rows,
                                      int32_t K, int32_t D, const int64_t* indices,
                                      const int64_t* offsets, int32_t B, int32_t L, float* out,
                                      int32_t* err_flag, void* stream) {
  if (K < 1 || D < 1 || L < 1 || B < 0) return DLRM_ERR_INVALID_ARG;
  if (K > DLRM_MAX_TABLES) return DLRM_ERR_UNSUPPORTED;
  if (!tables || !rows) return DLRM_ERR_INVALID_ARG;
  if (B == 0) return DLRM_OK;
  if (!indices || !offsets || !out) return DLRM_ERR_INVALID_ARG;
  if (!dlrm::aligned_to(indices, sizeof(int64_t)) || !dlrm::aligned_to(offsets, sizeof(int64_t)) ||
      !dlrm::aligned_to(out, sizeof(float)) || !dlrm::aligned_to(err_flag, sizeof(int32_t)))
    return DLRM_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * L > (int64_t(1) << 31)) return DLRM_ERR_UNSUPPORTED;
  dlrm::GatherTables tabs{};
  for (int t = 0; t < K; ++t) {
    if (!tables[t] || rows[t] < 0 || !dlrm::aligned_to(tables[t], sizeof(float)))
      return DLRM_ERR_INVALID_ARG;
    tabs.ptr[t] = tables[t];
    tabs.rows[t] = rows[t];
  }
  return cuda_status(dlrm::launch_gather(tabs, K, D, indices, offsets, B, L, out, err_flag,
                                         static_cast<cudaStream_t>(stream)));
}

dlrm_status_t embedding_bag_multi_ex(const float* const* tables, const int64_t* rows, int32_t K,
                                     int32_t D, const void* indices, int64_t n_idx,
                                     const void* offsets, int32_t B,
                                     const dlrm_bag_options_t* options, float* out,
                                     int32_t* err_flag, void* stream) {
  if (!options) return DLRM_ERR_INVALID_ARG;
  const int mode = options->mode;
  if (K < 1 || D < 1 || B < 0 || n_idx < 0) return DLRM_ERR_INVALID_ARG;
  if (mode != DLRM_BAG_SUM && mode != DLRM_BAG_MEAN && mode != DLRM_BAG_MAX)
    return DLRM_ERR_INVALID_ARG;
  if (options->index_bits != 32 && options->index_bits != 64) return DLRM_ERR_INVALID_ARG;
  if (options->index_bits == 32 && n_idx > INT32_MAX) return DLRM_ERR_INVALID_ARG;
  if (options->per_sample_weights && mode != DLRM_BAG_SUM) return DLRM_ERR_INVALID_ARG;
  if (K > DLRM_MAX_TABLES) return DLRM_ERR_UNSUPPORTED;
  if (!tables || !rows) return DLRM_ERR_INVALID_ARG;
  if (B == 0) return DLRM_OK;
  if ((n_idx > 0 && !indices) || !offsets || !out) return DLRM_ERR_INVALID_ARG;
  const size_t index_bytes = static_cast<size_t>(options->index_bits / 8);
  if (!dlrm::aligned_to(indices, index_bytes) || !dlrm::aligned_to(offsets, index_bytes) ||
      !dlrm::aligned_to(options->per_sample_weights, sizeof(float)) ||
      !dlrm::aligned_to(out, sizeof(float)) || !dlrm::aligned_to(err_flag, sizeof(int32_t)))
    return DLRM_ERR_INVALID_ARG;
  dlrm::GatherTables tabs{};
  for (int t = 0; t < K; ++t) {
    if (!tables[t] || rows[t] < 0 || !dlrm::aligned_to(tables[t], sizeof(float)))
      return DLRM_ERR_INVALID_ARG;
    tabs.ptr[t] = tables[t];
    tabs.rows[t] = rows[t];
  }
  const int64_t padding = options->padding_idx >= 0 ? options->padding_idx : -1;
  return cuda_status(dlrm::launch_gather_general(
      tabs, K, D, indices, n_idx, offsets, options->index_bits, B, mode,
      options->per_sample_weights, padding, out, err_flag, static_cast<cudaStream_t>(stream)));
}

dlrm_status_t embedding_bag_multi(const float* const* tables, const int64_t* rows, int32_t K,
                                  int32_t D, const int64_t* indices, int64_t n_idx,
                                  const int64_t* offsets, int32_t B, int32_t mode, float* out,
                                  int32_t* err_flag, void* stream) {
  const dlrm_bag_options_t opt{mode, 64, nullptr, -1};
  return embedding_bag_multi_ex(tables, rows, K, D, indices, n_idx, offsets, B, &opt, out,
                                err_flag, stream);
}

dlrm_status_t pairwise_dot_lower_tri(const float* dense, int32_t ld_dense, const float* emb,
                                     int32_t B, int32_t K, int32_t D, float* out,
                                     int32_t ld_out, int32_t copy_dense, void* stream) {
  if (B < 0 || K < 0 || D < 1 || ld_dense < D) return DLRM_ERR_INVALID_ARG;
  const int64_t f = static_cast<int64_t>(K) + 1;
  const int64_t p = f * (f - 1) / 2;
  if (ld_out < (copy_dense ? D : 0) + p) return DLRM_ERR_INVALID_ARG;
  if (B == 0) return DLRM_OK;
  if (!dense || !out || (K > 0 && !emb)) return DLRM_ERR_INVALID_ARG;
  if (!dlrm::aligned_to(dense, sizeof(float)) || !dlrm::aligned_to(emb, sizeof(float)) ||
      !dlrm::aligned_to(out, sizeof(float)))
    return DLRM_ERR_INVALID_ARG;
  if (p > (int64_t(1) << 30)) return DLRM_ERR_UNSUPPORTED;
  if (dlrm::interaction_smem_per_sample(K, D) > dlrm::device_max_smem_optin())
    return DLRM_ERR_UNSUPPORTED;
  return cuda_status(dlrm::launch_interaction(dense, ld_dense, emb, B, K, D, out, ld_out,
                                              copy_dense ? 1 : 0,
                                              static_cast<cudaStream_t>(stream)));
}

dlrm_status_t pairwise_pair_map(int32_t F, int32_t* i_out, int32_t* j_out, void* stream) {
  if (F < 2 || F > 46341 || !i_out || !j_out) return DLRM_ERR_INVALID_ARG;
  if (!dlrm::aligned_to(i_out, sizeof(int32_t)) || !dlrm::aligned_to(j_out, sizeof(int32_t)))
    return DLRM_ERR_INVALID_ARG;
  return cuda_status(dlrm::launch_pair_map(F, i_out, j_out, static_cast<cudaStream_t>(stream)));
}

dlrm_status_t linear_bias_act(const float* x, int32_t ld_x, const float* W, const float* bias,
                              float* y, int32_t ld_y, int32_t M, int32_t N, int32_t K,
                              dlrm_act_t act, dlrm_math_t math, void* stream) {
  if (M < 0 || N < 1 || K < 1 || ld_x < K || ld_y < N) return DLRM_ERR_INVALID_ARG;
  if (act != DLRM_ACT_NONE && act != DLRM_ACT_RELU && act != DLRM_ACT_SIGMOID)
    return DLRM_ERR_INVALID_ARG;
  if (math != DLRM_MATH_FP32 && math != DLRM_MATH_TF32 && math != DLRM_MATH_BF16 &&
      math != DLRM_MATH_TF32X3 && math != DLRM_MATH_FP32_FFMA)
    return DLRM_ERR_INVALID_ARG;
  if (M == 0) return DLRM_OK;
  if (!x || !W || !y) return DLRM_ERR_INVALID_ARG;
  if (!dlrm::aligned_to(x, sizeof(float)) || !dlrm::aligned_to(W, sizeof(float)) ||
      !dlrm::aligned_to(bias, sizeof(float)) || !dlrm::aligned_to(y, sizeof(float)))
    return DLRM_ERR_INVALID_ARG;
  const size_t ybytes = (static_cast<size_t>(M - 1) * ld_y + N) * sizeof(float);
  const size_t xbytes = (static_cast<size_t>(M - 1) * ld_x + K) * sizeof(float);
  const size_t wbytes = static_cast<size_t>(N) * K * sizeof(float);
  if (ranges_overlap(y, ybytes, x, xbytes) || ranges_overlap(y, ybytes, W, wbytes))
    return DLRM_ERR_INVALID_ARG;
  if (!fp32_math(math))
    return cuda_status(dlrm::launch_linear_tc(x, ld_x, W, K, bias, y, ld_y, M, N, K, act,
                                              static_cast<int>(math), nullptr,
                                              static_cast<cudaStream_t>(stream)));
  return cuda_status(dlrm::launch_linear_fp32(x, ld_x, W, K, bias, y, ld_y, M, N, K, act,
                                              static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
