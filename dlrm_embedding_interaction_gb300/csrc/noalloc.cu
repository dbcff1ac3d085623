// dlrm_forward_noalloc: the forward without a handle and without any device
// allocation, for callers that cannot allocate when they run the model (see
// include/dlrm.h). The working buffers (bag sums, two activation buffers, the
// interaction output) are slices of one fixed file-scope device array.
#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = DLRM_NOALLOC_SCRATCH_BYTES;

// The scratch. In host code this name is only a host-side stand-in for the
// symbol: kernels must be given the device address looked up below.
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch on the current device. Looked up on every
// call (cudaGetSymbolAddress is cheap): an address cached across calls would
// dangle after a device reset, which reloads the module elsewhere.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (!p) return cudaErrorInvalidSymbol;
  *out = p;
  return cudaSuccess;
}

size_t slice(size_t& cursor, size_t bytes) {
  const size_t at = cursor;
  cursor = static_cast<size_t>(dlrm::round_up(static_cast<int64_t>(cursor + bytes), 256));
  return at;
}

}  // namespace

extern "C" dlrm_status_t dlrm_forward_noalloc(
    const dlrm_config_t* cfg, const float* const* tables, const float* const* bot_w,
    const float* const* bot_b, const float* const* top_w, const float* const* top_b,
    const float* dense, const int64_t* indices, const int64_t* offsets, float* out,
    int32_t batch, int32_t* err_flag, void* stream) {
  // Shape checks as in dlrm_create.
  if (!cfg || !tables || !bot_w || !bot_b || !top_w || !top_b) return DLRM_ERR_INVALID_ARG;
  if (!dense || !indices || !offsets || !out || batch < 1) return DLRM_ERR_INVALID_ARG;
  if (!cfg->ln_bot || !cfg->ln_top || !cfg->rows) return DLRM_ERR_INVALID_ARG;
  if (cfg->n_bot < 1 || cfg->n_top < 1) return DLRM_ERR_INVALID_ARG;
  if (cfg->n_bot > DLRM_MAX_LAYERS || cfg->n_top > DLRM_MAX_LAYERS) return DLRM_ERR_UNSUPPORTED;
  if (cfg->n_tables < 1 || cfg->emb_dim < 1 || cfg->bag_size < 1) return DLRM_ERR_INVALID_ARG;
  if (cfg->n_tables > DLRM_MAX_TABLES) return DLRM_ERR_UNSUPPORTED;
  for (int l = 0; l <= cfg->n_bot; ++l) if (cfg->ln_bot[l] < 1) return DLRM_ERR_INVALID_ARG;
  for (int l = 0; l <= cfg->n_top; ++l) if (cfg->ln_top[l] < 1) return DLRM_ERR_INVALID_ARG;
  const int k = cfg->n_tables, d = cfg->emb_dim, bag = cfg->bag_size;
  const int64_t f = k + 1;
  const int64_t p = f * (f - 1) / 2;
  if (cfg->ln_bot[cfg->n_bot] != d || cfg->ln_top[0] != d + p || cfg->ln_top[cfg->n_top] != 1)
    return DLRM_ERR_INVALID_ARG;
  if (cfg->math != DLRM_MATH_FP32 && cfg->math != DLRM_MATH_FP32_FFMA) return DLRM_ERR_UNSUPPORTED;
  dlrm::GatherTables tabs{};
  if (!dlrm::aligned_to(dense, sizeof(float)) || !dlrm::aligned_to(indices, sizeof(int64_t)) ||
      !dlrm::aligned_to(offsets, sizeof(int64_t)) || !dlrm::aligned_to(out, sizeof(float)) ||
      !dlrm::aligned_to(err_flag, sizeof(int32_t)))
    return DLRM_ERR_INVALID_ARG;
  for (int t = 0; t < k; ++t) {
    if (!tables[t] || cfg->rows[t] < 1 || !dlrm::aligned_to(tables[t], sizeof(float)))
      return DLRM_ERR_INVALID_ARG;
    tabs.ptr[t] = tables[t];
    tabs.rows[t] = cfg->rows[t];
  }
  for (int side = 0; side < 2; ++side) {
    const float* const* ws = side == 0 ? bot_w : top_w;
    const float* const* bs = side == 0 ? bot_b : top_b;
    for (int l = 0; l < (side == 0 ? cfg->n_bot : cfg->n_top); ++l)
      if (!ws[l] || !bs[l] || !dlrm::aligned_to(ws[l], sizeof(float)) ||
          !dlrm::aligned_to(bs[l], sizeof(float)))
        return DLRM_ERR_INVALID_ARG;
  }
  if (static_cast<int64_t>(batch) * bag > (int64_t(1) << 31)) return DLRM_ERR_UNSUPPORTED;
  if (dlrm::interaction_smem_per_sample(k, d) > dlrm::device_max_smem_optin())
    return DLRM_ERR_UNSUPPORTED;

  // Scratch layout for this batch; reject what does not fit.
  int widest = 4;
  for (int l = 1; l <= cfg->n_bot; ++l) widest = std::max(widest, cfg->ln_bot[l]);
  for (int l = 1; l < cfg->n_top; ++l) widest = std::max(widest, cfg->ln_top[l]);
  const int ld_act = static_cast<int>(dlrm::round_up(widest, 4));
  const int ld_r = static_cast<int>(dlrm::round_up(cfg->ln_top[0], 4));
  const size_t nb = static_cast<size_t>(batch);
  size_t cursor = 0;
  const size_t off_emb = slice(cursor, nb * k * d * sizeof(float));
  const size_t off_a0 = slice(cursor, nb * ld_act * sizeof(float));
  const size_t off_a1 = slice(cursor, nb * ld_act * sizeof(float));
  const size_t off_r = slice(cursor, nb * ld_r * sizeof(float));
  if (cursor > kScratchBytes) return DLRM_ERR_UNSUPPORTED;

  void* base_v = nullptr;
  if (scratch_address(&base_v) != cudaSuccess) return DLRM_ERR_CUDA;
  char* base = static_cast<char*>(base_v);
  float* emb = reinterpret_cast<float*>(base + off_emb);
  float* act[2] = {reinterpret_cast<float*>(base + off_a0), reinterpret_cast<float*>(base + off_a1)};
  float* r = reinterpret_cast<float*>(base + off_r);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (dlrm::launch_gather(tabs, k, d, indices, offsets, batch, bag, emb, err_flag, s) !=
      cudaSuccess)
    return DLRM_ERR_CUDA;
  const float* in = dense;
  int ld_in = cfg->ln_bot[0];
  for (int l = 0; l < cfg->n_bot; ++l) {
    float* o = act[l & 1];
    if (dlrm::launch_linear_fp32(in, ld_in, bot_w[l], cfg->ln_bot[l], bot_b[l], o, ld_act, batch,
                                 cfg->ln_bot[l + 1], cfg->ln_bot[l], DLRM_ACT_RELU, s) !=
        cudaSuccess)
      return DLRM_ERR_CUDA;
    in = o;
    ld_in = ld_act;
  }
  if (dlrm::launch_interaction(in, ld_in, emb, batch, k, d, r, ld_r, 1, s) != cudaSuccess)
    return DLRM_ERR_CUDA;
  in = r;
  ld_in = ld_r;
  for (int l = 0; l < cfg->n_top; ++l) {
    const bool last = (l == cfg->n_top - 1);
    float* o = last ? out : act[l & 1];
    const int ld_o = last ? 1 : ld_act;
    if (dlrm::launch_linear_fp32(in, ld_in, top_w[l], cfg->ln_top[l], top_b[l], o, ld_o, batch,
                                 cfg->ln_top[l + 1], cfg->ln_top[l],
                                 last ? DLRM_ACT_SIGMOID : DLRM_ACT_RELU, s) != cudaSuccess)
      return DLRM_ERR_CUDA;
    in = o;
    ld_in = ld_o;
  }
  return DLRM_OK;
}
