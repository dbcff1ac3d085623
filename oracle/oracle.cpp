// CPU oracle for the DLRMv1 inference forward. TEST INFRASTRUCTURE ONLY.
//
// Only the tests, the smoke check and the bench's CPU-baseline leg may load
// this library. It shares no code, header, table or helper with the CUDA path
// and imports nothing from it. Every routine below is the plain definition of
// one step, computed in the order the pages give it, with fp64 accumulation:
// no blocking, fusion or reordering.
//
// Sources (Luminal compare pages on the DLRMv1 forward):
//  [P1] compare modal_ci_ready...vanilla-pytorch, commit message
//       "vanilla-PyTorch DLRMv1 fast paths" (emb-bag translator, pairwise-dot
//       kernels with the closed-form pair index, linear_bias_(relu|sigmoid)).
//  [P4] compare dlrm-fused-kernels...dlrm-pt2-megakernel:
//       crates/luminal_cuda_lite/src/kernel/dlrm_megakernel.rs (body steps
//       1-6: bottom MLP, lookups, dot interaction, concat, top MLP + sigmoid;
//       validate()), LessonsLearned "EmbeddingBag translator gap", and
//       translator/movement.rs translate_embedding_bag.
//
// Readings where the pages are silent (each also listed in the design notes):
//  * Bags use general offsets: bag b of table t is
//    indices[t][offsets[t][b] : offsets[t][b+1]] (the last bag ends at N);
//    an empty bag sums to zeros. An index outside [0, rows) contributes zeros
//    and the call returns ORACLE_INDEX_OOB.
//  * Pair p maps to (i, j) by i = floor((1 + sqrt(1 + 8p)) / 2),
//    j = p - i(i-1)/2, followed by an integer fix-up so rounding in sqrt can
//    never mis-map.
//  * The sigmoid is 1 / (1 + exp(-a)) in double.
//
// Pins: the tests check this file against bag-size-1 == index_select,
// permutation invariance inside a bag, the lower triangle of a brute-force
// Z Z^T, an exhaustive pair-map check for F <= 256, closed-form special cases
// (zero top weights, identity bottom MLP) and hand-computed integer examples.

#include <cmath>
#include <cstdint>
#include <thread>
#include <vector>

namespace {

enum { ORACLE_OK = 0, ORACLE_INVALID = 1, ORACLE_INDEX_OOB = 5 };
enum { ACT_NONE = 0, ACT_RELU = 1, ACT_SIGMOID = 2 };

double activate(double a, int act) {
  if (act == ACT_RELU) return a > 0.0 ? a : 0.0;
  if (act == ACT_SIGMOID) return 1.0 / (1.0 + std::exp(-a));
  return a;
}

// One Linear layer on one sample: y[n] = act(b[n] + sum_k x[k] * W[n][k]),
// W in PyTorch (out, in) row-major layout ([P4] dlrm_megakernel.rs, input
// layout note and body step 2).
void linear_row(const double* x, int k_in, int n_out, const float* w, const float* b,
                int act, double* y) {
  for (int n = 0; n < n_out; ++n) {
    double a = b ? static_cast<double>(b[n]) : 0.0;
    for (int k = 0; k < k_in; ++k) a += x[k] * static_cast<double>(w[(int64_t)n * k_in + k]);
    y[n] = activate(a, act);
  }
}

// Bag sum of one (sample, table) ([P4] LessonsLearned "EmbeddingBag
// translator gap": output[b] = sum of weight rows indices[offsets[b]:offsets[b+1]]).
int bag_sum(const float* table, int64_t rows, int d, const int64_t* idx, int64_t n_idx,
            const int64_t* off, int64_t batch, int64_t b, double* out) {
  int status = ORACLE_OK;
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  int64_t begin = off[b];
  int64_t end = (b + 1 < batch) ? off[b + 1] : n_idx;
  for (int64_t n = begin; n < end; ++n) {
    int64_t r = idx[n];
    if (r < 0 || r >= rows) { status = ORACLE_INDEX_OOB; continue; }
    const float* row = table + r * d;
    for (int c = 0; c < d; ++c) out[c] += static_cast<double>(row[c]);
  }
  return status;
}

// One (sample, table) bag under a reduction mode, over general offsets
// ([P4] LessonsLearned "EmbeddingBag translator gap": output[b] =
// reduce_op(weight[indices[offsets[b]:offsets[b+1]]]), reduce_op one of
// sum / mean / max). Readings where the pages are silent: the last bag ends
// at N; an index outside [0, rows) is left out of its bag (flag bit 1); mean
// divides by the number of rows kept; a bag with no rows kept is zeros in
// every mode; bounds with begin < 0, end > N or begin > end make the bag
// zeros (flag bit 2). Returns the flag bits.
enum { BAG_SUM = 0, BAG_MEAN = 1, BAG_MAX = 2 };
enum { BAG_FLAG_OOB = 1, BAG_FLAG_OFFSETS = 2 };
//
// PyTorch's per_sample_weights and padding_idx ([P4] LessonsLearned and the
// translator's guards name both as cases the pages leave out): with weights
// (sum only) row n is scaled by w[n] before it is added; an index equal to
// padding_idx (>= 0) is left out of its bag like an out-of-range one, but
// without a flag.
int bag_reduce(const float* table, int64_t rows, int d, const int64_t* idx, int64_t n_idx,
               const int64_t* off, int64_t batch, int64_t b, int mode, const float* psw,
               int64_t padding_idx, double* out) {
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  const int64_t begin = off[b];
  const int64_t end = (b + 1 < batch) ? off[b + 1] : n_idx;
  if (begin < 0 || end > n_idx || begin > end) return BAG_FLAG_OFFSETS;
  int flags = 0;
  int64_t kept = 0;
  for (int64_t n = begin; n < end; ++n) {
    const int64_t r = idx[n];
    if (padding_idx >= 0 && r == padding_idx) continue;
    if (r < 0 || r >= rows) { flags |= BAG_FLAG_OOB; continue; }
    const float* row = table + r * d;
    const double w = psw ? static_cast<double>(psw[n]) : 1.0;
    for (int c = 0; c < d; ++c) {
      const double v = w * static_cast<double>(row[c]);
      if (mode == BAG_MAX) out[c] = (kept == 0 || v > out[c]) ? v : out[c];
      else out[c] += v;
    }
    ++kept;
  }
  if (mode == BAG_MEAN && kept > 0)
    for (int c = 0; c < d; ++c) out[c] /= static_cast<double>(kept);
  return flags;
}

// Strict lower triangle of the Gram matrix of the F feature vectors, i-major
// then j ([P4] dlrm_megakernel.rs step 4: "for i in 0..n_feat for j in 0..i",
// Vec[0] = x, Vec[k+1] = table k). z must hold F(F-1)/2 values.
void interact_row(const double* const* vec, int f, int d, double* z) {
  int64_t p = 0;
  for (int i = 0; i < f; ++i) {
    for (int j = 0; j < i; ++j) {
      double s = 0.0;
      for (int c = 0; c < d; ++c) s += vec[i][c] * vec[j][c];
      z[p++] = s;
    }
  }
}

template <class Fn>
void parallel_for(int64_t n, int threads, Fn fn) {
  if (threads <= 1 || n < 2) { for (int64_t i = 0; i < n; ++i) fn(i); return; }
  if (threads > n) threads = static_cast<int>(n);
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t) {
    pool.emplace_back([=, &fn] {
      for (int64_t i = t; i < n; i += threads) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

int oracle_version() { return 3; }

// Pair index p -> (i, j), i > j >= 0 ([P1] PairwiseDotLowerTriStackedKernel:
// "(1+sqrt(1+8p))/2"; the floor and j = p - i(i-1)/2 are the reading).
void oracle_pair_from_index(int64_t p, int64_t* i_out, int64_t* j_out) {
  int64_t i = static_cast<int64_t>(std::floor((1.0 + std::sqrt(1.0 + 8.0 * (double)p)) / 2.0));
  while (i * (i - 1) / 2 > p) --i;
  while ((i + 1) * i / 2 <= p) ++i;
  *i_out = i;
  *j_out = p - i * (i - 1) / 2;
}

// Pairs in the enumeration order of [P4] step 4, for pinning the closed form.
void oracle_pair_enumerate(int f, int64_t* i_out, int64_t* j_out) {
  int64_t p = 0;
  for (int i = 0; i < f; ++i)
    for (int j = 0; j < i; ++j) { i_out[p] = i; j_out[p] = j; ++p; }
}

// Multi-table bag sum: out (B, K, D) double.
//   tables[t]  host pointer to table t, (rows[t], D) float row-major
//   indices    (K, n_idx) int64, table-major
//   offsets    (K, B) int64, bag starts (include_last_offset = false)
int oracle_embedding_bag_sum(int k_tables, const float* const* tables, const int64_t* rows,
                             int d, const int64_t* indices, int64_t n_idx,
                             const int64_t* offsets, int64_t batch, double* out,
                             int threads) {
  if (k_tables <= 0 || d <= 0 || batch < 0 || n_idx < 0) return ORACLE_INVALID;
  std::vector<int> status(batch, ORACLE_OK);
  parallel_for(batch, threads, [&](int64_t b) {
    for (int t = 0; t < k_tables; ++t) {
      int s = bag_sum(tables[t], rows[t], d, indices + (int64_t)t * n_idx, n_idx,
                      offsets + (int64_t)t * batch, batch, b, out + (b * k_tables + t) * d);
      if (s != ORACLE_OK) status[b] = s;
    }
  });
  for (int64_t b = 0; b < batch; ++b) if (status[b] != ORACLE_OK) return status[b];
  return ORACLE_OK;
}

// Multi-table EmbeddingBag with a reduction mode (0 sum, 1 mean, 2 max) over
// general offsets: out (B, K, D) double; *flags receives the OR of the bags'
// flag bits (1: an index out of range, 2: bad bag bounds).
//   psw: (K, n_idx) float per-sample weights or null (sum mode only)
//   padding_idx: a row index left out of every bag, or < 0 for none
int oracle_embedding_bag(int k_tables, const float* const* tables, const int64_t* rows, int d,
                         const int64_t* indices, int64_t n_idx, const int64_t* offsets,
                         int64_t batch, int mode, const float* psw, int64_t padding_idx,
                         double* out, int* flags, int threads) {
  if (k_tables <= 0 || d <= 0 || batch < 0 || n_idx < 0 || mode < BAG_SUM || mode > BAG_MAX)
    return ORACLE_INVALID;
  if (psw && mode != BAG_SUM) return ORACLE_INVALID;
  std::vector<int> f(batch, 0);
  parallel_for(batch, threads, [&](int64_t b) {
    for (int t = 0; t < k_tables; ++t)
      f[b] |= bag_reduce(tables[t], rows[t], d, indices + (int64_t)t * n_idx, n_idx,
                         offsets + (int64_t)t * batch, batch, b, mode,
                         psw ? psw + (int64_t)t * n_idx : nullptr, padding_idx,
                         out + (b * k_tables + t) * d);
  });
  int all = 0;
  for (int64_t b = 0; b < batch; ++b) all |= f[b];
  if (flags) *flags = all;
  return ORACLE_OK;
}

// y (M, N) = act(x (M, K) W^T + b); W (N, K) float, b (N) float or null.
int oracle_linear(int64_t m, int k_in, int n_out, const double* x, const float* w,
                  const float* b, int act, double* y, int threads) {
  if (m < 0 || k_in <= 0 || n_out <= 0) return ORACLE_INVALID;
  parallel_for(m, threads, [&](int64_t r) {
    linear_row(x + r * k_in, k_in, n_out, w, b, act, y + r * n_out);
  });
  return ORACLE_OK;
}

// Interaction + concat: R (B, D + F(F-1)/2) = [x, z] ([P4] steps 4-5).
//   x (B, D) double, e (B, K, D) double
int oracle_interaction(int64_t batch, int k_tables, int d, const double* x, const double* e,
                       double* r, int threads) {
  if (batch < 0 || k_tables < 0 || d <= 0) return ORACLE_INVALID;
  const int f = k_tables + 1;
  const int64_t p = (int64_t)f * (f - 1) / 2;
  parallel_for(batch, threads, [&](int64_t b) {
    std::vector<const double*> vec(f);
    vec[0] = x + b * d;
    for (int t = 0; t < k_tables; ++t) vec[t + 1] = e + (b * k_tables + t) * d;
    double* row = r + b * (d + p);
    for (int c = 0; c < d; ++c) row[c] = x[b * d + c];
    interact_row(vec.data(), f, d, row + d);
  });
  return ORACLE_OK;
}

// Full forward on a list of samples ([P4] dlrm_megakernel.rs steps 1-6).
//   ln_bot (n_bot + 1 widths), ln_top (n_top + 1 widths), host arrays
//   dense (B, ln_bot[0]) float; indices (K, n_idx); offsets (K, B)
//   sample_ids: the samples to evaluate (null = all B, in order)
//   out: one double per evaluated sample
int oracle_forward(int64_t batch, int n_bot, const int* ln_bot, const float* const* bot_w,
                   const float* const* bot_b, int k_tables, const float* const* tables,
                   const int64_t* rows, int d, const int64_t* indices, int64_t n_idx,
                   const int64_t* offsets, int n_top, const int* ln_top,
                   const float* const* top_w, const float* const* top_b, const float* dense,
                   const int64_t* sample_ids, int64_t n_samples, double* out, int threads) {
  // Shape checks of [P4] validate().
  if (n_bot < 1 || n_top < 1 || k_tables < 1 || d <= 0) return ORACLE_INVALID;
  if (ln_bot[n_bot] != d) return ORACLE_INVALID;
  const int f = k_tables + 1;
  const int p = f * (f - 1) / 2;
  if (ln_top[0] != d + p || ln_top[n_top] != 1) return ORACLE_INVALID;
  int widest = 0;
  for (int l = 0; l <= n_bot; ++l) widest = ln_bot[l] > widest ? ln_bot[l] : widest;
  for (int l = 0; l <= n_top; ++l) widest = ln_top[l] > widest ? ln_top[l] : widest;
  const int64_t count = sample_ids ? n_samples : batch;
  std::vector<int> status(count, ORACLE_OK);

  parallel_for(count, threads, [&](int64_t s) {
    const int64_t b = sample_ids ? sample_ids[s] : s;
    std::vector<double> h(widest), g(widest);
    // 1-2. Bottom MLP, ReLU after every layer including the last.
    for (int c = 0; c < ln_bot[0]; ++c) h[c] = dense[b * ln_bot[0] + c];
    for (int l = 0; l < n_bot; ++l) {
      linear_row(h.data(), ln_bot[l], ln_bot[l + 1], bot_w[l], bot_b[l], ACT_RELU, g.data());
      h.swap(g);
    }
    std::vector<double> x(h.begin(), h.begin() + d);
    // 3. Bag sums, one per table.
    std::vector<double> e((size_t)k_tables * d);
    for (int t = 0; t < k_tables; ++t) {
      int st = bag_sum(tables[t], rows[t], d, indices + (int64_t)t * n_idx, n_idx,
                       offsets + (int64_t)t * batch, batch, b, e.data() + (size_t)t * d);
      if (st != ORACLE_OK) status[s] = st;
    }
    // 4-5. Interaction; R = [x, z].
    std::vector<const double*> vec(f);
    vec[0] = x.data();
    for (int t = 0; t < k_tables; ++t) vec[t + 1] = e.data() + (size_t)t * d;
    std::vector<double> r((size_t)d + p);
    for (int c = 0; c < d; ++c) r[c] = x[c];
    interact_row(vec.data(), f, d, r.data() + d);
    // 6. Top MLP: ReLU on all but the last layer, sigmoid on the last.
    for (int c = 0; c < d + p; ++c) h[c] = r[c];
    for (int l = 0; l < n_top; ++l) {
      int act = (l == n_top - 1) ? ACT_SIGMOID : ACT_RELU;
      linear_row(h.data(), ln_top[l], ln_top[l + 1], top_w[l], top_b[l], act, g.data());
      h.swap(g);
    }
    out[s] = h[0];
  });
  for (int64_t s = 0; s < count; ++s) if (status[s] != ORACLE_OK) return status[s];
  return ORACLE_OK;
}

}  // extern "C"
