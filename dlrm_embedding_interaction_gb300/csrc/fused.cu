// Fused single-launch DLRMv1 forward (fp32): host planning and the launch of
// the instances without phase-trace stamps (the kernel is in
// fused_kernel.cuh; fused_trace.cu holds the instances with stamps).
#include "fused_kernel.cuh"

namespace dlrm {

cudaError_t fused_prepare(int bm, int cw, int lda) {
  cudaError_t e = prepare_fused_instances<false>(bm, cw, lda);
  if (e == cudaSuccess) e = fused_prepare_traced(bm, cw, lda);
  return e;
}

cudaError_t launch_fused(const FusedParams& p, int bm, cudaStream_t stream) {
  if (p.trace) return launch_fused_traced(p, bm, stream);
  return launch_fused_instances<false>(p, bm, stream);
}

// ---------------------------------------------------------------- host plan

namespace {

// Chunk swizzle of staged row `row` when a row holds `cpr` 16-byte chunks:
// 8 consecutive rows then hit 8 distinct 16-byte bank groups.
int swizzle_of(int row, int cpr) {
  return cpr == 2 ? ((row >> 2) & 1) : (cpr == 4 ? ((row >> 1) & 3) : (row & 7));
}

size_t align128(size_t x) { return (x + 127) / 128 * 128; }

// k-slices a stage of layer L is cut into among the 8 computing warps (the
// partial-sum sets of each output): 1 for layers wider than 256 columns (8
// column groups of 64 per pass), 4 for 256 columns (2 column groups of 128),
// else 8 / column groups, with n_pad / 64 column groups (at least one).
int fused_kslices(const FusedGemm& L) {
  if (L.ksplit == 1) return 1;
  return L.n_pad == 256 ? 4 : 8 / std::max(1, L.n_pad / 64);
}

}  // namespace

bool fused_plan(int n_dense, int k_tables, int d, int bag, const std::vector<int>& ln_bot,
                const std::vector<int>& ln_top, const std::vector<std::vector<float>>& w,
                const std::vector<std::vector<float>>& b, const GatherTables& tabs,
                int max_batch, int sms, size_t smem_limit, int cw, FusedPlan* plan) {
  if (cw != 8) return false;
  const int ksl = 16;           // k per stage at ksplit 1 (32 at ksplit 2)
  const int n_bot = static_cast<int>(ln_bot.size()) - 1;
  const int n_top = static_cast<int>(ln_top.size()) - 1;
  const int n_gemm = n_bot + n_top - 1;
  if (d % 4 != 0 || ln_top.back() != 1 || n_gemm > kFusedMaxGemm || n_bot < 1) return false;
  for (int t = 0; t < k_tables; ++t)
    if (reinterpret_cast<uintptr_t>(tabs.ptr[t]) % 16 != 0) return false;
  FusedParams& p = plan->params;
  p = FusedParams{};
  p.n_dense = n_dense;
  p.k_tables = k_tables;
  p.d = d;
  p.bag = bag;
  p.n_bot = n_bot;
  p.n_top = n_top;
  p.n_gemm = n_gemm;
  p.cw = cw;
  const int f = k_tables + 1;
  const int pairs = f * (f - 1) / 2;

  // layer shapes
  std::vector<int> kin(n_gemm), nout(n_gemm);
  for (int g = 0; g < n_gemm; ++g) {
    kin[g] = g < n_bot ? ln_bot[g] : ln_top[g - n_bot];
    nout[g] = g < n_bot ? ln_bot[g + 1] : ln_top[g - n_bot + 1];
  }
  // Layer shapes. Wider than 256 columns: 32 x 8-column warps in two column
  // groups per pass (ksplit 1), n_pad a multiple of 256. Otherwise one column
  // group of n_pad = 32 * tn (a power of two >= 32) and two k-slices.
  int widest = 0;
  int bias_floats = 0;
  for (int g = 0; g < n_gemm; ++g) {
    FusedGemm& L = p.gemm[g];
    L.n = nout[g];
    if (L.n > 256) {
      L.tn = 8;
      L.ksplit = 1;
      L.n_pad = static_cast<int>(round_up(L.n, 256));
      L.passes = (L.n_pad + 511) / 512;
    } else {
      int np = 32;
      while (np < L.n) np *= 2;
      L.n_pad = np;
      L.tn = np / 32;
      L.ksplit = 2;
      L.passes = 1;
    }
    L.k_pad = static_cast<int>(round_up(kin[g], ksl * L.ksplit));
    L.n_kst = L.k_pad / (ksl * L.ksplit);
    L.b_off = bias_floats;
    bias_floats += L.n_pad;
    // the k-slices' partial sums sit side by side in the rows of the two
    // activation buffers
    widest = std::max({widest, L.k_pad, L.n_pad * ((fused_kslices(L) + 1) / 2)});
  }
  p.k_last = static_cast<int>(round_up(ln_top[n_top - 1], 4));
  p.b_last = bias_floats;
  bias_floats += 4;
  p.bias_floats = bias_floats;
  widest = std::max({widest, p.k_last, d + pairs});
  p.lda = static_cast<int>(round_up(widest, 32)) + 16;
  p.ldz = static_cast<int>(round_up(d, 4)) + 4;

  // shared-memory carve: stages | act0 | act1 | z | rowidx | bias | wlast | barriers
  // Preference: every bag row of the tile prefetched at kernel start (bags of
  // one row, or every row of bags of L > 1 rows when they fit: the rows land
  // during the bottom MLP and are summed at the interaction); else two group
  // buffers streamed with cp.async (bag 1); else one group buffer filled with
  // summed loads at the interaction (bags of L > 1). The 16-row tile is kept
  // first (one wave of tiles), then a weight stage is given up.
  const size_t per_sample_z = static_cast<size_t>(k_tables) * p.ldz * sizeof(float);
  bool placed = false;
  // Tile height: the kernel is persistent (one CTA per SM looping over
  // tiles), so a launch takes rounds = ceil(tiles / SMs) tile times. A tile's
  // time grows about linearly with its rows, as if it had ~12 rows more (2048
  // samples: ~24 us at 4 rows, ~42 us at 14). Take the height with the least
  // rounds x (rows + 12), the smaller on a tie.
  int first_bm = 4;
  int64_t best = INT64_MAX;
  for (int bm : {4, 8, 12, 14, 16}) {
    const int64_t tiles = (max_batch + bm - 1) / bm;
    const int64_t rounds = (tiles + sms - 1) / std::max(sms, 1);
    const int64_t cost = rounds * (bm + 12);
    if (cost < best) {
      best = cost;
      first_bm = bm;
    }
  }
  for (int bm : {16, 14, 12, 8, 4}) {
    if (bm > first_bm) continue;
    for (int mode = 0; mode < 3 && !placed; ++mode) {
      // bags of several rows: every row prefetched (mode 0) when they fit and
      // each computing thread holds at most kFusedBagRowSums bag sums, else
      // summed by loads at the interaction (mode 2)
      // (they run on the instances with a run-time activation stride, which
      // carry that code: fused_instance_lda)
      const int lb = (bag > 1 && mode == 0) ? bag : 1;
      if (bag != 1 && mode == 1) continue;
      if (lb > 1 && static_cast<int64_t>(bm) * k_tables * (d / 4) >
                        static_cast<int64_t>(kFusedBagRowSums) * cw * kWarp)
        continue;
      // the deepest ring that fits: a CTA's weight feed is bounded by the
      // bytes it keeps in flight (~80 GB/s per SM at four 32 KB stages)
      for (int stages : {6, 5, 4, 3}) {
        const size_t off = static_cast<size_t>(stages) * kFusedStageFloats * sizeof(float);
        const size_t act = align128(static_cast<size_t>(bm) * p.lda * sizeof(float));
        const size_t rowidx = align128(static_cast<size_t>(bm) * k_tables * lb * sizeof(int));
        const size_t tail = rowidx + align128(bias_floats * sizeof(float)) +
                            align128(p.k_last * sizeof(float)) + align128(2 * stages * 8 + 16);
        const size_t fixed = off + 2 * act + tail;
        if (fixed >= smem_limit) continue;
        const size_t room = smem_limit - fixed;
        int sg = 0, zbuf = 1;
        if (mode == 0) {
          if (room < bm * per_sample_z * lb) continue;
          sg = bm;
        } else if (mode == 1) {
          sg = static_cast<int>(std::min<size_t>(bm, room / (2 * per_sample_z)));
          zbuf = 2;
          // groups of one or two samples leave the pair dots one pair per
          // thread (four times the shared-memory reads of 4 x 4 blocks) and
          // cost a sync and copy round trip per sample: a weight stage is
          // given up for groups of three (32 tables at 14-row tiles: the
          // interaction 38.6 -> ~9 us)
          if (sg < std::min(bm, 3) && stages > 3) continue;
        } else {
          sg = static_cast<int>(std::min<size_t>(bm, room / per_sample_z));
        }
        if (sg < 1) continue;
        p.stages = stages;
        p.off_act0 = static_cast<int>(off);
        p.off_act1 = static_cast<int>(off + act);
        p.off_z = static_cast<int>(off + 2 * act);
        const size_t zbytes = align128(static_cast<size_t>(zbuf) * sg * per_sample_z * lb);
        p.off_rowidx = static_cast<int>(p.off_z + zbytes);
        p.off_bias = static_cast<int>(p.off_rowidx + rowidx);
        p.off_wlast = static_cast<int>(p.off_bias + align128(bias_floats * sizeof(float)));
        p.off_bar = static_cast<int>(p.off_wlast + align128(p.k_last * sizeof(float)));
        p.smem_bytes = static_cast<int>(p.off_bar + align128(2 * stages * 8 + 16));
        p.sg = sg;
        p.prefetch_z = mode == 0 ? 1 : 0;
        p.bag_rows = lb > 1 ? 1 : 0;
        p.zbuf = zbuf;
        plan->bm = bm;
        placed = true;
        break;
      }
      if (placed) break;
    }
  }
  if (!placed || static_cast<size_t>(p.smem_bytes) > smem_limit) return false;

  // packed weight stream in consumption order, and its stage table
  plan->wstream.clear();
  plan->stage_tab.clear();
  for (int g = 0; g < n_gemm; ++g) {
    const FusedGemm& L = p.gemm[g];
    const int ks = ksl * L.ksplit;
    const std::vector<float>& W = w[g];
    for (int pass = 0; pass < L.passes; ++pass) {
      const int rows = gemm_rows(L, pass);
      for (int kst = 0; kst < L.n_kst; ++kst) {
        const size_t base = plan->wstream.size();
        if (base > 0xffffffffu) return false;
        plan->stage_tab.push_back(make_uint2(static_cast<unsigned>(base),
                                             static_cast<unsigned>(rows * ks * sizeof(float))));
        plan->wstream.resize(base + static_cast<size_t>(rows) * ks, 0.f);
        for (int rr = 0; rr < rows; ++rr) {
          const int n = pass * gemm_cols_per_pass(L) + rr;
          if (n >= L.n) continue;
          for (int kk = 0; kk < ks; ++kk) {
            const int kg = kst * ks + kk;
            if (kg >= kin[g]) break;
            const int chunk = (kk / 4) ^ swizzle_of(rr, ks / 4);
            plan->wstream[base + static_cast<size_t>(rr) * ks + chunk * 4 + kk % 4] =
                W[static_cast<size_t>(n) * kin[g] + kg];
          }
        }
      }
    }
  }
  p.n_stages = static_cast<int>(plan->stage_tab.size());
  p.stream_floats = plan->wstream.size();
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
