// Fused single-launch DLRMv1 forward (fp32): the kernel, included by fused.cu
// (the instances without the phase-trace stamps) and fused_trace.cu (those
// with them), so the two halves of the instances compile in parallel.
//
// A CTA runs the whole forward for a tile of BM samples (Luminal compare
// dlrm-fused-kernels...dlrm-pt2-megakernel, dlrm_megakernel.rs steps 1-6:
// bottom Linear+ReLU on every layer, lookups, i-major pairwise dots with
// Vec[0] = x, R = [x, z], top Linear+ReLU then Linear+sigmoid). The launch is
// persistent: at most one CTA per SM, each taking tiles c, c + grid, ... in
// turn while the weight stream flows on through the same ring.
//
// The pages' megakernel keeps one batch row per thread with activations in
// registers; at 512-wide layers that cannot hold. Here the tile's activations
// stay in shared memory for the whole forward and every layer is a CTA-wide
// GEMM of the tile's rows against weights streamed through shared memory:
//  * the weights of all layers form one stream, pre-packed at create time in
//    consumption order, each 32 KB stage one contiguous block whose 16-byte
//    chunks are XOR-swizzled so the warps' reads are bank-conflict free. It
//    flows through a ring of stages filled by 1-D bulk async copies
//    (cp.async.bulk) completing on mbarriers, issued by four lanes of one
//    producer warp that each copy a quarter of every stage (one thread's
//    copies are serialised), running ahead across layer boundaries while
//    eight warps compute.
//  * a computing warp covers all BM rows of the tile and 64 columns (fewer
//    in layers of 32 columns) of one k-slice of each stage: lane bit 0
//    picks the row parity and the other bits a group of columns, so each
//    128-bit shared load reads two activation rows or eight weight columns
//    per half-warp, one wavefront each. The lane's register tile (BM / 2
//    rows x 4 columns: 7 x 4 at 14-row tiles) accumulates with packed
//    fma.rn.f32x2, and the k-slices' partial sums meet in shared memory.
//  * biases and the last layer's weights are fetched with cp.async once per
//    CTA; per tile, one round of global loads checks the bags and fetches
//    the dense rows, and (bag size 1) the tile's embedding rows follow by
//    cp.async and land during the bottom MLP; bag sums and pair dots then run
//    from shared memory and build R = [x, z] in place; the N = 1 sigmoid
//    layer is a warp-per-row dot.
// Every mbarrier wait is bounded (%globaltimer; 2 s unless the launch sets
// another limit): on expiry the kernel sets DLRM_ERRBIT_TIMEOUT, stops
// waiting and finishes its control flow; before exiting it waits (bounded)
// for any copies still in flight.
// Rows past the batch are computed on zeros and never stored.
#pragma once

#include <atomic>

#include "common.cuh"
#include "fused.cuh"
#include "ring.cuh"

namespace dlrm {
namespace {

static_assert(kFusedStageFloats == kRingStageFloats, "one stage size for the plan and the ring");

// Phase trace (profiling): the consumer leader stamps when tile `tile`
// finishes phase `slot`, and (kloop_stamp) where GEMM layer g's leader stamps
// the end of its k-loop (trace slot 20 + g; slot 30 + g then receives the SM
// cycles warp 0 spent waiting for the layer's weight stages), or null.
// The stamps and the k-loop's wait timer exist only in the TRACE instances
// of the kernel (fused_trace.cu, launched while a trace buffer is set):
// compiled into the plain instances, untaken, they cost the 2048-sample,
// 3-table forward 3.6 us (47.0 against 43.4 us), most of it the timer branch
// inside every k-loop stage.
template <bool TRACE>
__device__ __forceinline__ unsigned long long* kloop_stamp(const FusedParams& p, int tile, int g) {
  // slots 20.. are free only while the phase stamps (up to n_gemm + 3) end below
  return (TRACE && p.trace && p.n_gemm + 3 < 20 && 30 + g < kFusedTraceSlots)
             ? p.trace + static_cast<size_t>(tile) * kFusedTraceSlots + 20 + g
             : nullptr;
}

template <bool TRACE>
__device__ __forceinline__ void stamp(const FusedParams& p, int tile, int slot) {
  if (TRACE && p.trace && threadIdx.x == 0)
    p.trace[static_cast<size_t>(tile) * kFusedTraceSlots + slot] = global_ns();
}

// Output columns one pass covers: 2 / ksplit column groups of 32 * tn.
__host__ __device__ __forceinline__ int gemm_cols_per_pass(const FusedGemm& L) {
  return (2 / L.ksplit) * 32 * L.tn;
}

// Staged weight rows (output columns) of pass `pass`.
__host__ __device__ __forceinline__ int gemm_rows(const FusedGemm& L, int pass) {
  const int per_pass = gemm_cols_per_pass(L);
  const int left = L.n_pad - pass * per_pass;
  return left < per_pass ? left : per_pass;
}

// ---------------------------------------------------------------- consumers

// C (BM x n_pad; zero beyond n) = act(A (BM x k_pad) W^T + b). `pos` is the
// warp's place in the stage sequence shared with the producer.
//
// Lane roles: every warp covers all BM rows. Lane bit 0 picks a row parity
// (the lane's TM = BM / 2 rows are rg, rg + 2, ...) and the other lane bits
// one of 16 lane column groups: lane column group lcg = lane / 2 owns the
// warp's columns lcg + 16 j (j < TN), WCOLS = 16 TN columns in all.
// Warp roles: warp w takes column group w % CGS of a pass (CGS = the pass's
// columns / WCOLS) and k-slice w / CGS of every stage (KSLICES = CW / CGS
// slices of KSL = KS / KSLICES values of k, KSL / 4 steps of 4).
// Shared-memory cost: a 128-bit load is served per half-warp, in one
// wavefront when the half-warp's distinct 16-byte words sit in distinct bank
// groups. A half-warp's activation load reads two rows (adjacent rows are
// sixteen banks apart: lda = 16 mod 32) and its weight load eight consecutive
// staged columns (the chunk swizzle puts eight consecutive rows of a stage
// in eight bank groups), so every load costs two wavefronts per warp: per
// 4-wide k step (TM + TN) loads, 2 (TM + TN) wavefronts, for 2 TM TN packed
// FMAs (the even-k and odd-k partial sums of an output in one float2):
// 0.39 wavefronts per packed FMA at 7 x 4, against 1/2 SM cycle of FMA
// pipe; the bulk copy that writes the stage adds 2 / BM.
// The k-slices' partial sums meet in the output buffer (set q at columns
// q * n_pad of each row) and, for the sets past lda / n_pad, the input
// buffer (the planner makes lda >= ceil(KSLICES / 2) * n_pad), where all threads add
// them, the bias and the activation. Layers split into several k-slices have
// a single pass (n_pad <= 256).
constexpr int kDoubleBufferMax = 56;   // lane tile outputs that leave room for it

template <int BM, int TN, int CGS, int KSPLIT, int CW, int LDA, bool TRACE>
__device__ void gemm_layer(const FusedGemm& L, float* a_s, float* c_s, int lda_rt,
                           const float* __restrict__ bias_s, int act, const Ring& r, RingPos& pos,
                           unsigned long long* kstamp) {
  // the activation row stride: a compile-time constant for the common
  // widths (row addresses become immediate offsets), else the plan's
  const int lda = LDA > 0 ? LDA : lda_rt;
  constexpr int R = 2;                         // row parities per warp
  constexpr int TM = BM / R;                   // rows per lane
  constexpr int LCG = kWarp / R;               // lane column groups
  constexpr int WCOLS = LCG * TN;              // columns of one warp
  constexpr int KSLICES = CW / CGS;
  constexpr int KS = 16 * KSPLIT;              // k per stage
  constexpr int KSL = KS / KSLICES;            // k per warp per stage
  constexpr int STEPS = KSL / 4;               // 4-wide k steps per warp per stage
  constexpr int CPR = KS / 4;                  // 16-byte chunks per staged row
  static_assert(BM % R == 0 && CW % CGS == 0 && KS % KSLICES == 0 && STEPS >= 1, "warp slots");
  static_assert(KSLICES == 1 || KSPLIT == 2, "k-sliced layers are the single-pass ones");
  // fragments of step s + 1 load while step s computes, when registers allow
  constexpr bool kDoubleBuffer = TM * TN <= kDoubleBufferMax;
  const int tid = threadIdx.x;
  const int warp = tid / kWarp;
  const int lane = tid % kWarp;
  const int rg = lane % R;
  const int lcg = lane / R;
  const int cg = warp % CGS;
  const int kslice = warp / CGS;
  // chunk swizzle of the lane's staged rows cg * WCOLS + 16 j + lcg: the
  // same for every j (16 j and cg * WCOLS are multiples of 8)
  const int sw = CPR == 4 ? ((lcg >> 1) & 3) : (lcg & 7);
  int ph[STEPS];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) ph[s] = ((kslice * STEPS + s) ^ sw) * 4;
  const float* a_base = a_s + rg * lda + kslice * KSL;
  const int per_pass = CGS * WCOLS;
  long long waited = 0;   // profiling: cycles spent waiting for stages

  for (int pass = 0; pass < L.passes; ++pass) {
    const bool active = cg * WCOLS < gemm_rows(L, pass);
    float2 acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = make_float2(0.f, 0.f);

    for (int kst = 0; kst < L.n_kst; ++kst, pos.advance(r.s_count)) {
      const uint32_t st = pos.slot;
      if (TRACE && kstamp) {   // profiling (uniform): time the wait
        const long long t0 = clock64();
        wait_phase<true>(smem_u32(&r.full[st]), pos.phase, r.abort_flag, r.err, r.limit_ns);
        waited += clock64() - t0;
      } else {
        wait_phase<true>(smem_u32(&r.full[st]), pos.phase, r.abort_flag, r.err, r.limit_ns);
      }
      // In the instances with a compile-time row stride (the workload
      // models') every warp runs the k-loop, also one whose column group lies
      // past the pass's staged rows (the last pass of a layer wider than 512):
      // it reads stale rows inside the stage buffer and its sums are never
      // stored (the epilogue checks `active`). A branch here cost the
      // 2048-sample forward 0.7-1 us although always taken there; the run-time
      // stride instances (the 64-wide model: 0.5 us the other way) keep it.
      if (LDA > 0 || active) {
        const float* ws = r.stages + st * kFusedStageFloats + (cg * WCOLS + lcg) * KS;
        const float* as = a_base + kst * KS;
        if (kDoubleBuffer) {
          float4 wv[2][TN], av[2][TM];
#pragma unroll
          for (int j = 0; j < TN; ++j)
            wv[0][j] = *reinterpret_cast<const float4*>(ws + LCG * j * KS + ph[0]);
#pragma unroll
          for (int i = 0; i < TM; ++i)
            av[0][i] = *reinterpret_cast<const float4*>(as + R * i * lda);
#pragma unroll
          for (int step = 0; step < STEPS; ++step) {
            const int cur = step & 1;
            if (step + 1 < STEPS) {
#pragma unroll
              for (int j = 0; j < TN; ++j)
                wv[cur ^ 1][j] =
                    *reinterpret_cast<const float4*>(ws + LCG * j * KS + ph[step + 1]);
#pragma unroll
              for (int i = 0; i < TM; ++i)
                av[cur ^ 1][i] =
                    *reinterpret_cast<const float4*>(as + R * i * lda + 4 * (step + 1));
            }
            // component-outer: TM * TN independent accumulators between the
            // two dependent updates of each
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
              for (int j = 0; j < TN; ++j)
                acc[i][j] = __ffma2_rn(make_float2(av[cur][i].x, av[cur][i].y),
                                       make_float2(wv[cur][j].x, wv[cur][j].y), acc[i][j]);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
              for (int j = 0; j < TN; ++j)
                acc[i][j] = __ffma2_rn(make_float2(av[cur][i].z, av[cur][i].w),
                                       make_float2(wv[cur][j].z, wv[cur][j].w), acc[i][j]);
          }
        } else {
#pragma unroll
          for (int step = 0; step < STEPS; ++step) {
            float4 wf[TN];
#pragma unroll
            for (int j = 0; j < TN; ++j)
              wf[j] = *reinterpret_cast<const float4*>(ws + LCG * j * KS + ph[step]);
#pragma unroll
            for (int i = 0; i < TM; ++i) {
              const float4 a = *reinterpret_cast<const float4*>(as + R * i * lda + 4 * step);
#pragma unroll
              for (int j = 0; j < TN; ++j)
                acc[i][j] = __ffma2_rn(make_float2(a.x, a.y), make_float2(wf[j].x, wf[j].y),
                                       acc[i][j]);
#pragma unroll
              for (int j = 0; j < TN; ++j)
                acc[i][j] = __ffma2_rn(make_float2(a.z, a.w), make_float2(wf[j].z, wf[j].w),
                                       acc[i][j]);
            }
          }
        }
      }
      ring_release(r, st);
    }

    // profiling: the leader stamps the end of the layer's k-loop and the
    // cycles it waited for weight stages
    if (TRACE && kstamp && pass + 1 == L.passes && threadIdx.x == 0) {
      kstamp[0] = global_ns();
      kstamp[10] = static_cast<unsigned long long>(waited);
    }
    // The lanes' scalar stores below hit row parities rg = 0, 1 at columns
    // lcg + 16 j: with lda = 16 mod 32 the two parities' 16 banks are
    // disjoint, one wavefront per store (two at lda = 4 mod 32).
    const int c0 = pass * per_pass + cg * WCOLS + lcg;   // the lane's first column
    if (KSLICES == 1) {
      if (active) {
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          const int n = c0 + LCG * j;
          const float bv = bias_s[L.b_off + n];
#pragma unroll
          for (int i = 0; i < TM; ++i) {
            const float v = apply_act((acc[i][j].x + acc[i][j].y) + bv, act);
            c_s[(rg + R * i) * lda + n] = (n < L.n) ? v : 0.f;
          }
        }
      }
      consumer_sync<CW>();
    } else {
      // Parallel reduction (one pass: c0 is the column within n_pad). The
      // k-slices' partial sums go to the output buffer, set q at columns
      // q * n_pad for q < qo = lda / n_pad, and the rest to the input buffer
      // (dead once every warp is past its k-loop) at columns (q - qo) *
      // n_pad; then all threads add the sets, the bias and the activation,
      // writing over set 0.
      const int np = L.n_pad;
      const int qo = lda / np;
      if (KSLICES > qo) consumer_sync<CW>();   // the input becomes scratch
      if (active) {
        float* dst = (kslice < qo ? c_s + kslice * np : a_s + (kslice - qo) * np) + c0;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
          for (int j = 0; j < TN; ++j)
            dst[(rg + R * i) * lda + LCG * j] = acc[i][j].x + acc[i][j].y;
      }
      consumer_sync<CW>();
      const int q_shift = 31 - __clz(np >> 2);          // np / 4 is a power of two
      for (int e = tid; e < BM * (np >> 2); e += CW * kWarp) {
        const int m = e >> q_shift;
        const int n = (e - (m << q_shift)) << 2;
        const float* base = c_s + m * lda + n;
        const float* base_a = a_s + m * lda + n;
        float4 v = *reinterpret_cast<const float4*>(base);
#pragma unroll
        for (int q = 1; q < KSLICES; ++q) {
          const float4 u =
              *reinterpret_cast<const float4*>(q < qo ? base + q * np : base_a + (q - qo) * np);
          v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
        }
        const float4 bv = *reinterpret_cast<const float4*>(bias_s + L.b_off + n);
        v.x = (n + 0 < L.n) ? apply_act(v.x + bv.x, act) : 0.f;
        v.y = (n + 1 < L.n) ? apply_act(v.y + bv.y, act) : 0.f;
        v.z = (n + 2 < L.n) ? apply_act(v.z + bv.z, act) : 0.f;
        v.w = (n + 3 < L.n) ? apply_act(v.w + bv.w, act) : 0.f;
        *reinterpret_cast<float4*>(c_s + m * lda + n) = v;
      }
      consumer_sync<CW>();
    }
  }
}

template <int BM, int CW, int LDA, bool TRACE>
__device__ void gemm_dispatch(const FusedGemm& L, float* a_s, float* c_s, int lda,
                              const float* bias_s, int act, int zero_to, const Ring& r,
                              RingPos& pos, unsigned long long* kstamp) {
  // Stage geometry (fused_plan): wider than 256 columns, 512 columns x 16 k
  // per stage (8 warp column groups of 64); 256 columns x 32 k, 2 column
  // groups of 128 (lane tiles BM / 2 x 8) x 4 k-slices; else n_pad = 32 * tn
  // columns x 32 k, cut into n_pad / 64 column groups (at least one) and the
  // rest of the warps as k-slices.
#define DLRM_GEMM_CASE(TN_, CGS_, KSPLIT_) \
  gemm_layer<BM, TN_, CGS_, KSPLIT_, CW, LDA, TRACE>(L, a_s, c_s, lda, bias_s, act, r, pos, kstamp)
  if (L.ksplit == 1) {
    DLRM_GEMM_CASE(4, 8, 1);
  } else {
    switch (L.tn) {
      case 8: DLRM_GEMM_CASE(8, 2, 2); break;     // 256 columns
      case 4: DLRM_GEMM_CASE(4, 2, 2); break;     // 128
      case 2: DLRM_GEMM_CASE(4, 1, 2); break;     // 64
      default: DLRM_GEMM_CASE(2, 1, 2); break;    // 32
    }
  }
#undef DLRM_GEMM_CASE
  const int extra = zero_to - L.n_pad;
  for (int e = threadIdx.x; e < BM * extra; e += CW * kWarp) {
    const int m = e / extra;
    c_s[m * lda + L.n_pad + (e - m * extra)] = 0.f;
  }
  consumer_sync<CW>();
}

// One tile of BM samples, rows m0 = tile * BM on. `first`: the CTA's first
// tile, which also fetches the biases and last-layer weights (they stay in
// shared memory for the CTA's later tiles). `pos` carries the CTA's place in
// the weight stream from tile to tile.
template <int BM, int CW, int LDA, bool TRACE>
__device__ void consume(const FusedParams& p, const Ring& ring, float* act0, float* act1, float* zs,
                        int* rowidx_s, float* bias_s, float* wlast_s, int tile, bool first,
                        RingPos& pos) {
  constexpr int kConsumers = CW * kWarp;
  // Whole-bag prefetch (bags of a few rows) is compiled into the instances
  // with a run-time row stride only: the workload models' instances (bags
  // of one row) keep the exact code they had, which matters here because
  // this kernel's instructions are fetched cold after every L2 flush (the
  // 2048-sample, 3-table forward ran 4 us slower with the extra code inline).
  constexpr bool kBagRows = LDA == 0;
  // Bag-row mode: each compile-time-stride instance takes one mode (528: every
  // bag row prefetched at tile start; 624: rows streamed through two group
  // buffers), so the other modes' code is not in it; fused_instance_lda sends
  // every other plan to the run-time-stride instances, which take any mode.
  const bool pz = LDA == 528 ? true : (LDA == 624 ? false : p.prefetch_z != 0);
  const bool zb2 = LDA == 624 ? true : (LDA == 528 ? false : p.zbuf == 2);
  const int lda = LDA > 0 ? LDA : p.lda;   // activation row stride
  const int tid = threadIdx.x;
  const int m0 = tile * BM;
  const int rows = min(BM, p.batch - m0);
  const int k = p.k_tables, d = p.d, d4 = d >> 2;
  const int f = k + 1;
  const int pairs = f * (f - 1) / 2;
  // quotients by these on the tile's paths come from quot (no divisions)
  const float r_k = __frcp_rn(static_cast<float>(k));
  const float r_d4 = __frcp_rn(static_cast<float>(d4));
  bool oob = false, bad_off = false;

  // Prologue: bias block + last-layer weights (group 0); global loads, two
  // per thread in flight before either is used, that check every bag of
  // size 1 (its row, or -1, kept in shared memory) and fetch the dense
  // features into act0 (zero-padded to the first layer's k_pad); then the
  // tile's embedding rows when they are prefetched whole (group 1).
  stamp<TRACE>(p, tile, 0);
  if (first) {
    for (int c = tid; c < p.bias_floats / 4; c += kConsumers)
      cp_async16(bias_s + 4 * c, p.bias + 4 * c);
    for (int c = tid; c < p.k_last / 4; c += kConsumers) cp_async16(wlast_s + 4 * c, p.wlast + 4 * c);
  }
  cp_async_commit();
  {
    // bag rows to fetch: one per bag, or (bag_rows) every row of every bag,
    // element e = (sample * k + table) * L + l
    const int lb = (kBagRows && p.bag_rows) ? p.bag : 1;
    const int n_bag = (pz || zb2) ? BM * k * lb : 0;
    const int kp = p.gemm[0].k_pad;
    const float r_kp = __frcp_rn(static_cast<float>(kp));
    const float r_lb = kBagRows ? __frcp_rn(static_cast<float>(lb)) : 1.f;
    const int n_dense = BM * kp;
    const int n_all = n_bag > n_dense ? n_bag : n_dense;
    // two elements per thread, both loads in flight before either is used
    for (int e0 = 0; e0 < n_all; e0 += 2 * kConsumers) {
      int64_t start[2], row[2];
      float dv[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = e0 + h * kConsumers + tid;
        start[h] = row[h] = 0;
        dv[h] = 0.f;
        if (e < n_bag) {
          const int sk = kBagRows ? quot(e, lb, r_lb) : e, l = e - sk * lb;
          const int s = quot(sk, k, r_k), t = sk - s * k;
          if (s < rows) {
            const int64_t b = m0 + s;
            start[h] = __ldg(p.offsets + static_cast<int64_t>(t) * p.batch + b);
            row[h] = __ldg(p.indices + (static_cast<int64_t>(t) * p.batch + b) * lb + l);
          }
        }
        if (e < n_dense) {
          const int m = quot(e, kp, r_kp), c = e - m * kp;
          if (m < rows && c < p.n_dense)
            dv[h] = __ldg(p.dense + static_cast<int64_t>(m0 + m) * p.n_dense + c);
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = e0 + h * kConsumers + tid;
        if (e < n_bag) {
          const int sk = kBagRows ? quot(e, lb, r_lb) : e;
          const int s = quot(sk, k, r_k), t = sk - s * k;
          int row32 = -1;
          if (s < rows) {
            // a bag that does not start at b * L is zeros (every one of its
            // rows sees the same start)
            if (start[h] != static_cast<int64_t>(m0 + s) * lb) bad_off = true;
            else if (row[h] < 0 || row[h] >= p.tabs.rows[t]) oob = true;
            else row32 = static_cast<int>(row[h]);
          }
          rowidx_s[e] = row32;
        }
        if (e < n_dense) {
          const int m = quot(e, kp, r_kp);
          act0[m * lda + (e - m * kp)] = dv[h];
        }
      }
    }
  }
  consumer_sync<CW>();
  if (pz) {
    const int lb = (kBagRows && p.bag_rows) ? p.bag : 1;
    const float r_lb = kBagRows ? __frcp_rn(static_cast<float>(lb)) : 1.f;
    for (int e = tid; e < BM * k * lb * d4; e += kConsumers) {
      const int sk = quot(e, d4, r_d4);   // (sample * k + table) * L + l
      const int c4 = e - sk * d4;
      const int sb = kBagRows ? quot(sk, lb, r_lb) : sk;
      const float* table = p.tabs.ptr[sb - quot(sb, k, r_k) * k];
      float* dst = zs + sk * p.ldz + 4 * c4;
      const int row = rowidx_s[sk];
      if (row >= 0) cp_async16(dst, table + static_cast<int64_t>(row) * d + 4 * c4);
      else cp_async16_zero(dst, table);
    }
  }
  cp_async_commit();
  cp_async_wait<1>();
  consumer_sync<CW>();
  stamp<TRACE>(p, tile, 1);

  // Bag-size-1 rows streamed by sample group into two buffers (zbuf == 2).
  const float r_kd4 = __frcp_rn(static_cast<float>(k * d4));
  auto issue_group = [&](int g0, int buf) {
    float* zb = zs + buf * p.sg * k * p.ldz;
    const int ns = min(p.sg, BM - g0);
    for (int e = tid; e < ns * k * d4; e += kConsumers) {
      const int s = quot(e, k * d4, r_kd4);
      const int rem = e - s * k * d4;
      const int t = quot(rem, d4, r_d4);
      const int c4 = rem - t * d4;
      const int row = rowidx_s[(g0 + s) * k + t];
      float* dst = zb + (s * k + t) * p.ldz + 4 * c4;
      const float* table = p.tabs.ptr[t];
      if (row >= 0) cp_async16(dst, table + static_cast<int64_t>(row) * d + 4 * c4);
      else cp_async16_zero(dst, table);
    }
    cp_async_commit();
  };
  if (zb2) {
    // the first two groups land while the bottom MLP runs
    issue_group(0, 0);
    if (p.sg < BM) issue_group(p.sg, 1);
    else cp_async_commit();
  }

  float* in = act0;
  float* out = act1;
  for (int g = 0; g < p.n_bot; ++g) {
    const int zero_to = (g + 1 < p.n_bot) ? p.gemm[g + 1].k_pad : p.gemm[g].n_pad;
    gemm_dispatch<BM, CW, LDA, TRACE>(p.gemm[g], in, out, lda, bias_s, DLRM_ACT_RELU, zero_to, ring, pos,
                          kloop_stamp<TRACE>(p, tile, g));
    float* t = in; in = out; out = t;
    stamp<TRACE>(p, tile, 2 + g);
  }
  const float* x = in;       // bottom output (BM, d)
  float* r = out;            // R = [x, z]

  // Interaction: R[m] = [x[m], z[m]], zero to the next layer's k_pad.
  // x by 16-byte words, and the padding past d + pairs zeroed; the pair dots
  // fill the columns between.
  const int rk = (p.n_top > 1) ? p.gemm[p.n_bot].k_pad : p.k_last;
  for (int e = tid; e < BM * d4; e += kConsumers) {
    const int m = quot(e, d4, r_d4);
    const int c4 = e - m * d4;
    *reinterpret_cast<float4*>(r + m * lda + 4 * c4) =
        *reinterpret_cast<const float4*>(x + m * lda + 4 * c4);
  }
  const int r_pad = rk - d - pairs;
  const float r_rpad = __frcp_rn(static_cast<float>(max(r_pad, 1)));
  for (int e = tid; e < BM * r_pad; e += kConsumers) {
    const int m = quot(e, r_pad, r_rpad);
    r[m * lda + d + pairs + (e - m * r_pad)] = 0.f;
  }
  if (pz) cp_async_wait<0>();
  if (kBagRows && p.bag_rows) {
    // every row of every bag landed at [(sample * k + table) * L + l]: sum
    // each bag's L rows (in order) into registers, then, once all have read,
    // write the sums to rows sample * k + table, the layout of bags of one row
    consumer_sync<CW>();
    constexpr int kMaxSums = kFusedBagRowSums;
    float4 sums[kMaxSums];
    const int lb = p.bag;
#pragma unroll
    for (int i = 0; i < kMaxSums; ++i) {
      const int e = tid + i * kConsumers;
      sums[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < BM * k * d4) {
        const int sk = quot(e, d4, r_d4), c4 = e - sk * d4;
        for (int l = 0; l < lb; ++l) {
          const float4 u = *reinterpret_cast<const float4*>(zs + (sk * lb + l) * p.ldz + 4 * c4);
          sums[i].x += u.x; sums[i].y += u.y; sums[i].z += u.z; sums[i].w += u.w;
        }
      }
    }
    consumer_sync<CW>();
#pragma unroll
    for (int i = 0; i < kMaxSums; ++i) {
      const int e = tid + i * kConsumers;
      if (e < BM * k * d4) {
        const int sk = quot(e, d4, r_d4), c4 = e - sk * d4;
        *reinterpret_cast<float4*>(zs + sk * p.ldz + 4 * c4) = sums[i];
      }
    }
  }
  // zbuf == 2: groups 0 and 1 were issued in the prologue; group g + 2
  // streams into buffer g % 2 once group g's pair dots are done.
  for (int g0 = 0, gi = 0; g0 < BM; g0 += p.sg, ++gi) {
    const int ns = min(p.sg, BM - g0);
    if (zb2) {
      cp_async_wait<1>();   // group gi has landed (only gi + 1 may be pending)
    } else if (!pz) {
      for (int e = tid; e < ns * k * d4; e += kConsumers) {
        const int s = quot(e, k * d4, r_kd4);
        const int rem = e - s * k * d4;
        const int t = quot(rem, d4, r_d4);
        const int c4 = rem - t * d4;
        const int m = g0 + s;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m < rows) {
          const int64_t b = m0 + m;
          const int64_t start = __ldg(p.offsets + static_cast<int64_t>(t) * p.batch + b);
          if (start != b * p.bag) {
            bad_off = true;
          } else {
            const int64_t* idx = p.indices + static_cast<int64_t>(t) * p.batch * p.bag + start;
            const float4* table = reinterpret_cast<const float4*>(p.tabs.ptr[t]);
            const int64_t nrows = p.tabs.rows[t];
            for (int l = 0; l < p.bag; ++l) {
              const int64_t row = __ldg(idx + l);
              if (row >= 0 && row < nrows) {
                const float4 u = __ldg(table + row * d4 + c4);
                v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
              } else {
                oob = true;
              }
            }
          }
        }
        *reinterpret_cast<float4*>(zs + (s * k + t) * p.ldz + 4 * c4) = v;
      }
    }
    consumer_sync<CW>();
    const float* zg = zs + (pz ? g0 * k * p.ldz : (zb2 ? (gi & 1) * p.sg * k * p.ldz : 0));
    // Pair dots; row 0 is x. In 4 x 4 register blocks (gram_block) when the
    // group has a block task for at least every other thread, else one pair
    // per thread: a block reads 8 rows for 16 dots where single pairs read
    // 32, so blocks win on shared-memory traffic even with half the threads
    // idle.
    const int nblk = gram_blocks(f);
    if (2 * ns * nblk >= kConsumers) {
      const float r_nblk = __frcp_rn(static_cast<float>(nblk));
      for (int e = tid; e < ns * nblk; e += kConsumers) {
        const int s = quot(e, nblk, r_nblk);
        const int q = e - s * nblk;
        const float* xrow = x + (g0 + s) * lda;
        const float* zsam = zg + s * k * p.ldz;
        float acc[4][4];
        int bi, bj;
        gram_block([&](int rr) { return rr == 0 ? xrow : zsam + (rr - 1) * p.ldz; }, f, d4, q,
                   bi, bj, acc);
        float* o = r + (g0 + s) * lda + d;
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int q2 = gram_block_pair(f, bi, bj, a, c);
            if (q2 >= 0) o[q2] = acc[a][c];
          }
      }
    } else {
      const float r_pairs = __frcp_rn(static_cast<float>(pairs));
      for (int e = tid; e < ns * pairs; e += kConsumers) {
        const int s = quot(e, pairs, r_pairs);
        const int q = e - s * pairs;
        int i, j;
        pair_from_index(q, i, j);
        const float* vi = (i == 0) ? x + (g0 + s) * lda : zg + (s * k + i - 1) * p.ldz;
        const float* vj = (j == 0) ? x + (g0 + s) * lda : zg + (s * k + j - 1) * p.ldz;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int c4 = 0; c4 < d4; ++c4) {
          const float4 u = *reinterpret_cast<const float4*>(vi + 4 * c4);
          const float4 w = *reinterpret_cast<const float4*>(vj + 4 * c4);
          a.x = fmaf(u.x, w.x, a.x);
          a.y = fmaf(u.y, w.y, a.y);
          a.z = fmaf(u.z, w.z, a.z);
          a.w = fmaf(u.w, w.w, a.w);
        }
        r[(g0 + s) * lda + d + q] = (a.x + a.y) + (a.z + a.w);
      }
    }
    consumer_sync<CW>();
    if (zb2) {
      if (g0 + 2 * p.sg < BM) issue_group(g0 + 2 * p.sg, gi & 1);
      else cp_async_commit();
    }
  }
  if (p.err) {
    if (oob) atomicOr(reinterpret_cast<unsigned int*>(p.err), DLRM_ERRBIT_INDEX_OOB);
    if (bad_off) atomicOr(reinterpret_cast<unsigned int*>(p.err), DLRM_ERRBIT_OFFSETS);
  }

  stamp<TRACE>(p, tile, 2 + p.n_bot);
  // Top MLP: ReLU layers, then the N = 1 sigmoid layer.
  in = r;
  out = (r == act0) ? act1 : act0;
  for (int g = p.n_bot; g < p.n_gemm; ++g) {
    const int zero_to = (g + 1 < p.n_gemm) ? p.gemm[g + 1].k_pad : p.k_last;
    gemm_dispatch<BM, CW, LDA, TRACE>(p.gemm[g], in, out, lda, bias_s, DLRM_ACT_RELU, zero_to, ring, pos,
                          kloop_stamp<TRACE>(p, tile, g));
    float* t = in; in = out; out = t;
    stamp<TRACE>(p, tile, 3 + g);
  }
  const int warp = tid / kWarp, lane = tid % kWarp;
  const int k4 = p.k_last / 4;
  const float bl = bias_s[p.b_last];
  for (int m = warp; m < rows; m += CW) {
    float acc = 0.f;
    for (int q = lane; q < k4; q += kWarp) {
      const float4 a = *reinterpret_cast<const float4*>(in + m * lda + 4 * q);
      const float4 w = *reinterpret_cast<const float4*>(wlast_s + 4 * q);
      acc = fmaf(a.x, w.x, acc);
      acc = fmaf(a.y, w.y, acc);
      acc = fmaf(a.z, w.z, acc);
      acc = fmaf(a.w, w.w, acc);
    }
#pragma unroll
    for (int o = kWarp / 2; o > 0; o /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) p.out[m0 + m] = apply_act(acc + bl, DLRM_ACT_SIGMOID);
  }
  // the next tile overwrites the activation, bag-row and row-index buffers
  consumer_sync<CW>();
  stamp<TRACE>(p, tile, 2 + p.n_gemm + 1);
}

// Warps: CW = 8 computing warps (warpgroups 0 and 1) and a producer
// warpgroup (warps 8-11) of which warp 8 streams the weights. At launch
// every thread has kLaunchRegs registers (the cap for 12 warps: three share
// one sub-partition's 16K); the producer warpgroup then gives most of its
// registers back (setmaxnreg.dec to kProducerRegs) and the computing
// warpgroups take them (setmaxnreg.inc to kComputeRegs), so a computing
// thread holds a BM / 2 x 8 lane tile with double-buffered operands. The
// split adds up exactly to the launch allocation (checked below); the host
// refuses an instance that ptxas built with a different launch count.
constexpr int kFusedWarps = 12;
constexpr int kLaunchRegs = 168;
constexpr int kProducerRegs = 40;
constexpr int kComputeRegs = 232;
static_assert(8 * kWarp * kComputeRegs + 4 * kWarp * kProducerRegs <=
                  kFusedWarps * kWarp * kLaunchRegs,
              "register split exceeds the launch allocation");

template <int BM, int CW, int LDA, bool TRACE>
__global__ void __launch_bounds__(kFusedWarps * 32, 1)
fused_forward_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* stages = reinterpret_cast<float*>(smem_raw);
  float* act0 = reinterpret_cast<float*>(smem_raw + p.off_act0);
  float* act1 = reinterpret_cast<float*>(smem_raw + p.off_act1);
  float* zs = reinterpret_cast<float*>(smem_raw + p.off_z);
  float* bias_s = reinterpret_cast<float*>(smem_raw + p.off_bias);
  float* wlast_s = reinterpret_cast<float*>(smem_raw + p.off_wlast);
  int* rowidx_s = reinterpret_cast<int*>(smem_raw + p.off_rowidx);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + p.off_bar);
  uint64_t* empty = full + p.stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + p.stages);
  const Ring r{stages, full, empty, abort_flag, static_cast<uint32_t>(p.stages), p.err,
               wait_limit_ns(p.wait)};
  const int warp = threadIdx.x / kWarp;
  // persistent: CTA c runs tiles c, c + gridDim.x, ...
  const int n_tiles = (p.batch + BM - 1) / BM;
  const int my_tiles = (n_tiles - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), CW);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  static_assert(CW == 8, "two computing warpgroups");
  if (warp >= CW) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs) : "memory");
    if (warp > CW) return;
    // the L2 prefetch from a lane that issues no copies: a thread's bulk
    // operations run one after another
    if (threadIdx.x % kWarp == kWarp - 1) prefetch_stream_l2(p.wstream, p.stream_floats);
    produce(r, p.wstream, p.stage_tab, static_cast<uint32_t>(p.n_stages),
            static_cast<uint32_t>(my_tiles), p.wait.withhold_last != 0);
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kComputeRegs) : "memory");
  RingPos pos;
  for (int i = 0; i < my_tiles; ++i)
    consume<BM, CW, LDA, TRACE>(p, r, act0, act1, zs, rowidx_s, bias_s, wlast_s,
                    static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x), i == 0, pos);
}

template <int BM, int CW, int LDA, bool TRACE>
cudaError_t enable_smem_one() {
  // the register split in the kernel assumes exactly kLaunchRegs per thread
  // at launch: any other count could leave setmaxnreg.inc waiting forever
  cudaFuncAttributes attr{};
  cudaError_t e = cudaFuncGetAttributes(&attr, fused_forward_kernel<BM, CW, LDA, TRACE>);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(fused_forward_kernel<BM, CW, LDA, TRACE>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(device_max_smem_optin()));
}

template <int BM, int CW, int LDA, bool TRACE>
cudaError_t enable_smem() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = enable_smem_one<BM, CW, LDA, TRACE>();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Kernel instances: every tile height with a run-time activation row stride,
// and the tile heights of 8 rows and more with the strides the workload
// models take (528: widest layer or interaction row <= 512 floats; 624: the
// 32-table models' 592-wide interaction rows) as compile-time constants.
#define DLRM_FUSED_SWITCH(BM_VAR, LDA_VAR, CALL)                                     \
  switch ((BM_VAR) * 10000 + (((BM_VAR) >= 8 && ((LDA_VAR) == 528 || (LDA_VAR) == 624)) \
                                  ? (LDA_VAR)                                          \
                                  : 0)) {                                              \
    case 16 * 10000 + 528: CALL(16, 528); break;                                       \
    case 16 * 10000 + 624: CALL(16, 624); break;                                       \
    case 16 * 10000: CALL(16, 0); break;                                               \
    case 14 * 10000 + 528: CALL(14, 528); break;                                       \
    case 14 * 10000 + 624: CALL(14, 624); break;                                       \
    case 14 * 10000: CALL(14, 0); break;                                               \
    case 12 * 10000 + 528: CALL(12, 528); break;                                       \
    case 12 * 10000 + 624: CALL(12, 624); break;                                       \
    case 12 * 10000: CALL(12, 0); break;                                               \
    case 8 * 10000 + 528: CALL(8, 528); break;                                         \
    case 8 * 10000 + 624: CALL(8, 624); break;                                         \
    case 8 * 10000: CALL(8, 0); break;                                                 \
    case 4 * 10000: CALL(4, 0); break;                                                 \
    default: return cudaErrorInvalidValue;                                             \
  }


// Instance selection and launch of the TRACE or plain instances.
template <bool TRACE>
cudaError_t prepare_fused_instances(int bm, int cw, int lda) {
  if (cw != 8) return cudaErrorInvalidValue;
#define DLRM_PREPARE(BM_, LDA_) return enable_smem<BM_, 8, LDA_, TRACE>()
  DLRM_FUSED_SWITCH(bm, lda, DLRM_PREPARE)
#undef DLRM_PREPARE
}

template <bool TRACE>
cudaError_t launch_fused_instances(const FusedParams& p, int bm, cudaStream_t stream) {
  if (p.batch == 0) return cudaSuccess;
  // persistent: at most one CTA per SM, each looping over its tiles
  const int64_t tiles = (p.batch + bm - 1) / bm;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(tiles, device_sm_count()));
  const int ilda = fused_instance_lda(p);
  cudaError_t e = prepare_fused_instances<TRACE>(bm, p.cw, ilda);
  if (e != cudaSuccess) return e;
  const unsigned threads = static_cast<unsigned>(kFusedWarps * kWarp);
#define DLRM_LAUNCH(BM_, LDA_) \
  fused_forward_kernel<BM_, 8, LDA_, TRACE><<<grid, threads, p.smem_bytes, stream>>>(p)
  DLRM_FUSED_SWITCH(bm, ilda, DLRM_LAUNCH)
#undef DLRM_LAUNCH
  return cudaGetLastError();
}

}  // namespace
}  // namespace dlrm
