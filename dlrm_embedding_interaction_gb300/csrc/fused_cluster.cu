// Cluster-split fused DLRMv1 forward (fp32) for small batches.
//
// The same forward as fused.cu (Luminal compare
// dlrm-fused-kernels...dlrm-pt2-megakernel, dlrm_megakernel.rs steps 1-6:
// bottom Linear+ReLU on every layer, lookups, i-major pairwise dots with
// Vec[0] = x, R = [x, z], top Linear+ReLU then Linear+sigmoid) for a tile of
// bm samples, but run by a cluster of C CTAs instead of one. A single CTA
// would stream every layer's weights through its own shared memory for
// only a few samples, which bounds small batches by one SM's weight feed.
// Here CTA q of the cluster holds output columns [q s, (q + 1) s) of every
// layer (s = n_pad / C): it streams only that 1/C share of the weights
// through its ring, computes the tile's outputs in those columns, and pushes
// them into the activation buffers of all C CTAs with st.async, each store
// signalling the receiver's exchange mbarrier with its bytes (distributed
// shared memory). A CTA starts layer g + 1 once its barrier has counted all
// of layer g's bytes. The interaction is split by samples (CTA q builds the
// R rows of samples q, q + C, ...) and exchanged the same way; the N = 1
// sigmoid layer is split by samples and stored directly.
//
// Exchange protocol. Exchange e (the bottom layers, the interaction, then
// the top layers but the last) lands on barrier e & 1 in phase e >> 1. A
// CTA arms exchange e + 1 (expect_tx of its byte count) before it pushes any
// byte of exchange e; a peer pushes exchange e + 1 only after receiving all
// of exchange e, so no byte can reach a barrier before its phase is armed.
// Outputs alternate between two activation buffers, and a peer writes
// layer g + 1's outputs into the buffer this CTA read layer g from only
// after this CTA has pushed layer g, i.e. finished reading it.
//
// Bounded waits: ring stages and exchanges give up after the launch's wait
// limit (DLRM_ERRBIT_TIMEOUT); a CTA that gave up still pushes all its bytes
// (then garbage), so every exchange completes. A cluster barrier at start
// (barriers initialised before any push) and one at exit (no CTA leaves
// while a peer may still write into it) are reached by every thread.
#include <atomic>

#include "common.cuh"
#include "fused_cluster.cuh"
#include "ring.cuh"

namespace dlrm {
namespace {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
  return d;
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// 16 bytes into a peer's shared memory; the peer's mbarrier `bar` counts them.
__device__ __forceinline__ void push16(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, "
      "[%5];" ::"r"(addr),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}

// Bounded wait for an exchange phase (bytes pushed by the cluster's CTAs):
// acquire at cluster scope. False when this or another thread gave up.
__device__ __forceinline__ bool wait_exchange(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int32_t* err,
                                              uint64_t limit_ns) {
  auto test = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
  };
  if (test()) return true;
  if (*abort_flag) return false;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (test()) return true;
    if ((i & 15) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        if (err) atomicOr(reinterpret_cast<unsigned int*>(err), DLRM_ERRBIT_TIMEOUT);
        return false;
      }
    }
  }
}

// Bytes exchange e brings every CTA of the cluster.
__device__ __forceinline__ uint32_t exchange_bytes(const ClusterParams& p, int e) {
  if (e == p.n_bot) return static_cast<uint32_t>(p.bm * p.ld_r * 4);
  const int g = e < p.n_bot ? e : e - 1;
  return static_cast<uint32_t>(p.bm * p.gemm[g].s * p.csize * 4);
}

// The exchange after GEMM layer g (bottom layers 0.., then the interaction,
// then the top layers).
__device__ __forceinline__ int exchange_of_gemm(const ClusterParams& p, int g) {
  return g < p.n_bot ? g : g + 1;
}

struct Cta {
  uint32_t q;             // rank in the cluster
  uint32_t xbar0, xbar1;  // local addresses of the exchange barriers
  volatile int* abort_flag;
  uint64_t limit_ns;
  __device__ __forceinline__ uint32_t xbar(int e) const { return (e & 1) ? xbar1 : xbar0; }
};

// Arms exchange e (if it exists: there are n_gemm + 1, the last after the
// last top GEMM layer) on this CTA: one arrival plus its bytes.
__device__ __forceinline__ void arm_exchange(const ClusterParams& p, const Cta& c, int e) {
  if (e <= p.n_gemm && threadIdx.x == 0) mbar_arrive_expect_tx(c.xbar(e), exchange_bytes(p, e));
}

// Sends a float4 of this CTA's outputs to `count` ranks rk = first, first +
// stride, ... of the cluster (the same address in each).
__device__ __forceinline__ void push_ranks(uint32_t dst, uint32_t bar, float4 v, int first,
                                           int stride, int csize) {
  for (int rk = first; rk < csize; rk += stride)
    push16(map_rank(dst, static_cast<uint32_t>(rk)), v, map_rank(bar, static_cast<uint32_t>(rk)));
}

// GEMM layer g on this CTA's column slice; the outputs (bias, ReLU) pushed
// to the out buffer of every CTA of the cluster, then this CTA waits for the
// whole layer. `last`: the last exchange of the forward; once its bytes have
// left, this CTA arrives on the exit barrier (it pushes nothing more).
template <int BM>
__device__ void cluster_gemm(const ClusterParams& p, const Cta& c, int g, const float* a_s,
                             float* out_s, float* scratch, const float* bias_s, const Ring& r,
                             RingPos& pos, bool last) {
  const ClusterGemm& L = p.gemm[g];
  const int tid = threadIdx.x;
  const int lda = p.lda;
  const int half = L.s >> 1;               // a power of two
  const int cg = tid & (half - 1);
  const int ks = tid >> (31 - __clz(half));
  const int k4v = (L.k + 3) >> 2;
  // kslices = 512 / s is a power of two: shifts, not divisions, per stage
  // (k_here is a multiple of 4 kslices; the inputs left are rounded up by
  // the shift, every operand non-negative)
  const int kshift = 31 - __clz(L.kslices);
  float2 acc[BM][2];
#pragma unroll
  for (int m = 0; m < BM; ++m) acc[m][0] = acc[m][1] = make_float2(0.f, 0.f);

  for (int kst = 0; kst < L.n_kst; ++kst, pos.advance(r.s_count)) {
    wait_phase<true>(smem_u32(&r.full[pos.slot]), pos.phase, r.abort_flag, r.err, r.limit_ns);
    const float4* w = reinterpret_cast<const float4*>(r.stages + pos.slot * kRingStageFloats);
    const int k_here = min(L.kst_k, L.k_pad - kst * L.kst_k);
    const int steps = k_here >> (2 + kshift);
    const int k4_0 = kst * (L.kst_k >> 2) + ks;
    // the thread's steps that reach inputs below k (k4_0 + kslices i < k4v)
    const int n = k4_0 < k4v ? min(steps, (k4v - k4_0 + L.kslices - 1) >> kshift) : 0;
    const float* a0 = a_s + 4 * k4_0;
#pragma unroll 4
    for (int i = 0; i < n; ++i) {
      const float4 w0 = w[(2 * i) * kClusterThreads + tid];
      const float4 w1 = w[(2 * i + 1) * kClusterThreads + tid];
      const float* ai = a0 + 4 * L.kslices * i;
#pragma unroll
      for (int m = 0; m < BM; ++m) {
        const float4 a = *reinterpret_cast<const float4*>(ai + m * lda);
        acc[m][0] = __ffma2_rn(make_float2(a.x, a.y), make_float2(w0.x, w0.y), acc[m][0]);
        acc[m][1] = __ffma2_rn(make_float2(a.x, a.y), make_float2(w1.x, w1.y), acc[m][1]);
        acc[m][0] = __ffma2_rn(make_float2(a.z, a.w), make_float2(w0.z, w0.w), acc[m][0]);
        acc[m][1] = __ffma2_rn(make_float2(a.z, a.w), make_float2(w1.z, w1.w), acc[m][1]);
      }
    }
    ring_release(r, pos.slot);
  }
  // k-slice partial sums: scratch[slice * kstride + m * s + column]. The
  // slices sit kstride = BM s + 4 floats apart: BM s is a multiple of 32
  // floats, and without the skew the G lanes that sum one output float4
  // (consecutive slices) would read one bank group, G ways conflicted.
  const int kstride = BM * L.s + 4;
#pragma unroll
  for (int m = 0; m < BM; ++m)
    *reinterpret_cast<float2*>(scratch + ks * kstride + m * L.s + 2 * cg) =
        make_float2(acc[m][0].x + acc[m][0].y, acc[m][1].x + acc[m][1].y);
  const int e = exchange_of_gemm(p, g);
  arm_exchange(p, c, e + 1);   // before any byte of exchange e leaves this CTA
  consumer_sync<kClusterWarps>();
  // Each float4 of outputs is summed over the k-slices by a group of G
  // consecutive lanes (G a power of two: 32 when the outputs are few), then
  // the group's lanes push it to the cluster's ranks between them.
  const int s4 = L.s >> 2;
  const int s4shift = 31 - __clz(s4);
  static_assert(BM == 4 || BM == 8 || BM == 16, "tile heights");
  constexpr int kLog2BM = BM == 4 ? 2 : (BM == 8 ? 3 : 4);
  const int oshift = kLog2BM + s4shift;     // outs = BM * s4, a power of two
  const int outs = 1 << oshift;
  int gsz = oshift >= 8 ? 1 : min(kClusterThreads >> oshift, 32);
  if (gsz > L.kslices) gsz = L.kslices;
  const int gshift = 31 - __clz(gsz);
  const int gl = tid & (gsz - 1);
  const uint32_t bar = c.xbar(e);
  const uint32_t base = smem_u32(out_s) + 4u * (c.q * L.s);
  for (int t0 = 0; t0 < outs * gsz; t0 += kClusterThreads) {
    const int o = (t0 + tid) >> gshift;
    const bool live = o < outs;
    const int m = live ? o >> s4shift : 0;
    const int c4 = live ? o & (s4 - 1) : 0;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
      for (int kk = gl; kk < L.kslices; kk += gsz) {
        const float4 u =
            *reinterpret_cast<const float4*>(scratch + kk * kstride + m * L.s + 4 * c4);
        v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
      }
    }
    for (int off = gsz >> 1; off > 0; off >>= 1) {
      v.x += __shfl_xor_sync(0xffffffffu, v.x, off);
      v.y += __shfl_xor_sync(0xffffffffu, v.y, off);
      v.z += __shfl_xor_sync(0xffffffffu, v.z, off);
      v.w += __shfl_xor_sync(0xffffffffu, v.w, off);
    }
    if (live) {
      const float4 bv = *reinterpret_cast<const float4*>(bias_s + L.b_off + 4 * c4);
      v.x = fmaxf(v.x + bv.x, 0.f);
      v.y = fmaxf(v.y + bv.y, 0.f);
      v.z = fmaxf(v.z + bv.z, 0.f);
      v.w = fmaxf(v.w + bv.w, 0.f);
      push_ranks(base + 4u * (m * lda + 4 * c4), bar, v, gl, gsz, p.csize);
    }
  }
  if (last) cluster_arrive();
  wait_exchange(bar, (e >> 1) & 1, c.abort_flag, p.err, c.limit_ns);
}

template <int BM>
__device__ void cluster_consume(const ClusterParams& p, const Cta& c, const Ring& ring,
                                float* act0, float* act1, float* scratch, float* zs, int* rowidx_s,
                                float* bias_s, float* wlast_s) {
  const int tid = threadIdx.x;
  const int lda = p.lda;
  const int C = p.csize;
  const int m0 = static_cast<int>(cluster_id()) * BM;
  const int rows = min(BM, p.batch - m0);
  const int k = p.k_tables, d = p.d, d4 = d >> 2;
  const int f = k + 1;
  const int pairs = f * (f - 1) / 2;
  const int cshift = 31 - __clz(C);       // clusters of 2 to 16 CTAs
  const float r_k = __frcp_rn(static_cast<float>(k));
  const float r_d4 = __frcp_rn(static_cast<float>(d4));
  bool oob = false, bad_off = false;

  // Prologue: this rank's bias block and the last layer's weights (group
  // 0); the tile's dense rows (zero-padded to a multiple of 4 columns); the
  // bags of this CTA's interaction rows q, q + C, ... checked and, with bags
  // of one row, their table rows fetched (group 1).
  for (int i = tid; i < p.bias_floats / 4; i += kClusterThreads)
    cp_async16(bias_s + 4 * i, p.bias + static_cast<size_t>(c.q) * p.bias_floats + 4 * i);
  for (int i = tid; i < p.k_last / 4; i += kClusterThreads) cp_async16(wlast_s + 4 * i, p.wlast + 4 * i);
  cp_async_commit();
  // One round of global loads, both elements of a thread in flight before
  // either is used: dense features and (bags of one row) bag starts and rows.
  const int kd = (p.n_dense + 3) & ~3;
  const float r_kd = __frcp_rn(static_cast<float>(kd));
  const int n_dense = BM * kd;
  const int n_bag = p.bag == 1 ? p.zrows * k : 0;
  const int n_all = max(n_dense, n_bag);
  for (int e0 = 0; e0 < n_all; e0 += 2 * kClusterThreads) {
    float dv[2];
    int64_t start[2], row[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = e0 + h * kClusterThreads + tid;
      dv[h] = 0.f;
      start[h] = row[h] = 0;
      if (e < n_dense) {
        const int m = quot(e, kd, r_kd), col = e - m * kd;
        if (m < rows && col < p.n_dense)
          dv[h] = __ldg(p.dense + static_cast<int64_t>(m0 + m) * p.n_dense + col);
      }
      if (e < n_bag) {
        const int j = quot(e, k, r_k), t = e - j * k;
        const int m = static_cast<int>(c.q) + C * j;
        if (m < rows) {
          start[h] = __ldg(p.offsets + static_cast<int64_t>(t) * p.batch + m0 + m);
          row[h] = __ldg(p.indices + static_cast<int64_t>(t) * p.batch + m0 + m);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = e0 + h * kClusterThreads + tid;
      if (e < n_dense) {
        const int m = quot(e, kd, r_kd);
        act0[m * lda + (e - m * kd)] = dv[h];
      }
      if (e < n_bag) {
        const int j = quot(e, k, r_k), t = e - j * k;
        const int m = static_cast<int>(c.q) + C * j;
        int row32 = -1;
        if (m < rows) {
          if (start[h] != m0 + m) bad_off = true;
          else if (row[h] < 0 || row[h] >= p.tabs.rows[t]) oob = true;
          else row32 = static_cast<int>(row[h]);
        }
        rowidx_s[e] = row32;
      }
    }
  }
  if (p.bag == 1) {
    consumer_sync<kClusterWarps>();
    for (int e = tid; e < p.zrows * k * d4; e += kClusterThreads) {
      const int jt = quot(e, d4, r_d4);   // row * k + table
      const int c4 = e - jt * d4;
      const float* table = p.tabs.ptr[jt - quot(jt, k, r_k) * k];
      float* dst = zs + jt * p.ldz + 4 * c4;
      const int rw = rowidx_s[jt];
      if (rw >= 0) cp_async16(dst, table + static_cast<int64_t>(rw) * d + 4 * c4);
      else cp_async16_zero(dst, table);
    }
  }
  cp_async_commit();
  cp_async_wait<1>();
  consumer_sync<kClusterWarps>();
  // every CTA of the cluster has its exchange barriers armed before any push
  cluster_wait();

  RingPos pos;
  float* in = act0;
  float* out = act1;
  for (int g = 0; g < p.n_bot; ++g) {
    cluster_gemm<BM>(p, c, g, in, out, scratch, bias_s, ring, pos, false);
    float* t = in; in = out; out = t;
  }
  const float* x = in;       // bottom output (BM, d), every row
  float* rbuf = out;         // R = [x, z], filled by the exchange

  // Interaction rows q, q + C, ... of the tile: bag sums (bags of one row:
  // already fetched), then x and the pair dots staged in scratch.
  if (p.bag == 1) {
    cp_async_wait<0>();
  } else {
    for (int e = tid; e < p.zrows * k * d4; e += kClusterThreads) {
      const int jt = quot(e, d4, r_d4);
      const int c4 = e - jt * d4;
      const int j = quot(jt, k, r_k), t = jt - j * k;
      const int m = static_cast<int>(c.q) + C * j;
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
      *reinterpret_cast<float4*>(zs + jt * p.ldz + 4 * c4) = v;
    }
  }
  consumer_sync<kClusterWarps>();
  const int ld_r = p.ld_r;
  // rows q, q + C, ... below BM
  const int nmine = max(BM - static_cast<int>(c.q) + C - 1, 0) >> cshift;
  for (int j = 0; j < nmine; ++j) {
    const int m = static_cast<int>(c.q) + C * j;
    for (int col = tid; col < ld_r; col += kClusterThreads)
      scratch[j * ld_r + col] = col < d ? x[m * lda + col] : 0.f;   // pairs overwrite [d, d + pairs) below
  }
  consumer_sync<kClusterWarps>();
  // Pair dots (row 0 is x) of this CTA's rows: in 4 x 4 register blocks
  // (gram_block), or one pair per group of G lanes that split D and meet by
  // shuffles, whichever the cost estimate (block or step latencies per
  // round of 256 threads) finds shorter for these few rows.
  const int nblk = gram_blocks(f);
  const int block_cost = (nmine * nblk + kClusterThreads - 1) / kClusterThreads * d4 * 64;
  int gsz = 0, lane_cost = block_cost;
  for (int lg = 0; lg <= 5 && (1 << lg) <= d4; ++lg) {
    const int gg = 1 << lg;
    const int rounds = (nmine * pairs * gg + kClusterThreads - 1) / kClusterThreads;
    const int cost = rounds * (((d4 + gg - 1) >> lg) * 40 + 120);
    if (cost < lane_cost) {
      lane_cost = cost;
      gsz = gg;
    }
  }
  if (gsz == 0) {
    const float r_nblk = __frcp_rn(static_cast<float>(nblk));
    for (int e = tid; e < nmine * nblk; e += kClusterThreads) {
      const int j = quot(e, nblk, r_nblk);
      const int qb = e - j * nblk;
      const int m = static_cast<int>(c.q) + C * j;
      const float* xrow = x + m * lda;
      const float* zsam = zs + j * k * p.ldz;
      float acc[4][4];
      int bi, bj;
      gram_block([&](int rr) { return rr == 0 ? xrow : zsam + (rr - 1) * p.ldz; }, f, d4, qb,
                 bi, bj, acc);
      float* o = scratch + j * ld_r + d;
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int q2 = gram_block_pair(f, bi, bj, a, cc);
          if (q2 >= 0) o[q2] = acc[a][cc];
        }
    }
  } else {
    const int gl = tid & (gsz - 1);
    const int gshift = 31 - __clz(gsz);
    const float r_pairs = __frcp_rn(static_cast<float>(pairs));
    const int tasks = nmine * pairs;
    for (int t0 = 0; t0 < tasks * gsz; t0 += kClusterThreads) {
      const int task = (t0 + tid) >> gshift;
      float a = 0.f;
      int j = 0, q = 0;
      if (task < tasks) {
        j = quot(task, pairs, r_pairs);
        q = task - j * pairs;
        int i, jj;
        pair_from_index(q, i, jj);
        const int m = static_cast<int>(c.q) + C * j;
        const float* zsam = zs + j * k * p.ldz;
        const float* vi = i == 0 ? x + m * lda : zsam + (i - 1) * p.ldz;
        const float* vj = jj == 0 ? x + m * lda : zsam + (jj - 1) * p.ldz;
        for (int c4 = gl; c4 < d4; c4 += gsz) {
          const float4 u = *reinterpret_cast<const float4*>(vi + 4 * c4);
          const float4 w = *reinterpret_cast<const float4*>(vj + 4 * c4);
          a = fmaf(u.x, w.x, a);
          a = fmaf(u.y, w.y, a);
          a = fmaf(u.z, w.z, a);
          a = fmaf(u.w, w.w, a);
        }
      }
      for (int off = gsz >> 1; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
      if (task < tasks && gl == 0) scratch[j * ld_r + d + q] = a;
    }
  }
  {
    const int e_int = p.n_bot;
    arm_exchange(p, c, e_int + 1);
    consumer_sync<kClusterWarps>();
    const uint32_t bar = c.xbar(e_int);
    const uint32_t base = smem_u32(rbuf);
    const int r4 = ld_r >> 2;
    // each float4 of R by C consecutive threads, one rank each
    for (int j = 0; j < nmine; ++j) {
      const int m = static_cast<int>(c.q) + C * j;
      for (int e = tid; e < r4 * C; e += kClusterThreads) {
        const int c4 = e >> cshift, rk = e & (C - 1);
        const float4 v = *reinterpret_cast<const float4*>(scratch + j * ld_r + 4 * c4);
        push_ranks(base + 4u * (m * lda + 4 * c4), bar, v, rk, C, C);
      }
    }
    wait_exchange(bar, (e_int >> 1) & 1, c.abort_flag, p.err, c.limit_ns);
  }
  (void)pairs;

  // Top MLP: ReLU layers, then the N = 1 sigmoid layer by rows q, q + C, ...
  in = rbuf;
  out = (rbuf == act0) ? act1 : act0;
  for (int g = p.n_bot; g < p.n_gemm; ++g) {
    cluster_gemm<BM>(p, c, g, in, out, scratch, bias_s, ring, pos, g + 1 == p.n_gemm);
    float* t = in; in = out; out = t;
  }
  const int warp = tid / kWarp, lane = tid % kWarp;
  const int k4 = p.k_last / 4;
  for (int m = static_cast<int>(c.q) + C * warp; m < rows; m += C * kClusterWarps) {
    float a = 0.f;
    for (int i = lane; i < k4; i += kWarp) {
      const float4 u = *reinterpret_cast<const float4*>(in + m * lda + 4 * i);
      const float4 w = *reinterpret_cast<const float4*>(wlast_s + 4 * i);
      a = fmaf(u.x, w.x, a);
      a = fmaf(u.y, w.y, a);
      a = fmaf(u.z, w.z, a);
      a = fmaf(u.w, w.w, a);
    }
#pragma unroll
    for (int o = kWarp / 2; o > 0; o /= 2) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) p.out[m0 + m] = apply_act(a + p.b_last, DLRM_ACT_SIGMOID);
  }
  if (p.err) {
    if (oob) atomicOr(reinterpret_cast<unsigned int*>(p.err), DLRM_ERRBIT_INDEX_OOB);
    if (bad_off) atomicOr(reinterpret_cast<unsigned int*>(p.err), DLRM_ERRBIT_OFFSETS);
  }
}

template <int BM>
__global__ void __launch_bounds__(kClusterThreads + kWarp, 1)
fused_cluster_kernel(const __grid_constant__ ClusterParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* stages = reinterpret_cast<float*>(smem_raw);
  float* act0 = reinterpret_cast<float*>(smem_raw + p.off_act0);
  float* act1 = reinterpret_cast<float*>(smem_raw + p.off_act1);
  float* scratch = reinterpret_cast<float*>(smem_raw + p.off_scratch);
  float* zs = reinterpret_cast<float*>(smem_raw + p.off_z);
  int* rowidx_s = reinterpret_cast<int*>(smem_raw + p.off_rowidx);
  float* bias_s = reinterpret_cast<float*>(smem_raw + p.off_bias);
  float* wlast_s = reinterpret_cast<float*>(smem_raw + p.off_wlast);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + p.off_bar);
  uint64_t* empty = full + p.stages;
  uint64_t* xbar = empty + p.stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(xbar + 2);
  const uint64_t limit = wait_limit_ns(p.wait);
  const Ring r{stages, full, empty, abort_flag, static_cast<uint32_t>(p.stages), p.err, limit};
  Cta c;
  c.q = cluster_rank();
  c.xbar0 = smem_u32(&xbar[0]);
  c.xbar1 = smem_u32(&xbar[1]);
  c.abort_flag = abort_flag;
  c.limit_ns = limit;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kClusterWarps);
    }
    mbar_init(c.xbar0, 1);
    mbar_init(c.xbar1, 1);
    *abort_flag = 0;
    mbar_arrive_expect_tx(c.xbar0, exchange_bytes(p, 0));   // exchange 0 armed
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  cluster_arrive();   // this CTA's barriers are ready for the cluster's pushes
  const int warp = threadIdx.x / kWarp;
  // Exit barrier: no CTA leaves while a peer may still write into it. The
  // computing threads arrive on it once their last push has left (in the
  // last top GEMM layer), the producer once its stream is issued.
  if (warp == kClusterWarps) {
    produce(r, p.wstream, p.stage_tab + static_cast<size_t>(c.q) * p.rank_stages,
            static_cast<uint32_t>(p.rank_stages), 1u, p.wait.withhold_last != 0);
    cluster_wait();
    cluster_arrive();
  } else {
    cluster_consume<BM>(p, c, r, act0, act1, scratch, zs, rowidx_s, bias_s, wlast_s);
  }
  cluster_wait();
  if (*abort_flag && threadIdx.x == 0) {
    // after a wait gave up, pushes of peers may still be in flight toward
    // this CTA: let them land before its shared memory is released
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 50000) __nanosleep(1000);
  }
  __syncthreads();
}

template <int BM>
cudaError_t enable_cluster_kernel() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(fused_cluster_kernel<BM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(device_max_smem_optin()));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_cluster_kernel<BM>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <int BM>
void* cluster_kernel_fn() {
  return reinterpret_cast<void*>(fused_cluster_kernel<BM>);
}

cudaLaunchConfig_t cluster_config(int grid, int csize, int smem, cudaStream_t stream,
                                  cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kClusterThreads + kWarp);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  return cfg;
}

}  // namespace

int fused_cluster_max_active(int bm, int csize, int smem_bytes) {
  void* fn = nullptr;
  cudaError_t e;
  switch (bm) {
    case 4: e = enable_cluster_kernel<4>(); fn = cluster_kernel_fn<4>(); break;
    case 8: e = enable_cluster_kernel<8>(); fn = cluster_kernel_fn<8>(); break;
    case 16: e = enable_cluster_kernel<16>(); fn = cluster_kernel_fn<16>(); break;
    default: return 0;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(csize, csize, smem_bytes, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_fused_cluster(const ClusterParams& p, cudaStream_t stream) {
  if (p.batch == 0) return cudaSuccess;
  const int tiles = (p.batch + p.bm - 1) / p.bm;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = cluster_config(tiles * p.csize, p.csize, p.smem_bytes, stream, attr);
  cudaError_t e;
  switch (p.bm) {
    case 4:
      e = enable_cluster_kernel<4>();
      if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, fused_cluster_kernel<4>, p);
      break;
    case 8:
      e = enable_cluster_kernel<8>();
      if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, fused_cluster_kernel<8>, p);
      break;
    case 16:
      e = enable_cluster_kernel<16>();
      if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, fused_cluster_kernel<16>, p);
      break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- host plan

namespace {

size_t align128(size_t x) { return (x + 127) / 128 * 128; }

int next_pow2(int x) {
  int p = 1;
  while (p < x) p *= 2;
  return p;
}

}  // namespace

bool fused_cluster_plan(int n_dense, int k_tables, int d, int bag, const std::vector<int>& ln_bot,
                        const std::vector<int>& ln_top, const std::vector<std::vector<float>>& w,
                        const std::vector<std::vector<float>>& b, const GatherTables& tabs,
                        int csize, size_t smem_limit, ClusterPlan* plan) {
  *plan = ClusterPlan{};
  if (csize < 2 || csize > 16 || (csize & (csize - 1)) != 0) return false;
  const int n_bot = static_cast<int>(ln_bot.size()) - 1;
  const int n_top = static_cast<int>(ln_top.size()) - 1;
  const int n_gemm = n_bot + n_top - 1;
  if (d % 4 != 0 || ln_top.back() != 1 || n_gemm > kClusterMaxGemm || n_bot < 1 || n_top < 2)
    return false;
  for (int t = 0; t < k_tables; ++t)
    if (reinterpret_cast<uintptr_t>(tabs.ptr[t]) % 16 != 0) return false;
  ClusterParams base{};
  base.n_dense = n_dense;
  base.k_tables = k_tables;
  base.d = d;
  base.bag = bag;
  base.n_bot = n_bot;
  base.n_top = n_top;
  base.n_gemm = n_gemm;
  base.csize = csize;
  const int f = k_tables + 1;
  const int pairs = f * (f - 1) / 2;

  // layer shapes
  int widest = static_cast<int>(round_up(n_dense, 4));
  int bias_floats = 0;
  for (int g = 0; g < n_gemm; ++g) {
    ClusterGemm& L = base.gemm[g];
    L.k = g < n_bot ? ln_bot[g] : ln_top[g - n_bot];
    L.n = g < n_bot ? ln_bot[g + 1] : ln_top[g - n_bot + 1];
    L.s = std::max(4, next_pow2((L.n + csize - 1) / csize));
    if (L.s > 512) return false;
    L.kslices = 512 / L.s;
    const int kstep = 4 * L.kslices;
    L.k_pad = static_cast<int>(round_up(L.k, kstep));
    L.kst_k = std::min(L.k_pad, kRingStageFloats / L.s / kstep * kstep);
    L.n_kst = (L.k_pad + L.kst_k - 1) / L.kst_k;
    L.b_off = bias_floats;
    bias_floats += L.s;
    widest = std::max({widest, L.s * csize, static_cast<int>(round_up(L.k, 4))});
  }
  base.ld_r = static_cast<int>(round_up(d + pairs, 4));
  widest = std::max(widest, base.ld_r);
  base.k_last = static_cast<int>(round_up(ln_top[n_top - 1], 4));
  widest = std::max(widest, base.k_last);
  base.bias_floats = static_cast<int>(round_up(bias_floats, 4));
  base.lda = static_cast<int>(round_up(widest, 32)) + 4;
  base.ldz = static_cast<int>(round_up(d, 4)) + 4;
  base.b_last = b[n_gemm][0];

  // per-rank weight streams in consumption order, and their stage tables
  std::vector<int> rank_stages(csize, 0);
  for (int r = 0; r < csize; ++r) {
    for (int g = 0; g < n_gemm; ++g) {
      const ClusterGemm& L = base.gemm[g];
      const int kstep = 4 * L.kslices;
      const int half = L.s / 2;
      const std::vector<float>& W = w[g];
      for (int kst = 0; kst < L.n_kst; ++kst) {
        const int k_here = std::min(L.kst_k, L.k_pad - kst * L.kst_k);
        const int steps = k_here / kstep;
        const size_t off = plan->wstream.size();
        const size_t floats = static_cast<size_t>(steps) * 2 * kClusterThreads * 4;
        if (off > 0xffffffffu) return false;
        plan->stage_tab.push_back(make_uint2(static_cast<unsigned>(off),
                                             static_cast<unsigned>(floats * sizeof(float))));
        plan->wstream.resize(off + floats, 0.f);
        for (int i = 0; i < steps; ++i)
          for (int j = 0; j < 2; ++j)
            for (int t = 0; t < kClusterThreads; ++t) {
              const int col = 2 * (t % half) + j;
              const int ks = t / half;
              const int k4 = kst * (L.kst_k / 4) + ks + L.kslices * i;
              const int n = r * L.s + col;
              if (n >= L.n) continue;
              for (int e = 0; e < 4; ++e) {
                const int kk = 4 * k4 + e;
                if (kk >= L.k) break;
                plan->wstream[off + ((static_cast<size_t>(2 * i + j) * kClusterThreads + t) * 4) + e] =
                    W[static_cast<size_t>(n) * L.k + kk];
              }
            }
        ++rank_stages[r];
      }
    }
  }
  for (int r = 1; r < csize; ++r)
    if (rank_stages[r] != rank_stages[0]) return false;
  base.rank_stages = rank_stages[0];
  plan->bias.assign(static_cast<size_t>(csize) * base.bias_floats, 0.f);
  for (int r = 0; r < csize; ++r)
    for (int g = 0; g < n_gemm; ++g) {
      const ClusterGemm& L = base.gemm[g];
      for (int col = 0; col < L.s; ++col) {
        const int n = r * L.s + col;
        if (n < L.n) plan->bias[static_cast<size_t>(r) * base.bias_floats + L.b_off + col] = b[g][n];
      }
    }
  plan->wlast.assign(base.k_last, 0.f);
  for (int i = 0; i < ln_top[n_top - 1]; ++i) plan->wlast[i] = w[n_gemm][i];
  base.tabs = tabs;

  // shared-memory carve per tile height: stages | act0 | act1 | scratch | z |
  // rowidx | bias | wlast | barriers; the deepest ring (up to 6 stages, or
  // the whole rank stream) that fits
  bool any = false;
  for (int hi = 0; hi < 3; ++hi) {
    const int bm = kClusterTileRows[hi];
    ClusterParams p = base;
    p.bm = bm;
    p.zrows = (bm + csize - 1) / csize;
    const size_t act = align128(static_cast<size_t>(bm) * p.lda * sizeof(float));
    // k-slice partial sums (512 / s slices of bm s floats, each skewed by 4)
    // or the interaction rows staged for the exchange
    const size_t scratch = align128(std::max<size_t>(static_cast<size_t>(512) * bm + 4 * 128,
                                                     static_cast<size_t>(p.zrows) * p.ld_r) *
                                    sizeof(float));
    const size_t z = align128(static_cast<size_t>(p.zrows) * k_tables * p.ldz * sizeof(float));
    const size_t rowidx = align128(static_cast<size_t>(p.zrows) * k_tables * sizeof(int));
    const size_t bias = align128(static_cast<size_t>(p.bias_floats) * sizeof(float));
    const size_t wl = align128(static_cast<size_t>(p.k_last) * sizeof(float));
    const int max_st = std::min(6, p.rank_stages);
    for (int st = max_st; st >= 2; --st) {
      const size_t bars = align128(static_cast<size_t>(2 * st + 2) * 8 + 16);
      const size_t ring = static_cast<size_t>(st) * kRingStageFloats * sizeof(float);
      const size_t total = ring + 2 * act + scratch + z + rowidx + bias + wl + bars;
      if (total > smem_limit) continue;
      p.stages = st;
      p.off_act0 = static_cast<int>(ring);
      p.off_act1 = static_cast<int>(ring + act);
      p.off_scratch = static_cast<int>(ring + 2 * act);
      p.off_z = static_cast<int>(p.off_scratch + scratch);
      p.off_rowidx = static_cast<int>(p.off_z + z);
      p.off_bias = static_cast<int>(p.off_rowidx + rowidx);
      p.off_wlast = static_cast<int>(p.off_bias + bias);
      p.off_bar = static_cast<int>(p.off_wlast + wl);
      p.smem_bytes = static_cast<int>(p.off_bar + bars);
      plan->params[hi] = p;
      plan->fits[hi] = true;
      any = true;
      break;
    }
  }
  plan->csize = csize;
  return any;
}

}  // namespace dlrm
