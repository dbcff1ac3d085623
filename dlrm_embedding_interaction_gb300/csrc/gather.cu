// Multi-table EmbeddingBag sum, all K tables in one launch.
//
// Computes out[b][t][:] = sum_{l < L} W_t[indices[t][offsets[t][b] + l]][:]
// (Luminal compare modal_ci_ready...vanilla-pytorch, commit message:
// MultiTableEmbeddingBagSumKernel, (batch, num_tables, d) F32 in one launch;
// compare dlrm-fused-kernels...dlrm-pt2-megakernel, LessonsLearned
// "EmbeddingBag translator gap": output[b] = sum over indices[offsets[b]:
// offsets[b+1]], uniform bags).
//
// GB300 design: the gather is HBM-bound (one random D*4-byte row per index),
// so the kernel is built for bytes in flight, not arithmetic:
//  * a group of TPB lanes owns one (sample, table) bag; each lane moves
//    CHUNKS 16-byte vectors of every row (128-bit loads, a D=128 row is one
//    fully coalesced 512-byte warp load);
//  * bag indices are loaded once per group (one lane per index) and
//    broadcast by shuffle; rows are fetched U at a time before any add, so a
//    warp keeps U * 512 bytes outstanding per group;
//  * bags are numbered t * B + b (table-major): the groups in flight at one
//    time work on one or two tables, so with skewed (Zipf) indices the hot
//    rows of the current table share all of L2 instead of every table's hot
//    rows competing for it, and consecutive groups read consecutive indices;
//    each group still writes its whole output row (D * 4 bytes) at once;
//  * no shared-memory staging: each row is read exactly once and consumed in
//    registers, so a TMA or cp.async copy would only add a round trip.
// Bounds: every index is checked against rows[t]; a bad index contributes
// zeros and sets DLRM_ERRBIT_INDEX_OOB. The bag start must equal b * L (the
// uniform stride), which also keeps every index read inside (K, B*L); a bag
// whose offset differs is written as zeros with DLRM_ERRBIT_OFFSETS.
//
// The general form (embedding_bag_multi) is the runtime segment reduction the
// same LessonsLearned entry names as the follow-up: bag b of table t spans
// indices[t][offsets[t][b] : offsets[t][b+1]] (the last bag runs to N), with
// reduce_op sum, mean or max. The same lane groups walk bags of any length;
// an out-of-range index is left out of its bag, mean divides by the rows
// kept, a bag with no rows is zeros, and bounds outside [0, N] or reversed
// give zeros with DLRM_ERRBIT_OFFSETS.
#include "common.cuh"

namespace dlrm {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ void flag_error(int32_t* err, uint32_t bit) {
  if (err) atomicOr(reinterpret_cast<unsigned int*>(err), bit);
}

__device__ __forceinline__ void add4(float4& a, const float4& v) {
  a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
}

__device__ __forceinline__ void fma4(float4& a, float w, const float4& v) {
  a.x = fmaf(w, v.x, a.x); a.y = fmaf(w, v.y, a.y); a.z = fmaf(w, v.z, a.z); a.w = fmaf(w, v.w, a.w);
}

__device__ __forceinline__ void max4(float4& a, const float4& v) {
  a.x = fmaxf(a.x, v.x); a.y = fmaxf(a.y, v.y); a.z = fmaxf(a.z, v.z); a.w = fmaxf(a.w, v.w);
}

// The weighted sum (per_sample_weights) is a fourth, internal reduction.
constexpr int kBagWeightedSum = 3;

// A row left out of its bag, in the vector kernel's 32-bit row numbers.
constexpr uint32_t kSkip = 0xFFFFFFFFu;

// Bag bounds: the uniform stride (GENERAL false: start must equal b * bag)
// or consecutive offsets with the last bag running to N.
template <bool GENERAL, typename IDX>
__device__ __forceinline__ bool bag_bounds(const IDX* offs, int b, int batch, int bag,
                                           int64_t n_idx, int64_t& start, int& len) {
  start = static_cast<int64_t>(offs[b]);
  if (!GENERAL) {
    len = bag;
    return start == static_cast<int64_t>(b) * bag;
  }
  const int64_t end = (b + 1 < batch) ? static_cast<int64_t>(offs[b + 1]) : n_idx;
  len = static_cast<int>(end - start);
  return start >= 0 && end <= n_idx && start <= end && end - start <= INT32_MAX;
}

// Vector path: D % 4 == 0, tables and out 16-byte aligned.
// TPB lanes per bag (power of two <= 32); each lane owns CHUNKS float4 columns
// col4 = lane + c * TPB (< D/4). GENERAL: bag bounds from consecutive offsets
// (else the uniform stride L); MODE: DLRM_BAG_SUM, _MEAN, _MAX or the weighted
// sum; IDX: the index and offset type. An index equal to `padding`, when that
// is >= 0, is left out of its bag without a flag (a negative `padding` is none).
// Six CTAs of 256 threads per SM (at most 40 registers a thread) keep the
// most rows in flight. Each index is checked once, by the lane that loads
// it, and passed on as a 32-bit row number (tables of fewer than 2^32 - 1
// rows; the scalar kernel takes larger ones), which keeps the row loop's
// state within those registers.
template <int TPB, int CHUNKS, int MODE, bool GENERAL, typename IDX>
__global__ void __launch_bounds__(kGatherThreads, CHUNKS == 1 ? 6 : 1)
gather_vec_kernel(const __grid_constant__ GatherTables tabs, int k_tables, int d4,
                  const IDX* __restrict__ indices, const IDX* __restrict__ offsets,
                  const float* __restrict__ psw, int64_t padding, int batch, int bag,
                  int64_t n_idx, float* __restrict__ out, int32_t* err) {
  pdl_wait();     // launched after the previous kernel may still run
  pdl_trigger();

  constexpr bool kWeighted = MODE == kBagWeightedSum;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t bag_id = gtid / TPB;
  const int lane = threadIdx.x & (TPB - 1);
  const unsigned lane_in_warp = threadIdx.x & (kWarp - 1);
  const unsigned gmask = (TPB == 32) ? 0xffffffffu
                                     : (((1u << TPB) - 1u) << (lane_in_warp & ~(TPB - 1u)));
  if (bag_id >= static_cast<int64_t>(batch) * k_tables) return;  // whole group leaves
  const int t = static_cast<int>(bag_id / batch);                 // table-major
  const int b = static_cast<int>(bag_id - static_cast<int64_t>(t) * batch);

  const float init = MODE == DLRM_BAG_MAX ? -INFINITY : 0.f;
  float4 acc[CHUNKS];
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) acc[c] = make_float4(init, init, init, init);

  int64_t start;
  int len;
  const bool good =
      bag_bounds<GENERAL>(offsets + static_cast<int64_t>(t) * batch, b, batch, bag, n_idx, start, len);
  int kept = 0;
  if (!good) {
    if (lane == 0) flag_error(err, DLRM_ERRBIT_OFFSETS);
  } else {
    const int64_t base = static_cast<int64_t>(t) * n_idx + start;
    const IDX* idx = indices + base;
    const float4* table = reinterpret_cast<const float4*>(tabs.ptr[t]);
    const uint64_t rows = static_cast<uint64_t>(tabs.rows[t]);   // < 2^32 - 1 (host check)
    bool oob = false;
    for (int l0 = 0; l0 < len; l0 += TPB) {
      const int cnt = min(TPB, len - l0);
      // The lane that owns an index checks it once: its row as a 32-bit
      // number, or kSkip when the row is left out (past the bag, the padding
      // row, out of range), so the unrolled loop below only shuffles,
      // compares, loads and adds.
      uint32_t mine = kSkip;
      float mine_w = 1.f;
      if (lane < cnt) {
        const int64_t r = static_cast<int64_t>(__ldg(idx + l0 + lane));
        const bool pad = GENERAL && padding >= 0 && r == padding;
        const bool in = static_cast<uint64_t>(r) < rows;
        oob |= !pad && !in;
        if (in && !pad) mine = static_cast<uint32_t>(r);
        if (kWeighted) mine_w = __ldg(psw + base + l0 + lane);
      }
      if (MODE == DLRM_BAG_MEAN || MODE == DLRM_BAG_MAX)
        kept += __popc(__ballot_sync(gmask, mine != kSkip) & gmask);
      for (int u0 = 0; u0 < cnt; u0 += kUnroll) {
        // a row left out loads the identity of the reduction: 0 for sums,
        // -inf for max
        float4 v[kUnroll][CHUNKS];
        float wq[kUnroll];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
          const uint32_t r = __shfl_sync(gmask, mine, (u0 + q) & (TPB - 1), TPB);
          if (kWeighted) wq[q] = __shfl_sync(gmask, mine_w, (u0 + q) & (TPB - 1), TPB);
          // (u0 + q) < cnt: for groups narrower than the unroll the source
          // lane wraps around to a row already taken
          const bool ok = r != kSkip && (u0 + q) < cnt;
#pragma unroll
          for (int c = 0; c < CHUNKS; ++c) {
            const int col4 = lane + c * TPB;
            v[q][c] = (ok && col4 < d4)
                          ? __ldg(table + static_cast<uint64_t>(r) * static_cast<uint32_t>(d4) + col4)
                          : make_float4(init, init, init, init);
          }
        }
#pragma unroll
        for (int q = 0; q < kUnroll; ++q)
#pragma unroll
          for (int c = 0; c < CHUNKS; ++c) {
            if (MODE == DLRM_BAG_MAX) max4(acc[c], v[q][c]);
            else if (kWeighted) fma4(acc[c], wq[q], v[q][c]);
            else add4(acc[c], v[q][c]);
          }
      }
    }
    if (__any_sync(gmask, oob) && lane == 0) flag_error(err, DLRM_ERRBIT_INDEX_OOB);
  }
  // no rows kept: zeros in every mode (a sum of none is already zero); mean
  // divides by the rows kept
  float4* dst = reinterpret_cast<float4*>(out) + (static_cast<int64_t>(b) * k_tables + t) * d4;
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    const int col4 = lane + c * TPB;
    if (col4 >= d4) continue;
    float4 r = acc[c];
    if ((MODE == DLRM_BAG_MEAN || MODE == DLRM_BAG_MAX) && kept == 0) {
      r = make_float4(0.f, 0.f, 0.f, 0.f);
    } else if (MODE == DLRM_BAG_MEAN) {
      r = make_float4(r.x / static_cast<float>(kept), r.y / static_cast<float>(kept),
                      r.z / static_cast<float>(kept), r.w / static_cast<float>(kept));
    }
    dst[col4] = r;
  }
}

// Scalar path for any D and alignment: TPB = 32 lanes per bag, lane owns
// columns lane, lane + 32, ...; indices re-read per column from L1.
template <int MODE, bool GENERAL, typename IDX>
__global__ void __launch_bounds__(kGatherThreads)
gather_scalar_kernel(const __grid_constant__ GatherTables tabs, int k_tables, int d,
                     const IDX* __restrict__ indices, const IDX* __restrict__ offsets,
                     const float* __restrict__ psw, int64_t padding, int batch, int bag,
                     int64_t n_idx, float* __restrict__ out, int32_t* err) {
  pdl_wait();     // launched after the previous kernel may still run
  pdl_trigger();

  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t bag_id = gtid / kWarp;
  const int lane = threadIdx.x & (kWarp - 1);
  if (bag_id >= static_cast<int64_t>(batch) * k_tables) return;
  const int t = static_cast<int>(bag_id / batch);                 // table-major
  const int b = static_cast<int>(bag_id - static_cast<int64_t>(t) * batch);
  float* dst = out + (static_cast<int64_t>(b) * k_tables + t) * d;
  int64_t start;
  int len;
  if (!bag_bounds<GENERAL>(offsets + static_cast<int64_t>(t) * batch, b, batch, bag, n_idx, start,
                           len)) {
    if (lane == 0) flag_error(err, DLRM_ERRBIT_OFFSETS);
    for (int c = lane; c < d; c += kWarp) dst[c] = 0.f;
    return;
  }
  const int64_t base = static_cast<int64_t>(t) * n_idx + start;
  const IDX* idx = indices + base;
  const float* table = tabs.ptr[t];
  const int64_t rows = tabs.rows[t];
  bool oob = false;
  for (int c = lane; c < d; c += kWarp) {
    float acc = MODE == DLRM_BAG_MAX ? -INFINITY : 0.f;
    int kept = 0;
    for (int l = 0; l < len; ++l) {
      const int64_t r = static_cast<int64_t>(__ldg(idx + l));
      if (GENERAL && padding >= 0 && r == padding) continue;
      if (r >= 0 && r < rows) {
        const float v = __ldg(table + r * d + c);
        if (MODE == DLRM_BAG_MAX) acc = fmaxf(acc, v);
        else if (MODE == kBagWeightedSum) acc = fmaf(__ldg(psw + base + l), v, acc);
        else acc += v;
        ++kept;
      } else {
        oob = true;
      }
    }
    if (kept == 0) acc = 0.f;
    else if (MODE == DLRM_BAG_MEAN) acc = acc / static_cast<float>(kept);
    dst[c] = acc;
  }
  if (d == 0) return;
  if (__any_sync(0xffffffffu, oob) && lane == 0) flag_error(err, DLRM_ERRBIT_INDEX_OOB);
}

template <int TPB, int CHUNKS, int MODE, bool GENERAL, typename IDX>
cudaError_t launch_vec(const GatherTables& tabs, int k, int d, const IDX* indices,
                       const IDX* offsets, const float* psw, int64_t padding, int b, int l,
                       int64_t n_idx, float* out, int32_t* err, cudaStream_t stream) {
  const int64_t bags = static_cast<int64_t>(b) * k;
  const int64_t per_block = kGatherThreads / TPB;
  const int64_t grid = (bags + per_block - 1) / per_block;
  return launch_pdl(gather_vec_kernel<TPB, CHUNKS, MODE, GENERAL, IDX>,
                    dim3(static_cast<unsigned>(grid)), dim3(kGatherThreads), 0, stream, tabs, k,
                    d / 4, indices, offsets, psw, padding, b, l, n_idx, out, err);
}

// Lane-group width and columns per lane by D, vector or scalar path.
template <int MODE, bool GENERAL, typename IDX>
cudaError_t launch_any(const GatherTables& tabs, int k, int d, const IDX* indices,
                       const IDX* offsets, const float* psw, int64_t padding, int b, int l,
                       int64_t n_idx, float* out, int32_t* err, cudaStream_t stream) {
  bool vec = (d % 4 == 0) && (reinterpret_cast<uintptr_t>(out) % 16 == 0);
  for (int t = 0; t < k && vec; ++t)
    vec = reinterpret_cast<uintptr_t>(tabs.ptr[t]) % 16 == 0 &&
          static_cast<uint64_t>(tabs.rows[t]) < static_cast<uint64_t>(kSkip);
  const int d4 = d / 4;
#define DLRM_VEC(TPB_, CH_)                                                                     \
  launch_vec<TPB_, CH_, MODE, GENERAL, IDX>(tabs, k, d, indices, offsets, psw, padding, b, l, \
                                            n_idx, out, err, stream)
  if (vec && d4 <= 256) {
    if (d4 <= 1) return DLRM_VEC(1, 1);
    if (d4 <= 2) return DLRM_VEC(2, 1);
    if (d4 <= 4) return DLRM_VEC(4, 1);
    if (d4 <= 8) return DLRM_VEC(8, 1);
    if (d4 <= 16) return DLRM_VEC(16, 1);
    if (d4 <= 32) return DLRM_VEC(32, 1);
    if (d4 <= 64) return DLRM_VEC(32, 2);
    if (d4 <= 128) return DLRM_VEC(32, 4);
    return DLRM_VEC(32, 8);
  }
#undef DLRM_VEC
  const int64_t bags = static_cast<int64_t>(b) * k;
  const int64_t per_block = kGatherThreads / kWarp;
  const int64_t grid = (bags + per_block - 1) / per_block;
  return launch_pdl(gather_scalar_kernel<MODE, GENERAL, IDX>, dim3(static_cast<unsigned>(grid)),
                    dim3(kGatherThreads), 0, stream, tabs, k, d, indices, offsets, psw, padding, b,
                    l, n_idx, out, err);
}

template <typename IDX>
cudaError_t launch_general(const GatherTables& tabs, int k, int d, const IDX* indices,
                           int64_t n_idx, const IDX* offsets, int b, int mode, const float* psw,
                           int64_t padding, float* out, int32_t* err, cudaStream_t stream) {
  if (psw) {
    if (mode != DLRM_BAG_SUM) return cudaErrorInvalidValue;
    return launch_any<kBagWeightedSum, true, IDX>(tabs, k, d, indices, offsets, psw, padding, b,
                                                  0, n_idx, out, err, stream);
  }
  switch (mode) {
    case DLRM_BAG_SUM:
      return launch_any<DLRM_BAG_SUM, true, IDX>(tabs, k, d, indices, offsets, nullptr, padding,
                                                 b, 0, n_idx, out, err, stream);
    case DLRM_BAG_MEAN:
      return launch_any<DLRM_BAG_MEAN, true, IDX>(tabs, k, d, indices, offsets, nullptr, padding,
                                                  b, 0, n_idx, out, err, stream);
    case DLRM_BAG_MAX:
      return launch_any<DLRM_BAG_MAX, true, IDX>(tabs, k, d, indices, offsets, nullptr, padding,
                                                 b, 0, n_idx, out, err, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gather(const GatherTables& tabs, int k, int d, const int64_t* indices,
                          const int64_t* offsets, int b, int l, float* out, int32_t* err,
                          cudaStream_t stream) {
  if (b == 0) return cudaSuccess;
  return launch_any<DLRM_BAG_SUM, false, int64_t>(tabs, k, d, indices, offsets, nullptr, -1, b, l,
                                                  static_cast<int64_t>(b) * l, out, err, stream);
}

cudaError_t launch_gather_general(const GatherTables& tabs, int k, int d, const void* indices,
                                  int64_t n_idx, const void* offsets, int index_bits, int b,
                                  int mode, const float* psw, int64_t padding, float* out,
                                  int32_t* err, cudaStream_t stream) {
  if (b == 0) return cudaSuccess;
  if (index_bits == 32)
    return launch_general<int32_t>(tabs, k, d, static_cast<const int32_t*>(indices), n_idx,
                                   static_cast<const int32_t*>(offsets), b, mode, psw, padding,
                                   out, err, stream);
  return launch_general<int64_t>(tabs, k, d, static_cast<const int64_t*>(indices), n_idx,
                                 static_cast<const int64_t*>(offsets), b, mode, psw, padding, out,
                                 err, stream);
}

}  // namespace dlrm
