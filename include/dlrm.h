/*
 * dlrm.h -- C ABI of libdlrm_gb300.so, a single-GPU (GB300, sm_103a) DLRMv1
 * inference forward: multi-table EmbeddingBag sum, bottom MLP, strict-lower-
 * triangular pairwise-dot interaction with the dense vector concatenated in
 * front, and a top MLP ending in a sigmoid.
 *
 * Sources (Luminal compare pages on the DLRMv1 forward):
 *  [P1] compare modal_ci_ready...vanilla-pytorch, commit message "vanilla-
 *       PyTorch DLRMv1 fast paths": multi_table_embedding_bag_sum (K tables in
 *       one launch, (batch, num_tables, d) F32 out), pairwise-dot kernels
 *       (block-per-batch, closed-form pair index), linear_bias_(relu|sigmoid).
 *  [P4] compare dlrm-fused-kernels...dlrm-pt2-megakernel:
 *       dlrm_megakernel.rs (shape struct, validate(), body steps 1-6),
 *       LessonsLearned "EmbeddingBag translator gap", translate_embedding_bag.
 *
 * Conventions for every call below:
 *  - Pointers are DEVICE pointers unless marked "host".
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Every call only enqueues work on it and never synchronises it,
 *    except dlrm_get_error and dlrm_create/dlrm_destroy as documented.
 *  - All float data is fp32, row-major; integer indices/offsets are int64.
 *  - Every pointer sits at its element's natural alignment (4 bytes for fp32
 *    and int32, 8 for int64 and uint64); any other is DLRM_ERR_INVALID_ARG,
 *    returned before anything is launched.
 *  - Argument problems detectable on the host are returned as a status
 *    before anything is launched. Problems only visible on the device (an
 *    index outside its table, offsets that are not the uniform stride) never
 *    trap: the affected bag contributes zeros and a bit is set in a device
 *    error word, read with dlrm_get_error (handle path) or by the caller
 *    (standalone path, err_flag argument).
 *  - Nothing here allocates except dlrm_create.
 */
#ifndef DLRM_GB300_H
#define DLRM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DLRM_OK = 0,
  DLRM_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or shape */
  DLRM_ERR_UNSUPPORTED = 2,  /* valid request outside what is implemented */
  DLRM_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  DLRM_ERR_OOM = 4,          /* device allocation failed (dlrm_create only) */
  DLRM_ERR_INDEX_OOB = 5,    /* device saw an index outside [0, rows) */
  DLRM_ERR_TIMEOUT = 6       /* a bounded device wait gave up */
} dlrm_status_t;

/* Arithmetic of the MLP GEMMs.
 * FP32 is the parity mode: results within the fp32 tolerance. The fused plan
 * and every small GEMM run on the FP32 FFMA pipe; the layer-wise plan runs
 * each GEMM of 64 or more inputs and 16 or more outputs (but the first
 * bottom layer, which reads the caller's buffer) as split-TF32 on the
 * tcgen05 tensor cores: every fp32 operand is split into a tf32 head and
 * its exact remainder and three products are summed in fp32 (head*head +
 * head*rest + rest*head, about 2^-21 relative per product).
 * FP32_FFMA is FP32 with every GEMM on the FFMA pipe.
 * TF32 and BF16 run the MLPs on the tensor cores with fp32 accumulation in
 * TMEM (opt-in; results within rel 2e-2 of fp32). In the layer-wise plan BF16
 * runs every layer but the first with tf32 operands on the TMA tensor-core
 * GEMM, which has no bf16 form (tf32 keeps more precision than bf16).
 * TF32X3 is split-TF32 on the tensor cores for every GEMM of 64 or more
 * inputs and 16 or more outputs, in the layer-wise plan and in
 * linear_bias_act; it has no fused plan. */
typedef enum {
  DLRM_MATH_FP32 = 0,
  DLRM_MATH_TF32 = 1,
  DLRM_MATH_BF16 = 2,
  DLRM_MATH_TF32X3 = 3,
  DLRM_MATH_FP32_FFMA = 4
} dlrm_math_t;

/* Kernel plan of a forward handle. AUTO takes the fused single-launch forward
 * when the shape fits it (activations of a tile of samples resident in shared
 * memory) and either the math is fp32 with bags of one row (the fp32 fused
 * kernel is persistent, one CTA per SM looping over tiles, so any batch) or
 * the batch is at most two waves of tiles; else the layer-wise launches.
 * FUSED fails dlrm_create with DLRM_ERR_UNSUPPORTED when the shape does not
 * fit; LAYERWISE always launches one kernel per step. */
typedef enum { DLRM_PATH_AUTO = 0, DLRM_PATH_LAYERWISE = 1, DLRM_PATH_FUSED = 2 } dlrm_path_t;

/* Epilogue activation of linear_bias_act. */
typedef enum { DLRM_ACT_NONE = 0, DLRM_ACT_RELU = 1, DLRM_ACT_SIGMOID = 2 } dlrm_act_t;

/* Reduction of embedding_bag_multi over the rows of a bag. */
typedef enum { DLRM_BAG_SUM = 0, DLRM_BAG_MEAN = 1, DLRM_BAG_MAX = 2 } dlrm_bag_mode_t;

/* Device error word bits (1u << code) set by kernels. */
#define DLRM_ERRBIT_INDEX_OOB (1u << DLRM_ERR_INDEX_OOB)
#define DLRM_ERRBIT_OFFSETS   (1u << DLRM_ERR_UNSUPPORTED)
#define DLRM_ERRBIT_TIMEOUT   (1u << DLRM_ERR_TIMEOUT)

#define DLRM_MAX_TABLES 128   /* K limit (kernel-parameter pointer table) */
#define DLRM_MAX_LAYERS 16    /* Linear layers per MLP */

/* Model shape ([P4] dlrm_megakernel.rs shape struct and validate()):
 *   ln_bot  host, n_bot + 1 widths: ln_bot[0] = dense features,
 *           ln_bot[n_bot] = emb_dim (the bottom output is the first feature
 *           vector); ReLU follows every bottom layer, including the last.
 *   rows    host, n_tables row counts (V_t); every table is (V_t, emb_dim).
 *   ln_top  host, n_top + 1 widths: ln_top[0] = emb_dim + F(F-1)/2 with
 *           F = n_tables + 1; ln_top[n_top] = 1. ReLU follows every top layer
 *           but the last, which is followed by a sigmoid.
 *   bag_size  L >= 1 indices per bag, uniform (offsets[t][b] = b * L).
 *   max_batch largest batch a forward call may pass; sizes the workspace.
 *   path      kernel plan (dlrm_path_t); ignored by dlrm_forward_noalloc. */
typedef struct {
  int32_t n_bot;
  const int32_t* ln_bot;
  int32_t n_tables;
  const int64_t* rows;
  int32_t emb_dim;
  int32_t n_top;
  const int32_t* ln_top;
  int32_t bag_size;
  int32_t max_batch;
  dlrm_math_t math;
  int32_t path;
} dlrm_config_t;

typedef struct dlrm_handle_s* dlrm_handle_t;

/* Library version (major * 10000 + minor * 100 + patch). */
int32_t dlrm_version(void);

/* Static string for a status code. */
const char* dlrm_status_string(int32_t status);

/* Build a forward plan on the current CUDA device.
 *   tables  host array of n_tables DEVICE pointers, each (rows[t], emb_dim)
 *           fp32 row-major, 16-byte aligned. BORROWED: the handle keeps the
 *           pointers and never copies the tables (a 13 GB table set stays
 *           where the caller put it); the caller keeps them alive and
 *           unchanged in shape until dlrm_destroy.
 *   bot_w/bot_b/top_w/top_b  host arrays of n_bot / n_top pointers (host or
 *           device memory, read with cudaMemcpyDefault) to the Linear weights
 *           in PyTorch (out, in) row-major layout and their (out) biases. The
 *           handle COPIES them (padded, and converted for TF32/BF16) into its
 *           own device memory; the caller may free them afterwards.
 * Allocates the handle's workspace for max_batch samples (bag sums, hidden
 * activations, the interaction output, staging for dlrm_forward_host) and
 * synchronises the device once. Returns INVALID_ARG for a null pointer, any
 * shape violation of [P4] validate(), an unknown math mode or path; OOM if an
 * allocation fails; UNSUPPORTED for n_tables > DLRM_MAX_TABLES, more than
 * DLRM_MAX_LAYERS layers a side, max_batch * bag_size > 2^31, an interaction
 * that needs more shared memory per sample than the device has, or path
 * FUSED when the model does not fit the fused kernel of its math (always for
 * TF32X3). dlrm_plan_query gives the same answer on the host. */
dlrm_status_t dlrm_create(const dlrm_config_t* cfg, const float* const* tables,
                          const float* const* bot_w, const float* const* bot_b,
                          const float* const* top_w, const float* const* top_b,
                          dlrm_handle_t* out);

/* The kernel plan dlrm_create would take for cfg on a device with sm_count
 * SMs and smem_per_block bytes of opt-in shared memory per block (GB300: 152
 * and 232448), assuming 16-byte aligned tables. Host-only: touches no device,
 * needs no weights (the plan depends on shapes alone). Returns the status
 * dlrm_create would return for the config's shape (INVALID_ARG, UNSUPPORTED
 * as documented there, UNSUPPORTED for path FUSED when the model does not fit
 * the fused kernel), and INVALID_ARG for a null cfg or info, sm_count < 1 or
 * smem_per_block < 1. On DLRM_OK, *info holds the plan. */
typedef struct {
  int32_t path;            /* DLRM_PATH_FUSED or DLRM_PATH_LAYERWISE */
  int32_t fused_fits;      /* 1: the model fits the fused kernel of its math */
  int32_t tensor_core;     /* 1: that fused kernel runs its GEMMs on tcgen05 */
  int32_t tile_samples;    /* samples per fused tile (0 unless fused_fits) */
  int64_t tiles;           /* fused tiles of max_batch samples */
  int32_t grid;            /* CTAs of one fused launch at max_batch (fp32: at
                              most one per SM, each looping over tiles) */
  int32_t smem_bytes;      /* dynamic shared memory per fused CTA */
  int32_t ring_stages;     /* depth of the fused weight ring */
  int32_t stream_copies;   /* bulk copies in one pass over the weight stream */
  int64_t stream_bytes;    /* packed MLP weight stream of the fused kernel */
  int32_t tensor_core_layers;  /* layer-wise plan: bit g set when Linear layer g
                                  (bottom layers first, then top) runs on the
                                  tcgen05 tensor cores; 0 for a fused plan */
  int32_t split_tf32;      /* 1: those layers compute split-TF32 (three tf32
                              products per fp32 product) */
  int64_t layerwise_from;  /* AUTO plan of fp32 math taking the fused kernel:
                              forwards of at least this many samples run the
                              layer-wise plan instead (its large GEMMs as
                              split-TF32 on the tensor cores); 0: never */
} dlrm_plan_info_t;

dlrm_status_t dlrm_plan_query(const dlrm_config_t* cfg, int32_t sm_count,
                              int64_t smem_per_block, dlrm_plan_info_t* info);

/* One forward pass for `batch` samples ([P4] dlrm_megakernel.rs steps 1-6).
 *   dense    (batch, ln_bot[0]) fp32
 *   indices  (n_tables, batch * bag_size) int64, table-major
 *   offsets  (n_tables, batch) int64, bag starts; must be b * bag_size
 *            (include_last_offset = false, [P4] translate_embedding_bag)
 *   out      (batch) fp32 click probabilities
 * 1 <= batch <= max_batch. Enqueued on `stream`; no host synchronisation;
 * capturable in a CUDA graph. Device-side problems (index out of range,
 * non-uniform offsets) set the handle's error word (see dlrm_get_error).
 * Calls on one handle must be serialised on one stream (shared workspace). */
dlrm_status_t dlrm_forward(dlrm_handle_t h, const float* dense, const int64_t* indices,
                           const int64_t* offsets, float* out, int32_t batch, void* stream);

/* dlrm_forward from HOST buffers, all on `stream`. A pinned (page-locked,
 * mapped) buffer is read or written in place by the kernels through its
 * device address (on GB300 host memory is coherent over NVLink-C2C): no copy.
 * Any other buffer is copied host-to-device into the handle's staging buffers
 * before the forward (dense, indices, offsets) or device-to-host after it
 * (out). Buffers must stay valid and unchanged until the stream has passed
 * this call (e.g. after cudaStreamSynchronize or dlrm_get_error). */
dlrm_status_t dlrm_forward_host(dlrm_handle_t h, const float* dense_host,
                                const int64_t* indices_host, const int64_t* offsets_host,
                                float* out_host, int32_t batch, void* stream);

/* Synchronises `stream`, returns the first error recorded on the device
 * since the last call (INDEX_OOB before UNSUPPORTED before TIMEOUT; OK if
 * none) and clears it. */
dlrm_status_t dlrm_get_error(dlrm_handle_t h, void* stream);

/* Test hook of the failure detection; no counterpart on the pages. Every
 * wait of the library's kernels on another party (a weight stage or tile
 * landing in shared memory, a ring slot being released, tensor-core work
 * completing) is bounded: on expiry the kernel sets DLRM_ERRBIT_TIMEOUT in the
 * handle's error word, stops waiting, waits (bounded) for the copies and
 * tensor-core work it issued, frees its tensor memory and returns, so the
 * context stays usable and dlrm_get_error reports DLRM_ERR_TIMEOUT. This call
 * sets, for every later dlrm_forward on h, the limit of those waits in
 * nanoseconds (0: the default, 2 s) and, with withhold_last != 0, makes each
 * kernel skip the last copy or tensor-core commit of its stream (the fused
 * kernels' last weight stage or tile, the layer-wise tensor-core GEMMs' last
 * K block commit), so that the wait on it runs out after the limit. Results
 * of such a forward are undefined. dlrm_test_stall(h, 0, 0) restores normal
 * operation. INVALID_ARG for a null handle or a negative limit. */
dlrm_status_t dlrm_test_stall(dlrm_handle_t h, int64_t wait_limit_ns, int32_t withhold_last);

/* The kernels one forward of `batch` samples on h runs: */
#define DLRM_KERNELS_LAYERWISE 1      /* one launch per step */
#define DLRM_KERNELS_FUSED 2          /* the fused kernel, one CTA per tile */
#define DLRM_KERNELS_FUSED_CLUSTER 3  /* the fused kernel on thread-block clusters */
#define DLRM_KERNELS_FUSED_TC 4       /* the fused tensor-core kernel (TF32 / BF16) */
/* -1 for a null handle or a batch outside [1, max_batch]. An AUTO handle of
 * fp32 math on the fused plan runs the layer-wise plan from
 * dlrm_plan_info_t.layerwise_from samples (large batches: split-TF32 GEMMs
 * on the tensor cores beat the FFMA kernel), the cluster kernel up to the
 * cluster batch limit below, the one-CTA-per-tile kernel between. While
 * per-stage timing or a phase trace is on, a handle keeps its own plan. */
int32_t dlrm_forward_kernels(dlrm_handle_t h, int32_t batch);

/* Small batches of the fp32 fused plan of a model with 1 MiB or more of
 * packed MLP weights run on a second kernel: each layer's output columns
 * split over the CTAs of a thread-block cluster (8 CTAs up to 32 samples, 4
 * above), every CTA streaming only its share of the weights and the layer's
 * outputs exchanged through distributed shared memory. A forward of at most
 * `limit` samples takes that kernel, a larger one the persistent
 * single-CTA-per-tile kernel (and so does every forward while a phase-trace
 * buffer is set). dlrm_set_cluster_batch_limit sets the limit: 0 turns the
 * cluster kernel off, -1 restores the default (the samples one wave of
 * clusters holds at the tallest tile that fits, at most 256). UNSUPPORTED when the handle has no cluster plan
 * (layer-wise or tensor-core plans, or a model the kernel does not take) and
 * limit > 0; INVALID_ARG for a null handle or limit < -1.
 * dlrm_get_cluster_batch_limit reads the current limit (0 when there is no
 * cluster plan). */
dlrm_status_t dlrm_set_cluster_batch_limit(dlrm_handle_t h, int32_t limit);
dlrm_status_t dlrm_get_cluster_batch_limit(dlrm_handle_t h, int32_t* limit);

/* Bytes of device memory the handle owns (workspace + packed weights). */
int64_t dlrm_workspace_bytes(dlrm_handle_t h);

/* The plan the handle resolved at create time: DLRM_PATH_LAYERWISE or
 * DLRM_PATH_FUSED (-1 for a null handle). */
int32_t dlrm_path(dlrm_handle_t h);

/* Number of kernel launches one dlrm_forward enqueues (its stages). */
int32_t dlrm_num_stages(dlrm_handle_t h);

/* Static name of stage i ("gather", "bottom0", ..., "interaction", "top0", ...),
 * or NULL when i is out of range. */
const char* dlrm_stage_name(dlrm_handle_t h, int32_t i);

/* Per-stage timing (off by default). With enable != 0 the handle creates one
 * CUDA event per stage boundary and every later dlrm_forward records them on
 * its stream, then WAITS for its last event and adds each stage's
 * event-to-event time to a running total; this mode synchronises the host
 * and must not be used inside graph capture. enable = 0 destroys the events
 * and clears the totals. With DLRM_PROFILE=1 in the environment, dlrm_create
 * turns it on and dlrm_destroy prints the mean time per call of every stage
 * to stderr. */
dlrm_status_t dlrm_set_profiling(dlrm_handle_t h, int32_t enable);

/* Phase trace of the fused plan (profiling; off by default). With a non-null
 * device buffer of `capacity` uint64 words, every later dlrm_forward on a
 * fused handle writes, per tile t of *tile_rows samples (the plan's tile
 * height: 4, 8, 12, 14 or 16 rows in fp32, 16 in TF32/BF16), the %globaltimer
 * nanoseconds at which the tile finished each phase to
 * buf[t * DLRM_TRACE_SLOTS + s]: s = 0 the tile's start (the kernel's start
 * for a CTA's first tile), 1 prologue (biases and inputs loaded), 2 .. 1+n_bot
 * the bottom layers, 2+n_bot the interaction, 3+n_bot .. 1+n_bot+n_top the top
 * layers but the last, 2+n_bot+n_top the end (sigmoid layer written). While
 * those slots end below 20, the slots from 20 on profile each GEMM layer g
 * (bottom layers, then top layers but the last): fp32 (for g < 10), slot
 * 20 + g = when its k-loop ended and slot 30 + g = the SM clock cycles
 * computing warp 0 spent waiting for the layer's weight stages; TF32/BF16,
 * slots 20 + 2g and 21 + 2g = nanoseconds the MMA thread waited for the
 * layer's input activations and for its weight tiles.
 * Needs capacity >= tiles(max_batch) * DLRM_TRACE_SLOTS (INVALID_ARG
 * otherwise; UNSUPPORTED on a layer-wise handle); NULL switches it off.
 * Returns the tile height in *tile_rows. */
#define DLRM_TRACE_SLOTS 40
dlrm_status_t dlrm_set_phase_trace(dlrm_handle_t h, uint64_t* buf, int64_t capacity,
                                   int32_t* tile_rows);

/* Copies up to `capacity` per-stage totals (milliseconds, summed over the
 * profiled forward calls) into total_ms and the number of profiled calls into
 * *calls; returns the number of stages, or -1 for a null handle. */
int32_t dlrm_stage_times(dlrm_handle_t h, double* total_ms, int32_t capacity, int64_t* calls);

/* Synchronises the device and frees everything the handle owns (not the
 * borrowed tables). Null is a no-op. */
void dlrm_destroy(dlrm_handle_t h);

/* Size of the fixed scratch array behind dlrm_forward_noalloc (16 MiB). */
#define DLRM_NOALLOC_SCRATCH_BYTES (16u << 20)

/* The same forward as dlrm_forward, for callers that cannot allocate device
 * memory when they run it. No counterpart exists on the pages; this is a
 * service of this library. Typical callers: a plug-in inside another
 * framework whose caching allocator owns the GPU's memory (a raw cudaMalloc
 * there bypasses its accounting and limits), a serving loop that must never
 * take cudaMalloc's implicit device-wide synchronisation, or code that runs
 * under a device-memory budget fixed at start-up.
 *
 * There is no handle: the caller passes the shape (cfg; cfg->math must be
 * DLRM_MATH_FP32 or DLRM_MATH_FP32_FFMA, both the FFMA fused kernel here;
 * cfg->max_batch is ignored), the DEVICE pointers of the
 * tables and of the Linear weights (PyTorch (out, in) layout, contiguous) and
 * biases, and the inputs and output exactly as for dlrm_forward. err_flag is
 * an optional device int32 word into which the DLRM_ERRBIT_* bits of this
 * call are OR-ed (it is never cleared here).
 *
 * Scratch: the bag sums, hidden activations and the interaction output live
 * in one file-scope __device__ array of DLRM_NOALLOC_SCRATCH_BYTES, which
 * every GPU that uses this entry point holds until the process exits. A
 * batch whose scratch would exceed it is rejected with DLRM_ERR_UNSUPPORTED
 * before anything is launched (the 2048-sample, 3-table, 512-wide model needs
 * about 10 MiB). Nothing in the scratch has to start at zero: every value a
 * call reads was written earlier in the same call. All calls share the one
 * array, so calls whose work overlaps on the GPU (different streams, or
 * different host threads, without ordering between them) race and corrupt
 * each other's results: serialise them, e.g. on one stream.
 * Set-up: every call looks up the array's device address on the current
 * device (cudaGetSymbolAddress), so calls stay valid after a device reset.
 * The first call on a device may load the library's device code: make that
 * first call before any stream capture. The call allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine. */
dlrm_status_t dlrm_forward_noalloc(const dlrm_config_t* cfg, const float* const* tables,
                                   const float* const* bot_w, const float* const* bot_b,
                                   const float* const* top_w, const float* const* top_b,
                                   const float* dense, const int64_t* indices,
                                   const int64_t* offsets, float* out, int32_t batch,
                                   int32_t* err_flag, void* stream);

/* Multi-table EmbeddingBag sum in one launch ([P1] MultiTableEmbeddingBagSum;
 * [P4] LessonsLearned "EmbeddingBag translator gap"):
 *   out[b][t][:] = sum_{l < L} tables[t][indices[t][offsets[t][b] + l]][:]
 *   tables   host array of K device pointers, table t is (rows[t], D) fp32
 *            row-major; rows is a host array of K row counts
 *   indices  (K, B * L) int64 table-major;  offsets (K, B) int64
 *   out      (B, K, D) fp32
 *   err_flag device int32 error word or NULL; bits DLRM_ERRBIT_INDEX_OOB (an
 *            index outside [0, rows[t]): that row contributes zeros) and
 *            DLRM_ERRBIT_OFFSETS (offsets[t][b] != b * L: the bag is zeros)
 *            are OR-ed in; it is never cleared here.
 * Sum order within a bag is the index order, in fp32; with L = 1 the result
 * is the row itself (an index_select), bit for bit.
 * 1 <= K <= DLRM_MAX_TABLES, D >= 1, L >= 1, B >= 0 (B = 0 is a no-op). */
dlrm_status_t embedding_bag_sum_multi(const float* const* tables, const int64_t* rows,
                                      int32_t K, int32_t D, const int64_t* indices,
                                      const int64_t* offsets, int32_t B, int32_t L, float* out,
                                      int32_t* err_flag, void* stream);

/* Multi-table EmbeddingBag over general offsets, in one launch: the runtime
 * segment reduction of [P4] LessonsLearned "EmbeddingBag translator gap",
 *   out[b][t][:] = reduce_op(tables[t][indices[t][n]][:] for n in bag(t, b)),
 *   bag(t, b) = [offsets[t][b], offsets[t][b+1])  (the last bag ends at N),
 * reduce_op = sum, mean or max (mode).
 *   tables   host array of K device pointers, table t is (rows[t], D) fp32
 *            row-major; rows is a host array of K row counts
 *   indices  (K, N) int64 table-major, N = n_idx >= 0 indices per table
 *   offsets  (K, B) int64 bag starts (PyTorch include_last_offset = false)
 *   out      (B, K, D) fp32
 *   err_flag device int32 error word or NULL; bits DLRM_ERRBIT_INDEX_OOB (an
 *            index outside [0, rows[t]) is left out of its bag) and
 *            DLRM_ERRBIT_OFFSETS (a bag with begin < 0, end > N or
 *            begin > end is written as zeros) are OR-ed in, never cleared.
 * A bag with no rows kept is zeros in every mode; mean divides by the rows
 * kept; sums run in index order in fp32; max is exact (fmaxf).
 * Returns DLRM_ERR_INVALID_ARG for null pointers, K < 1, D < 1, B < 0,
 * n_idx < 0 or an unknown mode; DLRM_ERR_UNSUPPORTED for K > DLRM_MAX_TABLES;
 * DLRM_ERR_CUDA if the launch fails. B = 0 is a no-op. Asynchronous on
 * stream; pointers are borrowed for the call only. */
dlrm_status_t embedding_bag_multi(const float* const* tables, const int64_t* rows, int32_t K,
                                  int32_t D, const int64_t* indices, int64_t n_idx,
                                  const int64_t* offsets, int32_t B, int32_t mode, float* out,
                                  int32_t* err_flag, void* stream);

/* Options of embedding_bag_multi_ex, PyTorch's EmbeddingBag arguments beyond
 * the mode.
 *   mode                DLRM_BAG_SUM, DLRM_BAG_MEAN or DLRM_BAG_MAX
 *   index_bits          64: indices and offsets are int64_t; 32: int32_t
 *   per_sample_weights  device (K, N) fp32 or NULL: with DLRM_BAG_SUM,
 *                       out[b][t] = sum_n w[t][n] * tables[t][indices[t][n]]
 *                       (fp32 fused multiply-adds in index order); any other
 *                       mode with weights is DLRM_ERR_INVALID_ARG
 *   padding_idx         a row index (>= 0) left out of every bag without a
 *                       flag (not counted by mean), or -1 for none */
typedef struct {
  int32_t mode;
  int32_t index_bits;
  const float* per_sample_weights;
  int64_t padding_idx;
} dlrm_bag_options_t;

/* embedding_bag_multi with options: the same operation and error behaviour,
 * indices and offsets of either width, per-sample weights and a padding row.
 * indices and offsets point to (K, N) and (K, B) arrays of the type
 * index_bits names. Returns DLRM_ERR_INVALID_ARG for a null options pointer,
 * index_bits other than 32 or 64, N > INT32_MAX with 32-bit indices, or the
 * cases of embedding_bag_multi. */
dlrm_status_t embedding_bag_multi_ex(const float* const* tables, const int64_t* rows, int32_t K,
                                     int32_t D, const void* indices, int64_t n_idx,
                                     const void* offsets, int32_t B,
                                     const dlrm_bag_options_t* options, float* out,
                                     int32_t* err_flag, void* stream);

/* Strict-lower-triangular pairwise-dot interaction ([P1]
 * PairwiseDotLowerTriStackedKernel; [P4] dlrm_megakernel.rs steps 4-5):
 * per sample, Z = [dense; emb[0..K-1]] is (F, D) with F = K + 1, and
 *   z[p] = <Z_i, Z_j>,  p = i(i-1)/2 + j,  0 <= j < i < F   (i-major order),
 * so i = floor((1 + sqrt(1 + 8p)) / 2), j = p - i(i-1)/2.
 *   dense  (B, D) fp32 with row stride ld_dense >= D
 *   emb    (B, K, D) fp32 contiguous
 *   out    (B, ld_out) fp32; copy_dense = 1 writes out[b] = [dense[b], z]
 *          (the concat R = [x, z] fused; ld_out >= D + P), copy_dense = 0
 *          writes out[b] = z (ld_out >= P). Columns past the written width
 *          are left untouched.
 * K >= 0 (K = 0 gives no pairs), D >= 1, B >= 0. Needs F * (D + 4) * 4 bytes
 * of shared memory per sample (UNSUPPORTED if that exceeds the device). */
dlrm_status_t pairwise_dot_lower_tri(const float* dense, int32_t ld_dense, const float* emb,
                                     int32_t B, int32_t K, int32_t D, float* out,
                                     int32_t ld_out, int32_t copy_dense, void* stream);

/* Test-mode export of the device pair map used by pairwise_dot_lower_tri:
 * i_out[p], j_out[p] (device int32, P = F(F-1)/2 entries each) for F >= 2. */
dlrm_status_t pairwise_pair_map(int32_t F, int32_t* i_out, int32_t* j_out, void* stream);

/* Fused Linear + bias + activation ([P1] linear_bias_(relu|sigmoid) over the
 * fused Matmul2D kernel; [P4] body steps 2 and 6):
 *   y[m][n] = act(sum_k x[m][k] * W[n][k] + bias[n])
 *   x     (M, K) fp32, row stride ld_x >= K
 *   W     (N, K) fp32 row-major (PyTorch nn.Linear layout), contiguous
 *   bias  (N) fp32 or NULL (no bias)
 *   y     (M, N) fp32, row stride ld_y >= N; must not overlap x or W
 * act: DLRM_ACT_NONE / RELU / SIGMOID (1 / (1 + exp(-a))).
 * math: DLRM_MATH_FP32 or DLRM_MATH_FP32_FFMA (both on the FFMA pipe here),
 * or an opt-in tensor-core mode.
 * M >= 0 (0 is a no-op), N >= 1, K >= 1. */
dlrm_status_t linear_bias_act(const float* x, int32_t ld_x, const float* W, const float* bias,
                              float* y, int32_t ld_y, int32_t M, int32_t N, int32_t K,
                              dlrm_act_t act, dlrm_math_t math, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DLRM_GB300_H */
