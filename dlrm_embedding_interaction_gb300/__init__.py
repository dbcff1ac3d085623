"""Python binding of libdlrm_gb300.so, the GB300 DLRMv1 inference forward.

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels (include/dlrm.h documents each entry point). PyTorch supplies
device memory and streams. There is no CPU or PyTorch fallback: if the
library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdlrm_gb300.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_INDEX_OOB, ERR_TIMEOUT = range(7)
MATH_FP32, MATH_TF32, MATH_BF16, MATH_TF32X3, MATH_FP32_FFMA = 0, 1, 2, 3, 4
PATH_AUTO, PATH_LAYERWISE, PATH_FUSED = 0, 1, 2
ACT_NONE, ACT_RELU, ACT_SIGMOID = 0, 1, 2
ERRBIT_INDEX_OOB = 1 << ERR_INDEX_OOB
ERRBIT_OFFSETS = 1 << ERR_UNSUPPORTED
MAX_TABLES = 128
MAX_LAYERS = 16

# Every symbol include/dlrm.h declares.
EXPORTS = ("dlrm_version", "dlrm_status_string", "dlrm_create", "dlrm_forward",
           "dlrm_forward_host", "dlrm_get_error", "dlrm_workspace_bytes", "dlrm_destroy",
           "dlrm_path", "dlrm_num_stages", "dlrm_stage_name", "dlrm_set_profiling", "dlrm_stage_times",
           "dlrm_forward_noalloc", "dlrm_set_phase_trace", "dlrm_plan_query",
           "embedding_bag_sum_multi", "embedding_bag_multi", "embedding_bag_multi_ex",
           "pairwise_dot_lower_tri",
           "pairwise_pair_map", "linear_bias_act", "dlrm_test_stall",
           "dlrm_set_cluster_batch_limit", "dlrm_get_cluster_batch_limit",
           "dlrm_forward_kernels")
NOALLOC_SCRATCH_BYTES = 16 << 20
TRACE_SLOTS = 40

_lib = None


class DlrmError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _status_string(status)
        super().__init__(f"{where}: status {status} ({msg})")
        self.status = status


class _BagOptions(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("index_bits", ctypes.c_int32),
                ("per_sample_weights", ctypes.c_void_p), ("padding_idx", ctypes.c_int64)]


class _Config(ctypes.Structure):
    _fields_ = [("n_bot", ctypes.c_int32), ("ln_bot", ctypes.POINTER(ctypes.c_int32)),
                ("n_tables", ctypes.c_int32), ("rows", ctypes.POINTER(ctypes.c_int64)),
                ("emb_dim", ctypes.c_int32), ("n_top", ctypes.c_int32),
                ("ln_top", ctypes.POINTER(ctypes.c_int32)), ("bag_size", ctypes.c_int32),
                ("max_batch", ctypes.c_int32), ("math", ctypes.c_int), ("path", ctypes.c_int32)]


class _PlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("fused_fits", ctypes.c_int32),
                ("tensor_core", ctypes.c_int32), ("tile_samples", ctypes.c_int32),
                ("tiles", ctypes.c_int64), ("grid", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("ring_stages", ctypes.c_int32),
                ("stream_copies", ctypes.c_int32), ("stream_bytes", ctypes.c_int64),
                ("tensor_core_layers", ctypes.c_int32), ("split_tf32", ctypes.c_int32),
                ("layerwise_from", ctypes.c_int64)]


def _bind(lib):
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    st = ctypes.c_int
    sig = {
        "dlrm_version": ([], i32),
        "dlrm_status_string": ([i32], ctypes.c_char_p),
        "dlrm_create": ([ctypes.POINTER(_Config), vp, vp, vp, vp, vp, ctypes.POINTER(vp)], st),
        "dlrm_forward": ([vp, vp, vp, vp, vp, i32, vp], st),
        "dlrm_forward_host": ([vp, vp, vp, vp, vp, i32, vp], st),
        "dlrm_get_error": ([vp, vp], st),
        "dlrm_test_stall": ([vp, i64, i32], st),
        "dlrm_set_cluster_batch_limit": ([vp, i32], st),
        "dlrm_forward_kernels": ([vp, i32], i32),
        "dlrm_get_cluster_batch_limit": ([vp, vp], st),
        "dlrm_workspace_bytes": ([vp], i64),
        "dlrm_destroy": ([vp], None),
        "dlrm_path": ([vp], i32),
        "dlrm_num_stages": ([vp], i32),
        "dlrm_stage_name": ([vp, i32], ctypes.c_char_p),
        "dlrm_set_profiling": ([vp, i32], st),
        "dlrm_stage_times": ([vp, ctypes.c_void_p, i32, ctypes.POINTER(i64)], i32),
        "dlrm_forward_noalloc": ([ctypes.POINTER(_Config), vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                  i32, vp, vp], st),
        "dlrm_set_phase_trace": ([vp, vp, i64, ctypes.POINTER(i32)], st),
        "dlrm_plan_query": ([ctypes.POINTER(_Config), i32, i64, ctypes.POINTER(_PlanInfo)], st),
        "embedding_bag_sum_multi": ([vp, vp, i32, i32, vp, vp, i32, i32, vp, vp, vp], st),
        "embedding_bag_multi": ([vp, vp, i32, i32, vp, i64, vp, i32, i32, vp, vp, vp], st),
        "embedding_bag_multi_ex": ([vp, vp, i32, i32, vp, i64, vp, i32,
                                    ctypes.POINTER(_BagOptions), vp, vp, vp], st),
        "pairwise_dot_lower_tri": ([vp, i32, vp, i32, i32, i32, vp, i32, i32, vp], st),
        "pairwise_pair_map": ([i32, vp, vp, vp], st),
        "linear_bias_act": ([vp, i32, vp, vp, vp, i32, i32, i32, i32, st, st, vp], st),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def lib():
    """The loaded library. Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m "
                "dlrm_embedding_interaction_gb300.build` (nvcc, sm_103a). "
                "There is no fallback path.")
        _lib = _bind(ctypes.CDLL(LIB_PATH))
    return _lib


def _status_string(status: int) -> str:
    try:
        return lib().dlrm_status_string(status).decode()
    except Exception:  # pragma: no cover - library not loadable
        return "?"


def _check(status: int, where: str) -> None:
    if status != OK:
        raise DlrmError(status, where)


def _stream(stream) -> ctypes.c_void_p:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t, dtype, name, cuda=True):
    import torch
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")


# Model shape of every handle dlrm_create returned in this process (the C
# handle is opaque): the forward bindings check their tensors against it.
_HANDLE_SHAPES: dict = {}


def _check_forward_io(n_dense: int, k: int, bag: int, max_batch: Optional[int], dense,
                      indices, offsets, out, where: str, on_cuda: bool) -> int:
    """Checks a forward's inputs and output before the library sees them and
    returns the batch. dense (B, n_dense) float32, indices (K, B * bag) and
    offsets (K, B) int64, out float32 with at least B elements, all
    contiguous; CUDA tensors when ``on_cuda``, else host (CPU) tensors. The
    library reads and writes these buffers by the sizes the model implies, so
    a short or mistyped tensor would be accessed past its end on the device:
    refused here with TypeError / ValueError instead. Checks run in the order
    dtype, shape, layout, device."""
    import torch
    for t, dt, name in ((dense, torch.float32, "dense"), (indices, torch.int64, "indices"),
                        (offsets, torch.int64, "offsets"), (out, torch.float32, "out")):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{where}: {name} must be a torch.Tensor")
        if t.dtype != dt:
            raise TypeError(f"{where}: {name}: expected {dt}, got {t.dtype}")
    if dense.dim() != 2 or dense.shape[1] != n_dense:
        raise ValueError(f"{where}: dense: expected (batch, {n_dense}), got {tuple(dense.shape)}")
    b = int(dense.shape[0])
    if b < 1 or (max_batch is not None and b > max_batch):
        raise ValueError(f"{where}: batch {b} outside [1, {max_batch}]")
    if indices.numel() != k * b * bag or (indices.dim() == 2 and indices.shape[0] != k):
        raise ValueError(f"{where}: indices: expected ({k}, {b * bag}) = {k * b * bag} "
                         f"elements, got {tuple(indices.shape)}")
    if offsets.numel() != k * b or (offsets.dim() == 2 and offsets.shape[0] != k):
        raise ValueError(f"{where}: offsets: expected ({k}, {b}), got {tuple(offsets.shape)}")
    if out.numel() < b:
        raise ValueError(f"{where}: out: needs at least {b} elements, has {out.numel()}")
    for t, name in ((dense, "dense"), (indices, "indices"), (offsets, "offsets"), (out, "out")):
        if not t.is_contiguous():
            raise ValueError(f"{where}: {name} must be contiguous")
    for t, name in ((dense, "dense"), (indices, "indices"), (offsets, "offsets"), (out, "out")):
        if on_cuda and not t.is_cuda:
            raise ValueError(f"{where}: {name} must be a CUDA tensor")
        if not on_cuda and t.device.type != "cpu":
            raise ValueError(f"{where}: {name} must be a host (CPU) tensor")
    if on_cuda and len({t.device for t in (dense, indices, offsets, out)}) != 1:
        raise ValueError(f"{where}: dense, indices, offsets and out must be on one device")
    return b


def _check_model_params(ln_bot, ln_top, tables, bot_w, bot_b, top_w, top_b, where: str,
                        on_cuda: bool) -> int:
    """Checks the tables and Linear parameters against the layer widths and
    returns the embedding width D: every table (rows, D) with one D, W[l]
    (ln[l+1], ln[l]) and b[l] (ln[l+1],) per side, all float32 and
    contiguous, and CUDA tensors when ``on_cuda`` (checked last, after every
    dtype and shape). Raises TypeError / ValueError."""
    import torch
    if len(tables) < 1:
        raise ValueError(f"{where}: need at least one table")
    if len(bot_w) != len(ln_bot) - 1 or len(bot_b) != len(ln_bot) - 1:
        raise ValueError(f"{where}: expected {len(ln_bot) - 1} bottom weights and biases")
    if len(top_w) != len(ln_top) - 1 or len(top_b) != len(ln_top) - 1:
        raise ValueError(f"{where}: expected {len(ln_top) - 1} top weights and biases")
    d = int(tables[0].shape[1]) if tables[0].dim() == 2 else -1
    named = [(t, f"tables[{i}]", None) for i, t in enumerate(tables)]
    for side, ln, ws, bs in (("bot", ln_bot, bot_w, bot_b), ("top", ln_top, top_w, top_b)):
        for l in range(len(ln) - 1):
            named.append((ws[l], f"{side}_w[{l}]", (ln[l + 1], ln[l])))
            named.append((bs[l], f"{side}_b[{l}]", (ln[l + 1],)))
    for t, name, shape in named:
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{where}: {name} must be a torch.Tensor")
        if t.dtype != torch.float32:
            raise TypeError(f"{where}: {name}: expected torch.float32, got {t.dtype}")
        if shape is None:
            if t.dim() != 2 or t.shape[1] != d or t.shape[0] < 1:
                raise ValueError(f"{where}: {name}: expected (rows, {d}), got {tuple(t.shape)}")
        elif tuple(t.shape) != tuple(shape):
            raise ValueError(f"{where}: {name}: expected {tuple(shape)}, got {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{where}: {name} must be contiguous")
    for t, name, _ in named:
        if on_cuda and not t.is_cuda:
            raise ValueError(f"{where}: {name} must be a CUDA tensor")
    return d


def _row_stride(t, name) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name}: expected a 2-D tensor with unit column stride")
    return t.stride(0)


def version() -> int:
    return int(lib().dlrm_version())


# ---------------------------------------------------------------- standalone ops

def embedding_bag_sum_multi(tables: Sequence, indices, offsets, out, bag_size: int,
                            err_flag=None, stream=None) -> None:
    """out (B, K, D) = per-table bag sums; indices (K, B*L), offsets (K, B) int64."""
    import torch
    k = len(tables)
    if k == 0:
        raise ValueError("need at least one table")
    d = tables[0].shape[1]
    for i, t in enumerate(tables):
        _need(t, torch.float32, f"tables[{i}]")
        if t.dim() != 2 or t.shape[1] != d or not t.is_contiguous():
            raise ValueError(f"tables[{i}]: expected contiguous (rows, {d})")
    _need(indices, torch.int64, "indices")
    _need(offsets, torch.int64, "offsets")
    _need(out, torch.float32, "out")
    b = offsets.shape[1]
    if (tuple(indices.shape) != (k, b * bag_size) or tuple(offsets.shape) != (k, b)
            or tuple(out.shape) != (b, k, d)):
        raise ValueError("shape mismatch among indices/offsets/out")
    if not (indices.is_contiguous() and offsets.is_contiguous() and out.is_contiguous()):
        raise ValueError("indices, offsets and out must be contiguous")
    if err_flag is not None:
        _need(err_flag, torch.int32, "err_flag")
    ptrs = (ctypes.c_void_p * k)(*[t.data_ptr() for t in tables])
    rows = (ctypes.c_int64 * k)(*[t.shape[0] for t in tables])
    _check(lib().embedding_bag_sum_multi(ptrs, rows, k, d, _ptr(indices), _ptr(offsets), b,
                                         bag_size, _ptr(out), _ptr(err_flag), _stream(stream)),
           "embedding_bag_sum_multi")


BAG_SUM, BAG_MEAN, BAG_MAX = 0, 1, 2


def embedding_bag_multi(tables: Sequence, indices, offsets, out, mode: int = BAG_SUM,
                        per_sample_weights=None, padding_idx: int = -1, err_flag=None,
                        stream=None) -> None:
    """out (B, K, D) = per-table bag reductions over general offsets.

    indices (K, N) and offsets (K, B), both int64 or both int32; offsets are bag
    starts (the last bag runs to N); mode BAG_SUM, BAG_MEAN or BAG_MAX.
    per_sample_weights (K, N) fp32 scales each row (BAG_SUM only); an index equal
    to padding_idx (>= 0) is left out of its bag.
    """
    import torch
    k = len(tables)
    if k == 0:
        raise ValueError("need at least one table")
    d = tables[0].shape[1]
    for i, t in enumerate(tables):
        _need(t, torch.float32, f"tables[{i}]")
        if t.dim() != 2 or t.shape[1] != d or not t.is_contiguous():
            raise ValueError(f"tables[{i}]: expected contiguous (rows, {d})")
    if indices.dtype not in (torch.int64, torch.int32) or offsets.dtype != indices.dtype:
        raise ValueError("indices and offsets must both be int64 or both int32")
    _need(indices, indices.dtype, "indices")
    _need(offsets, offsets.dtype, "offsets")
    _need(out, torch.float32, "out")
    b = offsets.shape[1]
    if (indices.dim() != 2 or indices.shape[0] != k or tuple(offsets.shape) != (k, b)
            or tuple(out.shape) != (b, k, d)):
        raise ValueError("shape mismatch among indices/offsets/out")
    if not (indices.is_contiguous() and offsets.is_contiguous() and out.is_contiguous()):
        raise ValueError("indices, offsets and out must be contiguous")
    if per_sample_weights is not None:
        _need(per_sample_weights, torch.float32, "per_sample_weights")
        if (tuple(per_sample_weights.shape) != tuple(indices.shape)
                or not per_sample_weights.is_contiguous()):
            raise ValueError("per_sample_weights must be a contiguous tensor shaped like indices")
    if err_flag is not None:
        _need(err_flag, torch.int32, "err_flag")
    ptrs = (ctypes.c_void_p * k)(*[t.data_ptr() for t in tables])
    rows = (ctypes.c_int64 * k)(*[t.shape[0] for t in tables])
    opt = _BagOptions(int(mode), 64 if indices.dtype == torch.int64 else 32,
                      _ptr(per_sample_weights), int(padding_idx))
    _check(lib().embedding_bag_multi_ex(ptrs, rows, k, d, _ptr(indices), indices.shape[1],
                                        _ptr(offsets), b, ctypes.byref(opt), _ptr(out),
                                        _ptr(err_flag), _stream(stream)),
           "embedding_bag_multi_ex")


def pairwise_dot_lower_tri(dense, emb, out, copy_dense: bool = True, stream=None) -> None:
    """out[b] = [dense[b], z[b]] (copy_dense) or z[b]; dense (B, D), emb (B, K, D)."""
    import torch
    _need(dense, torch.float32, "dense")
    _need(emb, torch.float32, "emb")
    _need(out, torch.float32, "out")
    b, d = dense.shape
    if emb.dim() != 3 or emb.shape[0] != b or emb.shape[2] != d or not emb.is_contiguous():
        raise ValueError("emb: expected contiguous (B, K, D)")
    k = emb.shape[1]
    ld_dense = _row_stride(dense, "dense")
    ld_out = _row_stride(out, "out")
    if out.shape[0] != b:
        raise ValueError("out: batch mismatch")
    _check(lib().pairwise_dot_lower_tri(_ptr(dense), ld_dense, _ptr(emb), b, k, d, _ptr(out),
                                        ld_out, 1 if copy_dense else 0, _stream(stream)),
           "pairwise_dot_lower_tri")


def pairwise_pair_map(f: int, i_out, j_out, stream=None) -> None:
    import torch
    _need(i_out, torch.int32, "i_out")
    _need(j_out, torch.int32, "j_out")
    p = f * (f - 1) // 2
    if i_out.numel() < p or j_out.numel() < p:
        raise ValueError("i_out/j_out too small")
    _check(lib().pairwise_pair_map(f, _ptr(i_out), _ptr(j_out), _stream(stream)),
           "pairwise_pair_map")


def linear_bias_act(x, w, bias, y, act: int = ACT_NONE, math: int = MATH_FP32,
                    stream=None) -> None:
    """y = act(x W^T + bias); x (M, K), W (N, K) contiguous, y (M, N)."""
    import torch
    _need(x, torch.float32, "x")
    _need(w, torch.float32, "W")
    _need(y, torch.float32, "y")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    m, k = x.shape
    n = w.shape[0]
    if w.dim() != 2 or w.shape[1] != k or not w.is_contiguous():
        raise ValueError("W: expected contiguous (N, K)")
    if y.shape[0] != m or y.shape[1] != n:
        raise ValueError("y: expected (M, N)")
    _check(lib().linear_bias_act(_ptr(x), _row_stride(x, "x"), _ptr(w), _ptr(bias), _ptr(y),
                                 _row_stride(y, "y"), m, n, k, act, math, _stream(stream)),
           "linear_bias_act")


# ---------------------------------------------------------------- forward plan

def dlrm_create(ln_bot: Sequence[int], ln_top: Sequence[int], tables: Sequence,
                bot_w: Sequence, bot_b: Sequence, top_w: Sequence, top_b: Sequence,
                bag_size: int, max_batch: int, math: int = MATH_FP32,
                path: int = PATH_AUTO) -> int:
    """Build a forward plan; returns the opaque handle (an int).

    ``tables`` are CUDA tensors the handle borrows (keep them alive); the MLP
    parameters may be CPU or CUDA float32 tensors and are copied.
    """
    k = len(tables)
    d = _check_model_params(ln_bot, ln_top, tables, bot_w, bot_b, top_w, top_b, "dlrm_create",
                            on_cuda=False)
    for i, t in enumerate(tables):
        if not t.is_cuda:
            raise ValueError(f"dlrm_create: tables[{i}] must be a CUDA tensor (borrowed)")
    lb = (ctypes.c_int32 * len(ln_bot))(*ln_bot)
    lt = (ctypes.c_int32 * len(ln_top))(*ln_top)
    rows = (ctypes.c_int64 * k)(*[int(t.shape[0]) for t in tables])
    cfg = _Config(len(ln_bot) - 1, lb, k, rows, d, len(ln_top) - 1, lt, bag_size, max_batch,
                  math, path)

    def arr(ts):
        return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])

    h = ctypes.c_void_p()
    _check(lib().dlrm_create(ctypes.byref(cfg), arr(tables), arr(bot_w), arr(bot_b),
                             arr(top_w), arr(top_b), ctypes.byref(h)), "dlrm_create")
    _HANDLE_SHAPES[h.value] = (int(ln_bot[0]), k, int(bag_size), int(max_batch))
    return h.value


GB300_SMS = 152
GB300_SMEM_PER_BLOCK = 232448


def dlrm_plan_query(ln_bot: Sequence[int], ln_top: Sequence[int], rows: Sequence[int],
                    emb_dim: int, bag_size: int, max_batch: int, math: int = MATH_FP32,
                    path: int = PATH_AUTO, sm_count: int = GB300_SMS,
                    smem_per_block: int = GB300_SMEM_PER_BLOCK) -> dict:
    """The plan ``dlrm_create`` would take for this model on a device with
    ``sm_count`` SMs and ``smem_per_block`` bytes of opt-in shared memory per
    block (a GB300's by default), as a dict of the header's plan fields.
    Host-only: no device and no weights are needed."""
    k = len(rows)
    lb = (ctypes.c_int32 * len(ln_bot))(*ln_bot)
    lt = (ctypes.c_int32 * len(ln_top))(*ln_top)
    rw = (ctypes.c_int64 * k)(*rows)
    cfg = _Config(len(ln_bot) - 1, lb, k, rw, emb_dim, len(ln_top) - 1, lt, bag_size, max_batch,
                  math, path)
    info = _PlanInfo()
    _check(lib().dlrm_plan_query(ctypes.byref(cfg), sm_count, smem_per_block, ctypes.byref(info)),
           "dlrm_plan_query")
    return {name: getattr(info, name) for name, _ in _PlanInfo._fields_}


def _handle_shape(h: int, where: str):
    shape = _HANDLE_SHAPES.get(h)
    if shape is None:
        raise ValueError(f"{where}: {h!r} is not a live handle from dlrm_create")
    return shape


def dlrm_forward(h: int, dense, indices, offsets, out, stream=None) -> None:
    """One forward on CUDA tensors: dense (B, n_dense) float32, indices (K, B*L)
    and offsets (K, B) int64, out (>= B) float32; asynchronous on ``stream``."""
    n_dense, k, bag, max_batch = _handle_shape(h, "dlrm_forward")
    batch = _check_forward_io(n_dense, k, bag, max_batch, dense, indices, offsets, out,
                              "dlrm_forward", on_cuda=True)
    _check(lib().dlrm_forward(ctypes.c_void_p(h), _ptr(dense), _ptr(indices), _ptr(offsets),
                              _ptr(out), batch, _stream(stream)), "dlrm_forward")


def dlrm_forward_host(h: int, dense, indices, offsets, out, stream=None) -> None:
    """Host-buffer forward (CPU tensors, pinned or not; shapes as dlrm_forward);
    asynchronous on ``stream``."""
    n_dense, k, bag, max_batch = _handle_shape(h, "dlrm_forward_host")
    batch = _check_forward_io(n_dense, k, bag, max_batch, dense, indices, offsets, out,
                              "dlrm_forward_host", on_cuda=False)
    _check(lib().dlrm_forward_host(ctypes.c_void_p(h), _ptr(dense), _ptr(indices),
                                   _ptr(offsets), _ptr(out), batch, _stream(stream)),
           "dlrm_forward_host")


def dlrm_forward_noalloc(ln_bot: Sequence[int], ln_top: Sequence[int], tables: Sequence,
                         bot_w: Sequence, bot_b: Sequence, top_w: Sequence, top_b: Sequence,
                         bag_size: int, dense, indices, offsets, out, err_flag=None,
                         stream=None) -> None:
    """The forward with no handle and no device allocation (fixed library scratch).

    For callers that must not allocate device memory when they run the model.
    Every tensor is a CUDA tensor the caller owns; weights are (out, in)
    contiguous. Calls share one scratch array: serialise them (one stream).
    """
    import torch
    k = len(tables)
    d = _check_model_params(ln_bot, ln_top, tables, bot_w, bot_b, top_w, top_b,
                            "dlrm_forward_noalloc", on_cuda=True)
    batch = _check_forward_io(int(ln_bot[0]), k, int(bag_size), None, dense, indices, offsets,
                              out, "dlrm_forward_noalloc", on_cuda=True)
    if err_flag is not None:
        _need(err_flag, torch.int32, "err_flag")
        if err_flag.numel() < 1:
            raise ValueError("dlrm_forward_noalloc: err_flag needs one element")
    lb = (ctypes.c_int32 * len(ln_bot))(*ln_bot)
    lt = (ctypes.c_int32 * len(ln_top))(*ln_top)
    rows = (ctypes.c_int64 * k)(*[int(t.shape[0]) for t in tables])
    cfg = _Config(len(ln_bot) - 1, lb, k, rows, d, len(ln_top) - 1, lt, bag_size, batch,
                  MATH_FP32, PATH_AUTO)

    def arr(ts):
        return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])

    _check(lib().dlrm_forward_noalloc(ctypes.byref(cfg), arr(tables), arr(bot_w), arr(bot_b),
                                      arr(top_w), arr(top_b), _ptr(dense), _ptr(indices),
                                      _ptr(offsets), _ptr(out), batch,
                                      _ptr(err_flag), _stream(stream)),
           "dlrm_forward_noalloc")


def dlrm_get_error(h: int, stream=None) -> int:
    return int(lib().dlrm_get_error(ctypes.c_void_p(h), _stream(stream)))


def dlrm_test_stall(h: int, wait_limit_ns: int = 0, withhold_last: bool = False) -> None:
    """Failure-detection test hook: the limit of every bounded device wait of
    later forwards on ``h`` (0: the default) and, with ``withhold_last``, each
    kernel skips the last copy or tensor-core commit of its stream so that the
    wait on it runs out (``dlrm_get_error`` then reports ERR_TIMEOUT).
    ``dlrm_test_stall(h)`` restores normal operation."""
    _handle_shape(h, "dlrm_test_stall")
    _check(lib().dlrm_test_stall(ctypes.c_void_p(h), int(wait_limit_ns), 1 if withhold_last else 0),
           "dlrm_test_stall")


KERNELS_LAYERWISE, KERNELS_FUSED, KERNELS_FUSED_CLUSTER, KERNELS_FUSED_TC = 1, 2, 3, 4


def dlrm_forward_kernels(h: int, batch: int) -> int:
    """Which kernels a forward of ``batch`` samples on ``h`` runs (KERNELS_*)."""
    _handle_shape(h, "dlrm_forward_kernels")
    r = int(lib().dlrm_forward_kernels(ctypes.c_void_p(h), int(batch)))
    if r < 0:
        raise ValueError(f"dlrm_forward_kernels: batch {batch} outside [1, max_batch]")
    return r


def dlrm_set_cluster_batch_limit(h: int, limit: int) -> None:
    """Forwards of at most ``limit`` samples on ``h`` take the cluster-split
    fused kernel (0: never; -1: the default)."""
    _handle_shape(h, "dlrm_set_cluster_batch_limit")
    _check(lib().dlrm_set_cluster_batch_limit(ctypes.c_void_p(h), int(limit)),
           "dlrm_set_cluster_batch_limit")


def dlrm_get_cluster_batch_limit(h: int) -> int:
    """The largest batch ``h`` runs on the cluster-split kernel (0: none)."""
    _handle_shape(h, "dlrm_get_cluster_batch_limit")
    v = ctypes.c_int32(0)
    _check(lib().dlrm_get_cluster_batch_limit(ctypes.c_void_p(h), ctypes.byref(v)),
           "dlrm_get_cluster_batch_limit")
    return int(v.value)


def dlrm_workspace_bytes(h: int) -> int:
    return int(lib().dlrm_workspace_bytes(ctypes.c_void_p(h)))


def dlrm_path(h: int) -> int:
    return int(lib().dlrm_path(ctypes.c_void_p(h)))


def dlrm_num_stages(h: int) -> int:
    return int(lib().dlrm_num_stages(ctypes.c_void_p(h)))


def dlrm_stage_name(h: int, i: int) -> str:
    name = lib().dlrm_stage_name(ctypes.c_void_p(h), i)
    return name.decode() if name is not None else ""


def dlrm_set_profiling(h: int, enable: bool) -> None:
    _check(lib().dlrm_set_profiling(ctypes.c_void_p(h), 1 if enable else 0),
           "dlrm_set_profiling")


def dlrm_stage_times(h: int):
    """(names, total_ms per stage, profiled calls)."""
    n = dlrm_num_stages(h)
    buf = (ctypes.c_double * max(n, 1))()
    calls = ctypes.c_int64()
    lib().dlrm_stage_times(ctypes.c_void_p(h), buf, n, ctypes.byref(calls))
    return [dlrm_stage_name(h, i) for i in range(n)], list(buf)[:n], calls.value


def dlrm_destroy(h: Optional[int]) -> None:
    if h:
        _HANDLE_SHAPES.pop(h, None)
        lib().dlrm_destroy(ctypes.c_void_p(h))


class DlrmModel:
    """Owns a forward plan and keeps the borrowed tables alive."""

    def __init__(self, ln_bot, ln_top, tables, bot_w, bot_b, top_w, top_b, bag_size: int,
                 max_batch: int, math: int = MATH_FP32, path: int = PATH_AUTO):
        self.tables = list(tables)
        self.ln_bot, self.ln_top = tuple(ln_bot), tuple(ln_top)
        self.bag_size, self.max_batch, self.math = bag_size, max_batch, math
        self.handle = dlrm_create(ln_bot, ln_top, self.tables, bot_w, bot_b, top_w, top_b,
                                  bag_size, max_batch, math, path)

    def forward(self, dense, indices, offsets, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty(dense.shape[0], dtype=torch.float32, device=dense.device)
        dlrm_forward(self.handle, dense, indices, offsets, out, stream)
        return out

    def forward_host(self, dense, indices, offsets, out, stream=None):
        dlrm_forward_host(self.handle, dense, indices, offsets, out, stream)
        return out

    def error(self, stream=None) -> int:
        return dlrm_get_error(self.handle, stream)

    def workspace_bytes(self) -> int:
        return dlrm_workspace_bytes(self.handle)

    @property
    def path(self) -> int:
        return dlrm_path(self.handle)

    def stage_names(self):
        return [dlrm_stage_name(self.handle, i) for i in range(dlrm_num_stages(self.handle))]

    def kernels(self, batch: int) -> int:
        """Which kernels a forward of ``batch`` samples runs (KERNELS_*)."""
        return dlrm_forward_kernels(self.handle, batch)

    @property
    def cluster_batch_limit(self) -> int:
        """Forwards of at most this many samples take the cluster-split kernel."""
        return dlrm_get_cluster_batch_limit(self.handle)

    @cluster_batch_limit.setter
    def cluster_batch_limit(self, limit: int) -> None:
        dlrm_set_cluster_batch_limit(self.handle, limit)

    def set_profiling(self, enable: bool) -> None:
        dlrm_set_profiling(self.handle, enable)

    def stage_times(self):
        return dlrm_stage_times(self.handle)

    def set_phase_trace(self, buf) -> int:
        """Fused plan only: per-tile phase stamps into ``buf`` (int64 CUDA tensor of at
        least tiles * TRACE_SLOTS words) or off with None; returns the tile height."""
        rows = ctypes.c_int32()
        cap = 0 if buf is None else buf.numel()
        _check(lib().dlrm_set_phase_trace(ctypes.c_void_p(self.handle), _ptr(buf), cap,
                                          ctypes.byref(rows)), "dlrm_set_phase_trace")
        return rows.value

    def phase_names(self):
        """Names of the trace phases 1.. (slot 0 is the kernel start)."""
        nb, nt = len(self.ln_bot) - 1, len(self.ln_top) - 1
        return (["prologue"] + [f"bottom{l}" for l in range(nb)] + ["interaction"]
                + [f"top{l}" for l in range(nt - 1)] + [f"top{nt - 1}_sigmoid"])

    def close(self):
        if self.handle:
            dlrm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
