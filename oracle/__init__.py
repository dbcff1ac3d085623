"""CPU oracle for the DLRMv1 inference forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
may import this package. The product path (the CUDA library and its binding)
never imports, links or calls it, and it never imports the product.

This is a thin ctypes marshalling layer over ``oracle.cpp`` (plain C++,
fp64 accumulation); see that file for the definitions it follows and the
readings taken where the Luminal DLRM pages are silent. Stage functions take
the fp32 arrays a GPU stage consumed and return float64 results, so stage
errors never compound.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

OK, INVALID, INDEX_OOB = 0, 1, 5
ACT_NONE, ACT_RELU, ACT_SIGMOID = 0, 1, 2


def build(force: bool = False, extra_flags: Sequence[str] = (), out: Optional[str] = None) -> str:
    """Compile the oracle with g++ -O2 (no fast-math, no -march=native)."""
    out = out or _LIB_PATH
    if (not force and not extra_flags and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
                           *extra_flags, _SRC, "-o", tmp])
    os.replace(tmp, out)
    return out


def _bind(lib):
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.oracle_pair_from_index.argtypes = [i64, vp, vp]
    lib.oracle_pair_from_index.restype = None
    lib.oracle_pair_enumerate.argtypes = [i32, vp, vp]
    lib.oracle_pair_enumerate.restype = None
    lib.oracle_embedding_bag_sum.argtypes = [i32, vp, vp, i32, vp, i64, vp, i64, vp, i32]
    lib.oracle_embedding_bag.argtypes = [i32, vp, vp, i32, vp, i64, vp, i64, i32, vp, i64, vp,
                                         vp, i32]
    lib.oracle_linear.argtypes = [i64, i32, i32, vp, vp, vp, i32, vp, i32]
    lib.oracle_interaction.argtypes = [i64, i32, i32, vp, vp, vp, i32]
    lib.oracle_forward.argtypes = [i64, i32, vp, vp, vp, i32, vp, vp, i32, vp, i64, vp,
                                   i32, vp, vp, vp, vp, vp, i64, vp, i32]
    for f in (lib.oracle_embedding_bag_sum, lib.oracle_embedding_bag, lib.oracle_linear,
              lib.oracle_interaction, lib.oracle_forward):
        f.restype = ctypes.c_int
    return lib


def load(path: Optional[str] = None):
    """Load the oracle library (building it first if needed)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _threads(threads: Optional[int]) -> int:
    return threads if threads else (os.cpu_count() or 1)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int64)


def _ptr_array(arrays) -> ctypes.Array:
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


class OracleError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"oracle {where} returned status {code}")
        self.code = code


def _check(rc: int, where: str, allow_oob: bool) -> int:
    if rc == OK or (rc == INDEX_OOB and allow_oob):
        return rc
    raise OracleError(rc, where)


def pair_from_index(p: int, lib=None):
    lib = lib or load()
    i, j = ctypes.c_int64(), ctypes.c_int64()
    lib.oracle_pair_from_index(p, ctypes.byref(i), ctypes.byref(j))
    return i.value, j.value


def pair_enumerate(f: int, lib=None):
    lib = lib or load()
    n = f * (f - 1) // 2
    i, j = np.zeros(n, np.int64), np.zeros(n, np.int64)
    lib.oracle_pair_enumerate(f, i.ctypes.data, j.ctypes.data)
    return i, j


def embedding_bag_sum(tables, indices, offsets, allow_oob: bool = False,
                      threads: Optional[int] = None, lib=None, return_status: bool = False):
    """Bag sums, (B, K, D) float64. ``indices`` (K, N), ``offsets`` (K, B)."""
    lib = lib or load()
    tables = [_f32(t) for t in tables]
    indices, offsets = _i64(indices), _i64(offsets)
    k = len(tables)
    d = tables[0].shape[1]
    b = offsets.shape[1]
    rows = np.array([t.shape[0] for t in tables], np.int64)
    out = np.zeros((b, k, d), np.float64)
    rc = lib.oracle_embedding_bag_sum(k, _ptr_array(tables), rows.ctypes.data, d,
                                      indices.ctypes.data, indices.shape[1],
                                      offsets.ctypes.data, b, out.ctypes.data,
                                      _threads(threads))
    rc = _check(rc, "embedding_bag_sum", allow_oob)
    return (out, rc) if return_status else out


BAG_SUM, BAG_MEAN, BAG_MAX = 0, 1, 2
BAG_FLAG_OOB, BAG_FLAG_OFFSETS = 1, 2


def embedding_bag(tables, indices, offsets, mode: int = BAG_SUM, per_sample_weights=None,
                  padding_idx: int = -1, threads: Optional[int] = None, lib=None):
    """Bags under a reduction mode over general offsets: ((B, K, D) float64, flags).

    Bag b of table t is indices[t][offsets[t][b] : offsets[t][b+1]] (the last
    bag ends at N = indices.shape[1]); mode BAG_SUM, BAG_MEAN or BAG_MAX. An
    index out of range is left out of its bag (flag BAG_FLAG_OOB); mean divides
    by the rows kept; a bag with no rows is zeros; bad bounds (begin < 0,
    end > N, begin > end) give zeros and flag BAG_FLAG_OFFSETS.
    per_sample_weights (K, N) float scales each row (sum only); an index equal
    to padding_idx (>= 0) is left out without a flag.
    """
    lib = lib or load()
    tables = [_f32(t) for t in tables]
    indices, offsets = _i64(indices), _i64(offsets)
    k = len(tables)
    d = tables[0].shape[1]
    b = offsets.shape[1]
    rows = np.array([t.shape[0] for t in tables], np.int64)
    out = np.zeros((b, k, d), np.float64)
    flags = ctypes.c_int(0)
    psw = None if per_sample_weights is None else _f32(per_sample_weights)
    if psw is not None and psw.shape != indices.shape:
        raise ValueError("per_sample_weights must match indices")
    rc = lib.oracle_embedding_bag(k, _ptr_array(tables), rows.ctypes.data, d,
                                  indices.ctypes.data, indices.shape[1], offsets.ctypes.data, b,
                                  int(mode), None if psw is None else psw.ctypes.data,
                                  int(padding_idx), out.ctypes.data, ctypes.byref(flags),
                                  _threads(threads))
    if rc != OK:
        raise OracleError(rc, "embedding_bag")
    return out, flags.value


def linear(x, w, b=None, act: int = ACT_NONE, threads: Optional[int] = None, lib=None):
    """act(x W^T + b), float64 (M, N). ``w`` is (N, K) as in nn.Linear."""
    lib = lib or load()
    x, w = _f64(x), _f32(w)
    bb = None if b is None else _f32(b)
    m, k = x.shape
    n = w.shape[0]
    y = np.zeros((m, n), np.float64)
    rc = lib.oracle_linear(m, k, n, x.ctypes.data, w.ctypes.data,
                           None if bb is None else bb.ctypes.data, act, y.ctypes.data,
                           _threads(threads))
    _check(rc, "linear", False)
    return y


def interaction(x, e, threads: Optional[int] = None, lib=None):
    """R = [x, z] (B, D + F(F-1)/2) float64 from x (B, D) and e (B, K, D)."""
    lib = lib or load()
    x, e = _f64(x), _f64(e)
    b, d = x.shape
    k = e.shape[1]
    f = k + 1
    r = np.zeros((b, d + f * (f - 1) // 2), np.float64)
    rc = lib.oracle_interaction(b, k, d, x.ctypes.data, e.ctypes.data, r.ctypes.data,
                                _threads(threads))
    _check(rc, "interaction", False)
    return r


def forward(inputs: dict, sample_ids=None, allow_oob: bool = False,
            threads: Optional[int] = None, lib=None):
    """Full forward, float64 (n,) for the given samples (all when None).

    ``inputs`` holds dense (B, n_dense), tables [K x (V_t, D)], indices (K, N),
    offsets (K, B), bot_w/bot_b/top_w/top_b lists ((out, in) weights).
    """
    lib = lib or load()
    dense = _f32(inputs["dense"])
    tables = [_f32(t) for t in inputs["tables"]]
    indices, offsets = _i64(inputs["indices"]), _i64(inputs["offsets"])
    bot_w = [_f32(w) for w in inputs["bot_w"]]
    bot_b = [_f32(v) for v in inputs["bot_b"]]
    top_w = [_f32(w) for w in inputs["top_w"]]
    top_b = [_f32(v) for v in inputs["top_b"]]
    ln_bot = np.array([bot_w[0].shape[1]] + [w.shape[0] for w in bot_w], np.int32)
    ln_top = np.array([top_w[0].shape[1]] + [w.shape[0] for w in top_w], np.int32)
    b = dense.shape[0]
    k = len(tables)
    d = tables[0].shape[1]
    rows = np.array([t.shape[0] for t in tables], np.int64)
    ids = None if sample_ids is None else _i64(sample_ids)
    n = b if ids is None else ids.shape[0]
    out = np.zeros(n, np.float64)
    rc = lib.oracle_forward(b, len(bot_w), ln_bot.ctypes.data, _ptr_array(bot_w),
                            _ptr_array(bot_b), k, _ptr_array(tables), rows.ctypes.data, d,
                            indices.ctypes.data, indices.shape[1], offsets.ctypes.data,
                            len(top_w), ln_top.ctypes.data, _ptr_array(top_w),
                            _ptr_array(top_b), dense.ctypes.data,
                            None if ids is None else ids.ctypes.data, n, out.ctypes.data,
                            _threads(threads))
    _check(rc, "forward", allow_oob)
    return out
