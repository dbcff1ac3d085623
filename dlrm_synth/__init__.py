"""Seeded synthetic inputs for the DLRMv1 inference forward.

This module only draws random numbers; it holds none of the forward's
arithmetic. The CUDA path's tests, the bench and the CPU oracle all consume
what it produces, and it imports neither of them.

The named workloads follow the DLRMv1 shapes the Luminal DLRM pages describe
(``dlrm_megakernel.rs`` shape struct: dense width, bottom widths, K tables of
width m_spa, top widths ending in 1):

* ``tiny_b64_k3``      batch 64, bottom 13-64-16, 3 x 1000 x 16 tables, bags of 2,
                       top 22-64-1
* ``b2048_k3``         batch 2048, bottom 13-512-256-64, 3 x 100k x 64, bag 1,
                       top 70-512-256-1
* ``b2048_k32``        batch 2048, same bottom, 32 x 100k x 64, bag 1,
                       top 592-512-256-1
* ``b65536_k26_zipf``  batch 65536, bottom 13-512-256-128, 26 x 1M x 128 (13.3 GB),
                       bags of 20 drawn Zipf(1.05), top 479-1024-1024-512-256-1
* ``sweep_b{B}_k{K}``  100k x 64 tables, bag 1, bottom 13-512-256-64,
                       top (64 + P)-512-256-1
* ``mini_b2048_k3_d4`` the pages' megakernel unit-test shape: bottom 13-8-4,
                       tables of 10/20/30 rows x 4, top 10-8-1

Distributions: dense ~ N(0, 1); tables ~ U(-r, r) with r = 0.05 (tiny, mini) or
0.01; MLP weights and biases ~ U(-1/sqrt(fan_in), 1/sqrt(fan_in)) (the PyTorch
``nn.Linear`` default, Kaiming-uniform with a = sqrt(5)); indices uniform over
rows, or truncated Zipf(s) over ranks with rank k mapped to row k - 1; offsets
are the uniform stride b * L.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
from typing import Dict, List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libdlrm_synth.so")
_lib = None

# Stream ids: one independent SplitMix64 stream per tensor.
STREAM_DENSE = 1
STREAM_TABLE = 1000
STREAM_INDEX = 2000
STREAM_BOT = 3000
STREAM_TOP = 4000
STREAM_BAG_LEN = 5000
STREAM_BAG_WEIGHT = 6000


def build(force: bool = False) -> str:
    """Compile the generator library with the host C compiler (seconds)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, u64, dbl, i32, vp = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_double,
                                  ctypes.c_int, ctypes.c_void_p)
        lib.synth_uniform_f32.argtypes = [vp, i64, u64, u64, dbl, dbl, i32]
        lib.synth_normal_f32.argtypes = [vp, i64, u64, u64, i32]
        lib.synth_uniform_i64.argtypes = [vp, i64, u64, u64, i64, i32]
        lib.synth_zipf_cdf.argtypes = [vp, i64, dbl]
        lib.synth_zipf_i64.argtypes = [vp, i64, u64, u64, vp, i64, i32]
        lib.synth_element.argtypes = [u64, u64, u64]
        lib.synth_element.restype = u64
        lib.synth_raw.argtypes = [u64, u64]
        lib.synth_raw.restype = u64
        for f in (lib.synth_uniform_f32, lib.synth_normal_f32, lib.synth_uniform_i64,
                  lib.synth_zipf_cdf, lib.synth_zipf_i64):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _threads(threads: Optional[int]) -> int:
    return threads if threads else (os.cpu_count() or 1)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"dlrm_synth: {what} failed with code {rc}")


def _contig(a: np.ndarray, dtype) -> None:
    if a.dtype != dtype or not a.flags["C_CONTIGUOUS"]:
        raise ValueError(f"need a C-contiguous {np.dtype(dtype)} array, got {a.dtype}")


def element(seed: int, stream: int, i: int) -> int:
    """Raw 64-bit element i of stream (seed, stream); used to pin the generator."""
    return int(_load().synth_element(seed, stream, i))


def raw(key: int, i: int) -> int:
    """Element i of the plain SplitMix64 sequence started at state ``key``."""
    return int(_load().synth_raw(key, i))


def fill_uniform(out: np.ndarray, seed: int, stream: int, lo: float, hi: float,
                 threads: Optional[int] = None) -> np.ndarray:
    _contig(out, np.float32)
    _check(_load().synth_uniform_f32(out.ctypes.data, out.size, seed, stream, lo, hi,
                                     _threads(threads)), "uniform")
    return out


def fill_normal(out: np.ndarray, seed: int, stream: int,
                threads: Optional[int] = None) -> np.ndarray:
    _contig(out, np.float32)
    _check(_load().synth_normal_f32(out.ctypes.data, out.size, seed, stream,
                                    _threads(threads)), "normal")
    return out


def fill_index_uniform(out: np.ndarray, seed: int, stream: int, rows: int,
                       threads: Optional[int] = None) -> np.ndarray:
    _contig(out, np.int64)
    _check(_load().synth_uniform_i64(out.ctypes.data, out.size, seed, stream, rows,
                                     _threads(threads)), "uniform index")
    return out


_CDF_CACHE: Dict = {}


def zipf_cdf(rows: int, s: float) -> np.ndarray:
    key = (rows, s)
    if key not in _CDF_CACHE:
        cdf = np.empty(rows, dtype=np.float64)
        _check(_load().synth_zipf_cdf(cdf.ctypes.data, rows, s), "zipf cdf")
        _CDF_CACHE[key] = cdf
    return _CDF_CACHE[key]


def fill_index_zipf(out: np.ndarray, seed: int, stream: int, rows: int, s: float,
                    threads: Optional[int] = None) -> np.ndarray:
    _contig(out, np.int64)
    cdf = zipf_cdf(rows, s)
    _check(_load().synth_zipf_i64(out.ctypes.data, out.size, seed, stream,
                                  cdf.ctypes.data, rows, _threads(threads)), "zipf index")
    return out


@dataclasses.dataclass(frozen=True)
class DlrmConfig:
    """Shape and distribution of one synthetic DLRMv1 workload."""
    name: str
    batch: int
    ln_bot: tuple          # (n_dense, ..., D)
    rows: tuple            # rows per table, len K
    emb_dim: int           # D
    bag_size: int          # L (uniform)
    ln_top: tuple          # (D + P, ..., 1)
    table_range: float = 0.01
    index_dist: str = "uniform"   # "uniform" | "zipf"
    zipf_s: float = 1.05

    @property
    def n_tables(self) -> int:
        return len(self.rows)

    @property
    def n_features(self) -> int:
        return self.n_tables + 1

    @property
    def n_pairs(self) -> int:
        f = self.n_features
        return f * (f - 1) // 2

    @property
    def n_dense(self) -> int:
        return self.ln_bot[0]

    def with_batch(self, batch: int) -> "DlrmConfig":
        return dataclasses.replace(self, batch=batch)


def _top(d: int, k: int, hidden: Sequence[int]) -> tuple:
    f = k + 1
    return (d + f * (f - 1) // 2,) + tuple(hidden) + (1,)


def sweep_config(batch: int, n_tables: int) -> DlrmConfig:
    return DlrmConfig(f"sweep_b{batch}_k{n_tables}", batch, (13, 512, 256, 64),
                      (100_000,) * n_tables, 64, 1, _top(64, n_tables, (512, 256)))


SWEEP_BATCHES = (1, 8, 32, 64, 128, 256, 512, 1024, 2048, 4096, 8192)
SWEEP_TABLES = (1, 3, 8, 16, 32)

CONFIGS: Dict[str, DlrmConfig] = {
    "tiny_b64_k3": DlrmConfig("tiny_b64_k3", 64, (13, 64, 16), (1000,) * 3, 16, 2,
                              _top(16, 3, (64,)), table_range=0.05),
    "b2048_k3": DlrmConfig("b2048_k3", 2048, (13, 512, 256, 64), (100_000,) * 3, 64, 1,
                           _top(64, 3, (512, 256))),
    "b2048_k32": DlrmConfig("b2048_k32", 2048, (13, 512, 256, 64), (100_000,) * 32, 64, 1,
                            _top(64, 32, (512, 256))),
    "b65536_k26_zipf": DlrmConfig("b65536_k26_zipf", 65536, (13, 512, 256, 128),
                                  (1_000_000,) * 26, 128, 20,
                                  _top(128, 26, (1024, 1024, 512, 256)),
                                  index_dist="zipf", zipf_s=1.05),
    "mini_b2048_k3_d4": DlrmConfig("mini_b2048_k3_d4", 2048, (13, 8, 4), (10, 20, 30), 4, 1,
                                   (10, 8, 1), table_range=0.05),
}


def get_config(name: str) -> DlrmConfig:
    if name in CONFIGS:
        return CONFIGS[name]
    if name.startswith("sweep_b"):
        b, k = name[len("sweep_b"):].split("_k")
        return sweep_config(int(b), int(k))
    raise KeyError(f"unknown workload {name!r}")


def make_table(cfg: DlrmConfig, seed: int, t: int, out: Optional[np.ndarray] = None,
               threads: Optional[int] = None) -> np.ndarray:
    if out is None:
        out = np.empty((cfg.rows[t], cfg.emb_dim), dtype=np.float32)
    return fill_uniform(out, seed, STREAM_TABLE + t, -cfg.table_range, cfg.table_range,
                        threads)


def make_mlp(cfg: DlrmConfig, seed: int, which: str):
    widths = cfg.ln_bot if which == "bot" else cfg.ln_top
    base = STREAM_BOT if which == "bot" else STREAM_TOP
    ws, bs = [], []
    for l in range(len(widths) - 1):
        fan_in, fan_out = widths[l], widths[l + 1]
        bound = 1.0 / np.sqrt(fan_in)
        ws.append(fill_uniform(np.empty((fan_out, fan_in), np.float32), seed,
                               base + 2 * l, -bound, bound))
        bs.append(fill_uniform(np.empty((fan_out,), np.float32), seed,
                               base + 2 * l + 1, -bound, bound))
    return ws, bs


def make_dense(cfg: DlrmConfig, seed: int, batch: Optional[int] = None) -> np.ndarray:
    b = cfg.batch if batch is None else batch
    return fill_normal(np.empty((b, cfg.n_dense), np.float32), seed, STREAM_DENSE)


def make_indices(cfg: DlrmConfig, seed: int, batch: Optional[int] = None,
                 threads: Optional[int] = None) -> np.ndarray:
    """Indices, table-major (K, B * L) int64."""
    b = cfg.batch if batch is None else batch
    out = np.empty((cfg.n_tables, b * cfg.bag_size), np.int64)
    for t in range(cfg.n_tables):
        if cfg.index_dist == "zipf":
            fill_index_zipf(out[t], seed, STREAM_INDEX + t, cfg.rows[t], cfg.zipf_s, threads)
        else:
            fill_index_uniform(out[t], seed, STREAM_INDEX + t, cfg.rows[t], threads)
    return out


def make_offsets(cfg: DlrmConfig, batch: Optional[int] = None) -> np.ndarray:
    """Uniform-stride offsets, (K, B) int64: offsets[t][b] = b * L."""
    b = cfg.batch if batch is None else batch
    row = np.arange(b, dtype=np.int64) * cfg.bag_size
    return np.broadcast_to(row, (cfg.n_tables, b)).copy()


def make_variable_bags(cfg: DlrmConfig, seed: int, max_len: int, batch: Optional[int] = None,
                       threads: Optional[int] = None):
    """Bags of random lengths for the general-offsets EmbeddingBag.

    Table 0's bag lengths are uniform on 0..max_len (stream STREAM_BAG_LEN);
    every other table t takes the same lengths in its own order (sorted by keys
    from stream STREAM_BAG_LEN + t), so all tables hold the same number N of
    indices and no bag absorbs a remainder. Indices follow cfg.index_dist
    (stream STREAM_INDEX + t). Returns ((K, N) int64 indices, (K, B) int64
    offsets, (K, B) int64 lengths).
    """
    b = cfg.batch if batch is None else batch
    k = cfg.n_tables
    lens = np.empty((k, b), np.int64)
    fill_index_uniform(lens[0], seed, STREAM_BAG_LEN, max_len + 1, threads)
    keys = np.empty(b, np.int64)
    for t in range(1, k):
        fill_index_uniform(keys, seed, STREAM_BAG_LEN + t, 0xFFFFFFFF, threads)
        lens[t] = lens[0][np.argsort(keys, kind="stable")]
    n = int(lens[0].sum()) if b > 0 else 0
    offsets = np.zeros((k, b), np.int64)
    if b > 0:
        offsets[:, 1:] = np.cumsum(lens, axis=1)[:, :-1]
    indices = np.empty((k, n), np.int64)
    for t in range(k):
        if n == 0:
            continue
        if cfg.index_dist == "zipf":
            fill_index_zipf(indices[t], seed, STREAM_INDEX + t, cfg.rows[t], cfg.zipf_s, threads)
        else:
            fill_index_uniform(indices[t], seed, STREAM_INDEX + t, cfg.rows[t], threads)
    return indices, offsets, lens


def make_bag_weights(shape, seed: int, lo: float = -2.0, hi: float = 2.0,
                     threads: Optional[int] = None) -> np.ndarray:
    """Per-sample weights (K, N) fp32, uniform on [lo, hi) (stream STREAM_BAG_WEIGHT + t)."""
    out = np.empty(shape, np.float32)
    for t in range(shape[0]):
        fill_uniform(out[t], seed, STREAM_BAG_WEIGHT + t, lo, hi, threads)
    return out


def make_inputs(cfg: DlrmConfig, seed: int = 1234, batch: Optional[int] = None,
                with_tables: bool = True, threads: Optional[int] = None) -> dict:
    """All inputs and parameters of one workload as host numpy arrays."""
    bot_w, bot_b = make_mlp(cfg, seed, "bot")
    top_w, top_b = make_mlp(cfg, seed, "top")
    inp = dict(
        dense=make_dense(cfg, seed, batch),
        indices=make_indices(cfg, seed, batch, threads),
        offsets=make_offsets(cfg, batch),
        bot_w=bot_w, bot_b=bot_b, top_w=top_w, top_b=top_b,
    )
    if with_tables:
        inp["tables"] = [make_table(cfg, seed, t, threads=threads)
                         for t in range(cfg.n_tables)]
    return inp
