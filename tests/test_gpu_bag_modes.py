"""GPU parity of embedding_bag_multi (general offsets; sum, mean, max) against the oracle.

The operation is the runtime segment reduction of Luminal compare
dlrm-fused-kernels...dlrm-pt2-megakernel, LessonsLearned "EmbeddingBag
translator gap": output[b] = reduce_op(weight[indices[offsets[b]:offsets[b+1]]]).
Tolerances: max is exact (bit-exact against the oracle rounded to fp32); sum and
mean satisfy |gpu - oracle| <= 1e-5 + 1e-4 |oracle|; sums of one-row bags are
bit-exact row copies. Inputs are seeded bags of random lengths (dlrm_synth).
"""
import numpy as np
import pytest

import dlrm_synth as synth
import oracle

torch = pytest.importorskip("torch")
import dlrm_embedding_interaction_gb300 as dl  # noqa: E402

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-5, 1e-4
MODES = [(dl.BAG_SUM, oracle.BAG_SUM), (dl.BAG_MEAN, oracle.BAG_MEAN),
         (dl.BAG_MAX, oracle.BAG_MAX)]
MODE_IDS = ["sum", "mean", "max"]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    from dlrm_embedding_interaction_gb300 import build
    build.build()
    dl.lib()
    torch.cuda.set_device(0)


def cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _tables(rows, d, seed):
    cfg = synth.DlrmConfig("bags", 1, (13, d), tuple(rows), d, 1, (d + 1,), 0.05)
    return cfg, [synth.make_table(cfg, seed, t) for t in range(len(rows))]


def _run(tables, idx, off, mode, out=None):
    k, d = len(tables), tables[0].shape[1]
    b = off.shape[1]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if out is None:
        out = torch.full((b, k, d), float("nan"), device="cuda")
    dl.embedding_bag_multi([cu(t) for t in tables], cu(idx), cu(off), out, mode, err_flag=err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


def _flags(err):
    """The device error bits as the oracle's flag bits."""
    f = 0
    if err & dl.ERRBIT_INDEX_OOB:
        f |= oracle.BAG_FLAG_OOB
    if err & dl.ERRBIT_OFFSETS:
        f |= oracle.BAG_FLAG_OFFSETS
    return f


def _compare(got, ref, mode):
    if mode == dl.BAG_MAX:
        np.testing.assert_array_equal(got, ref.astype(np.float32))
    else:
        np.testing.assert_allclose(got.astype(np.float64), ref, atol=ATOL, rtol=RTOL)


# D picks every launch shape: lane groups of 1..32 lanes, 1..8 vectors per lane,
# and the scalar path (D % 4 != 0)
CASES = [
    # rows, D, B, max_len
    ((1000, 50, 7), 16, 37, 12),
    ((300,), 4, 129, 5),
    ((2000, 2000), 64, 200, 40),
    ((500,) * 3, 128, 97, 25),
    ((100, 100), 200, 33, 9),
    ((80,), 1024, 5, 70),
    ((64, 64), 13, 41, 8),
    ((10,), 1, 17, 3),
    ((20,) * 128, 8, 40, 6),          # DLRM_MAX_TABLES tables in one launch
]


@pytest.mark.parametrize("mode,omode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("rows,d,b,max_len", CASES)
def test_bag_modes_match_oracle(rows, d, b, max_len, mode, omode):
    cfg, tables = _tables(rows, d, seed=d + b)
    idx, off, lens = synth.make_variable_bags(cfg.with_batch(b), seed=b, max_len=max_len)
    assert (lens == 0).any() or max_len >= 40          # empty bags are covered
    got, err = _run(tables, idx, off, mode)
    ref, flags = oracle.embedding_bag(tables, idx, off, omode)
    assert flags == 0 and err == 0
    _compare(got, ref, mode)


@pytest.mark.parametrize("mode,omode", MODES, ids=MODE_IDS)
def test_one_long_bag_among_short_ones(mode, omode):
    """A 3000-row bag (many passes of one lane group) next to bags of 0..3 rows."""
    cfg, tables = _tables((5000, 5000), 64, seed=13)
    idx, off, lens = synth.make_variable_bags(cfg.with_batch(50), seed=14, max_len=3)
    extra = synth.make_indices(synth.DlrmConfig("x", 3000, (13, 64), (5000, 5000), 64, 1,
                                                (65,), 0.05), 15)
    # bag 20 of both tables grows by 3000 rows
    at = off[:, 20] + lens[:, 20]
    idx = np.stack([np.insert(idx[t], at[t], extra[t]) for t in range(2)])
    off = off.copy()
    off[:, 21:] += 3000
    got, err = _run(tables, idx, off, mode)
    ref, flags = oracle.embedding_bag(tables, idx, off, omode)
    assert err == 0 and flags == 0
    _compare(got, ref, mode)


def test_one_row_bags_are_row_copies():
    """Bags of one row over general offsets: the sum is the row itself, bit for bit."""
    cfg, tables = _tables((1000, 700, 33), 24, seed=3)
    b = 300
    idx = synth.make_indices(cfg.with_batch(b), 5)
    off = np.broadcast_to(np.arange(b, dtype=np.int64), (3, b)).copy()
    for mode in (dl.BAG_SUM, dl.BAG_MEAN, dl.BAG_MAX):
        got, err = _run(tables, idx, off, mode)
        assert err == 0
        for t in range(3):
            np.testing.assert_array_equal(got[:, t, :], np.take(tables[t], idx[t], axis=0))


@pytest.mark.parametrize("mode,omode", MODES, ids=MODE_IDS)
def test_out_of_range_rows_are_left_out_and_flagged(mode, omode):
    cfg, tables = _tables((400, 400), 32, seed=8)
    idx, off, _ = synth.make_variable_bags(cfg.with_batch(60), seed=9, max_len=10)
    idx = idx.copy()
    idx[0, 3] = 400          # one past the end
    idx[1, 17] = -1
    idx[1, 18] = 1 << 40
    got, err = _run(tables, idx, off, mode)
    ref, flags = oracle.embedding_bag(tables, idx, off, omode)
    assert flags == oracle.BAG_FLAG_OOB and _flags(err) == flags
    _compare(got, ref, mode)


@pytest.mark.parametrize("mode,omode", MODES, ids=MODE_IDS)
def test_bad_bag_bounds_give_zeros_and_flag(mode, omode):
    cfg, tables = _tables((300,), 16, seed=4)
    idx, off, _ = synth.make_variable_bags(cfg.with_batch(25), seed=2, max_len=6)
    n = idx.shape[1]
    off = off.copy()
    off[0, 4] = off[0, 5] + 1        # bag 4 reversed
    off[0, 10] = -2                  # bag 9 ends at -2 (< its start); bag 10 starts below 0
    off[0, 24] = n + 3               # the last bag starts past N
    got, err = _run(tables, idx, off, mode)
    ref, flags = oracle.embedding_bag(tables, idx, off, omode)
    assert flags & oracle.BAG_FLAG_OFFSETS and _flags(err) == flags
    _compare(got, ref, mode)
    for bb in (4, 9, 10, 24):
        assert not got[bb].any()


@pytest.mark.parametrize("mode", [dl.BAG_SUM, dl.BAG_MEAN, dl.BAG_MAX], ids=MODE_IDS)
def test_no_indices_at_all_gives_zeros(mode):
    _, tables = _tables((10, 10), 8, seed=1)
    idx = np.zeros((2, 0), np.int64)
    off = np.zeros((2, 7), np.int64)
    got, err = _run(tables, idx, off, mode)
    assert err == 0 and not got.any()


def test_empty_batch_is_a_noop_and_bad_mode_is_refused():
    _, tables = _tables((10,), 8, seed=1)
    out = torch.full((0, 1, 8), 1.0, device="cuda")
    dl.embedding_bag_multi([cu(tables[0])], cu(np.zeros((1, 0), np.int64)),
                           cu(np.zeros((1, 0), np.int64)), out, dl.BAG_SUM)
    with pytest.raises(dl.DlrmError) as ei:
        dl.embedding_bag_multi([cu(tables[0])], cu(np.zeros((1, 3), np.int64)),
                               cu(np.zeros((1, 2), np.int64)),
                               torch.empty((2, 1, 8), device="cuda"), 7)
    assert ei.value.status == dl.ERR_INVALID_ARG


@pytest.mark.parametrize("mode,omode", MODES, ids=MODE_IDS)
def test_unaligned_output_takes_the_scalar_path(mode, omode):
    """An output that is not 16-byte aligned runs the scalar kernel; same results."""
    cfg, tables = _tables((300, 300), 32, seed=6)
    idx, off, _ = synth.make_variable_bags(cfg.with_batch(45), seed=7, max_len=9)
    big = torch.full((45 * 2 * 32 + 1,), float("nan"), device="cuda")
    out = big[1:].view(45, 2, 32)
    got, err = _run(tables, idx, off, mode, out=out)
    ref, _ = oracle.embedding_bag(tables, idx, off, omode)
    assert err == 0
    _compare(got, ref, mode)


@pytest.mark.parametrize("mode,omode", MODES, ids=MODE_IDS)
def test_zipf_bags_of_the_large_workload_sampled(mode, omode):
    """The bench's variable-length workload shape (D = 128, Zipf(1.05) over 1M rows,
    lengths 0..40) on a slice of 2048 samples and 4 tables, all checked."""
    cfg = synth.DlrmConfig("vz", 2048, (13, 128), (1_000_000,) * 4, 128, 1, (129,), 0.01, "zipf")
    tables = [synth.make_table(cfg, 11, t) for t in range(4)]
    idx, off, _ = synth.make_variable_bags(cfg, seed=12, max_len=40)
    got, err = _run(tables, idx, off, mode)
    ref, flags = oracle.embedding_bag(tables, idx, off, omode)
    assert err == 0 and flags == 0
    _compare(got, ref, mode)


# ---------------------------------------------------------------- options

def _run_ex(tables, idx, off, mode, psw=None, padding_idx=-1, out=None):
    k, d = len(tables), tables[0].shape[1]
    b = off.shape[1]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if out is None:
        out = torch.full((b, k, d), float("nan"), device="cuda")
    dl.embedding_bag_multi([cu(t) for t in tables], cu(idx), cu(off), out, mode,
                           per_sample_weights=None if psw is None else cu(psw),
                           padding_idx=padding_idx, err_flag=err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("mode,omode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("d", [64, 13])
def test_int32_indices_and_offsets(mode, omode, d):
    """32-bit indices and offsets give what 64-bit ones give (and the oracle)."""
    cfg, tables = _tables((3000, 2000), d, seed=31)
    idx, off, _ = synth.make_variable_bags(cfg.with_batch(150), seed=32, max_len=15)
    got32, err = _run_ex(tables, idx.astype(np.int32), off.astype(np.int32), mode)
    got64, _ = _run_ex(tables, idx, off, mode)
    ref, _ = oracle.embedding_bag(tables, idx, off, omode)
    assert err == 0
    np.testing.assert_array_equal(got32, got64)
    _compare(got32, ref, mode)


@pytest.mark.parametrize("bits", [64, 32])
@pytest.mark.parametrize("d", [128, 24, 7])
def test_per_sample_weights(bits, d):
    cfg, tables = _tables((4000, 300, 50), d, seed=41)
    idx, off, _ = synth.make_variable_bags(cfg.with_batch(120), seed=42, max_len=20)
    w = synth.make_bag_weights(idx.shape, 43)
    dt = np.int64 if bits == 64 else np.int32
    got, err = _run_ex(tables, idx.astype(dt), off.astype(dt), dl.BAG_SUM, psw=w)
    ref, flags = oracle.embedding_bag(tables, idx, off, oracle.BAG_SUM, per_sample_weights=w)
    assert err == 0 and flags == 0
    _compare(got, ref, dl.BAG_SUM)


@pytest.mark.parametrize("mode,omode", MODES, ids=MODE_IDS)
def test_padding_idx_leaves_rows_out_without_a_flag(mode, omode):
    cfg, tables = _tables((500, 500), 32, seed=51)
    idx, off, _ = synth.make_variable_bags(cfg.with_batch(80), seed=52, max_len=6)
    idx = idx.copy()
    idx[:, ::3] = 7                     # a third of all entries are the padding row
    got, err = _run_ex(tables, idx, off, mode, padding_idx=7)
    ref, flags = oracle.embedding_bag(tables, idx, off, omode, padding_idx=7)
    assert err == 0 and flags == 0
    _compare(got, ref, mode)
    # and without padding_idx the same rows count
    got2, _ = _run_ex(tables, idx, off, mode)
    ref2, _ = oracle.embedding_bag(tables, idx, off, omode)
    _compare(got2, ref2, mode)


@pytest.mark.parametrize("mode,omode", MODES, ids=MODE_IDS)
def test_minus_one_is_out_of_range_without_padding(mode, omode):
    """With no padding row, an index of -1 is out of range: left out and flagged."""
    cfg, tables = _tables((200,), 16, seed=71)
    idx, off, _ = synth.make_variable_bags(cfg.with_batch(30), seed=72, max_len=5)
    idx = idx.copy()
    idx[0, 4] = -1
    got, err = _run_ex(tables, idx, off, mode)
    ref, flags = oracle.embedding_bag(tables, idx, off, omode)
    assert flags == oracle.BAG_FLAG_OOB and _flags(err) == flags
    _compare(got, ref, mode)


def test_weights_padding_and_bad_rows_together():
    cfg, tables = _tables((600,), 16, seed=61)
    idx, off, _ = synth.make_variable_bags(cfg.with_batch(64), seed=62, max_len=9)
    idx = idx.copy()
    idx[0, ::5] = 0
    idx[0, 3] = 600
    w = np.linspace(-1, 1, idx.size, dtype=np.float32).reshape(idx.shape)
    got, err = _run_ex(tables, idx, off, dl.BAG_SUM, psw=w, padding_idx=0)
    ref, flags = oracle.embedding_bag(tables, idx, off, oracle.BAG_SUM, per_sample_weights=w,
                                      padding_idx=0)
    assert flags == oracle.BAG_FLAG_OOB and _flags(err) == flags
    _compare(got, ref, dl.BAG_SUM)


def test_weights_need_sum_mode_and_matching_index_types():
    _, tables = _tables((10,), 8, seed=1)
    idx = cu(np.zeros((1, 4), np.int64))
    off = cu(np.zeros((1, 2), np.int64))
    out = torch.empty((2, 1, 8), device="cuda")
    w = torch.ones((1, 4), device="cuda")
    for mode in (dl.BAG_MEAN, dl.BAG_MAX):
        with pytest.raises(dl.DlrmError) as ei:
            dl.embedding_bag_multi([cu(tables[0])], idx, off, out, mode, per_sample_weights=w)
        assert ei.value.status == dl.ERR_INVALID_ARG
    with pytest.raises(ValueError):
        dl.embedding_bag_multi([cu(tables[0])], idx, off.int(), out, dl.BAG_SUM)
