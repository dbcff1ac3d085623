"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Nothing here compares the oracle with itself: each check uses an independent
library routine (numpy fancy indexing, matmul, tril_indices; torch CPU
modules), a closed form, an invariant, exhaustive enumeration, or a
hand-computed fixture under tests/golden/.
"""
import json
import math
import os

import numpy as np
import pytest

import dlrm_synth as synth
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _arr(x, dt):
    return np.array(x, dtype=dt)


# ---------------------------------------------------------------- pair map

def test_pair_closed_form_exhaustive_f_le_256(oracle_lib):
    """p -> (i, j) closed form equals the i-major enumeration for every F <= 256.

    Luminal compare modal_ci_ready...vanilla-pytorch, commit message,
    PairwiseDotLowerTriStackedKernel: pair (i, j) from p via (1+sqrt(1+8p))/2.
    The enumeration for F is a prefix of that for F+1, so F = 256 covers all.
    """
    f = 256
    ei, ej = oracle.pair_enumerate(f, oracle_lib)
    # the enumeration itself is the strict lower triangle, row-major
    ti, tj = np.tril_indices(f, -1)
    np.testing.assert_array_equal(ei, ti)
    np.testing.assert_array_equal(ej, tj)
    for p in range(f * (f - 1) // 2):
        assert oracle.pair_from_index(p, oracle_lib) == (ei[p], ej[p]), p


def test_pair_counts_and_shape_invariants():
    """F(F-1)/2 and ln_top[0] = D + P for the pages' mini shape and the workloads.

    dlrm_megakernel.rs tests shape_invariants: F = 4 -> 6 pairs, ln_top[0] = m_spa + n_pairs.
    """
    mini = synth.get_config("mini_b2048_k3_d4")
    assert mini.n_features == 4 and mini.n_pairs == 6
    assert mini.ln_top[0] == mini.emb_dim + mini.n_pairs == 10
    assert synth.get_config("b2048_k32").n_pairs == 528
    assert synth.get_config("b65536_k26_zipf").n_pairs == 351
    for name in ("tiny_b64_k3", "b2048_k3", "b2048_k32", "b65536_k26_zipf"):
        c = synth.get_config(name)
        assert c.ln_top[0] == c.emb_dim + c.n_pairs and c.ln_top[-1] == 1
        assert c.ln_bot[-1] == c.emb_dim


# ---------------------------------------------------------------- bag sum

def test_bag_size_one_is_index_select(oracle_lib):
    """With one index per bag the bag sum is a row lookup (index_select), bit-exact.

    LessonsLearned 'EmbeddingBag translator gap': for bag size 1 it is just an
    embedding lookup.
    """
    cfg = synth.sweep_config(257, 5)
    cfg = synth.DlrmConfig("t", 257, cfg.ln_bot, (1000, 700, 1, 33, 5000), 24, 1, cfg.ln_top)
    tables = [synth.make_table(cfg, 7, t) for t in range(cfg.n_tables)]
    idx = synth.make_indices(cfg, 7)
    off = synth.make_offsets(cfg)
    e = oracle.embedding_bag_sum(tables, idx, off, lib=oracle_lib)
    for t in range(cfg.n_tables):
        expect = np.take(tables[t], idx[t], axis=0)
        np.testing.assert_array_equal(e[:, t, :].astype(np.float32), expect)
        np.testing.assert_array_equal(e[:, t, :], expect.astype(np.float64))


def test_bag_sum_permutation_invariant(oracle_lib):
    """Permuting indices inside each bag leaves the bag sum unchanged (<= 1 ulp in fp32)."""
    cfg = synth.get_config("tiny_b64_k3")
    cfg = synth.DlrmConfig("t", 96, cfg.ln_bot, (1000,) * 3, 16, 7, cfg.ln_top, 0.05)
    tables = [synth.make_table(cfg, 3, t) for t in range(3)]
    idx = synth.make_indices(cfg, 3)
    off = synth.make_offsets(cfg)
    base = oracle.embedding_bag_sum(tables, idx, off, lib=oracle_lib).astype(np.float32)
    rng = np.random.default_rng(0)
    perm = idx.copy().reshape(3, 96, 7)
    for t in range(3):
        for b in range(96):
            perm[t, b] = perm[t, b][rng.permutation(7)]
    assert not np.array_equal(perm.reshape(3, -1), idx)
    got = oracle.embedding_bag_sum(tables, perm.reshape(3, -1), off,
                                   lib=oracle_lib).astype(np.float32)
    ulp = np.spacing(np.maximum(np.abs(base), np.abs(got)))
    assert np.all(np.abs(got - base) <= ulp)


def test_bag_sum_general_offsets_and_empty_bags(oracle_lib):
    """General offsets: bag b spans offsets[b]..offsets[b+1] (last bag to N); empty bag = 0."""
    table = np.arange(20, dtype=np.float32).reshape(10, 2)   # row r = [2r, 2r+1]
    idx = np.array([[3, 1, 4, 1, 5, 9, 2, 6]], np.int64)
    off = np.array([[0, 2, 2, 5]], np.int64)  # bags: {3,1}, {}, {4,1,5}, {9,2,6}
    e = oracle.embedding_bag_sum([table], idx, off, lib=oracle_lib)
    expect = np.array([[6 + 2, 7 + 3], [0, 0], [8 + 2 + 10, 9 + 3 + 11],
                       [18 + 4 + 12, 19 + 5 + 13]], np.float64)
    np.testing.assert_array_equal(e[:, 0, :], expect)


def test_bag_sum_out_of_range_index_flags(oracle_lib):
    """An index outside [0, rows) contributes zeros and reports INDEX_OOB."""
    table = np.ones((4, 3), np.float32)
    idx = np.array([[0, 7, -1, 2]], np.int64)
    off = np.array([[0, 2]], np.int64)
    e, rc = oracle.embedding_bag_sum([table], idx, off, allow_oob=True, lib=oracle_lib,
                                     return_status=True)
    assert rc == oracle.INDEX_OOB
    np.testing.assert_array_equal(e[:, 0, :], [[1, 1, 1], [1, 1, 1]])
    with pytest.raises(oracle.OracleError):
        oracle.embedding_bag_sum([table], idx, off, lib=oracle_lib)


def test_bag_sum_matches_torch_embedding_bag(oracle_lib):
    """Library cross-check: torch.nn.functional.embedding_bag(mode='sum') in float64."""
    torch = pytest.importorskip("torch")
    cfg = synth.get_config("tiny_b64_k3")
    inp = synth.make_inputs(cfg, seed=11)
    e = oracle.embedding_bag_sum(inp["tables"], inp["indices"], inp["offsets"], lib=oracle_lib)
    for t in range(cfg.n_tables):
        ref = torch.nn.functional.embedding_bag(
            torch.from_numpy(inp["indices"][t]), torch.from_numpy(inp["tables"][t]).double(),
            torch.from_numpy(inp["offsets"][t]), mode="sum").numpy()
        np.testing.assert_allclose(e[:, t, :], ref, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- bag modes

MODES = [("sum", oracle.BAG_SUM), ("mean", oracle.BAG_MEAN), ("max", oracle.BAG_MAX)]


def _variable_bags(rng, k, b, v, max_len, empty_every=7):
    """(K, N) indices and (K, B) offsets of bags of random lengths in [0, max_len],
    with every `empty_every`-th bag empty. All tables share N, so the last bag
    of a table with fewer indices runs on to N (include_last_offset = false)."""
    lens = rng.integers(1, max_len + 1, size=(k, b))
    lens[:, ::empty_every] = 0
    n = int(lens.sum(axis=1).max())
    idx = rng.integers(0, v, size=(k, n)).astype(np.int64)
    off = np.zeros((k, b), np.int64)
    for t in range(k):
        off[t, 1:] = np.cumsum(lens[t])[:-1]
    return idx, off, lens


def test_bag_modes_hand_fixture(oracle_lib):
    """Sum, mean and max over general offsets, worked by hand (tests/golden)."""
    g = _golden("hand_bag_modes.json")
    table = _arr(g["table"], np.float32)
    for case in g["cases"]:
        idx = _arr([case["indices"]], np.int64)
        off = _arr([case["offsets"]], np.int64)
        for name, mode in MODES:
            e, flags = oracle.embedding_bag([table], idx, off, mode, lib=oracle_lib)
            np.testing.assert_array_equal(e[:, 0, :], _arr(case[name], np.float64))
            assert flags == case["flags"], (name, flags)


@pytest.mark.parametrize("name,mode", MODES)
def test_bag_modes_match_torch_embedding_bag(oracle_lib, name, mode):
    """Library cross-check: torch.nn.functional.embedding_bag(mode=...) in float64 on
    bags of random lengths 0..9 over general offsets (the last bag runs to N)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(41)
    k, b, v, d = 3, 50, 300, 12
    tables = [rng.uniform(-1, 1, (v, d)).astype(np.float32) for _ in range(k)]
    idx, off, _ = _variable_bags(rng, k, b, v, 9)
    e, flags = oracle.embedding_bag(tables, idx, off, mode, lib=oracle_lib)
    assert flags == 0
    for t in range(k):
        ref = torch.nn.functional.embedding_bag(
            torch.from_numpy(idx[t]), torch.from_numpy(tables[t]).double(),
            torch.from_numpy(off[t]), mode=name).numpy()
        if mode == oracle.BAG_MAX:
            np.testing.assert_array_equal(e[:, t, :], ref)
        else:
            np.testing.assert_allclose(e[:, t, :], ref, rtol=1e-13, atol=1e-15)


def test_bag_modes_selection_matrix_brute_force(oracle_lib):
    """Brute force on tiny inputs in matrix form: with S[b, n] = 1 when index n lies
    in bag b and G = table[indices], sum = S G, mean = S G / |bag|, max = the column
    max of G over the rows S selects; empty bags are zeros."""
    rng = np.random.default_rng(5)
    v, d, b = 40, 6, 9
    table = rng.uniform(-2, 2, (v, d)).astype(np.float32)
    idx, off, _ = _variable_bags(rng, 1, b, v, 6, empty_every=4)
    n = idx.shape[1]
    ends = np.append(off[0, 1:], n)
    sel = np.zeros((b, n))
    for bb in range(b):
        sel[bb, off[0, bb]:ends[bb]] = 1.0
    g = table[idx[0]].astype(np.float64)
    count = sel.sum(axis=1)
    want_sum = sel @ g
    want_mean = np.where(count[:, None] > 0, want_sum / np.maximum(count, 1)[:, None], 0.0)
    masked = np.where(sel[:, :, None] > 0, g[None, :, :], -np.inf)
    want_max = np.where(count[:, None] > 0, masked.max(axis=1), 0.0)
    for (name, mode), want in zip(MODES, (want_sum, want_mean, want_max)):
        e, _ = oracle.embedding_bag([table], idx, off, mode, lib=oracle_lib)
        if mode == oracle.BAG_MAX:
            np.testing.assert_array_equal(e[:, 0, :], want)
        else:
            np.testing.assert_allclose(e[:, 0, :], want, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("name,mode", MODES)
def test_bag_modes_permutation_invariant(oracle_lib, name, mode):
    """Permuting indices inside each bag leaves every mode unchanged: max exactly,
    sum and mean within 1 ulp once rounded to fp32."""
    rng = np.random.default_rng(17)
    k, b, v, d = 2, 40, 500, 8
    tables = [rng.uniform(-1, 1, (v, d)).astype(np.float32) for _ in range(k)]
    idx, off, lens = _variable_bags(rng, k, b, v, 12)
    base, _ = oracle.embedding_bag(tables, idx, off, mode, lib=oracle_lib)
    perm = idx.copy()
    for t in range(k):
        for bb in range(b):
            lo = off[t, bb]
            hi = off[t, bb + 1] if bb + 1 < b else idx.shape[1]
            perm[t, lo:hi] = perm[t, lo:hi][rng.permutation(hi - lo)]
    assert not np.array_equal(perm, idx)
    got, _ = oracle.embedding_bag(tables, perm, off, mode, lib=oracle_lib)
    if mode == oracle.BAG_MAX:
        np.testing.assert_array_equal(got, base)
    else:
        b32, g32 = base.astype(np.float32), got.astype(np.float32)
        ulp = np.spacing(np.maximum(np.abs(b32), np.abs(g32)))
        assert np.all(np.abs(g32 - b32) <= ulp)


def test_bag_weighted_sum_and_padding_match_torch(oracle_lib):
    """Library cross-check of per_sample_weights (sum) and padding_idx (all modes):
    torch.nn.functional.embedding_bag in float64 over general offsets."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(23)
    k, b, v, d = 2, 40, 60, 7
    tables = [rng.uniform(-1, 1, (v, d)).astype(np.float32) for _ in range(k)]
    idx, off, _ = _variable_bags(rng, k, b, v, 8)
    idx[:, ::5] = 3                         # plenty of the padding row
    w = rng.uniform(-2, 2, idx.shape).astype(np.float32)
    e, flags = oracle.embedding_bag(tables, idx, off, oracle.BAG_SUM, per_sample_weights=w,
                                    lib=oracle_lib)
    assert flags == 0
    for t in range(k):
        ref = torch.nn.functional.embedding_bag(
            torch.from_numpy(idx[t]), torch.from_numpy(tables[t]).double(),
            torch.from_numpy(off[t]), mode="sum",
            per_sample_weights=torch.from_numpy(w[t]).double()).numpy()
        np.testing.assert_allclose(e[:, t, :], ref, rtol=1e-13, atol=1e-14)
    for name, mode in MODES:
        e, _ = oracle.embedding_bag(tables, idx, off, mode, padding_idx=3, lib=oracle_lib)
        for t in range(k):
            ref = torch.nn.functional.embedding_bag(
                torch.from_numpy(idx[t]), torch.from_numpy(tables[t]).double(),
                torch.from_numpy(off[t]), mode=name, padding_idx=3).numpy()
            if mode == oracle.BAG_MAX:
                np.testing.assert_array_equal(e[:, t, :], ref)
            else:
                np.testing.assert_allclose(e[:, t, :], ref, rtol=1e-13, atol=1e-14)


def test_bag_weighted_sum_selection_matrix(oracle_lib):
    """Brute force: the weighted sum is S diag(w) G; padding rows drop out of S."""
    rng = np.random.default_rng(8)
    v, d, b = 30, 5, 8
    table = rng.uniform(-1, 1, (v, d)).astype(np.float32)
    idx, off, _ = _variable_bags(rng, 1, b, v, 5, empty_every=3)
    idx[0, 1::4] = 0
    n = idx.shape[1]
    w = rng.uniform(-1, 1, (1, n)).astype(np.float32)
    ends = np.append(off[0, 1:], n)
    sel = np.zeros((b, n))
    for bb in range(b):
        sel[bb, off[0, bb]:ends[bb]] = 1.0
    sel[:, idx[0] == 0] = 0.0                 # padding_idx = 0
    want = sel @ (w[0][:, None].astype(np.float64) * table[idx[0]].astype(np.float64))
    e, _ = oracle.embedding_bag([table], idx, off, oracle.BAG_SUM, per_sample_weights=w,
                                padding_idx=0, lib=oracle_lib)
    np.testing.assert_allclose(e[:, 0, :], want, rtol=1e-13, atol=1e-14)


def test_bag_padding_hand_case(oracle_lib):
    """Hand-worked: padding rows leave the bag without a flag; mean counts the rest."""
    g = _golden("hand_bag_modes.json")
    table = _arr(g["table"], np.float32)
    idx = _arr([[2, 0, 4, 1, 0, 0, 2]], np.int64)
    off = _arr([[0, 2, 4, 6]], np.int64)     # bags {2,0}, {4,1}, {0,0}, {2}
    e, flags = oracle.embedding_bag([table], idx, off, oracle.BAG_MEAN, padding_idx=0,
                                    lib=oracle_lib)
    assert flags == 0
    np.testing.assert_array_equal(e[:, 0, :], [[5, 0], [-0.5, 3], [0, 0], [5, 0]])
    w = _arr([[2, 10, 0.5, -1, 3, 3, 1]], np.float32)
    e, _ = oracle.embedding_bag([table], idx, off, oracle.BAG_SUM, per_sample_weights=w,
                                padding_idx=0, lib=oracle_lib)
    np.testing.assert_array_equal(e[:, 0, :], [[10, 0], [4, -3], [0, 0], [5, 0]])
    with pytest.raises(oracle.OracleError):
        oracle.embedding_bag([table], idx, off, oracle.BAG_MAX, per_sample_weights=w,
                             lib=oracle_lib)


def test_bag_mean_of_one_repeated_row_is_that_row(oracle_lib):
    """Closed form: the mean of L copies of row r is row r, exactly."""
    rng = np.random.default_rng(2)
    table = rng.uniform(-1, 1, (30, 5)).astype(np.float32)
    rows = np.array([3, 17, 0, 29])
    lens = np.array([1, 7, 20, 3])
    idx = np.repeat(rows, lens)[None, :].astype(np.int64)
    off = np.concatenate([[0], np.cumsum(lens)[:-1]])[None, :].astype(np.int64)
    e, _ = oracle.embedding_bag([table], idx, off, oracle.BAG_MEAN, lib=oracle_lib)
    np.testing.assert_array_equal(e[:, 0, :], table[rows].astype(np.float64))


# ---------------------------------------------------------------- interaction

@pytest.mark.parametrize("k,d", [(1, 8), (3, 16), (8, 5), (32, 64), (26, 128)])
def test_interaction_is_lower_triangle_of_gram(oracle_lib, k, d):
    """z equals the strict lower triangle of Z Z^T read row-major, and R = [x, z].

    Luminal compare modal_ci_ready...vanilla-pytorch, commit message: the
    interaction is Z[:, li, lj] over bmm(cat(...), permute(..., [0,2,1])).
    """
    rng = np.random.default_rng(k * 1000 + d)
    b = 9
    x = rng.standard_normal((b, d))
    e = rng.standard_normal((b, k, d))
    r = oracle.interaction(x, e, lib=oracle_lib)
    z_stack = np.concatenate([x[:, None, :], e], axis=1)           # (B, F, D)
    gram = np.matmul(z_stack, np.transpose(z_stack, (0, 2, 1)))    # (B, F, F)
    li, lj = np.tril_indices(k + 1, -1)
    np.testing.assert_allclose(r[:, d:], gram[:, li, lj], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(r[:, :d], x)


def test_interaction_hand_fixture(oracle_lib):
    g = _golden("hand_interaction_f4.json")
    r = oracle.interaction(_arr(g["x"], np.float64), _arr(g["emb"], np.float64), lib=oracle_lib)
    np.testing.assert_array_equal(r, _arr(g["expected_R"], np.float64))
    ei, ej = oracle.pair_enumerate(4, oracle_lib)
    assert [list(p) for p in zip(ei.tolist(), ej.tolist())] == g["expected_pairs"]


# ---------------------------------------------------------------- linear

@pytest.mark.parametrize("act", [oracle.ACT_NONE, oracle.ACT_RELU, oracle.ACT_SIGMOID])
def test_linear_matches_matmul(oracle_lib, act):
    """y = act(x W^T + b) against numpy matmul; W is (out, in) as in nn.Linear."""
    rng = np.random.default_rng(act)
    x = rng.standard_normal((37, 19))
    w = rng.standard_normal((11, 19)).astype(np.float32)
    b = rng.standard_normal(11).astype(np.float32)
    y = oracle.linear(x, w, b, act, lib=oracle_lib)
    a = x @ w.astype(np.float64).T + b.astype(np.float64)
    ref = {oracle.ACT_NONE: a, oracle.ACT_RELU: np.maximum(a, 0.0),
           oracle.ACT_SIGMOID: 1.0 / (1.0 + np.exp(-a))}[act]
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    y0 = oracle.linear(x, w, None, act, lib=oracle_lib)
    a0 = x @ w.astype(np.float64).T
    ref0 = {oracle.ACT_NONE: a0, oracle.ACT_RELU: np.maximum(a0, 0.0),
            oracle.ACT_SIGMOID: 1.0 / (1.0 + np.exp(-a0))}[act]
    np.testing.assert_allclose(y0, ref0, rtol=1e-12, atol=1e-12)


def test_linear_non_square_orientation(oracle_lib):
    """A transposed weight would not even match shapes; check one element by hand."""
    x = np.array([[1.0, 2.0, 3.0]])
    w = np.array([[1, 0, 0], [0, 0, 10]], np.float32)    # out 2, in 3
    y = oracle.linear(x, w, np.array([0.5, -1], np.float32), oracle.ACT_NONE, lib=oracle_lib)
    np.testing.assert_array_equal(y, [[1.5, 29.0]])


# ---------------------------------------------------------------- forward

def _golden_inputs(g):
    return dict(
        dense=_arr(g["dense"], np.float32),
        tables=[_arr(t, np.float32) for t in g["tables"]],
        indices=_arr(g["indices"], np.int64), offsets=_arr(g["offsets"], np.int64),
        bot_w=[_arr(w, np.float32) for w in g["bot_w"]],
        bot_b=[_arr(v, np.float32) for v in g["bot_b"]],
        top_w=[_arr(w, np.float32) for w in g["top_w"]],
        top_b=[_arr(v, np.float32) for v in g["top_b"]])


def test_forward_hand_fixture(oracle_lib):
    """Hand-computed forward: ReLU after the last bottom layer, bag sums, pair
    order, concat position, top ReLU and final sigmoid all matter here."""
    g = _golden("hand_forward_f3.json")
    inp = _golden_inputs(g)
    out = oracle.forward(inp, lib=oracle_lib)
    np.testing.assert_allclose(out, g["expected_out"], rtol=0, atol=1e-15)
    x = oracle.linear(inp["dense"], inp["bot_w"][0], inp["bot_b"][0], oracle.ACT_RELU,
                      lib=oracle_lib)
    np.testing.assert_array_equal(x, g["expected_x"])
    e = oracle.embedding_bag_sum(inp["tables"], inp["indices"], inp["offsets"], lib=oracle_lib)
    np.testing.assert_array_equal(e, g["expected_bags"])
    np.testing.assert_array_equal(oracle.interaction(x, e, lib=oracle_lib), g["expected_R"])


def test_forward_sample_subset_matches_full(oracle_lib):
    cfg = synth.get_config("tiny_b64_k3")
    inp = synth.make_inputs(cfg, seed=5)
    full = oracle.forward(inp, lib=oracle_lib)
    ids = np.array([63, 0, 17, 17, 40])
    np.testing.assert_array_equal(oracle.forward(inp, sample_ids=ids, lib=oracle_lib), full[ids])
    # single-threaded gives the same bits (no reduction is split across threads)
    np.testing.assert_array_equal(oracle.forward(inp, threads=1, lib=oracle_lib), full)


def test_forward_zero_last_top_layer_is_sigmoid_of_bias(oracle_lib):
    """All-zero last top weights: out = sigmoid(b_last) for every sample; sigmoid(0) = 0.5."""
    cfg = synth.get_config("tiny_b64_k3")
    inp = synth.make_inputs(cfg, seed=9)
    inp["top_w"][-1] = np.zeros_like(inp["top_w"][-1])
    b_last = float(inp["top_b"][-1][0])
    out = oracle.forward(inp, lib=oracle_lib)
    np.testing.assert_allclose(out, 1.0 / (1.0 + math.exp(-b_last)), rtol=0, atol=1e-16)
    inp["top_b"][-1] = np.zeros_like(inp["top_b"][-1])
    np.testing.assert_array_equal(oracle.forward(inp, lib=oracle_lib), 0.5)


def test_forward_selectors_pin_concat_and_pairs(oracle_lib):
    """Identity bottom MLP and a one-hot single-layer top MLP read single entries of R.

    With W_bot = I, b_bot = 0 and dense >= 0, x = dense. A top layer whose
    weight is the unit vector e_c gives out = sigmoid(R[c]): c < D reads x[c],
    c = D + p reads the dot of pair p = (i, j), checked against numpy.
    """
    d, k, b = 4, 3, 16
    f = k + 1
    p_count = f * (f - 1) // 2
    rng = np.random.default_rng(1)
    dense = np.abs(rng.standard_normal((b, d))).astype(np.float32)
    tables = [rng.uniform(-1, 1, (50, d)).astype(np.float32) for _ in range(k)]
    idx = rng.integers(0, 50, (k, b * 2)).astype(np.int64)
    off = np.ascontiguousarray(np.broadcast_to(np.arange(b) * 2, (k, b))).astype(np.int64)
    bags = np.stack([np.take(tables[t], idx[t].reshape(b, 2), axis=0).astype(np.float64).sum(1)
                     for t in range(k)], axis=1)                          # (B, K, D)
    feats = np.concatenate([dense.astype(np.float64)[:, None, :], bags], axis=1)
    li, lj = np.tril_indices(f, -1)
    for c in range(d + p_count):
        w = np.zeros((1, d + p_count), np.float32)
        w[0, c] = 1.0
        inp = dict(dense=dense, tables=tables, indices=idx, offsets=off,
                   bot_w=[np.eye(d, dtype=np.float32)], bot_b=[np.zeros(d, np.float32)],
                   top_w=[w], top_b=[np.zeros(1, np.float32)])
        out = oracle.forward(inp, lib=oracle_lib)
        if c < d:
            val = dense[:, c].astype(np.float64)
        else:
            p = c - d
            val = np.einsum("bd,bd->b", feats[:, li[p]], feats[:, lj[p]])
        np.testing.assert_allclose(out, 1.0 / (1.0 + np.exp(-val)), rtol=1e-13, atol=1e-15)


def test_forward_matches_torch_modules(oracle_lib):
    """Library cross-check on the tiny workload: torch CPU float64 built from
    nn.functional.embedding_bag, linear, bmm and tril_indices."""
    torch = pytest.importorskip("torch")
    cfg = synth.get_config("tiny_b64_k3")
    inp = synth.make_inputs(cfg, seed=21)
    t64 = lambda a: torch.from_numpy(np.asarray(a)).double()
    h = t64(inp["dense"])
    for w, bb in zip(inp["bot_w"], inp["bot_b"]):
        h = torch.relu(torch.nn.functional.linear(h, t64(w), t64(bb)))
    embs = [torch.nn.functional.embedding_bag(torch.from_numpy(inp["indices"][t]),
                                              t64(inp["tables"][t]),
                                              torch.from_numpy(inp["offsets"][t]), mode="sum")
            for t in range(cfg.n_tables)]
    z = torch.stack([h] + embs, dim=1)
    gram = torch.bmm(z, z.transpose(1, 2))
    li, lj = torch.tril_indices(cfg.n_features, cfg.n_features, -1)
    r = torch.cat([h, gram[:, li, lj]], dim=1)
    for l, (w, bb) in enumerate(zip(inp["top_w"], inp["top_b"])):
        r = torch.nn.functional.linear(r, t64(w), t64(bb))
        r = torch.sigmoid(r) if l == len(inp["top_w"]) - 1 else torch.relu(r)
    out = oracle.forward(inp, lib=oracle_lib)
    np.testing.assert_allclose(out, r[:, 0].numpy(), rtol=1e-12, atol=1e-14)


def test_forward_rejects_inconsistent_shapes(oracle_lib):
    """validate(): ln_top[0] must be D + P and ln_top[-1] must be 1."""
    g = _golden("hand_forward_f3.json")
    inp = _golden_inputs(g)
    inp["top_w"][0] = np.zeros((2, 6), np.float32)     # 6 != D + P = 5
    with pytest.raises(oracle.OracleError):
        oracle.forward(inp, lib=oracle_lib)


# ---------------------------------------------------------------- generator

def test_generator_splitmix_reference_value():
    """SplitMix64 started at state 0 yields 0xE220A8397B1DCDAF first (Steele, Lea and
    Flood, OOPSLA 2014, reference implementation); streams are deterministic."""
    assert synth.raw(0, 0) == 0xE220A8397B1DCDAF
    a = [synth.element(1234, 5, i) for i in range(4)]
    assert len(set(a)) == 4 and a == [synth.element(1234, 5, i) for i in range(4)]
    assert synth.element(1234, 6, 0) != a[0] and synth.element(1235, 5, 0) != a[0]


def test_generator_distributions():
    u = synth.fill_uniform(np.empty(1 << 18, np.float32), 1, 2, -0.01, 0.01)
    assert u.min() >= -0.01 and u.max() <= 0.01 and abs(u.mean()) < 1e-4
    n = synth.fill_normal(np.empty(1 << 18, np.float32), 1, 3)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1) < 0.01
    z = synth.fill_index_zipf(np.empty(1 << 18, np.int64), 1, 4, 1_000_000, 1.05)
    ranks = np.arange(1, 1_000_001, dtype=np.float64)
    w = ranks ** -1.05
    head = w[:10_000].sum() / w.sum()
    assert abs((z < 10_000).mean() - head) < 0.005
    assert z.min() >= 0 and z.max() < 1_000_000


def test_generator_variable_bags_structure():
    """The general-offsets input recipe: table 0's lengths uniform on 0..max_len,
    every table the same lengths in its own order (the same N indices, no
    remainder bag), offsets the running sum from 0, indices inside each table,
    and the bench's 0..40 mixture averaging 20 rows with empty bags present."""
    cfg = synth.DlrmConfig("vb", 20000, (13, 8), (1000, 50, 7), 8, 1, (8 + 6,), 0.05)
    idx, off, lens = synth.make_variable_bags(cfg, seed=3, max_len=40)
    k, b = 3, 20000
    assert lens.shape == off.shape == (k, b) and idx.shape == (k, int(lens[0].sum()))
    for t in range(k):
        assert sorted(lens[t]) == sorted(lens[0])
        assert off[t, 0] == 0 and np.array_equal(np.diff(off[t]), lens[t, :-1])
        assert off[t, -1] + lens[t, -1] == idx.shape[1]
        assert idx[t].min() >= 0 and idx[t].max() < cfg.rows[t]
    assert not np.array_equal(lens[1], lens[0])         # a different order per table
    assert lens.min() == 0 and lens.max() == 40
    assert abs(lens[0].mean() - 20.0) < 0.3
    counts = np.bincount(lens[0], minlength=41)
    assert counts.min() > 0.8 * b / 41                  # every length 0..40 drawn evenly
    again = synth.make_variable_bags(cfg, seed=3, max_len=40)
    assert all(np.array_equal(x, y) for x, y in zip((idx, off, lens), again))


def test_generator_bag_weights():
    w = synth.make_bag_weights((2, 1 << 16), seed=5)
    assert w.dtype == np.float32 and w.min() >= -2.0 and w.max() < 2.0
    assert abs(w.mean()) < 0.02 and not np.array_equal(w[0], w[1])
    assert np.array_equal(w, synth.make_bag_weights((2, 1 << 16), seed=5))


def _splitmix64_output(state: int, i: int) -> int:
    """Output i of SplitMix64 from `state`, written from the published
    definition (Steele, Lea and Flood, OOPSLA 2014; the splitmix64.c finaliser)."""
    m = (1 << 64) - 1
    z = (state + (i + 1) * 0x9E3779B97F4A7C15) & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def test_generator_streams_follow_their_stated_recipe():
    """Every stream is a SplitMix64 sequence, and each distribution maps its
    elements as the recipe states: uniform floats lo + (hi - lo) * top24 / 2^24,
    uniform indices floor(top32 * V / 2^32), Zipf by the first CDF entry above
    top53 / 2^53. Checked element by element against a pure-Python restatement."""
    for i in (0, 1, 2, 7, 1000):
        assert synth.raw(12345, i) == _splitmix64_output(12345, i)
    seed, stream, n = 77, 3, 64
    e = [synth.element(seed, stream, i) for i in range(n)]
    u = synth.fill_uniform(np.empty(n, np.float32), seed, stream, -0.5, 1.5)
    assert np.array_equal(u, np.array([np.float32(-0.5 + 2.0 * ((x >> 40) / 2.0 ** 24)) for x in e]))
    v = 1_000_003
    idx = synth.fill_index_uniform(np.empty(n, np.int64), seed, stream, v)
    assert np.array_equal(idx, np.array([((x >> 32) * v) >> 32 for x in e]))
    cdf = synth.zipf_cdf(1000, 1.05)
    z = synth.fill_index_zipf(np.empty(n, np.int64), seed, stream, 1000, 1.05)
    assert np.array_equal(z, np.array([int(np.argmax(cdf > (x >> 11) / 2.0 ** 53)) for x in e]))
