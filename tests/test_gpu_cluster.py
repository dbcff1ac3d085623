"""The cluster-split fused forward (small batches of the fp32 fused plan)
against the CPU oracle.

Each layer's output columns are split over the CTAs of a cluster (8 up to
32 samples, 4 above) and the outputs exchanged through distributed shared
memory; the interaction and the
sigmoid layer are split by samples. The cases cover every tile height (4, 8
and 16 samples), partial tiles, one and several waves of clusters, column
slices from 4 to 512 wide (layers of 16 to 1024 outputs), padded input
widths, bags of one row (fetched at kernel start) and of several rows
(summed at the interaction), and the device flags. Tolerance: the fp32 bar,
|gpu - oracle| <= 1e-5 + 1e-4 |oracle|.
"""
import numpy as np
import pytest

import dlrm_synth as synth
import oracle

torch = pytest.importorskip("torch")
import dlrm_embedding_interaction_gb300 as dl  # noqa: E402

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-5, 1e-4


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


def close(gpu, ref):
    np.testing.assert_allclose(np.asarray(gpu, dtype=np.float64), ref, atol=ATOL, rtol=RTOL)


def make_model(cfg, inp, max_batch=None, path=dl.PATH_FUSED):
    return dl.DlrmModel(cfg.ln_bot, cfg.ln_top, [cu(t) for t in inp["tables"]],
                        [cu(w) for w in inp["bot_w"]], [cu(v) for v in inp["bot_b"]],
                        [cu(w) for w in inp["top_w"]], [cu(v) for v in inp["top_b"]],
                        cfg.bag_size, max_batch or cfg.batch, dl.MATH_FP32, path)


def forward(model, inp, batch):
    out = torch.full((batch,), float("nan"), device="cuda")
    model.forward(cu(inp["dense"]), cu(inp["indices"]), cu(inp["offsets"]), out)
    return out, model.error()


def test_default_limit_and_switch():
    """fp32 fused handles of models with 1 MiB or more of weights get a cluster
    plan (a positive default limit); limit 0 and -1 switch it off and back;
    layer-wise handles and the 20 KB tiny model have none."""
    cfg = synth.sweep_config(64, 3)
    inp = synth.make_inputs(cfg, seed=5)
    model = make_model(cfg, inp)
    default = model.cluster_batch_limit
    assert default == 256
    assert model.kernels(cfg.batch) == dl.KERNELS_FUSED_CLUSTER
    model.cluster_batch_limit = 0
    assert model.cluster_batch_limit == 0
    assert model.kernels(cfg.batch) == dl.KERNELS_FUSED
    a, st = forward(model, inp, cfg.batch)           # the persistent kernel
    assert st == dl.OK
    model.cluster_batch_limit = -1
    assert model.cluster_batch_limit == default
    b, st = forward(model, inp, cfg.batch)           # the cluster kernel
    assert st == dl.OK
    ref = oracle.forward(inp)
    close(a.cpu().numpy(), ref)
    close(b.cpu().numpy(), ref)
    model.close()
    lw = make_model(cfg, inp, path=dl.PATH_LAYERWISE)
    assert lw.cluster_batch_limit == 0
    with pytest.raises(dl.DlrmError) as e:
        lw.cluster_batch_limit = 16
    assert e.value.status == dl.ERR_UNSUPPORTED
    lw.cluster_batch_limit = 0                       # off is always accepted
    with pytest.raises(dl.DlrmError) as e:
        lw.cluster_batch_limit = -2
    assert e.value.status == dl.ERR_INVALID_ARG
    lw.close()
    tiny = synth.get_config("tiny_b64_k3")
    tin = synth.make_inputs(tiny, seed=5)
    small = make_model(tiny, tin)
    assert small.cluster_batch_limit == 0
    small.close()


SWEEP = [(b, k) for k in (1, 3, 8, 16, 32) for b in (1, 3, 8, 29, 64, 128, 256)]


@pytest.mark.parametrize("b,k", SWEEP, ids=[f"b{b}_k{k}" for b, k in SWEEP])
def test_sweep_cells_match_oracle(b, k):
    """The sweep's small cells (bottom 13-512-256-64, top 512-256-1) at the
    default limit: clusters of 8 CTAs up to 32 samples, of 4 above."""
    cfg = synth.sweep_config(b, k)
    inp = synth.make_inputs(cfg, seed=100 + b + k)
    model = make_model(cfg, inp)
    assert model.cluster_batch_limit == 256
    out, st = forward(model, inp, b)
    assert st == dl.OK
    close(out.cpu().numpy(), oracle.forward(inp))
    model.close()


@pytest.mark.parametrize("batch", [1, 4, 5, 17, 33, 61, 100, 255, 700])
def test_tile_heights_and_waves(batch):
    """With the limit raised every batch takes the cluster kernel: clusters of
    8 and of 4 CTAs, tiles of 4, 8 and 16 samples, partial last tiles, and
    more tiles than one wave of clusters holds (700 samples)."""
    cfg = synth.sweep_config(batch, 3)
    inp = synth.make_inputs(cfg, seed=batch)
    model = make_model(cfg, inp, max_batch=1024)
    model.cluster_batch_limit = 1024
    out, st = forward(model, inp, batch)
    assert st == dl.OK
    close(out.cpu().numpy(), oracle.forward(inp))
    model.close()


def test_odd_and_wide_layers():
    """Layers of 1024, 600, 100, 24 and 16 outputs (column slices of 128, 128,
    16, 4 and 4 per CTA) and inputs that are not multiples of 4."""
    cfg = synth.DlrmConfig("odd_cluster", 37, (13, 1024, 600, 24), (300, 500, 700), 24, 1,
                           (24 + 6, 100, 16, 1), table_range=0.05)
    inp = synth.make_inputs(cfg, seed=8)
    model = make_model(cfg, inp)
    out, st = forward(model, inp, cfg.batch)
    assert st == dl.OK
    close(out.cpu().numpy(), oracle.forward(inp))
    model.close()


@pytest.mark.parametrize("batch", [20, 48])
def test_long_bags(batch):
    """Bags of 20 rows (the 26-table model's shape, small tables): summed at
    the interaction by the CTA that owns each sample (clusters of 8 CTAs at
    20 samples, of 4 at 48)."""
    base = synth.get_config("b65536_k26_zipf")
    cfg = synth.DlrmConfig(f"b{batch}_k26_l20", batch, base.ln_bot, (5000,) * 26, base.emb_dim,
                           20, base.ln_top, index_dist="zipf", zipf_s=1.05)
    inp = synth.make_inputs(cfg, seed=12)
    model = make_model(cfg, inp)
    assert model.path == dl.PATH_FUSED
    assert model.kernels(cfg.batch) == dl.KERNELS_FUSED_CLUSTER
    out, st = forward(model, inp, cfg.batch)
    assert st == dl.OK
    close(out.cpu().numpy(), oracle.forward(inp))
    model.close()


def test_flags_bad_index_and_offsets():
    """An index out of range and a bag start other than b * L are flagged;
    the bag contributes zeros; every other sample is the oracle's."""
    cfg = synth.sweep_config(40, 3)
    inp = synth.make_inputs(cfg, seed=31)
    model = make_model(cfg, inp)
    bad = dict(inp)
    bad["indices"] = inp["indices"].copy()
    bad["indices"][2, 13] = cfg.rows[2] + 5            # sample 13, table 2
    out = torch.empty(cfg.batch, device="cuda")
    model.forward(cu(inp["dense"]), cu(bad["indices"]), cu(inp["offsets"]), out)
    assert model.error() == dl.ERR_INDEX_OOB
    got = out.cpu().numpy()
    keep = np.arange(cfg.batch) != 13
    close(got[keep], oracle.forward(inp)[keep])
    zeroed = dict(inp)
    zeroed["tables"] = list(inp["tables"])
    zeroed["tables"][2] = np.concatenate([inp["tables"][2],
                                          np.zeros((1, cfg.emb_dim), np.float32)])
    zeroed["indices"] = inp["indices"].copy()
    zeroed["indices"][2, 13] = cfg.rows[2]
    close(got[13:14], oracle.forward(zeroed, sample_ids=np.array([13])))
    off = inp["offsets"].copy()
    off[0, 7] = 3
    model.forward(cu(inp["dense"]), cu(inp["indices"]), cu(off), out)
    assert model.error() == dl.ERR_UNSUPPORTED
    model.close()


def test_graph_capture_and_replay():
    cfg = synth.sweep_config(64, 8)
    inp = synth.make_inputs(cfg, seed=9)
    model = make_model(cfg, inp)
    dense, idx, off = cu(inp["dense"]), cu(inp["indices"]), cu(inp["offsets"])
    out = torch.empty(cfg.batch, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        model.forward(dense, idx, off, out, stream=s)
    s.synchronize()
    ref = out.clone()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g, stream=s):
        model.forward(dense, idx, off, out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    torch.testing.assert_close(out, ref, rtol=0, atol=0)
    close(out.cpu().numpy(), oracle.forward(inp))
    model.close()
