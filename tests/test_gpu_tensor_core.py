"""Opt-in tensor-core modes (tcgen05, TF32 / BF16 operands, fp32 accumulation)
against the fp64 oracle.

Tolerance of these modes: rel 2e-2. For a GEMM output, where single elements
can cancel to ~0, the bound is |gpu - ref| <= 2e-2 * (|ref| + rms(ref)) per
element; for the forward's sigmoid outputs it is 2e-2 * |ref|.
"""
import numpy as np
import pytest

import dlrm_synth as synth
import oracle

torch = pytest.importorskip("torch")
import dlrm_embedding_interaction_gb300 as dl  # noqa: E402

pytestmark = pytest.mark.gpu

MODES = [dl.MATH_TF32, dl.MATH_BF16]
MODE_IDS = ["tf32", "bf16"]
ALL_MODES = MODES + [dl.MATH_TF32X3]
ALL_IDS = MODE_IDS + ["tf32x3"]


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


def tc_close(got, ref, rel=2e-2):
    got = np.asarray(got, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(got - ref)
    bound = rel * (np.abs(ref) + rms)
    worst = np.argmax(err - bound) if err.size else 0
    assert np.all(err <= bound), (
        f"max excess {float((err - bound).flat[worst]):.3e} at {np.unravel_index(worst, err.shape)}: "
        f"got {got.flat[worst]:.6f} ref {ref.flat[worst]:.6f}")
    return float(np.max(err / (np.abs(ref) + rms))) if err.size else 0.0


LINEAR_CASES = [
    (1, 16, 1), (7, 16, 5), (128, 128, 32), (128, 128, 64), (300, 200, 70), (2048, 512, 13),
    (2048, 256, 512), (2048, 64, 256), (257, 1024, 479), (65, 17, 16), (129, 130, 131),
    (4096, 512, 592),
]


@pytest.mark.parametrize("mode", ALL_MODES, ids=ALL_IDS)
@pytest.mark.parametrize("m,n,k", LINEAR_CASES)
def test_linear_tensor_core_matches_oracle(m, n, k, mode):
    rng = np.random.default_rng(m * 7 + n * 11 + k * 13 + mode)
    x = rng.standard_normal((m, k)).astype(np.float32)
    bound = 1.0 / np.sqrt(k)
    w = rng.uniform(-bound, bound, (n, k)).astype(np.float32)
    b = rng.uniform(-bound, bound, n).astype(np.float32)
    y = torch.full((m, n), float("nan"), device="cuda")
    dl.linear_bias_act(cu(x), cu(w), cu(b), y, dl.ACT_NONE, mode)
    torch.cuda.synchronize()
    ref = oracle.linear(x, w, b, oracle.ACT_NONE)
    if mode == dl.MATH_TF32X3:     # fp32 parity tolerance
        np.testing.assert_allclose(y.cpu().numpy(), ref, atol=1e-5, rtol=1e-4)
        return
    worst = tc_close(y.cpu().numpy(), ref)
    if mode == dl.MATH_TF32:
        assert worst < 5e-3     # tf32 keeps 10 mantissa bits: far inside the bound


@pytest.mark.parametrize("mode", ALL_MODES, ids=ALL_IDS)
@pytest.mark.parametrize("act", [dl.ACT_RELU, dl.ACT_SIGMOID])
def test_linear_tensor_core_epilogue(mode, act):
    rng = np.random.default_rng(act)
    x = rng.standard_normal((333, 96)).astype(np.float32)
    w = rng.uniform(-0.1, 0.1, (160, 96)).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, 160).astype(np.float32)
    y = torch.empty((333, 160), device="cuda")
    dl.linear_bias_act(cu(x), cu(w), cu(b), y, act, mode)
    torch.cuda.synchronize()
    tc_close(y.cpu().numpy(), oracle.linear(x, w, b, act))


def test_linear_tensor_core_strided_rows_and_no_bias():
    rng = np.random.default_rng(5)
    xf = rng.standard_normal((200, 75)).astype(np.float32)
    w = rng.uniform(-0.1, 0.1, (48, 70)).astype(np.float32)
    y = torch.empty((200, 48), device="cuda")
    dl.linear_bias_act(cu(xf)[:, :70], cu(w), None, y, dl.ACT_NONE, dl.MATH_TF32)
    torch.cuda.synchronize()
    tc_close(y.cpu().numpy(), oracle.linear(xf[:, :70], w, None, oracle.ACT_NONE))


def _model(cfg, inp, mode, path):
    return dl.DlrmModel(cfg.ln_bot, cfg.ln_top, [cu(t) for t in inp["tables"]],
                        [cu(w) for w in inp["bot_w"]], [cu(v) for v in inp["bot_b"]],
                        [cu(w) for w in inp["top_w"]], [cu(v) for v in inp["top_b"]],
                        cfg.bag_size, cfg.batch, mode, path)


@pytest.mark.parametrize("mode", ALL_MODES, ids=ALL_IDS)
@pytest.mark.parametrize("path", [dl.PATH_LAYERWISE, dl.PATH_FUSED], ids=["layerwise", "fused"])
@pytest.mark.parametrize("name", ["tiny_b64_k3", "b2048_k3", "b2048_k32", "sweep_b33_k8",
                                  "sweep_b1_k1", "sweep_b300_k16"])
def test_forward_tensor_core_matches_oracle(name, path, mode):
    """Both plans of the tensor-core modes against the oracle. The fused plan
    takes models whose tile fits shared memory; TF32X3 is layer-wise only.
    Other requests must be refused with UNSUPPORTED."""
    cfg = synth.get_config(name)
    inp = synth.make_inputs(cfg, seed=1234)
    if path == dl.PATH_FUSED and mode == dl.MATH_TF32X3:
        with pytest.raises(dl.DlrmError) as ei:
            _model(cfg, inp, mode, path)
        assert ei.value.status == dl.ERR_UNSUPPORTED
        return
    try:
        model = _model(cfg, inp, mode, path)
    except dl.DlrmError as e:
        assert path == dl.PATH_FUSED and e.status == dl.ERR_UNSUPPORTED
        pytest.skip("model does not fit the fused tensor-core tile")
    assert model.path == path
    out = model.forward(cu(inp["dense"]), cu(inp["indices"]), cu(inp["offsets"]))
    assert model.error() == dl.OK
    ref = oracle.forward(inp)
    if mode == dl.MATH_TF32X3:     # fp32 parity tolerance
        np.testing.assert_allclose(out.cpu().numpy(), ref, atol=1e-5, rtol=1e-4)
    else:
        np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=2e-2, atol=0)
    model.close()


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_fused_tensor_core_is_auto_choice_and_flags_bad_indices(mode):
    cfg = synth.get_config("b2048_k3")
    inp = synth.make_inputs(cfg, seed=7)
    model = _model(cfg, inp, mode, dl.PATH_AUTO)
    assert model.path == dl.PATH_FUSED
    idx = inp["indices"].copy()
    idx[1, 100] = cfg.rows[1]            # one index past its table
    out = model.forward(cu(inp["dense"]), cu(idx), cu(inp["offsets"]))
    assert model.error() == dl.ERR_INDEX_OOB
    # the bag with the bad index contributes zeros (the oracle's definition)
    inp2 = dict(inp)
    inp2["indices"] = idx
    ref = oracle.forward(inp2, allow_oob=True)
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=2e-2, atol=0)
    model.close()


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_fused_tensor_core_bags_of_two_flag_bad_index_and_offsets(mode):
    """Bags of two rows (the 64-sample model): an index past its table adds
    nothing to its bag and raises INDEX_OOB; an offset off the uniform stride
    zeroes that bag and raises the offsets flag."""
    cfg = synth.get_config("tiny_b64_k3")
    assert cfg.bag_size == 2
    inp = synth.make_inputs(cfg, seed=21)
    model = _model(cfg, inp, mode, dl.PATH_FUSED)
    idx = inp["indices"].copy()
    idx[0, 2 * 5 + 1] = -3                 # second row of sample 5's bag in table 0
    out = model.forward(cu(inp["dense"]), cu(idx), cu(inp["offsets"]))
    assert model.error() == dl.ERR_INDEX_OOB
    inp2 = dict(inp)
    inp2["indices"] = idx
    np.testing.assert_allclose(out.cpu().numpy(), oracle.forward(inp2, allow_oob=True),
                               rtol=2e-2, atol=0)
    off = inp["offsets"].copy()
    off[1, 9] = 2 * 9 + 1
    out = model.forward(cu(inp["dense"]), cu(inp["indices"]), cu(off)).cpu().numpy()
    assert model.error() == dl.ERR_UNSUPPORTED
    keep = np.arange(cfg.batch) != 9
    np.testing.assert_allclose(out[keep], oracle.forward(inp)[keep], rtol=2e-2, atol=0)
    model.close()


def test_fused_plan_rejects_tf32x3():
    cfg = synth.get_config("b2048_k3")
    inp = synth.make_inputs(cfg, seed=1)
    with pytest.raises(dl.DlrmError) as ei:
        _model(cfg, inp, dl.MATH_TF32X3, dl.PATH_FUSED)
    assert ei.value.status == dl.ERR_UNSUPPORTED


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_fused_tensor_core_flags_non_uniform_offsets(mode):
    cfg = synth.get_config("b2048_k3")
    inp = synth.make_inputs(cfg, seed=9)
    model = _model(cfg, inp, mode, dl.PATH_FUSED)
    off = inp["offsets"].copy()
    off[2, 40] = 41
    out = model.forward(cu(inp["dense"]), cu(inp["indices"]), cu(off)).cpu().numpy()
    assert model.error() == dl.ERR_UNSUPPORTED
    keep = np.arange(cfg.batch) != 40
    np.testing.assert_allclose(out[keep], oracle.forward(inp)[keep], rtol=2e-2, atol=0)
    model.close()


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_fused_tensor_core_phase_trace_and_host_buffers(mode):
    """The fused tensor-core plan's phase stamps rise phase by phase, and the
    host-buffer call (pinned buffers used in place) equals the device call."""
    cfg = synth.get_config("sweep_b300_k3")
    inp = synth.make_inputs(cfg, seed=4)
    model = _model(cfg, inp, mode, dl.PATH_FUSED)
    buf = torch.zeros(((cfg.batch + 3) // 4) * dl.TRACE_SLOTS, dtype=torch.int64, device="cuda")
    rows = model.set_phase_trace(buf)
    assert rows == 16
    dev = model.forward(cu(inp["dense"]), cu(inp["indices"]), cu(inp["offsets"])).cpu().numpy()
    assert model.error() == dl.OK
    tiles = (cfg.batch + rows - 1) // rows
    t = buf.view(-1, dl.TRACE_SLOTS)[:tiles].cpu().numpy()
    n = len(model.phase_names())
    assert (t[:, :n + 1] > 0).all() and (np.diff(t[:, :n + 1], axis=1) >= 0).all()
    model.set_phase_trace(None)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    out = torch.full((cfg.batch,), -1.0).pin_memory()
    model.forward_host(pin(inp["dense"]), pin(inp["indices"]), pin(inp["offsets"]), out)
    assert model.error() == dl.OK
    np.testing.assert_array_equal(out.numpy(), dev)
    model.close()
