"""dlrm_forward_noalloc: the forward for callers that cannot allocate device
memory when they run it (a plug-in whose host framework owns the GPU's
memory, a serving loop that must not take cudaMalloc's device-wide sync, a
fixed memory budget). It uses a fixed scratch array inside the library.

Checked against the CPU oracle at the fp32 tolerance, on three workload
shapes that fit the scratch, two calls in a row each; and the device's free
memory is the same before and after repeated calls (nothing allocated).

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test. It passes alone in a fresh process
and after the rest of the suite.
"""
import numpy as np
import pytest

import dlrm_synth as synth
import oracle

torch = pytest.importorskip("torch")
import dlrm_embedding_interaction_gb300 as dl  # noqa: E402

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-5, 1e-4
SHAPES = ["b2048_k3", "tiny_b64_k3", "sweep_b512_k8"]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    from dlrm_embedding_interaction_gb300 import build
    build.build()
    dl.lib()
    torch.cuda.set_device(0)


def _cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _config(name):
    if name.startswith("sweep_"):
        b, k = name[len("sweep_b"):].split("_k")
        return synth.sweep_config(int(b), int(k))
    return synth.get_config(name)


def _device_inputs(cfg, seed):
    inp = synth.make_inputs(cfg, seed=seed)
    dev = dict(tables=[_cu(t) for t in inp["tables"]],
               bw=[_cu(w) for w in inp["bot_w"]], bb=[_cu(v) for v in inp["bot_b"]],
               tw=[_cu(w) for w in inp["top_w"]], tb=[_cu(v) for v in inp["top_b"]],
               dense=_cu(inp["dense"]), idx=_cu(inp["indices"]), off=_cu(inp["offsets"]))
    return inp, dev


def _call(cfg, dev, out, err):
    dl.dlrm_forward_noalloc(cfg.ln_bot, cfg.ln_top, dev["tables"], dev["bw"], dev["bb"],
                            dev["tw"], dev["tb"], cfg.bag_size, dev["dense"], dev["idx"],
                            dev["off"], out, err_flag=err)


@pytest.mark.parametrize("name", SHAPES)
def test_noalloc_forward_matches_the_oracle_twice_in_a_row(name):
    cfg = _config(name)
    inp, dev = _device_inputs(cfg, seed=4321)
    ref = oracle.forward(inp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full((cfg.batch,), float("nan"), device="cuda")
        _call(cfg, dev, out, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, call
        got = out.cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(got, ref, atol=ATOL, rtol=RTOL, err_msg=f"call {call}")


def test_noalloc_forward_agrees_with_the_handle_forward():
    cfg = _config("b2048_k3")
    inp, dev = _device_inputs(cfg, seed=99)
    model = dl.DlrmModel(cfg.ln_bot, cfg.ln_top, dev["tables"], dev["bw"], dev["bb"], dev["tw"],
                         dev["tb"], cfg.bag_size, cfg.batch)
    ref = model.forward(dev["dense"], dev["idx"], dev["off"])
    assert model.error() == dl.OK
    ref = ref.cpu().numpy()
    model.close()
    out = torch.empty(cfg.batch, device="cuda")
    _call(cfg, dev, out, None)
    torch.cuda.synchronize()
    np.testing.assert_allclose(out.cpu().numpy(), ref, atol=ATOL, rtol=RTOL)


def test_noalloc_forward_allocates_no_device_memory():
    """Every shape once to load the kernels it uses, then the device's free
    memory (cudaMemGetInfo) before and after three more rounds of calls: equal.
    All tensors are made before the first reading."""
    runs = []
    for name in SHAPES:
        cfg = _config(name)
        _, dev = _device_inputs(cfg, seed=7)
        runs.append((cfg, dev, torch.empty(cfg.batch, device="cuda")))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for cfg, dev, out in runs:
        _call(cfg, dev, out, err)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        for cfg, dev, out in runs:
            _call(cfg, dev, out, err)
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert int(err.item()) == 0
    assert free_after == free_before


def test_noalloc_rejects_a_batch_beyond_the_scratch():
    cfg = synth.get_config("b2048_k3").with_batch(4096)    # ~20 MiB of scratch > 16 MiB
    inp = synth.make_inputs(cfg, seed=1)
    tables = [_cu(t) for t in inp["tables"]]
    out = torch.empty(cfg.batch, device="cuda")
    with pytest.raises(dl.DlrmError) as ei:
        dl.dlrm_forward_noalloc(cfg.ln_bot, cfg.ln_top, tables,
                                [_cu(w) for w in inp["bot_w"]], [_cu(v) for v in inp["bot_b"]],
                                [_cu(w) for w in inp["top_w"]], [_cu(v) for v in inp["top_b"]],
                                cfg.bag_size, _cu(inp["dense"]), _cu(inp["indices"]),
                                _cu(inp["offsets"]), out)
    assert ei.value.status == dl.ERR_UNSUPPORTED
