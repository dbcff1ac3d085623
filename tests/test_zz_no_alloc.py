"""dlrm_forward_noalloc: the forward for callers that cannot allocate device
memory when they run it (a plug-in whose host framework owns the GPU's
memory, a serving loop that must not take cudaMalloc's device-wide sync, a
fixed memory budget). It uses a fixed scratch array inside the library.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test. It passes alone in a fresh process
and after the rest of the suite.
"""
import numpy as np
import pytest

import dlrm_synth as synth

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


def _cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_noalloc_forward_matches_handle_forward_twice_in_a_row():
    cfg = synth.get_config("b2048_k3")
    inp = synth.make_inputs(cfg, seed=4321)
    tables = [_cu(t) for t in inp["tables"]]
    bw, bb = [_cu(w) for w in inp["bot_w"]], [_cu(v) for v in inp["bot_b"]]
    tw, tb = [_cu(w) for w in inp["top_w"]], [_cu(v) for v in inp["top_b"]]
    dense, idx, off = _cu(inp["dense"]), _cu(inp["indices"]), _cu(inp["offsets"])

    model = dl.DlrmModel(cfg.ln_bot, cfg.ln_top, tables, bw, bb, tw, tb, cfg.bag_size,
                         cfg.batch)
    ref = model.forward(dense, idx, off)
    assert model.error() == dl.OK
    ref = ref.cpu().numpy()
    model.close()

    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full((cfg.batch,), float("nan"), device="cuda")
        dl.dlrm_forward_noalloc(cfg.ln_bot, cfg.ln_top, tables, bw, bb, tw, tb, cfg.bag_size,
                                dense, idx, off, out, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, call
        np.testing.assert_allclose(out.cpu().numpy(), ref, atol=ATOL, rtol=RTOL)


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
