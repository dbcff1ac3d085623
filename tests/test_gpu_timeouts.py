"""Failure detection on the GPU: a bounded device wait that runs out.

Every wait of the library's kernels on another party (a weight stage or
tile landing, a ring slot being released, tensor-core work completing) is
bounded. Here the test hook dlrm_test_stall shortens that bound to 100 us
and makes each kernel withhold the last copy or tensor-core commit of its
stream, so that the wait on it cannot complete. Nothing faults, traps or
hangs: the launch returns, dlrm_get_error reports DLRM_ERR_TIMEOUT, and the
next normal forward on the same handle matches the oracle.

Covered: the fused fp32 kernel (one tile per CTA, and several tiles per CTA
on the persistent path), the cluster-split fp32 kernel of small batches
(weight stages and the exchanges between the cluster's CTAs), the fused
tensor-core kernel (BF16 and TF32), and
the layer-wise tensor-core GEMM (TF32X3 and BF16).
"""
import time

import numpy as np
import pytest

import dlrm_synth as synth
import oracle

torch = pytest.importorskip("torch")
import dlrm_embedding_interaction_gb300 as dl  # noqa: E402

pytestmark = pytest.mark.gpu

LIMIT_NS = 100_000        # 100 us: far above any wait of a healthy forward here


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


CASES = [
    # workload, math, path, tolerance (atol, rtol)
    ("b2048_k3", dl.MATH_FP32, dl.PATH_FUSED, (1e-5, 1e-4)),
    ("sweep_b8192_k3", dl.MATH_FP32, dl.PATH_FUSED, (1e-5, 1e-4)),   # several tiles per CTA
    ("sweep_b64_k3", dl.MATH_FP32, dl.PATH_FUSED, (1e-5, 1e-4)),     # cluster kernel, 4 CTAs
    ("sweep_b16_k3", dl.MATH_FP32, dl.PATH_FUSED, (1e-5, 1e-4)),     # cluster kernel, 8 CTAs
    ("b2048_k3", dl.MATH_BF16, dl.PATH_FUSED, (2e-2, 2e-2)),
    ("tiny_b64_k3", dl.MATH_TF32, dl.PATH_FUSED, (2e-2, 2e-2)),
    ("tiny_b64_k3", dl.MATH_TF32X3, dl.PATH_LAYERWISE, (1e-5, 1e-4)),
    ("b2048_k3", dl.MATH_BF16, dl.PATH_LAYERWISE, (2e-2, 2e-2)),
]
IDS = ["fp32-fused", "fp32-fused-persistent", "fp32-fused-cluster4", "fp32-fused-cluster8",
       "bf16-fused", "tf32-fused", "tf32x3-layerwise",
       "bf16-layerwise"]


@pytest.mark.parametrize("name,math,path,tol", CASES, ids=IDS)
def test_a_wait_that_runs_out_reports_timeout_and_the_handle_recovers(name, math, path, tol):
    cfg = synth.get_config(name)
    inp = synth.make_inputs(cfg, seed=77)
    model = dl.DlrmModel(cfg.ln_bot, cfg.ln_top, [cu(t) for t in inp["tables"]],
                         [cu(w) for w in inp["bot_w"]], [cu(v) for v in inp["bot_b"]],
                         [cu(w) for w in inp["top_w"]], [cu(v) for v in inp["top_b"]],
                         cfg.bag_size, cfg.batch, math, path)
    assert model.path == path
    dense, idx, off = cu(inp["dense"]), cu(inp["indices"]), cu(inp["offsets"])
    out = torch.empty(cfg.batch, device="cuda")

    # a healthy forward under the short limit: no wait comes near it
    dl.dlrm_test_stall(model.handle, LIMIT_NS, False)
    model.forward(dense, idx, off, out)
    assert model.error() == dl.OK

    # the last copy or commit withheld: the wait on it runs out
    dl.dlrm_test_stall(model.handle, LIMIT_NS, True)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    model.forward(dense, idx, off, out)
    status = model.error()            # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status == dl.ERR_TIMEOUT
    assert elapsed < 0.5, elapsed     # the 100 us bound, not the 2 s default
    assert model.error() == dl.OK     # the error word was read and cleared

    # normal operation again on the same handle and context
    dl.dlrm_test_stall(model.handle)
    out.fill_(float("nan"))
    model.forward(dense, idx, off, out)
    assert model.error() == dl.OK
    ref = oracle.forward(inp)
    np.testing.assert_allclose(out.cpu().numpy().astype(np.float64), ref, atol=tol[0],
                               rtol=tol[1])
    model.close()


def test_stall_hook_checks_its_arguments():
    with pytest.raises(ValueError):
        dl.dlrm_test_stall(12345, LIMIT_NS, True)          # not a live handle
    import ctypes
    assert dl.lib().dlrm_test_stall(ctypes.c_void_p(0), 0, 0) == dl.ERR_INVALID_ARG
    cfg = synth.get_config("tiny_b64_k3")
    inp = synth.make_inputs(cfg, seed=3)
    model = dl.DlrmModel(cfg.ln_bot, cfg.ln_top, [cu(t) for t in inp["tables"]],
                         [cu(w) for w in inp["bot_w"]], [cu(v) for v in inp["bot_b"]],
                         [cu(w) for w in inp["top_w"]], [cu(v) for v in inp["top_b"]],
                         cfg.bag_size, cfg.batch)
    assert dl.lib().dlrm_test_stall(ctypes.c_void_p(model.handle), -1, 0) == dl.ERR_INVALID_ARG
    model.close()
