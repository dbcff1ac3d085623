"""Table-wise sharded forward with the library's CUDA kernels, on one GPU.

Every rank's part (its tables' bag sums in one launch, and the dense part as
a forward over the receive chunks) runs the real kernels; the all-to-all of
a multi-GPU run is replaced by the same copies done in this one process, in
stream order, after every rank's bag sums. Nothing waits across ranks. The
outputs of all ranks must match the unsharded CPU oracle at the fp32
tolerance.
"""
import numpy as np
import pytest

import dlrm_synth as synth
import oracle

torch = pytest.importorskip("torch")
import dlrm_embedding_interaction_gb300 as dl  # noqa: E402
from dlrm_embedding_interaction_gb300 import sharded  # noqa: E402

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


class InProcessBackend(sharded.CudaBackend):
    """The library's kernels; the exchange is left to the test."""

    def exchange(self, recv, send, recv_splits, send_splits):
        pass


def cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def exchange_all(ranks):
    """What the all-to-all does, for ranks living in one process: rank q's
    receive chunk from s is s's send slice for q."""
    for q, rq in enumerate(ranks):
        at = 0
        for s, rs in enumerate(ranks):
            n = rs.send_splits[q]
            rq.recv[at:at + n].copy_(rs.send[q * n:(q + 1) * n])
            at += n


@pytest.mark.parametrize("name,world,path", [
    ("b2048_k32", 2, dl.PATH_FUSED), ("b2048_k32", 3, dl.PATH_LAYERWISE),
    ("tiny_b64_k3", 2, dl.PATH_AUTO), ("tiny_b64_k3", 4, dl.PATH_AUTO)])
def test_sharded_forward_on_one_gpu_matches_the_oracle(name, world, path):
    cfg = synth.get_config(name)
    inp = synth.make_inputs(cfg, seed=31)
    batch = cfg.batch // world
    g = batch * world                      # the global batch the ranks share
    part = sharded.partition_tables(cfg.rows, world)
    backend = InProcessBackend()
    ranks = []
    for r in range(world):
        ranks.append(sharded.TableShardedForward(
            cfg.ln_bot, cfg.ln_top, [cu(inp["tables"][t]) for t in part[r]], cfg.rows,
            cfg.emb_dim, [cu(w) for w in inp["bot_w"]], [cu(v) for v in inp["bot_b"]],
            [cu(w) for w in inp["top_w"]], [cu(v) for v in inp["top_b"]], cfg.bag_size,
            batch, r, world, path=path, backend=backend))
    idx = inp["indices"][:, :g * cfg.bag_size]
    off = inp["offsets"][:, :g]
    for r, fr in enumerate(ranks):
        i_mine, o_mine = sharded.local_sparse_inputs(idx, off, part, r)
        fr.bag_sums(cu(i_mine), cu(o_mine))
    exchange_all(ranks)
    outs = []
    for r, fr in enumerate(ranks):
        out = torch.full((batch,), float("nan"), device="cuda")
        fr.dense(cu(inp["dense"][r * batch:(r + 1) * batch]), out)
        assert fr.model.error() == dl.OK
        outs.append(out.cpu().numpy())
    ref = oracle.forward(dict(inp, dense=inp["dense"][:g], indices=idx, offsets=off))
    np.testing.assert_allclose(np.concatenate(outs).astype(np.float64), ref, atol=ATOL,
                               rtol=RTOL)
    for fr in ranks:
        fr.close()
