"""Table-wise sharded forward (dlrm_embedding_interaction_gb300.sharded) on CPU.

The host logic (table partition, the all-to-all's splits, the receive-chunk
indexing of the dense part) runs here on gloo ranks, world sizes 2 and 3,
with the CPU oracle as the compute backend; every rank's outputs must match
the unsharded oracle forward of its samples. The same module runs the
library's CUDA kernels and NCCL by default (tests/test_gpu_sharded.py runs
those kernels on one GPU with the exchange done in one process)."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import dlrm_synth as synth  # noqa: E402
from dlrm_embedding_interaction_gb300 import sharded  # noqa: E402

ATOL, RTOL = 1e-5, 1e-4


class OracleBackend:
    """Test backend: the CPU oracle computes, gloo exchanges."""

    def bag_sums(self, tables, indices, offsets, out, bag_size, stream=None):
        import oracle
        e = oracle.embedding_bag_sum([t.numpy() for t in tables], indices.numpy(),
                                     offsets.numpy())
        out.copy_(torch.from_numpy(e.astype(np.float32)))

    def exchange(self, recv, send, recv_splits, send_splits):
        dist.all_to_all_single(recv, send, output_split_sizes=recv_splits,
                               input_split_sizes=send_splits)

    def make_dense(self, ln_bot, ln_top, tables, bot_w, bot_b, top_w, top_b, batch, math, path):
        return dict(tables=tables, bot_w=bot_w, bot_b=bot_b, top_w=top_w, top_b=top_b)

    def dense_forward(self, model, dense, indices, offsets, out, stream=None):
        import oracle
        inp = dict(dense=dense.numpy(), tables=[t.numpy() for t in model["tables"]],
                   indices=indices.numpy(), offsets=offsets.numpy(),
                   bot_w=[w.numpy() for w in model["bot_w"]],
                   bot_b=[v.numpy() for v in model["bot_b"]],
                   top_w=[w.numpy() for w in model["top_w"]],
                   top_b=[v.numpy() for v in model["top_b"]])
        out.copy_(torch.from_numpy(oracle.forward(inp).astype(np.float32)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _config(rows, batch_per_rank, world, bag=2, d=16):
    k = len(rows)
    f = k + 1
    return synth.DlrmConfig(f"shard_k{k}", batch_per_rank * world, (13, 32, d), tuple(rows), d,
                            bag, (d + f * (f - 1) // 2, 32, 1), 0.05)


def _rank_main(rank, world, port, rows, batch, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        cfg = _config(rows, batch, world)
        inp = synth.make_inputs(cfg, seed=2024)
        part = sharded.partition_tables(cfg.rows, world)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
        mine = [t(inp["tables"][i]) for i in part[rank]]
        fwd = sharded.TableShardedForward(
            cfg.ln_bot, cfg.ln_top, mine, cfg.rows, cfg.emb_dim,
            [t(w) for w in inp["bot_w"]], [t(v) for v in inp["bot_b"]],
            [t(w) for w in inp["top_w"]], [t(v) for v in inp["top_b"]],
            cfg.bag_size, batch, rank, world, backend=OracleBackend(), device="cpu")
        idx_mine, off_mine = sharded.local_sparse_inputs(inp["indices"], inp["offsets"], part, rank)
        out = torch.full((batch,), float("nan"))
        fwd.forward(t(inp["dense"][rank * batch:(rank + 1) * batch]), t(idx_mine), t(off_mine), out)
        ref = oracle.forward(inp)[rank * batch:(rank + 1) * batch]
        q.put((rank, out.numpy().astype(np.float64), ref, part))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,rows", [(2, (300, 50, 200, 120, 77)), (3, (90, 40)),
                                        (2, (60, 60, 60))])
def test_sharded_forward_matches_the_unsharded_oracle_on_gloo_ranks(world, rows):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    batch = 6
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, rows, batch, q))
             for r in range(world)]
    for p in procs:
        p.start()
    try:
        got = [q.get(timeout=180) for _ in range(world)]
    finally:
        for p in procs:
            p.join(timeout=60)
    for p in procs:
        assert p.exitcode == 0
    for rank, out, ref, part in got:
        np.testing.assert_allclose(out, ref, atol=ATOL, rtol=RTOL, err_msg=f"rank {rank}")
    if world == 3 and len(rows) == 2:
        assert [] in got[0][3]            # a rank without tables still takes part


def test_partition_covers_every_table_once_and_balances_rows():
    rows = (1000, 10, 500, 500, 20, 990)
    for world in (1, 2, 3, 4, 8):
        part = sharded.partition_tables(rows, world)
        assert len(part) == world
        flat = sorted(t for p in part for t in p)
        assert flat == list(range(len(rows)))
        assert all(p == sorted(p) for p in part)
    # largest first onto the lightest rank: 1000 -> r0, 990 -> r1, 500 -> r1
    # (1490), 500 -> r0 (1500), 20 -> r1 (1510), 10 -> r0 (1510)
    assert sharded.partition_tables(rows, 2) == [[0, 1, 3], [2, 4, 5]]


def test_split_sizes_and_dense_indices_by_hand():
    part = [[0, 3], [1], [2, 4, 5]]
    send, recv = sharded.split_sizes(part, 2, batch=4, emb_dim=8)
    assert send == [4 * 3 * 8] * 3
    assert recv == [4 * 2 * 8, 4 * 1 * 8, 4 * 3 * 8]
    idx = sharded.dense_gather_indices(part, batch=4)
    # table 3 is rank 0's second table (K_0 = 2): rows 1, 3, 5, 7
    assert idx[3] == [1, 3, 5, 7]
    # table 5 is rank 2's third table (K_2 = 3): rows 2, 5, 8, 11
    assert idx[5] == [2, 5, 8, 11]
    assert idx[1] == [0, 1, 2, 3]
    assert sharded.owner_and_slot(part)[4] == (2, 1)
