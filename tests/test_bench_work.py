"""The algorithmic work behind every roofline fraction the bench reports.

bench.forward_work and bench.stage_work count the method's own flops and HBM
bytes (intermediates excluded, int64 indices). They are checked here against
the figures derived independently for the workloads: 1.318 GFLOP and 3.08 MB
for the 2048-sample 3-table model, 2.549 GFLOP and 20.3 MB for 32 tables,
320.0 GFLOP and 17.75 GB for the 65536-sample 26-table model, and the gather's
18.61 GB on the latter, plus hand counts on a tiny shape.
"""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
import dlrm_synth as synth  # noqa: E402


@pytest.mark.parametrize("name,gflop,mbytes", [
    ("b2048_k3", 1.318, 3.08),
    ("b2048_k32", 2.549, 20.3),
    ("b65536_k26_zipf", 320.0, 17750.0),
])
def test_forward_work_matches_the_derived_figures(name, gflop, mbytes):
    cfg = synth.get_config(name)
    flops, byts = bench.forward_work(cfg, cfg.batch)
    assert flops / 1e9 == pytest.approx(gflop, rel=2e-3)
    assert byts / 1e6 == pytest.approx(mbytes, rel=3e-3)


def test_gather_bytes_of_the_large_workload():
    cfg = synth.get_config("b65536_k26_zipf")
    flops, byts = bench.stage_work(cfg, "gather", cfg.batch)
    assert byts / 1e9 == pytest.approx(18.61, rel=1e-3)
    assert flops == cfg.batch * cfg.n_tables * (cfg.bag_size - 1) * cfg.emb_dim


def test_work_by_hand_on_a_tiny_shape():
    """B = 2, K = 2 tables of D = 4, bags of 3; bottom 3 -> 4, top (4 + 3) -> 5 -> 1."""
    cfg = synth.DlrmConfig("hand", 2, (3, 4), (10, 10), 4, 3, (7, 5, 1))
    flops, byts = bench.forward_work(cfg, 2)
    # MLP: 2 * B * (3*4 + 7*5 + 5*1); pairs: F = 3 -> P = 3, 2 * B * P * D; bag adds B*K*(L-1)*D
    assert flops == 2 * 2 * (12 + 35 + 5) + 2 * 2 * 3 * 4 + 2 * 2 * 2 * 4
    # rows 4*D*K*L*B, indices 8*K*L*B, offsets 8*K*B, dense 4*3*B, out 4*B, weights+biases
    w = 4 * ((3 * 4 + 4) + (7 * 5 + 5) + (5 * 1 + 1))
    assert byts == 4 * 4 * 2 * 3 * 2 + 8 * 2 * 3 * 2 + 8 * 2 * 2 + 4 * 3 * 2 + 4 * 2 + w
    assert bench.stage_work(cfg, "interaction", 2) == (2 * 2 * 3 * 4, 2 * 3 * 4 * 4 + 2 * 7 * 4)
    assert bench.stage_work(cfg, "top0", 2) == (2 * 2 * 7 * 5, 4 * (2 * 7 + 7 * 5 + 5 + 2 * 5))
