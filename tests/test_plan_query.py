"""The host-side plan (dlrm_plan_query): the same planner dlrm_create runs,
asked for a device's SM count and shared memory without a GPU.

The expected plans of the 2048-sample, 3-table model are the ones its GPU runs
reported (tile rows from the fused kernel's phase trace, CTAs and shared memory
from the launch), and the weight stream is counted by hand from the stage
layout. The rest are properties every plan must have.
"""
import numpy as np
import pytest

import dlrm_embedding_interaction_gb300 as dl
import dlrm_synth as synth

SMS = 152
SMEM = 232448


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dlrm_embedding_interaction_gb300 import build
    build.build()
    dl.lib()


def query(cfg, math=dl.MATH_FP32, path=dl.PATH_AUTO, batch=None, sms=SMS, smem=SMEM,
          bag=None):
    return dl.dlrm_plan_query(cfg.ln_bot, cfg.ln_top, cfg.rows, cfg.emb_dim,
                              cfg.bag_size if bag is None else bag,
                              cfg.batch if batch is None else batch, math, path, sms, smem)


def test_headline_model_plan_matches_the_gpu_runs():
    """2048 samples, 3 tables, fp32: the persistent fused kernel with 14-row
    tiles, 147 CTAs (one tile each) and 209,664 bytes of shared memory in a
    4-stage weight ring; BF16: the tensor-core kernel, 16-sample tiles, a
    9-slot ring in 223,104 bytes."""
    cfg = synth.get_config("b2048_k3")
    p = query(cfg)
    assert (p["path"], p["fused_fits"], p["tensor_core"]) == (dl.PATH_FUSED, 1, 0)
    assert (p["tile_samples"], p["tiles"], p["grid"]) == (14, 147, 147)
    assert (p["smem_bytes"], p["ring_stages"]) == (209664, 4)
    b = query(cfg, dl.MATH_BF16)
    assert (b["path"], b["tensor_core"], b["tile_samples"], b["tiles"]) == (dl.PATH_FUSED, 1, 16, 128)
    assert (b["smem_bytes"], b["ring_stages"]) == (223104, 9)


def test_fp32_weight_stream_counted_by_hand():
    """Stages of at most 32 KB: a layer wider than 256 columns stages 512
    columns x 16 k, a narrower one n_pad columns x 32 k, with k padded to the
    stage's k. Model 13-512-256-64 / 70-512-256-1 (the last layer is a dot,
    outside the stream):
      13->512   k 16:  1 stage  x 512*16*4 = 32 KB
      512->256  k 512: 16 stages x 256*32*4 = 32 KB
      256->64   k 256: 8 stages  x 64*32*4  =  8 KB
      70->512   k 80:  5 stages  x 512*16*4 = 32 KB
      512->256  k 512: 16 stages x 32 KB
    46 stages, 1,310,720 bytes."""
    p = query(synth.get_config("b2048_k3"))
    assert p["stream_copies"] == 1 + 16 + 8 + 5 + 16
    kb = 1024
    assert p["stream_bytes"] == 32 * kb + 16 * 32 * kb + 8 * 8 * kb + 5 * 32 * kb + 16 * 32 * kb


def test_bf16_weight_stream_counted_by_hand():
    """Tensor-core stream: 16 KB tiles of 128 output features x 64 bf16 k.
    13->512: 4 M-tiles x 1 K-block; 512->256: 2 x 8; 256->64: 1 x 4;
    70->512: 4 x 2; 512->256: 2 x 8. 48 tiles, 786,432 bytes."""
    b = query(synth.get_config("b2048_k3"), dl.MATH_BF16)
    assert b["stream_copies"] == 4 + 16 + 4 + 8 + 16
    assert b["stream_bytes"] == 48 * 16384


@pytest.mark.parametrize("batch,rows,grid", [(1, 4, 1), (64, 4, 16), (512, 4, 128),
                                             (4096, 14, 152), (8192, 14, 152)])
def test_tile_height_by_batch(batch, rows, grid):
    """The persistent kernel's tile height on 152 SMs: 4 rows while the
    4-row tiles fit one wave, 14 at 2048 samples and past it (8192: 586
    tiles, 3-4 per CTA, as the phase trace showed)."""
    p = query(synth.get_config("b2048_k3"), batch=batch)
    assert p["path"] == dl.PATH_FUSED
    assert (p["tile_samples"], p["grid"]) == (rows, grid)


def test_tile_height_follows_the_sm_count():
    """With fewer SMs the same 2048 samples take shorter tiles once 14-row
    tiles would need a second round (100 SMs: 12 rows, 171 tiles)."""
    p = query(synth.get_config("b2048_k3"), sms=100)
    assert (p["tile_samples"], p["tiles"], p["grid"]) == (12, 171, 100)


def test_auto_rules():
    """AUTO: the fp32 kernel with one-row bags at any batch; longer bags or the
    tensor-core kernel only up to two waves of tiles; TF32X3 is layer-wise."""
    big = synth.get_config("b65536_k26_zipf")          # bags of 20, 65536 samples
    p = query(big)
    assert p["fused_fits"] == 1 and p["path"] == dl.PATH_LAYERWISE
    small = query(big, batch=2 * SMS * p["tile_samples"])
    assert small["path"] == dl.PATH_FUSED
    assert query(big, batch=2 * SMS * p["tile_samples"] + 1)["path"] == dl.PATH_LAYERWISE
    cfg = synth.get_config("b2048_k3")
    assert query(cfg, dl.MATH_BF16, batch=2 * SMS * 16)["path"] == dl.PATH_FUSED
    assert query(cfg, dl.MATH_BF16, batch=2 * SMS * 16 + 1)["path"] == dl.PATH_LAYERWISE
    assert query(cfg, batch=65536)["path"] == dl.PATH_FUSED
    t = query(cfg, dl.MATH_TF32X3)
    assert (t["path"], t["fused_fits"]) == (dl.PATH_LAYERWISE, 0)


def test_explicit_paths():
    cfg = synth.get_config("b2048_k3")
    lw = query(cfg, path=dl.PATH_LAYERWISE)
    assert (lw["path"], lw["fused_fits"], lw["tile_samples"]) == (dl.PATH_LAYERWISE, 0, 0)
    assert query(cfg, path=dl.PATH_FUSED, batch=65536)["path"] == dl.PATH_FUSED
    with pytest.raises(dl.DlrmError) as e:
        query(cfg, dl.MATH_TF32X3, path=dl.PATH_FUSED)
    assert e.value.status == dl.ERR_UNSUPPORTED


def test_small_shared_memory_leaves_the_fused_kernel_out():
    """A device with 100 KB per block cannot hold the 512-wide model's tile
    plus its 32 KB ring stages: AUTO goes layer-wise and FUSED is refused."""
    cfg = synth.get_config("b2048_k3")
    p = query(cfg, smem=100 * 1024)
    assert (p["path"], p["fused_fits"]) == (dl.PATH_LAYERWISE, 0)
    with pytest.raises(dl.DlrmError) as e:
        query(cfg, path=dl.PATH_FUSED, smem=100 * 1024)
    assert e.value.status == dl.ERR_UNSUPPORTED


def test_layerwise_tensor_core_layers():
    """Which layer-wise GEMMs run on the tensor cores. The 26-table model has
    bottom 13-512-256-128 and top 479-1024-1024-512-256-1 (layers 0-2, 3-7):
    FP32 and TF32X3 take split-TF32 for every layer of >= 64 inputs and >= 16
    outputs but the first bottom layer (13 inputs; it reads the caller's
    buffer), FP32_FFMA none, TF32 and BF16 every layer of >= 16 outputs."""
    big = synth.get_config("b65536_k26_zipf")
    split_layers = 0b01111110            # layers 1..6; 7 is the N = 1 sigmoid layer
    for math in (dl.MATH_FP32, dl.MATH_TF32X3):
        p = query(big, math, path=dl.PATH_LAYERWISE)
        assert (p["tensor_core_layers"], p["split_tf32"]) == (split_layers, 1)
    p = query(big, dl.MATH_FP32_FFMA, path=dl.PATH_LAYERWISE)
    assert (p["tensor_core_layers"], p["split_tf32"]) == (0, 0)
    for math in (dl.MATH_TF32, dl.MATH_BF16):
        p = query(big, math, path=dl.PATH_LAYERWISE)
        assert (p["tensor_core_layers"], p["split_tf32"]) == (0b01111111, 0)
    # AUTO takes the layer-wise plan for this model in fp32: the same layers
    assert query(big)["tensor_core_layers"] == split_layers
    # a fused plan reports none
    cfg = synth.get_config("b2048_k3")
    assert query(cfg)["tensor_core_layers"] == 0


def test_ffma_mode_plans_like_fp32_when_fused():
    """FP32_FFMA takes the same fused plan as FP32 (the fused kernel is FFMA),
    but never the layer-wise split-TF32 plan at large batches."""
    switch = ("layerwise_from", "tensor_core_layers", "split_tf32")
    for name in ("b2048_k3", "tiny_b64_k3", "sweep_b8192_k16"):
        cfg = synth.get_config(name)
        a, b = query(cfg, dl.MATH_FP32_FFMA), query(cfg, dl.MATH_FP32)
        assert {k: v for k, v in a.items() if k not in switch} == \
            {k: v for k, v in b.items() if k not in switch}
        assert a["layerwise_from"] == 0


@pytest.mark.parametrize("k", [1, 3, 16, 32])
@pytest.mark.parametrize("max_batch", [4096, 16384])
def test_large_batches_switch_to_the_split_tf32_plan(k, max_batch):
    """AUTO fp32 on the fused plan runs the layer-wise split-TF32 plan from the
    first sample of a second round of fused tiles (one wave = SMs x tile
    samples); a handle whose max_batch fits one wave never switches, nor an
    explicit FUSED path, FFMA math or a model whose fused round is short."""
    cfg = synth.sweep_config(max_batch, k)
    p = query(cfg)
    assert p["path"] == dl.PATH_FUSED
    wave = SMS * p["tile_samples"]
    assert p["layerwise_from"] == wave + 1
    assert p["tensor_core_layers"] != 0 and p["split_tf32"] == 1
    one_wave = query(cfg, batch=wave)
    assert one_wave["layerwise_from"] == 0 or one_wave["layerwise_from"] > wave
    assert query(cfg, path=dl.PATH_FUSED)["layerwise_from"] == 0
    assert query(cfg, dl.MATH_FP32_FFMA)["layerwise_from"] == 0
    assert query(synth.get_config("tiny_b64_k3"), batch=65536)["layerwise_from"] == 0


def test_many_tables_trade_a_weight_stage_for_bag_row_groups():
    """32 tables at 14-row tiles: the bag rows (14 x 32 rows of 68 floats,
    122 KB) stream in groups; a 4-stage ring leaves room for groups of one
    sample, so the plan takes 3 stages and two 3-sample groups: 3 x 32,768
    (stages) + 2 x 34,944 (14 x 624-float activation buffers) + 9,472 (row
    indices, biases, last layer, barriers) + 2 x 3 x 8,704 (groups of 32
    rows of 68 floats) = 229,888 bytes. 16 tables keep every bag row
    resident (3 stages, no streaming) and 3 tables a 4-stage ring."""
    assert (query(synth.get_config("b2048_k32"))["ring_stages"],
            query(synth.get_config("b2048_k32"))["smem_bytes"]) == (3, 229888)
    assert query(synth.get_config("sweep_b2048_k16"))["ring_stages"] == 3
    assert query(synth.get_config("b2048_k3"))["ring_stages"] == 4


@pytest.mark.parametrize("math", [dl.MATH_FP32, dl.MATH_TF32, dl.MATH_BF16])
def test_every_sweep_plan_is_consistent(math):
    """Over the 11 x 5 batch x tables sweep: a fused plan fits the device's
    shared memory, its tiles cover the batch, the fp32 grid is at most one
    CTA per SM and the tensor-core grid one CTA per tile."""
    for b in synth.SWEEP_BATCHES:
        for k in synth.SWEEP_TABLES:
            cfg = synth.get_config(f"sweep_b{b}_k{k}")
            p = query(cfg, math)
            if not p["fused_fits"]:
                assert p["path"] == dl.PATH_LAYERWISE
                continue
            assert 0 < p["smem_bytes"] <= SMEM
            assert p["ring_stages"] >= 2
            assert p["tiles"] * p["tile_samples"] >= b > (p["tiles"] - 1) * p["tile_samples"]
            if math == dl.MATH_FP32:
                assert p["tile_samples"] in (4, 8, 12, 14, 16)
                assert p["grid"] == min(p["tiles"], SMS)
                assert p["path"] == dl.PATH_FUSED       # bags of one row
            else:
                assert p["tile_samples"] == 16 and p["grid"] == p["tiles"]


def test_query_checks_its_arguments_like_create():
    cfg = synth.get_config("tiny_b64_k3")
    with pytest.raises(dl.DlrmError) as e:
        query(cfg, sms=0)
    assert e.value.status == dl.ERR_INVALID_ARG
    with pytest.raises(dl.DlrmError) as e:
        query(cfg, smem=0)
    assert e.value.status == dl.ERR_INVALID_ARG
    with pytest.raises(dl.DlrmError) as e:   # ln_top[0] != D + P
        dl.dlrm_plan_query([13, 8, 4], [11, 8, 1], [10, 20, 30], 4, 1, 8)
    assert e.value.status == dl.ERR_INVALID_ARG
    with pytest.raises(dl.DlrmError) as e:   # bag 0
        dl.dlrm_plan_query([13, 8, 4], [10, 8, 1], [10, 20, 30], 4, 0, 8)
    assert e.value.status == dl.ERR_INVALID_ARG
    with pytest.raises(dl.DlrmError) as e:   # unknown path
        dl.dlrm_plan_query([13, 8, 4], [10, 8, 1], [10, 20, 30], 4, 1, 8, path=7)
    assert e.value.status == dl.ERR_INVALID_ARG
    with pytest.raises(dl.DlrmError) as e:   # more tables than the kernels take
        rows = [10] * (dl.MAX_TABLES + 1)
        f = len(rows) + 1
        dl.dlrm_plan_query([13, 4], [4 + f * (f - 1) // 2, 1], rows, 4, 1, 8)
    assert e.value.status == dl.ERR_UNSUPPORTED
    assert dl.lib().dlrm_plan_query(None, SMS, SMEM, None) == dl.ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("name,math", [
    ("tiny_b64_k3", dl.MATH_FP32), ("b2048_k3", dl.MATH_FP32), ("b2048_k3", dl.MATH_BF16),
    ("b2048_k32", dl.MATH_FP32), ("b2048_k32", dl.MATH_BF16), ("sweep_b8192_k3", dl.MATH_FP32),
    ("sweep_b8192_k3", dl.MATH_TF32), ("sweep_b300_k16", dl.MATH_TF32),
    ("b2048_k3", dl.MATH_TF32X3)])
def test_query_matches_create_on_the_device(name, math):
    """The host query, given this device's SM count and shared memory, names
    the path and tile height the handle built on the device took."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    props = torch.cuda.get_device_properties(0)
    smem = getattr(props, "shared_memory_per_block_optin", SMEM)
    cfg = synth.get_config(name)
    q = query(cfg, math, sms=props.multi_processor_count, smem=smem)
    inp = synth.make_inputs(cfg, seed=1)

    def cu(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    model = dl.DlrmModel(cfg.ln_bot, cfg.ln_top, [cu(t) for t in inp["tables"]],
                         [cu(w) for w in inp["bot_w"]], [cu(v) for v in inp["bot_b"]],
                         [cu(w) for w in inp["top_w"]], [cu(v) for v in inp["top_b"]],
                         cfg.bag_size, cfg.batch, math)
    try:
        assert model.path == q["path"]
        if q["path"] == dl.PATH_FUSED:
            assert model.set_phase_trace(None) == q["tile_samples"]
    finally:
        model.close()
