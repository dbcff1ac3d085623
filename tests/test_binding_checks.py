"""The Python binding refuses mistyped, misshapen, non-contiguous or
wrong-device tensors before the library is called (no GPU needed): the
library reads and writes these buffers by the sizes the model implies, so a
short tensor would otherwise be accessed past its end on the device."""
import pytest

torch = pytest.importorskip("torch")
import dlrm_embedding_interaction_gb300 as dl  # noqa: E402

N_DENSE, K, BAG, MAXB = 13, 3, 2, 8
LN_BOT, LN_TOP, D = [13, 8, 4], [10, 8, 1], 4
FAKE = 0x5eed0001     # a handle value registered below; never passed to the library


@pytest.fixture(autouse=True)
def fake_handle():
    dl._HANDLE_SHAPES[FAKE] = (N_DENSE, K, BAG, MAXB)
    yield
    dl._HANDLE_SHAPES.pop(FAKE, None)


def io(b=4, dense_dtype=torch.float32, idx_dtype=torch.int64, n_dense=N_DENSE, idx_len=None,
       off_len=None, out_len=None):
    dense = torch.zeros(b, n_dense, dtype=dense_dtype)
    idx = torch.zeros(K, idx_len if idx_len is not None else b * BAG, dtype=idx_dtype)
    off = torch.zeros(K, off_len if off_len is not None else b, dtype=torch.int64)
    out = torch.zeros(out_len if out_len is not None else b, dtype=torch.float32)
    return dense, idx, off, out


def check(*t, on_cuda=True, max_batch=MAXB):
    return dl._check_forward_io(N_DENSE, K, BAG, max_batch, *t, "test", on_cuda=on_cuda)


def test_well_formed_host_tensors_pass_and_give_the_batch():
    assert check(*io(b=4), on_cuda=False) == 4
    assert check(*io(b=4, out_len=9), on_cuda=False) == 4     # a longer out is fine


@pytest.mark.parametrize("bad, exc", [
    (dict(dense_dtype=torch.float64), TypeError),
    (dict(idx_dtype=torch.int32), TypeError),                  # int32 would be read as int64
    (dict(n_dense=12), ValueError),
    (dict(idx_len=4 * BAG - 1), ValueError),
    (dict(off_len=3), ValueError),
    (dict(out_len=3), ValueError),                             # too short: written past its end
    (dict(b=MAXB + 1), ValueError),
])
def test_forward_inputs_are_refused_before_the_library(bad, exc):
    with pytest.raises(exc):
        check(*io(**bad), on_cuda=False)
    with pytest.raises(exc):
        dl.dlrm_forward(FAKE, *io(**bad))
    with pytest.raises(exc):
        dl.dlrm_forward_host(FAKE, *io(**bad))


def test_non_contiguous_and_wrong_device_are_refused():
    dense, idx, off, out = io(b=4)
    with pytest.raises(ValueError, match="contiguous"):
        check(dense.t().contiguous().t(), idx, off, out, on_cuda=False)
    with pytest.raises(ValueError, match="contiguous"):
        check(dense, idx, off, torch.zeros(8)[::2], on_cuda=False)
    with pytest.raises(ValueError, match="CUDA"):
        dl.dlrm_forward(FAKE, dense, idx, off, out)            # host tensors to the device call


def test_unknown_handle_is_refused():
    with pytest.raises(ValueError, match="handle"):
        dl.dlrm_forward(FAKE + 1, *io(b=4))


def params(bot_w_shape=None, top_b_shape=None, table_d=None):
    tables = [torch.zeros(10, D), torch.zeros(20, table_d or D), torch.zeros(30, D)]
    bw = [torch.zeros(LN_BOT[l + 1], LN_BOT[l]) for l in range(len(LN_BOT) - 1)]
    bb = [torch.zeros(LN_BOT[l + 1]) for l in range(len(LN_BOT) - 1)]
    tw = [torch.zeros(LN_TOP[l + 1], LN_TOP[l]) for l in range(len(LN_TOP) - 1)]
    tb = [torch.zeros(LN_TOP[l + 1]) for l in range(len(LN_TOP) - 1)]
    if bot_w_shape:
        bw[1] = torch.zeros(*bot_w_shape)
    if top_b_shape:
        tb[0] = torch.zeros(*top_b_shape)
    return tables, bw, bb, tw, tb


def test_model_parameters_are_checked_against_the_widths():
    assert dl._check_model_params(LN_BOT, LN_TOP, *params(), "test", on_cuda=False) == D
    for bad in (dict(bot_w_shape=(4, 7)), dict(bot_w_shape=(8, 4)), dict(top_b_shape=(9,)),
                dict(table_d=5)):
        with pytest.raises(ValueError):
            dl._check_model_params(LN_BOT, LN_TOP, *params(**bad), "test", on_cuda=False)
    tables, bw, bb, tw, tb = params()
    with pytest.raises(TypeError):
        dl._check_model_params(LN_BOT, LN_TOP, tables, [w.double() for w in bw], bb, tw, tb,
                               "test", on_cuda=False)
    with pytest.raises(ValueError, match="CUDA"):
        dl._check_model_params(LN_BOT, LN_TOP, *params(), "test", on_cuda=True)


def test_noalloc_binding_refuses_bad_shapes_before_the_library():
    tables, bw, bb, tw, tb = params(bot_w_shape=(4, 7))
    dense, idx, off, out = io(b=4)
    with pytest.raises(ValueError):
        dl.dlrm_forward_noalloc(LN_BOT, LN_TOP, tables, bw, bb, tw, tb, BAG, dense, idx, off, out)
    tables, bw, bb, tw, tb = params()
    with pytest.raises(ValueError):
        dl.dlrm_forward_noalloc(LN_BOT, LN_TOP, tables, bw, bb, tw, tb, BAG,
                                *io(b=4, out_len=2))
    with pytest.raises(ValueError, match="CUDA"):
        dl.dlrm_forward_noalloc(LN_BOT, LN_TOP, tables, bw, bb, tw, tb, BAG, *io(b=4))
