"""The C-ABI library loads, exports every symbol include/dlrm.h declares, and
rejects bad arguments on the host before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

import dlrm_embedding_interaction_gb300 as dl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dlrm.h")


@pytest.fixture(scope="module")
def lib():
    from dlrm_embedding_interaction_gb300 import build
    build.build()
    return dl.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("dlrm_create", "dlrm_forward", "embedding_bag_sum_multi",
                     "pairwise_dot_lower_tri", "linear_bias_act"):
        assert required in names
    assert sorted(dl.EXPORTS) == names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert dl.version() == 100


def test_status_strings(lib):
    assert lib.dlrm_status_string(dl.OK) == b"ok"
    assert lib.dlrm_status_string(dl.ERR_INDEX_OOB) == b"index out of range"
    assert lib.dlrm_status_string(99) == b"unknown status"


def test_host_side_argument_checks(lib):
    vp = ctypes.c_void_p
    null = vp(0)
    # linear_bias_act: N < 1, K < 1, ld_x < K, bad act
    assert lib.linear_bias_act(null, 4, null, null, null, 4, 4, 0, 4, 0, 0, null) == dl.ERR_INVALID_ARG
    assert lib.linear_bias_act(null, 4, null, null, null, 4, 4, 4, 0, 0, 0, null) == dl.ERR_INVALID_ARG
    assert lib.linear_bias_act(null, 3, null, null, null, 4, 4, 4, 4, 0, 0, null) == dl.ERR_INVALID_ARG
    assert lib.linear_bias_act(null, 4, null, null, null, 4, 4, 4, 4, 7, 0, null) == dl.ERR_INVALID_ARG
    # unknown math mode; every known one (FP32_FFMA = 4 the last) passes the check
    assert lib.linear_bias_act(null, 4, null, null, null, 4, 0, 4, 4, 0, 5, null) == dl.ERR_INVALID_ARG
    for math in (dl.MATH_FP32, dl.MATH_TF32, dl.MATH_BF16, dl.MATH_TF32X3, dl.MATH_FP32_FFMA):
        assert lib.linear_bias_act(null, 4, null, null, null, 4, 0, 4, 4, 0, math, null) == dl.OK
    # M = 0 is a no-op
    assert lib.linear_bias_act(null, 4, null, null, null, 4, 0, 4, 4, 0, 0, null) == dl.OK
    # null pointers with M > 0
    assert lib.linear_bias_act(null, 4, null, null, null, 4, 2, 4, 4, 0, 0, null) == dl.ERR_INVALID_ARG
    # gather: K < 1, K > max, B = 0 no-op, null tables
    assert lib.embedding_bag_sum_multi(null, null, 0, 4, null, null, 1, 1, null, null, null) == dl.ERR_INVALID_ARG
    ptrs = (vp * 200)()
    rows = (ctypes.c_int64 * 200)()
    assert lib.embedding_bag_sum_multi(ptrs, rows, 200, 4, null, null, 1, 1, null, null, null) == dl.ERR_UNSUPPORTED
    assert lib.embedding_bag_sum_multi(ptrs, rows, 3, 4, null, null, 0, 1, null, null, null) == dl.OK
    assert lib.embedding_bag_sum_multi(ptrs, rows, 3, 4, null, null, 5, 1, null, null, null) == dl.ERR_INVALID_ARG
    # interaction: ld_out too small for [x, z]; B = 0 no-op
    assert lib.pairwise_dot_lower_tri(null, 4, null, 2, 3, 4, null, 9, 1, null) == dl.ERR_INVALID_ARG
    assert lib.pairwise_dot_lower_tri(null, 4, null, 0, 3, 4, null, 10, 1, null) == dl.OK
    assert lib.pairwise_pair_map(1, null, null, null) == dl.ERR_INVALID_ARG


def _create(lib, ln_bot, ln_top, rows, d, bag=1, max_batch=8, math=0, tables_ok=True,
            table=0x1000):
    k = len(rows)
    cfg = dl._Config(len(ln_bot) - 1, (ctypes.c_int32 * len(ln_bot))(*ln_bot), k,
                     (ctypes.c_int64 * k)(*rows), d, len(ln_top) - 1,
                     (ctypes.c_int32 * len(ln_top))(*ln_top), bag, max_batch, math, 0)
    fake = ctypes.c_void_p(table if tables_ok else 0)
    tabs = (ctypes.c_void_p * k)(*([fake] * k))
    w = (ctypes.c_void_p * 16)(*([ctypes.c_void_p(0x1000)] * 16))
    h = ctypes.c_void_p()
    return lib.dlrm_create(ctypes.byref(cfg), tabs, w, w, w, w, ctypes.byref(h)), h


def test_create_validates_shapes(lib):
    """dlrm_megakernel.rs validate(): ln_bot.last() = m_spa, ln_top[0] = m_spa + P,
    ln_top.last() = 1; plus the ABI's own limits."""
    assert _create(lib, [13, 8, 5], [10, 8, 1], [10, 20, 30], 4)[0] == dl.ERR_INVALID_ARG
    assert _create(lib, [13, 8, 4], [11, 8, 1], [10, 20, 30], 4)[0] == dl.ERR_INVALID_ARG
    assert _create(lib, [13, 8, 4], [10, 8, 2], [10, 20, 30], 4)[0] == dl.ERR_INVALID_ARG
    assert _create(lib, [13, 8, 4], [10, 8, 1], [10, 20, 30], 4, bag=0)[0] == dl.ERR_INVALID_ARG
    assert _create(lib, [13, 8, 4], [10, 8, 1], [10, 20, 30], 4, max_batch=0)[0] == dl.ERR_INVALID_ARG
    assert _create(lib, [13, 8, 4], [10, 8, 1], [10, 0, 30], 4)[0] == dl.ERR_INVALID_ARG
    assert _create(lib, [13, 8, 4], [10, 8, 1], [10, 20, 30], 4, tables_ok=False)[0] == dl.ERR_INVALID_ARG
    assert _create(lib, [13, 8, 4], [10, 8, 1], [10, 20, 30], 4, math=5)[0] != dl.OK
    assert lib.dlrm_create(None, None, None, None, None, None, None) == dl.ERR_INVALID_ARG


def test_forward_rejects_null_handle(lib):
    null = ctypes.c_void_p(0)
    assert lib.dlrm_forward(null, null, null, null, null, 1, null) == dl.ERR_INVALID_ARG
    assert lib.dlrm_forward_host(null, null, null, null, null, 1, null) == dl.ERR_INVALID_ARG
    assert lib.dlrm_get_error(null, null) == dl.ERR_INVALID_ARG
    assert lib.dlrm_workspace_bytes(null) == 0
    lib.dlrm_destroy(null)


def test_bag_calls_check_arguments_on_the_host(lib):
    """embedding_bag_multi(_ex) refuse bad shapes, modes, index widths and weight use
    before any launch; a batch of zero returns at once."""
    vp = ctypes.c_void_p
    null = vp(0)
    tabs = (vp * 2)(vp(16), vp(16))
    rows = (ctypes.c_int64 * 2)(10, 10)
    f = lib.embedding_bag_multi
    f.argtypes = [vp, vp, ctypes.c_int32, ctypes.c_int32, vp, ctypes.c_int64, vp,
                  ctypes.c_int32, ctypes.c_int32, vp, vp, vp]
    assert f(tabs, rows, 0, 8, null, 4, null, 2, 0, null, null, null) == dl.ERR_INVALID_ARG
    assert f(tabs, rows, 2, 0, null, 4, null, 2, 0, null, null, null) == dl.ERR_INVALID_ARG
    assert f(tabs, rows, 2, 8, null, -1, null, 2, 0, null, null, null) == dl.ERR_INVALID_ARG
    assert f(tabs, rows, 2, 8, null, 4, null, -1, 0, null, null, null) == dl.ERR_INVALID_ARG
    assert f(tabs, rows, 2, 8, null, 4, null, 2, 3, null, null, null) == dl.ERR_INVALID_ARG
    assert f(tabs, rows, 129, 8, null, 4, null, 2, 0, null, null, null) == dl.ERR_UNSUPPORTED
    assert f(null, rows, 2, 8, null, 4, null, 2, 0, null, null, null) == dl.ERR_INVALID_ARG
    assert f(tabs, rows, 2, 8, null, 4, null, 2, 0, null, null, null) == dl.ERR_INVALID_ARG
    assert f(tabs, rows, 2, 8, null, 4, null, 0, 0, null, null, null) == dl.OK
    g = lib.embedding_bag_multi_ex
    g.argtypes = [vp, vp, ctypes.c_int32, ctypes.c_int32, vp, ctypes.c_int64, vp,
                  ctypes.c_int32, ctypes.POINTER(dl._BagOptions), vp, vp, vp]
    g.restype = ctypes.c_int

    def ex(mode, bits, weights, n_idx=4, b=2):
        opt = dl._BagOptions(mode, bits, weights, -1)
        return g(tabs, rows, 2, 8, null, n_idx, null, b, ctypes.byref(opt), null, null, null)

    assert g(tabs, rows, 2, 8, null, 4, null, 2, None, null, null, null) == dl.ERR_INVALID_ARG
    assert ex(0, 16, None) == dl.ERR_INVALID_ARG
    assert ex(1, 64, 16) == dl.ERR_INVALID_ARG          # weights with mean
    assert ex(2, 32, 16) == dl.ERR_INVALID_ARG          # weights with max
    assert ex(0, 32, None, n_idx=1 << 31) == dl.ERR_INVALID_ARG
    assert ex(0, 32, 16, b=0) == dl.OK


def test_header_is_plain_c_and_links(tmp_path, lib):
    """include/dlrm.h compiles as C11 and a C program links against the library."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use.c"
    src.write_text(
        '#include "dlrm.h"\n'
        "int main(void) {\n"
        "  dlrm_bag_options_t o = {DLRM_BAG_MEAN, 64, 0, -1};\n"
        "  (void)o;\n"
        "  return dlrm_version() == 100 ? 0 : 1;\n"
        "}\n")
    cuda_inc = "/usr/local/cuda/include"
    exe = tmp_path / "use"
    libdir = os.path.dirname(dl.LIB_PATH)
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", cuda_inc, str(src), "-o", str(exe), "-L", libdir, "-ldlrm_gb300",
                        f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, run.stderr


def test_misaligned_pointers_are_refused_before_any_launch(lib):
    """Every pointer must sit at its element's natural alignment (4 bytes for
    fp32 and int32, 8 for int64); the calls refuse others with INVALID_ARG on
    the host instead of faulting on the device."""
    vp = ctypes.c_void_p
    f32, i64, odd = vp(0x1000), vp(0x1008), vp(0x1002)
    i64_on_4 = vp(0x1004)                               # int64 on a 4-byte boundary
    rows = (ctypes.c_int64 * 2)(10, 10)
    tabs = (vp * 2)(f32, f32)
    bad_tabs = (vp * 2)(f32, odd)
    null = vp(0)
    g = lib.embedding_bag_sum_multi
    assert g(bad_tabs, rows, 2, 8, i64, i64, 4, 1, f32, null, null) == dl.ERR_INVALID_ARG
    assert g(tabs, rows, 2, 8, i64_on_4, i64, 4, 1, f32, null, null) == dl.ERR_INVALID_ARG
    assert g(tabs, rows, 2, 8, i64, i64_on_4, 4, 1, f32, null, null) == dl.ERR_INVALID_ARG
    assert g(tabs, rows, 2, 8, i64, i64, 4, 1, odd, null, null) == dl.ERR_INVALID_ARG
    assert g(tabs, rows, 2, 8, i64, i64, 4, 1, f32, odd, null) == dl.ERR_INVALID_ARG

    ex = lib.embedding_bag_multi_ex
    ex.argtypes = [vp, vp, ctypes.c_int32, ctypes.c_int32, vp, ctypes.c_int64, vp,
                   ctypes.c_int32, ctypes.POINTER(dl._BagOptions), vp, vp, vp]
    ex.restype = ctypes.c_int
    o64 = dl._BagOptions(0, 64, None, -1)
    o32 = dl._BagOptions(0, 32, None, -1)
    assert ex(tabs, rows, 2, 8, i64_on_4, 8, i64, 4, ctypes.byref(o64), f32, null, null) == dl.ERR_INVALID_ARG
    assert ex(tabs, rows, 2, 8, odd, 8, f32, 4, ctypes.byref(o32), f32, null, null) == dl.ERR_INVALID_ARG
    assert ex(bad_tabs, rows, 2, 8, i64, 8, i64, 4, ctypes.byref(o64), f32, null, null) == dl.ERR_INVALID_ARG
    ow = dl._BagOptions(0, 64, 0x1002, -1)               # per-sample weights off by 2 bytes
    assert ex(tabs, rows, 2, 8, i64, 8, i64, 4, ctypes.byref(ow), f32, null, null) == dl.ERR_INVALID_ARG

    assert lib.pairwise_dot_lower_tri(odd, 8, f32, 2, 3, 8, f32, 20, 1, null) == dl.ERR_INVALID_ARG
    assert lib.pairwise_dot_lower_tri(f32, 8, odd, 2, 3, 8, f32, 20, 1, null) == dl.ERR_INVALID_ARG
    assert lib.pairwise_dot_lower_tri(f32, 8, f32, 2, 3, 8, odd, 20, 1, null) == dl.ERR_INVALID_ARG
    assert lib.pairwise_pair_map(4, odd, f32, null) == dl.ERR_INVALID_ARG
    w, y = vp(0x2000), vp(0x3000)
    assert lib.linear_bias_act(odd, 4, w, null, y, 4, 2, 4, 4, 0, 0, null) == dl.ERR_INVALID_ARG
    assert lib.linear_bias_act(f32, 4, w, odd, y, 4, 2, 4, 4, 0, 0, null) == dl.ERR_INVALID_ARG
    assert lib.linear_bias_act(f32, 4, w, null, vp(0x3001), 4, 2, 4, 4, 0, 0, null) == dl.ERR_INVALID_ARG

    # the forward handle borrows its tables: a misaligned one is refused at create
    assert _create(lib, [13, 8, 4], [10, 8, 1], [10, 20, 30], 4, table=0x1002)[0] == dl.ERR_INVALID_ARG


def test_noalloc_forward_refuses_misaligned_inputs(lib):
    vp = ctypes.c_void_p
    ln_bot, ln_top, rows = [13, 8, 4], [10, 8, 1], [10, 20, 30]
    cfg = dl._Config(2, (ctypes.c_int32 * 3)(*ln_bot), 3, (ctypes.c_int64 * 3)(*rows), 4, 2,
                     (ctypes.c_int32 * 3)(*ln_top), 1, 8, 0, 0)
    ok = vp(0x1000)
    tabs = (vp * 3)(ok, ok, ok)
    w = (vp * 16)(*([ok] * 16))
    f = lib.dlrm_forward_noalloc
    args = lambda dense, idx, off, out, wts=w: f(ctypes.byref(cfg), tabs, wts, wts, wts, wts, dense,
                                                 idx, off, out, 4, None, None)
    assert args(vp(0x1002), ok, ok, ok) == dl.ERR_INVALID_ARG
    assert args(ok, vp(0x1004), ok, ok) == dl.ERR_INVALID_ARG
    assert args(ok, ok, vp(0x1004), ok) == dl.ERR_INVALID_ARG
    assert args(ok, ok, ok, vp(0x1001)) == dl.ERR_INVALID_ARG
    bad_w = (vp * 16)(*([vp(0x1002)] * 16))
    assert args(ok, ok, ok, ok, bad_w) == dl.ERR_INVALID_ARG
