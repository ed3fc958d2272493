"""C-ABI checks that need no GPU: the library loads, exports every entry point
declared in include/wtconv.h, and rejects bad arguments with a status code
before it touches the device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

from memory_bound_cnn_wtconv2d_gb300 import build, wtconv


@pytest.fixture(scope="module")
def L():
    build.build()
    return wtconv.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "wtconv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(wtconv_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert set(wtconv.EXPORTS) <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code, name in [(0, "WTCONV_OK"), (1, "WTCONV_ERR_INVALID_ARG"), (2, "WTCONV_ERR_UNSUPPORTED"),
                       (3, "WTCONV_ERR_MISALIGNED"), (4, "WTCONV_ERR_WORKSPACE"), (5, "WTCONV_ERR_CUDA")]:
        assert L.wtconv_status_string(code).decode() == name


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def call_fwd(L, desc, x=FAKE, y=FAKE, w=FAKE):
    p = ctypes.c_void_p
    return L.wtconv_fwd(ctypes.byref(desc), p(x), p(w), None, p(w), p(w), p(w), p(y), None, 0, None)


@pytest.mark.parametrize("field,value,code", [
    ("k", 4, wtconv.WTCONV_ERR_INVALID_ARG), ("k", 1, wtconv.WTCONV_ERR_INVALID_ARG),
    ("k", 11, wtconv.WTCONV_ERR_INVALID_ARG), ("levels", 0, wtconv.WTCONV_ERR_INVALID_ARG),
    ("levels", 9, wtconv.WTCONV_ERR_INVALID_ARG), ("N", -1, wtconv.WTCONV_ERR_INVALID_ARG),
    ("C", 0, wtconv.WTCONV_ERR_INVALID_ARG), ("H", 0, wtconv.WTCONV_ERR_INVALID_ARG),
    ("dtype", 7, wtconv.WTCONV_ERR_INVALID_ARG), ("H", 8192, wtconv.WTCONV_ERR_UNSUPPORTED),
    ("levels", 5, wtconv.WTCONV_ERR_WORKSPACE),
])
def test_invalid_descriptors(L, field, value, code):
    # H = W = 8192: beyond 2^24 pixels per plane.  512 x 512 at 5 levels,
    # k = 5: not one CTA, and a tile's window (64-pixel halo) neither, so the
    # layer is computed as a fine pass and a coarse layer, which needs a
    # workspace (none given here).
    d = wtconv.make_desc(2, 3, 16, 16, 2, 5, 0)
    setattr(d, field, value)
    if field == "H" and value == 8192:
        d.W = 8192
    if field == "levels" and value == 5:
        d.H = d.W = 512
    assert call_fwd(L, d) == code
    assert L.wtconv_last_error().decode() != ""


def test_null_and_misaligned_pointers(L):
    d = wtconv.make_desc(2, 3, 16, 16, 2, 5, 0)
    assert call_fwd(L, d, x=0) == wtconv.WTCONV_ERR_INVALID_ARG
    assert call_fwd(L, d, w=0) == wtconv.WTCONV_ERR_INVALID_ARG
    assert call_fwd(L, d, x=FAKE + 2) == wtconv.WTCONV_ERR_MISALIGNED
    d16 = wtconv.make_desc(2, 3, 16, 16, 2, 5, 1)
    assert call_fwd(L, d16, y=FAKE + 1) == wtconv.WTCONV_ERR_MISALIGNED


def test_bwd_weight_workspace_checks(L):
    d = wtconv.make_desc(4, 8, 28, 28, 3, 5, 0)
    need = L.wtconv_workspace_size(ctypes.byref(d), wtconv.OP_BWD_WEIGHT)
    assert need > 0 and need % 256 == 0
    assert L.wtconv_workspace_size(ctypes.byref(d), wtconv.OP_FWD) == 0
    p = ctypes.c_void_p(FAKE)
    rc = L.wtconv_bwd_weight(ctypes.byref(d), p, p, p, None, p, p, p, p, None, p, p, p, p, need - 256, None)
    assert rc == wtconv.WTCONV_ERR_WORKSPACE
    rc = L.wtconv_bwd_weight(ctypes.byref(d), p, p, p, None, p, p, p, p, None, p, p, p, None, need, None)
    assert rc == wtconv.WTCONV_ERR_WORKSPACE
    rc = L.wtconv_bwd_weight(ctypes.byref(d), p, p, p, None, p, p, p, p, None, p, p, p,
                             ctypes.c_void_p(FAKE + 16), need, None)
    assert rc == wtconv.WTCONV_ERR_MISALIGNED


def test_workspace_size_invalid_desc_is_zero(L):
    d = wtconv.make_desc(4, 8, 28, 28, 3, 4, 0)
    assert L.wtconv_workspace_size(ctypes.byref(d), wtconv.OP_BWD_WEIGHT) == 0
    assert L.wtconv_workspace_size(None, wtconv.OP_BWD_WEIGHT) == 0


def test_plans_are_consistent_under_concurrent_calls(L):
    # Launch plans are cached per layer geometry inside the library and shared
    # by all threads; ctypes releases the interpreter lock during the call, so
    # these queries run concurrently in the library.  Every thread must see
    # the same workspace sizes as a single-threaded pass, for every call kind
    # (whole planes, planes beyond one CTA, the fused backward).
    import concurrent.futures
    shapes = [(N, C, H, W, lv, k, dt) for (N, C, H, W) in ((2, 3, 13, 17), (64, 96, 56, 56), (3, 4, 28, 28),
                                                          (2, 2, 150, 150), (1, 2, 57, 61), (9, 6, 7, 7))
              for lv in (1, 3) for k in (3, 5) for dt in (0, 1)]
    ops = (wtconv.OP_BWD_WEIGHT, wtconv.OP_BWD)

    def sizes():
        out = []
        for s in shapes:
            d = wtconv.make_desc(*s)
            out.append(tuple(L.wtconv_workspace_size(ctypes.byref(d), op) for op in ops))
        return out

    reference = sizes()
    assert all(a > 0 and b > 0 for a, b in reference)
    with concurrent.futures.ThreadPoolExecutor(8) as ex:
        results = list(ex.map(lambda _: sizes(), range(16)))
    for r in results:
        assert r == reference


def test_fused_backward_argument_checks(L):
    # wtconv_bwd validates everything before any launch: null and misaligned
    # activations, null required gradients, and a missing, short or
    # misaligned workspace each return their status code (no device needed).
    d = wtconv.make_desc(2, 4, 56, 56, 3, 5, 0)  # a layer the fused kernel takes
    need = L.wtconv_workspace_size(ctypes.byref(d), wtconv.OP_BWD)
    assert need > 0 and need % 256 == 0
    p = ctypes.c_void_p(FAKE)

    def call(x=FAKE, dy=FAKE, dx=FAKE, dw=FAKE, ws=FAKE, ws_bytes=None):
        v = lambda a: None if a == 0 else ctypes.c_void_p(a)
        return L.wtconv_bwd(ctypes.byref(d), v(x), v(dy), p, None, p, p, p, v(dx), v(dw), None, p, p, p, v(ws),
                            need if ws_bytes is None else ws_bytes, None)

    assert call(x=0) == wtconv.WTCONV_ERR_INVALID_ARG
    assert call(dx=0) == wtconv.WTCONV_ERR_INVALID_ARG
    assert call(dw=0) == wtconv.WTCONV_ERR_INVALID_ARG
    assert call(dy=FAKE + 2) == wtconv.WTCONV_ERR_MISALIGNED
    assert call(dx=FAKE + 1) == wtconv.WTCONV_ERR_MISALIGNED
    assert call(ws=0) == wtconv.WTCONV_ERR_WORKSPACE
    assert call(ws_bytes=need - 256) == wtconv.WTCONV_ERR_WORKSPACE
    assert call(ws=FAKE + 16) == wtconv.WTCONV_ERR_MISALIGNED
    bad = wtconv.make_desc(2, 4, 56, 56, 3, 4, 0)  # even k
    v = ctypes.c_void_p(FAKE)
    assert L.wtconv_bwd(ctypes.byref(bad), v, v, v, None, v, v, v, v, v, None, v, v, v, v, need, None) == \
        wtconv.WTCONV_ERR_INVALID_ARG
    assert L.wtconv_last_error().decode() != ""


def test_binding_argtypes_match_the_header(L):
    # every prototype's parameter count and pointer-or-integer kind, as the
    # binding declares them to ctypes
    from test_binding_host import header_params
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "wtconv.h")).read(), flags=re.S)
    for name, params in header_params().items():
        argtypes = getattr(L, name).argtypes
        assert argtypes is not None and len(argtypes) == len(params), name
        proto = re.search(r"\b" + name + r"\s*\(([^;{]*?)\)\s*;", src).group(1)
        for decl, t in zip([a.strip() for a in proto.split(",") if a.strip() not in ("", "void")], argtypes):
            if "*" in decl:
                assert t in (ctypes.c_void_p, ctypes.POINTER(wtconv.WtconvDesc)), (name, decl, t)
            elif decl.startswith("size_t"):
                assert t is ctypes.c_size_t, (name, decl, t)
            else:
                assert t is ctypes.c_int, (name, decl, t)


def test_split_layers_request_a_workspace_in_every_pass(L):
    # Layers whose tile window does not fit one CTA run as a fine pass plus a
    # coarse layer on the low-pass planes; their forward and input-gradient
    # calls need a workspace then (the low-pass and coarse-output planes), and
    # every pass's size covers the float32 low-pass planes at least.  Layers
    # that fit need none in those passes.
    split = wtconv.make_desc(2, 3, 512, 512, 5, 5, 0)  # 64-pixel halo at k = 5: split at 4 levels
    low = 2 * 3 * (512 >> 4) * (512 >> 4) * 4          # float32 bytes of the level-4 low-pass planes
    for op in (wtconv.OP_FWD, wtconv.OP_BWD_DATA):
        assert L.wtconv_workspace_size(ctypes.byref(split), op) >= 2 * low  # low-pass planes + coarse output
    assert L.wtconv_workspace_size(ctypes.byref(split), wtconv.OP_BWD_WEIGHT) >= 2 * low  # of x and of dy
    assert L.wtconv_workspace_size(ctypes.byref(split), wtconv.OP_BWD) >= 2 * low
    deep = wtconv.make_desc(1, 2, 1024, 1024, 8, 9, 1)  # the coarse layer splits again
    assert L.wtconv_workspace_size(ctypes.byref(deep), wtconv.OP_FWD) > 0
    for desc in (wtconv.make_desc(2, 3, 512, 512, 4, 5, 0), wtconv.make_desc(64, 96, 56, 56, 3, 5, 0),
                 wtconv.make_desc(2, 3, 512, 512, 5, 3, 0)):
        for op in (wtconv.OP_FWD, wtconv.OP_BWD_DATA):
            assert L.wtconv_workspace_size(ctypes.byref(desc), op) == 0, (desc.H, desc.levels, desc.k, op)
