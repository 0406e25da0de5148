"""Host-side checks of the C ABI: the library builds, loads and exports every
entry point include/still.h declares; host-only calls (argument checks,
workspace sizing, status strings) behave as documented.  No kernel runs."""
import ctypes as ct
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from linear_attention_linearization_gb300 import build, still
    build.build()
    return still.lib()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(still_[a-z_0-9]+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert {"still_score", "still_select", "still_prefill", "still_decode_step"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_binding_covers_every_symbol():
    from linear_attention_linearization_gb300 import still
    assert declared_symbols() <= set(still.SIGNATURES)


def test_status_strings_and_lambda(lib):
    from linear_attention_linearization_gb300 import still
    for code in range(7):
        assert lib.still_status_string(code).decode() == still.STATUS[code]
    assert lib.still_lambda(64, 288, 64) == 3
    assert lib.still_lambda(64, 288, 16) == 14
    assert lib.still_lambda(64, 128, 8) == 8
    assert lib.still_lambda(64, 32, 8) == -1
    assert lib.still_lambda(0, 0, 3) == 0


def test_workspace_size_and_argument_errors(lib):
    from linear_attention_linearization_gb300.still import Shape, DecodeStateC
    sh = Shape(1, 32, 8, 16384, 128, 128)
    ws = lib.still_prefill_workspace_size(ct.byref(sh), 64, 256, 288, 64)
    assert ws > 0 and ws % 256 == 0
    assert lib.still_prefill_workspace_size(ct.byref(Shape(1, 3, 2, 16, 64, 64)), 4, 4, 8, 2) == 0  # Hq % Hkv
    assert lib.still_prefill_workspace_size(ct.byref(sh), 64, 256, 32, 64) == 0                      # m < W
    # rejected on the host, before any CUDA call
    p = ct.c_void_p(16)
    bad = ct.c_void_p(18)
    args = lambda q, out: (ct.byref(sh), q, p, p, p, 64, 256, 288, 64, out, None, None, 0, None, None)
    assert lib.still_prefill(*args(None, p)) == 1            # null q
    assert lib.still_prefill(*args(bad, p)) == 1             # misaligned q
    assert lib.still_prefill(*args(p, None)) == 1            # null out
    sh_bad = Shape(1, 32, 8, 16384, 96, 96)
    assert lib.still_prefill(ct.byref(sh_bad), p, p, p, p, 64, 256, 288, 64, p, None, None, 0, None, None) == 2
    sh0 = Shape(1, 32, 8, 16384, 128, 128)
    assert lib.still_prefill(ct.byref(sh0), p, p, p, p, 0, 256, 64, 64, p, None, None, 0, None, None) == 1  # W=0, lambda>0
    assert lib.still_prefill(ct.byref(sh0), p, p, p, p, 64, 256, 288, 64, p, None, p, 100, None, None) == 6  # small ws
    st = DecodeStateC()
    assert lib.still_decode_step(ct.byref(sh), ct.byref(st), p, p, p, p, 64, 256, 288, 64, p, None) == 1
    assert lib.still_decode_step_gated(ct.byref(sh), ct.byref(st), p, p, p, None, p, 64, 256, 288, 64, p,
                                       None) == 1                    # no gate
    assert lib.still_score(ct.byref(sh), p, p, 0, p, None) == 1
    # routing metrics: unknown metric, missing inputs, windowed metric without a window
    assert lib.still_score_metric(ct.byref(sh), p, p, 64, 256, 288, 64, 6, 0, p, None) == 1
    assert lib.still_score_metric(ct.byref(sh), p, p, 64, 256, 288, 64, -1, 0, p, None) == 1
    assert lib.still_score_metric(ct.byref(sh), None, p, 64, 256, 288, 64, 2, 0, p, None) == 1   # q.k without q
    assert lib.still_score_metric(ct.byref(sh), p, None, 64, 256, 288, 64, 3, 0, p, None) == 1   # key norm without k
    assert lib.still_score_metric(ct.byref(sh), p, p, 64, 256, 288, 64, 4, 0, None, None) == 1   # no scores
    assert lib.still_score_metric(ct.byref(sh), p, p, 0, 256, 0, 64, 1, 0, p, None) == 1         # diagonal, W = 0
    assert lib.still_score_metric(ct.byref(sh), p, p, 64, 256, 32, 64, 4, 0, p, None) == 1       # m < W
    rargs = lambda metric, q: (ct.byref(sh), q, p, p, p, 64, 256, 288, 64, metric, 0, p, None, None, 0, None)
    assert lib.still_prefill_routed(*rargs(7, p)) == 1
    assert lib.still_prefill_routed(*rargs(2, None)) == 1
    assert lib.still_prefill_routed(*rargs(2, bad)) == 1



def test_backward_argument_errors(lib):
    from linear_attention_linearization_gb300.still import Shape
    p = ct.c_void_p(16)
    bad = ct.c_void_p(18)
    tr = Shape(8, 32, 8, 1024, 128, 128)
    assert lib.still_backward_workspace_size(ct.byref(tr), 64, 64, 288, 16) > 0
    assert lib.still_backward_workspace_size(ct.byref(tr), 64, 64, 32, 16) == 0          # m < W
    args = lambda sh, W, C, q, dWf: (ct.byref(sh), q, p, p, p, W, C, 288, 16, p, p, p, p, p, dWf, None, None, 0,
                                     None)
    tr_big = Shape(1, 32, 8, 1024, 128, 128)
    assert lib.still_backward(ct.byref(tr_big), p, p, p, p, 64, 256, 64 + 16 * 129, 16, p, p, p, p, p, p, None, None,
                              0, None) == 2                           # W < C with lambda > 128
    assert lib.still_backward(*args(Shape(1, 24, 3, 64, 128, 128), 64, 64, p, p)) == 2   # G = 8
    assert lib.still_backward(*args(Shape(1, 8, 2, 64, 128, 64), 64, 64, p, p)) == 2     # d != d_f
    assert lib.still_backward(*args(tr, 64, 64, None, p)) == 1        # null q
    assert lib.still_backward(*args(tr, 64, 64, bad, p)) == 1         # misaligned q
    assert lib.still_backward(*args(tr, 64, 64, p, None)) == 1        # null dWf
    assert lib.still_backward(ct.byref(tr), p, p, p, p, 64, 64, 288, 16, None, p, p, p, p, p, None, None, 0,
                              None) == 1                              # no selection with lambda > 0
    assert lib.still_backward(ct.byref(tr), p, p, p, p, 64, 64, 288, 16, p, p, p, p, p, p, None, p, 100,
                              None) == 6                              # workspace too small

def test_oracle_library_shares_nothing_with_cuda_path():
    """The oracle is built from its own C file and links no CUDA library."""
    from oracle import ref
    path = ref.build()
    src = open(os.path.join(ROOT, "oracle", "still_ref.c")).read()
    assert "#include \"" not in src                 # no project header
    assert os.path.exists(path)
    for fn in os.listdir(os.path.join(ROOT, "linear_attention_linearization_gb300", "csrc")):
        body = open(os.path.join(ROOT, "linear_attention_linearization_gb300", "csrc", fn)).read()
        assert "oracle" not in body.lower()


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "linear_attention_linearization_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            body = open(os.path.join(pkg, fn)).read()
            assert "import oracle" not in body and "from oracle" not in body, fn
