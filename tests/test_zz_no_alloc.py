"""The allocation-free prefill entry point (still_prefill_noalloc).

Some callers may not allocate device memory while they run (an engine plug-in
whose execution step must not allocate, latency-critical code); for them the
library offers the prefill with its scratch in a fixed array of its own.  This
file checks, through the C ABI, that it gives the same result as still_prefill
with a caller workspace on two calls in a row, and that sizes needing more
scratch than the array holds are refused without launching anything.  It is
named so that pytest collects it last.
"""
import ctypes as ct

import numpy as np
import pytest
import torch

from linear_attention_linearization_gb300 import inputs
from linear_attention_linearization_gb300.inputs import to_f64

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2   # the tolerance of every output parity test of this suite


@pytest.fixture(scope="module")
def still(cuda_ok):
    from linear_attention_linearization_gb300 import build
    build.build()
    from linear_attention_linearization_gb300 import still as s
    return s


@pytest.mark.parametrize("name", ["tiny_prefill_n512", "llama32_1b_layer_prefill_4k"])
def test_noalloc_matches_prefill_twice(still, name):
    w = inputs.WORKLOADS[name]
    assert still.lib().still_prefill_noalloc_max_bytes() == 16 << 20
    dev = torch.device("cuda")
    for seed in (21, 22):                                  # two calls in a row, different data
        q, k, v, Wf = (t.to(dev) for t in inputs.make_inputs(w, seed=seed))
        assert still.workspace_size(q, k, Wf, w.W, w.C, w.m, w.T_max) <= still.lib().still_prefill_noalloc_max_bytes()
        ws = torch.empty(still.workspace_size(q, k, Wf, w.W, w.C, w.m, w.T_max), dtype=torch.uint8, device=dev)
        ref_out, ref_sel = still.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max, workspace=ws)
        out, sel = still.prefill_noalloc(q, k, v, Wf, w.W, w.C, w.m, w.T_max)
        torch.cuda.synchronize()
        a, b = to_f64(out), to_f64(ref_out)
        assert np.abs(a - b).max() <= OUT_TOL * np.abs(b).max()
        assert torch.equal(sel.cpu(), ref_sel.cpu())


def test_noalloc_refuses_sizes_beyond_its_array(still):
    w = inputs.WORKLOADS["llama3_8b_layer_prefill_16k"]          # needs about 45 MB of scratch
    sh = still.Shape(w.B, w.Hq, w.Hkv, w.N, w.d, w.df)
    assert still.lib().still_prefill_workspace_size(ct.byref(sh), w.W, w.C, w.m, w.T_max) > (16 << 20)
    p = ct.c_void_p(256)                                          # never dereferenced: refused on the host
    rc = still.lib().still_prefill_noalloc(ct.byref(sh), p, p, p, p, w.W, w.C, w.m, w.T_max, p, None, None, None)
    assert rc == 6                                                # STILL_ERR_WORKSPACE
