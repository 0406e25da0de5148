"""The allocation-free prefill entry point (still_prefill_noalloc).

Some callers may not allocate device memory while they run (an engine plug-in
whose execution step must not allocate, latency-critical code); for them the
library offers the prefill with its scratch in a fixed array of its own.  This
file checks, through the C ABI, that it gives the same result as still_prefill
with a caller workspace on two calls in a row, and that sizes needing more
scratch than the array holds are refused without launching anything, that
sizes still_prefill refuses are refused with the same status, and that the
call takes nothing from the device's stream-ordered memory pool (the one a
workspace-less still_prefill draws from).  It is named so that pytest collects
it last.
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


class _PoolProbe:
    """High-water mark of the memory pool cudaMallocAsync uses on the current
    device (CUDA driver API: CU_MEMPOOL_ATTR_USED_MEM_HIGH / _CURRENT)."""
    USED_CURRENT, USED_HIGH = 7, 8

    def __init__(self):
        self.cu = ct.CDLL("libcuda.so.1")
        dev = ct.c_int(0)
        assert self.cu.cuCtxGetDevice(ct.byref(dev)) == 0
        self.pool = ct.c_void_p()
        assert self.cu.cuDeviceGetMemPool(ct.byref(self.pool), dev) == 0

    def _get(self, attr):
        v = ct.c_uint64(0)
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ct.byref(v)) == 0
        return v.value

    def reset(self):
        zero = ct.c_uint64(0)
        assert self.cu.cuMemPoolSetAttribute(self.pool, self.USED_HIGH, ct.byref(zero)) == 0
        return self._get(self.USED_CURRENT)

    def high(self):
        return self._get(self.USED_HIGH)


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
        out, sel = torch.empty_like(ref_out), torch.empty_like(ref_sel)
        torch.cuda.synchronize()
        probe = _PoolProbe()
        base = probe.reset()
        still.prefill_noalloc(q, k, v, Wf, w.W, w.C, w.m, w.T_max, out=out, sel_idx=sel)
        torch.cuda.synchronize()
        assert probe.high() == base, "still_prefill_noalloc took memory from the stream-ordered pool"
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


def test_noalloc_refuses_what_prefill_refuses(still):
    """d outside {64, 128}: both entry points answer STILL_ERR_UNSUPPORTED."""
    sh = still.Shape(1, 2, 2, 64, 96, 96)
    p = ct.c_void_p(256)                                          # never dereferenced: refused on the host
    assert still.lib().still_prefill(ct.byref(sh), p, p, p, p, 8, 8, 16, 1, p, None, None, 0, None, None) == 2
    assert still.lib().still_prefill_noalloc(ct.byref(sh), p, p, p, p, 8, 8, 16, 1, p, None, None, None) == 2


def test_pool_probe_sees_a_workspace_allocation(still):
    """The probe above is live: a still_prefill without a workspace takes its
    workspace from that pool, and the high-water mark shows it."""
    w = inputs.WORKLOADS["tiny_prefill_n512"]
    q, k, v, Wf = (t.to("cuda") for t in inputs.make_inputs(w, seed=23))
    torch.cuda.synchronize()
    probe = _PoolProbe()
    base = probe.reset()
    still.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max)
    torch.cuda.synchronize()
    assert probe.high() >= base + still.workspace_size(q, k, Wf, w.W, w.C, w.m, w.T_max)
