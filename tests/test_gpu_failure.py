"""Failure detection on the GPU without a fault.

The prefill kernels bound every device-side wait.  A wait that gives up
writes STILL_ERR_TIMEOUT to the prefill's status word, its block lets the
copies and tensor-core operations it already issued complete, and the kernel
returns: nothing traps and nothing waits forever.  Here the row-side wait
limit is lowered to a few hundred clock cycles (far below the time a TMA copy
from HBM takes), so the waits give up for real; the status word must say so,
and the next call with the default limit must be exact again on the same
context.  Every parity case of the suite also reads the status word
(test_gpu_parity.prefill_checked).
"""
import numpy as np
import pytest
import torch

from linear_attention_linearization_gb300 import inputs
from linear_attention_linearization_gb300.inputs import to_f64
from oracle import brute, ref

pytestmark = pytest.mark.gpu

DEV = "cuda"
STILL_ERR_TIMEOUT = 4


@pytest.fixture(scope="module")
def still(cuda_ok):
    from linear_attention_linearization_gb300 import build
    build.build()
    ref.build()
    from linear_attention_linearization_gb300 import still as s
    return s


@pytest.mark.parametrize("name", ["tiny_prefill_n512", "llama32_1b_layer_prefill_4k"])
def test_timeout_is_reported_and_the_context_recovers(still, name):
    w = inputs.WORKLOADS[name]
    q, k, v, Wf = inputs.make_inputs(w, seed=31)
    qd, kd, vd, Wd = (t.to(DEV) for t in (q, k, v, Wf))
    ws = torch.empty(still.workspace_size(qd, kd, Wd, w.W, w.C, w.m, w.T_max), dtype=torch.uint8, device=DEV)
    still.debug_set_wait_limit(200)
    try:
        still.prefill(qd, kd, vd, Wd, w.W, w.C, w.m, w.T_max, workspace=ws)
        status = still.workspace_status(ws)
    finally:
        still.debug_set_wait_limit(0)
    assert status == STILL_ERR_TIMEOUT
    # the same context, default limit: the status word is clear and the layer exact
    out, sel = still.prefill(qd, kd, vd, Wd, w.W, w.C, w.m, w.T_max, workspace=ws)
    assert still.workspace_status(ws) == 0
    args = [to_f64(t) for t in (q, k, v, Wf)]
    y_ref, sc_ref, _ = ref.prefill(*args, w.W, w.C, w.m, w.T_max)
    sel_g = sel.cpu().numpy()
    for b in range(w.B):
        ties = set(brute.near_ties(sc_ref[b], w.C, w.lam, w.T_max))
        diff = {tuple(x) for x in np.argwhere((sel_g[b] != brute.select(sc_ref[b], w.C, w.lam, w.T_max)).any(-1))}
        assert diff <= ties
    if (sel_g != np.stack([brute.select(sc_ref[b], w.C, w.lam, w.T_max) for b in range(w.B)])).any():
        y_ref, _, _ = ref.prefill(*args, w.W, w.C, w.m, w.T_max, sel_override=sel_g)
    assert np.abs(to_f64(out) - y_ref).max() <= 1e-2 * np.abs(y_ref).max()
