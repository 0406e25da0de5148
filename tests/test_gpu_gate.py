"""Parity of the gated layer (still_prefill_gated) with the oracle's gate.

Reading of the pages' linear-branch gate ("STILL: Content-Aware Intra-Layer
Hybrid Attention for Efficient LLM Linearization", section "NP-Map:
Norm-Preserving Feature Map"): a per-channel sigmoid gate on the linear
branch's numerator.  Same bars as the ungated layer: selections exact outside
near ties, outputs within 1e-2 of max|y_ref|; the status word reads 0; the
benchmark shapes take the tensor-core kernel.
"""
import numpy as np
import pytest
import torch

from conftest import record_parity
from linear_attention_linearization_gb300 import inputs
from linear_attention_linearization_gb300.inputs import Workload, to_f64
from oracle import brute, ref

pytestmark = pytest.mark.gpu

DEV = "cuda"
OUT_TOL = 1e-2


@pytest.fixture(scope="module")
def still(cuda_ok):
    from linear_attention_linearization_gb300 import build
    build.build()
    ref.build()
    from linear_attention_linearization_gb300 import still as s
    return s


def run_gated(still, w, seed, name):
    q, k, v, Wf = inputs.make_inputs(w, seed=seed)
    a = inputs.make_gate(w, seed=seed)
    qd, kd, vd, ad, Wd = (t.to(DEV) for t in (q, k, v, a, Wf))
    ws = torch.empty(still.workspace_size(qd, kd, Wd, w.W, w.C, w.m, w.T_max), dtype=torch.uint8, device=DEV)
    still.timing_read()
    still.timing_enable(True)
    try:
        out, sel = still.prefill_gated(qd, kd, vd, ad, Wd, w.W, w.C, w.m, w.T_max, workspace=ws)
        assert still.workspace_status(ws) == 0
    finally:
        still.timing_enable(False)
    names = set(still.timing_read())
    args = [to_f64(t) for t in (q, k, v, Wf)]
    y_ref, sc_ref, _ = ref.prefill(*args, w.W, w.C, w.m, w.T_max, gate=to_f64(a))
    sel_g = sel.cpu().numpy()
    n_ties = n_diff = 0
    if w.lam > 0 and w.W >= 1:
        for b in range(w.B):
            ties = set(brute.near_ties(sc_ref[b], w.C, w.lam, w.T_max))
            n_ties += len(ties)
            sref = brute.select(sc_ref[b], w.C, w.lam, w.T_max)
            diff = {tuple(x) for x in np.argwhere((sel_g[b] != sref).any(-1))}
            assert diff <= ties
            n_diff += len(diff)
        if n_diff:
            y_ref, _, _ = ref.prefill(*args, w.W, w.C, w.m, w.T_max, gate=to_f64(a), sel_override=sel_g)
    err = np.abs(to_f64(out) - y_ref).max()
    record_parity(f"gated {name}", max_err_rel=float(err / np.abs(y_ref).max()), near_tie_chunks=n_ties,
                  sel_differs_in_ties=n_diff, sel_exact_outside_ties=True)
    assert err <= OUT_TOL * np.abs(y_ref).max()
    return out, names, (qd, kd, vd, ad, Wd)


@pytest.mark.parametrize("name", ["tiny_prefill_n512", "llama32_1b_layer_prefill_4k", "train_b8_n1k_chunk_parallel",
                                  "llama3_8b_layer_prefill_16k"])
def test_gated_workloads(still, name):
    _, names, _ = run_gated(still, inputs.WORKLOADS[name], seed=6, name=name)
    assert "hybrid_attn_gated" in names and "hybrid_attn_general_gated" not in names, names


EDGE = [
    Workload("e1", 2, 8, 2, 128, 515, 24, 40, 24 + 5 * 6, 6, 128),    # C not a multiple of 32: CUDA-core kernel
    Workload("e2", 1, 2, 1, 64, 400, 600, 64, 700, 4, 64),            # W >= N: no linear key
    Workload("e3", 1, 4, 2, 64, 300, 16, 32, 40, 8, 64),              # W < C, candidates in the tail
    Workload("e4", 1, 2, 2, 64, 333, 0, 16, 0, 4, 64),                # W = 0: linear only (CUDA-core kernel)
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
def test_gated_edge_cases(still, w):
    run_gated(still, w, seed=8, name=w.name)


def test_open_gate_equals_the_ungated_layer(still):
    w = inputs.WORKLOADS["llama32_1b_layer_prefill_4k"]
    q, k, v, Wf = (t.to(DEV) for t in inputs.make_inputs(w, seed=9))
    a = torch.full(q.shape, 40.0, dtype=torch.bfloat16, device=DEV)
    yg, sg = still.prefill_gated(q, k, v, a, Wf, w.W, w.C, w.m, w.T_max)
    y, s_ = still.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max)
    torch.cuda.synchronize()
    assert torch.equal(sg, s_)
    yg64, y64 = to_f64(yg), to_f64(y)
    assert np.abs(yg64 - y64).max() <= 2 ** -7 * np.abs(y64).max()


@pytest.mark.parametrize("w", [Workload("gdec_w_lt_c", 1, 8, 2, 64, 150, 16, 32, 16 + 4 * 6, 6, 64),
                               Workload("gdec_w_eq_c", 2, 4, 1, 128, 140, 32, 32, 32 + 3 * 5, 5, 128)],
                         ids=lambda w: w.name)
def test_gated_prefill_then_gated_decode_steps(still, w):
    # the gated layer's state is the ungated one's: a gated prefill of N0 tokens, exported,
    # continued by gated decode steps, equals the oracle's gated layer over all N tokens
    N0 = 96
    q, k, v, Wf = inputs.make_inputs(w, seed=5)
    a = inputs.make_gate(w, seed=5)
    qd, kd, vd, ad, Wd = (t.to(DEV) for t in (q, k, v, a, Wf))
    st = still.DecodeState(w.B, w.Hkv, w.d, w.df, w.C, w.m, device=DEV)
    y0, _ = still.prefill_gated(qd[:, :, :N0].contiguous(), kd[:, :, :N0].contiguous(), vd[:, :, :N0].contiguous(),
                                ad[:, :, :N0].contiguous(), Wd, w.W, w.C, w.m, w.T_max, export_state=st)
    ys = []
    for t in range(N0, w.N):
        ys.append(still.decode_step_gated(st, qd[:, :, t].contiguous(), kd[:, :, t].contiguous(),
                                          vd[:, :, t].contiguous(), ad[:, :, t].contiguous(), Wd, w.W, w.C, w.m,
                                          w.T_max))
    torch.cuda.synchronize()
    assert st.read_status() == 0
    y = torch.cat([y0, torch.stack(ys, dim=2)], dim=2)
    y_ref, _, _ = ref.prefill(*(to_f64(t) for t in (q, k, v, Wf)), w.W, w.C, w.m, w.T_max, gate=to_f64(a))
    err = np.abs(to_f64(y) - y_ref).max()
    record_parity(f"gated prefill {N0} + {w.N - N0} gated decode steps {w.name}",
                  max_err_rel=float(err / np.abs(y_ref).max()))
    assert err <= OUT_TOL * np.abs(y_ref).max()


def test_open_gate_decode_equals_ungated_decode(still):
    w = Workload("gdec_open", 1, 4, 2, 64, 120, 16, 32, 16 + 4 * 4, 4, 64)
    q, k, v, Wf = (t.to(DEV) for t in inputs.make_inputs(w, seed=6))
    sa = still.DecodeState(w.B, w.Hkv, w.d, w.df, w.C, w.m, device=DEV)
    sb = still.DecodeState(w.B, w.Hkv, w.d, w.df, w.C, w.m, device=DEV)
    still.prefill(q[:, :, :80].contiguous(), k[:, :, :80].contiguous(), v[:, :, :80].contiguous(), Wf,
                  w.W, w.C, w.m, w.T_max, export_state=sa)
    still.prefill(q[:, :, :80].contiguous(), k[:, :, :80].contiguous(), v[:, :, :80].contiguous(), Wf,
                  w.W, w.C, w.m, w.T_max, export_state=sb)
    open_gate = torch.full((w.B, w.Hq, w.d), 40.0, dtype=torch.bfloat16, device=DEV)
    for t in range(80, w.N):
        qt, kt, vt = (x[:, :, t].contiguous() for x in (q, k, v))
        ya = still.decode_step(sa, qt, kt, vt, Wf, w.W, w.C, w.m, w.T_max)
        yb = still.decode_step_gated(sb, qt, kt, vt, open_gate, Wf, w.W, w.C, w.m, w.T_max)
        assert torch.equal(ya, yb), t
