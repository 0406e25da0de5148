"""Parity of the backward pass (still_backward) with the gradient oracle.

The selection is the one the GPU forward made (still_prefill's sel_idx); the
oracle (oracle/grad.py) differentiates the layer with that selection held
fixed.  Bar: for each of dq, dk, dv and dWf, max|g_gpu - g_ref| <= 1e-2 *
max|g_ref| -- the output tolerance of the forward, applied tensor by tensor.
The GPU rounds P, dS, g, phi, the block states and Wf to bf16 as MMA
operands (unit roundoff 2^-8) and accumulates in fp32, so its normwise error
is a few times 2^-8 of the terms summed; the records in the pytest summary
show how far inside the bar each case lands.

The stabiliser's gradient goes to the key where the row maximum is attained.
The GPU reports its choice (cmax_idx); it must equal the oracle's except where
the two largest logits of the row differ by less than twice the bound on the
fp32 rounding of a logit (near-equal maxima, counted and reported), and there
the oracle is evaluated with the GPU's choice.  The bound: the products of
bf16 values are exact in fp32 and a sum of d of them in any order is within
d 2^-24 sum|q_i k_i| <= d 2^-24 ||q|| ||k|| of the exact sum, then scaled by
1/sqrt(d).
"""
import numpy as np
import pytest
import torch

from conftest import record_parity
from linear_attention_linearization_gb300 import inputs
from linear_attention_linearization_gb300.inputs import Workload, to_f64
from oracle import grad

pytestmark = pytest.mark.gpu

DEV = "cuda"
GRAD_TOL = 1e-2
U_F32 = 2.0 ** -24


def logit_rounding_bound(q, k):
    """[B, Hq, N]: d 2^-24 ||q_t|| max_j ||k_j|| / sqrt(d), a bound on the fp32
    rounding of any logit of row t (max over all keys of the row's kv head)."""
    B, Hq, N, d = q.shape
    G = Hq // k.shape[1]
    nq = np.linalg.norm(q, axis=-1)
    nk = np.linalg.norm(k, axis=-1).max(axis=-1)            # [B, Hkv]
    return d * U_F32 * nq * np.repeat(nk, G, axis=1)[..., None] / np.sqrt(d)


@pytest.fixture(scope="module")
def still(cuda_ok):
    from linear_attention_linearization_gb300 import build
    build.build()
    from linear_attention_linearization_gb300 import still as s
    return s


def gpu_backward(still, w, seed, timers=False):
    q, k, v, Wf = inputs.make_inputs(w, seed=seed)
    dy = inputs.make_dout(w, seed=seed)
    qd, kd, vd, Wd, dyd = (t.to(DEV) for t in (q, k, v, Wf, dy))
    _, sel = still.prefill(qd, kd, vd, Wd, w.W, w.C, w.m, w.T_max)
    cidx = torch.full((w.B, w.Hq, w.N), -7, dtype=torch.int32, device=DEV)
    if timers:
        still.timing_read()
        still.timing_enable(True)
    try:
        dq, dk, dv, dWf = still.backward(qd, kd, vd, Wd, w.W, w.C, w.m, w.T_max, sel, dyd, cmax_idx=cidx)
        torch.cuda.synchronize()
    finally:
        if timers:
            still.timing_enable(False)
    names = set(still.timing_read()) if timers else set()
    return (q, k, v, Wf, dy), sel.cpu().numpy(), cidx.cpu().numpy(), (dq, dk, dv, dWf), names


def check_against_oracle(name, w, host, sel, cidx, grads, seqs=None):
    q, k, v, Wf, dy = (to_f64(t) for t in host)
    seqs = range(w.B) if seqs is None else seqs
    errs = {n: 0.0 for n in ("dq", "dk", "dv")}
    refmax = {n: 0.0 for n in ("dq", "dk", "dv")}
    gq, gk, gv, gW = (t.cpu().double().numpy() for t in grads)
    dW_ref = np.zeros_like(Wf)
    n_gap = n_moved = 0
    for b in seqs:
        sl = slice(b, b + 1)
        _, dq_r, dk_r, dv_r, dW_r, c_r = grad.layer_grad(q[sl], k[sl], v[sl], Wf, w.W, w.C, sel[sl], dy[sl])
        moved = cidx[sl] != c_r
        if moved.any():
            near = grad.max_gaps(q[sl], k[sl], w.W, w.C, sel[sl]) < 2 * logit_rounding_bound(q[sl], k[sl])
            n_gap += int(near.sum())
            assert near[moved].all(), "the GPU took c at another key without a near-equal maximum"
            n_moved += int(moved.sum())
            _, dq_r, dk_r, dv_r, dW_r, _ = grad.layer_grad(q[sl], k[sl], v[sl], Wf, w.W, w.C, sel[sl], dy[sl],
                                                           cidx=cidx[sl].astype(np.int64))
        for n, g_gpu, g_ref in (("dq", gq[sl], dq_r), ("dk", gk[sl], dk_r), ("dv", gv[sl], dv_r)):
            errs[n] = max(errs[n], float(np.abs(g_gpu - g_ref).max()))
            refmax[n] = max(refmax[n], float(np.abs(g_ref).max()))
        dW_ref += dW_r
    if len(seqs) == w.B:
        errs["dWf"] = float(np.abs(gW - dW_ref).max())
        refmax["dWf"] = float(np.abs(dW_ref).max())
    rel = {n: errs[n] / refmax[n] if refmax[n] > 0 else errs[n] for n in errs}
    record_parity(f"backward {name}", **{f"{n}_err_rel": rel[n] for n in rel}, rows_cmax_moved=n_moved,
                  rows_near_equal_max=n_gap, seqs=len(seqs))
    for n in rel:
        assert rel[n] <= GRAD_TOL, (n, rel)
    return rel


CASES = [
    ("tiny_prefill_n512", inputs.WORKLOADS["tiny_prefill_n512"]),
    ("g4_d128_ragged", Workload("g4_d128_ragged", 2, 8, 2, 128, 333, 64, 64, 288, 16, 128, "dirnorm", 0.05)),
    ("g2_d64_w48_c32", Workload("g2_d64_w48_c32", 1, 4, 2, 64, 200, 48, 32, 48 + 3 * 7, 7, 64)),
    ("g1_d128_lam0", Workload("g1_d128_lam0", 1, 2, 2, 128, 150, 32, 32, 32, 4, 128)),
    ("g4_d64_w_ge_n", Workload("g4_d64_w_ge_n", 1, 4, 1, 64, 90, 128, 64, 128 + 4, 2, 64)),
    # W < C: kept keys stay linear keys of their own chunk's later queries
    ("g4_d64_w16_c32", Workload("g4_d64_w16_c32", 1, 8, 2, 64, 300, 16, 32, 16 + 4 * 9, 9, 64)),
    ("g2_d128_w24_c64_ragged", Workload("g2_d128_w24_c64_ragged", 2, 4, 2, 128, 333, 24, 64, 24 + 6 * 5, 5, 128)),
    ("g1_d64_w8_c48", Workload("g1_d64_w8_c48", 1, 2, 2, 64, 200, 8, 48, 8 + 20 * 4, 4, 64)),
    ("llama32_1b_shape_n1024", Workload("llama32_1b_shape_n1024", 1, 32, 8, 64, 1024, 64, 256, 288, 16, 64)),
]


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_the_gradient_oracle(still, name, w):
    host, sel, cidx, grads, _ = gpu_backward(still, w, seed=21)
    check_against_oracle(name, w, host, sel, cidx, grads)


def test_backward_training_workload(still):
    # the training-shaped batch (B = 8 sequences of 1024 tokens, lambda = 14) in the
    # launch configuration the benchmark times; the oracle checks every element of dq,
    # dk, dv and dWf, the timers show the backward's kernels ran
    w = inputs.WORKLOADS["train_b8_n1k_chunk_parallel"]
    host, sel, cidx, grads, names = gpu_backward(still, w, seed=4, timers=True)
    assert {"bwd_query", "bwd_key", "bwd_kept", "bwd_dwf"} <= names, names
    check_against_oracle("train_b8_n1k_chunk_parallel", w, host, sel, cidx, grads)
    assert np.isfinite(grads[3].cpu().numpy()).all()


def test_backward_1b_layer_4k(still):
    # the Llama-3.2-1B-shaped layer at 4K (W = 64 < C = 256, lambda = 14): every element of
    # dq, dk, dv and dWf against the oracle
    w = inputs.WORKLOADS["llama32_1b_layer_prefill_4k"]
    host, sel, cidx, grads, names = gpu_backward(still, w, seed=4, timers=True)
    assert "bwd_kept_lin" in names, names
    check_against_oracle("llama32_1b_layer_prefill_4k", w, host, sel, cidx, grads)


def test_backward_refuses_what_it_does_not_cover(still):
    w = Workload("g8", 1, 16, 2, 64, 128, 64, 64, 128, 8, 64)   # G = 8
    q, k, v, Wf = (t.to(DEV) for t in inputs.make_inputs(w, seed=0))
    sel = torch.full((1, w.Hkv, w.T_max, w.lam), -1, dtype=torch.int32, device=DEV)
    dy = torch.zeros_like(q)
    with pytest.raises(still.StillError) as ei:
        still.backward(q, k, v, Wf, w.W, w.C, w.m, w.T_max, sel, dy)
    assert ei.value.code == 2   # STILL_ERR_UNSUPPORTED


def test_backward_of_an_empty_sequence_zeroes_dwf(still):
    w = Workload("empty", 1, 4, 2, 64, 0, 32, 32, 64, 4, 64)
    q = torch.empty((1, 4, 0, 64), dtype=torch.bfloat16, device=DEV)
    k = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device=DEV)
    Wf = torch.randn(64, 64, device=DEV)
    dWf = torch.full((64, 64), 3.0, device=DEV)
    sel = torch.full((1, 2, 4, 8), -1, dtype=torch.int32, device=DEV)
    still.backward(q, k, k, Wf, w.W, w.C, w.m, w.T_max, sel, q,
                   grads=(torch.empty_like(q, dtype=torch.float32), torch.empty_like(k, dtype=torch.float32),
                          torch.empty_like(k, dtype=torch.float32), dWf))
    torch.cuda.synchronize()
    assert (dWf == 0).all()


def test_backward_repeated_calls_and_workspace(still):
    # dq has no atomic additions: bit-identical across calls; dk, dv, dWf take atomic
    # additions in an unspecified order: equal to within fp32 reassociation
    w = Workload("rep", 2, 8, 2, 128, 300, 64, 64, 288, 16, 128, "dirnorm", 0.05)
    q, k, v, Wf = (t.to(DEV) for t in inputs.make_inputs(w, seed=8))
    dy = inputs.make_dout(w, seed=8).to(DEV)
    _, sel = still.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max)
    ws = torch.empty(still.backward_workspace_size(q, k, Wf, w.W, w.C, w.m, w.T_max), dtype=torch.uint8, device=DEV)
    a = [t.clone() for t in still.backward(q, k, v, Wf, w.W, w.C, w.m, w.T_max, sel, dy)]
    b = still.backward(q, k, v, Wf, w.W, w.C, w.m, w.T_max, sel, dy, workspace=ws)
    c = still.backward(q, k, v, Wf, w.W, w.C, w.m, w.T_max, sel, dy, workspace=ws)
    torch.cuda.synchronize()
    for x, y, z in zip(a, b, c):
        scale = x.abs().max().item()
        assert (x - y).abs().max().item() <= 1e-5 * scale and (y - z).abs().max().item() <= 1e-5 * scale
    assert torch.equal(a[0], b[0]) and torch.equal(b[0], c[0])


def test_backward_ignores_selection_entries_out_of_range(still):
    # an entry past the sequence is no token (as -1): the kernels never read its row
    w = Workload("oor", 1, 4, 2, 64, 256, 32, 32, 32 + 4 * 8, 8, 64)
    q, k, v, Wf = (t.to(DEV) for t in inputs.make_inputs(w, seed=9))
    dy = inputs.make_dout(w, seed=9).to(DEV)
    _, sel = still.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max)
    sel_a = sel.clone()
    sel_a[:, :, 2, 1] = -1
    sel_b = sel.clone()
    sel_b[:, :, 2, 1] = w.N + 1000
    ga = still.backward(q, k, v, Wf, w.W, w.C, w.m, w.T_max, sel_a, dy)
    gb = still.backward(q, k, v, Wf, w.W, w.C, w.m, w.T_max, sel_b, dy)
    torch.cuda.synchronize()
    assert torch.equal(ga[0], gb[0])
    for x, y in zip(ga[1:], gb[1:]):
        assert (x - y).abs().max().item() <= 1e-5 * x.abs().max().item()


def test_autograd_op_matches_the_gradient_oracle(still):
    # still.hybrid_attention inside a torch autograd graph: the loss sum(y * dy) gives the
    # oracle's gradients (bf16 for q, k, v as the inputs, fp32 for Wf)
    w = Workload("ag", 1, 4, 2, 64, 200, 32, 32, 32 + 8 * 4, 8, 64)
    q, k, v, Wf = inputs.make_inputs(w, seed=12)
    dy = inputs.make_dout(w, seed=12)
    qd, kd, vd, Wd = (t.to(DEV).requires_grad_(True) for t in (q, k, v, Wf))
    y = still.hybrid_attention(qd, kd, vd, Wd, w.W, w.C, w.m, w.T_max)
    (y.float() * dy.to(DEV).float()).sum().backward()
    _, sel = still.prefill(qd.detach(), kd.detach(), vd.detach(), Wd.detach(), w.W, w.C, w.m, w.T_max)
    _, dq_r, dk_r, dv_r, dW_r, _ = grad.layer_grad(*(to_f64(t) for t in (q, k, v, Wf)), w.W, w.C,
                                                   sel.cpu().numpy(), to_f64(dy))
    assert qd.grad.dtype == torch.bfloat16 and Wd.grad.dtype == torch.float32
    for g_gpu, g_ref in ((qd.grad, dq_r), (kd.grad, dk_r), (vd.grad, dv_r), (Wd.grad, dW_r)):
        err = np.abs(g_gpu.detach().cpu().double().numpy() - g_ref).max()
        assert err <= GRAD_TOL * np.abs(g_ref).max()
