"""Pins of the gradient oracle (oracle/grad.py) against things other than itself.

* hand-derived gradients of two worked examples (tests/golden/grad_hand.txt),
  one of which fixes the stabiliser's gradient (a row with one softmax key
  sends nothing to that key's logit);
* central differences of the independent C streaming oracle (still_ref.c)
  along random directions of q, k, v and Wf, with the routing held fixed, for
  W >= C and W < C, grouped and ungrouped heads, and a ragged last chunk;
* the softmax-attention reduction (lambda = 0, W >= N): the gradient of
  torch's scaled_dot_product_attention, a library routine, and no gradient
  for Wf;
* the linear-attention reduction (W = 0, lambda = 0) against central
  differences, where only the NP-Map carries the gradient to q, k and Wf;
* for the gated layer: a hand-derived gated example, central differences of
  the C oracle's gated recurrence (including the gate's pre-activations), and
  the open-gate limit, which is the ungated gradient.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import brute, grad, ref

GOLD = os.path.join(os.path.dirname(__file__), "golden", "grad_hand.txt")


def _cases():
    cases, cur = [], None
    for line in open(GOLD):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        tag, *rest = line.split(None, 1)
        if tag == "case":
            name, *nums = rest[0].split()
            cur = dict(name=name, dims=[int(x) for x in nums], vals={}, expect=[])
            cases.append(cur)
        elif tag in ("q", "k", "v", "gate"):
            cur["vals"][tag] = [float(x) for x in rest[0].split()]
        elif tag in ("dq", "dk", "dv", "dgate"):
            t, expr = rest[0].split(None, 1)
            cur["expect"].append((tag, int(t), eval(expr, {"math": math})))
        elif tag == "dWf":
            cur["expect"].append(("dWf", 0, eval(rest[0], {"math": math})))
    return cases


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_derived_gradients(case):
    N, d, W, C, m, T_max = case["dims"]
    q, k, v = (np.array(case["vals"][n]).reshape(1, 1, N, d) for n in "qkv")
    Wf = np.zeros((d, 1))
    lam = brute.lam_of(m, W, T_max)
    sel = np.full((1, 1, T_max, lam), -1)
    if "gate" in case["vals"]:
        gate = np.array(case["vals"]["gate"]).reshape(1, 1, N, d)
        _, dq, dk, dv, dWf, _, dgate = grad.layer_grad(q, k, v, Wf, W, C, sel, np.ones_like(q), gate=gate)
    else:
        _, dq, dk, dv, dWf, _ = grad.layer_grad(q, k, v, Wf, W, C, sel, np.ones_like(q))
        dgate = None
    got = {"dq": dq[0, 0, :, 0], "dk": dk[0, 0, :, 0], "dv": dv[0, 0, :, 0]}
    if dgate is not None:
        got["dgate"] = dgate[0, 0, :, 0]
    for tag, t, want in case["expect"]:
        val = dWf[0, 0] if tag == "dWf" else got[tag][t]
        assert val == pytest.approx(want, rel=1e-12, abs=1e-12), (tag, t)


def _random_case(seed, B, Hq, Hkv, N, d, df, W, C, m, T_max):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    Wf = rng.standard_normal((d, df)) / np.sqrt(d)
    dy = rng.standard_normal((B, Hq, N, d))
    lam = brute.lam_of(m, W, T_max)
    sel = np.stack([brute.select(brute.kv_scores(q[b], k[b], W), C, lam, T_max) for b in range(B)]) \
        if W >= 1 else np.full((B, Hkv, T_max, lam), -1)
    return q, k, v, Wf, dy, sel, lam


def _loss_c(q, k, v, Wf, dy, W, C, m, T_max, sel, lam):
    y, _, _ = ref.prefill(q, k, v, Wf, W, C, m, T_max, sel_override=sel.astype(np.int32) if lam > 0 else None)
    return float((y * dy).sum())


FD_CASES = [
    # B, Hq, Hkv, N, d, df, W, C, m, T_max
    (1, 2, 1, 20, 4, 3, 3, 3, 9, 3),      # W = C, grouped heads, kept keys of earlier chunks
    (1, 2, 2, 23, 4, 5, 2, 5, 8, 4),      # W < C (own-chunk kept keys stay linear), ragged tail
    (2, 4, 2, 16, 3, 4, 4, 4, 10, 3),     # two sequences, groups of two
    (1, 1, 1, 12, 4, 4, 0, 4, 0, 2),      # W = 0, lambda = 0: pure linear attention
]


@pytest.mark.parametrize("cfg", FD_CASES, ids=[f"fd{i}" for i in range(len(FD_CASES))])
def test_gradient_matches_central_differences_of_the_streaming_oracle(cfg):
    B, Hq, Hkv, N, d, df, W, C, m, T_max = cfg
    q, k, v, Wf, dy, sel, lam = _random_case(11 + N, *cfg)
    y, dq, dk, dv, dWf, _ = grad.layer_grad(q, k, v, Wf, W, C, sel, dy)
    y_c, _, _ = ref.prefill(q, k, v, Wf, W, C, m, T_max, sel_override=sel.astype(np.int32) if lam > 0 else None)
    assert np.abs(y - y_c).max() <= 1e-12 * max(1.0, np.abs(y_c).max())
    rng = np.random.default_rng(5)
    h = 1e-5
    args = {"q": q, "k": k, "v": v, "Wf": Wf}
    grads = {"q": dq, "k": dk, "v": dv, "Wf": dWf}
    for name in args:
        for _ in range(3):
            dirn = rng.standard_normal(args[name].shape)
            plus = dict(args)
            minus = dict(args)
            plus[name] = args[name] + h * dirn
            minus[name] = args[name] - h * dirn
            fd = (_loss_c(plus["q"], plus["k"], plus["v"], plus["Wf"], dy, W, C, m, T_max, sel, lam)
                  - _loss_c(minus["q"], minus["k"], minus["v"], minus["Wf"], dy, W, C, m, T_max, sel, lam)) / (2 * h)
            an = float((grads[name] * dirn).sum())
            assert an == pytest.approx(fd, rel=1e-6, abs=1e-7), name


def _loss_c_gated(q, k, v, Wf, gate, dy, W, C, m, T_max, sel, lam):
    y, _, _ = ref.prefill(q, k, v, Wf, W, C, m, T_max, sel_override=sel.astype(np.int32) if lam > 0 else None,
                          gate=gate)
    return float((y * dy).sum())


@pytest.mark.parametrize("cfg", FD_CASES[:3], ids=[f"gated_fd{i}" for i in range(3)])
def test_gated_gradient_matches_central_differences_of_the_streaming_oracle(cfg):
    # the gated layer: the C oracle's own gated recurrence, differenced along
    # random directions of q, k, v, Wf and the gate's pre-activations
    B, Hq, Hkv, N, d, df, W, C, m, T_max = cfg
    q, k, v, Wf, dy, sel, lam = _random_case(29 + N, *cfg)
    gate = np.random.default_rng(7).normal(0.0, 2.0, q.shape)
    y, dq, dk, dv, dWf, _, dgate = grad.layer_grad(q, k, v, Wf, W, C, sel, dy, gate=gate)
    y_c, _, _ = ref.prefill(q, k, v, Wf, W, C, m, T_max, sel_override=sel.astype(np.int32) if lam > 0 else None,
                            gate=gate)
    assert np.abs(y - y_c).max() <= 1e-12 * max(1.0, np.abs(y_c).max())
    rng = np.random.default_rng(6)
    h = 1e-5
    args = {"q": q, "k": k, "v": v, "Wf": Wf, "gate": gate}
    grads = {"q": dq, "k": dk, "v": dv, "Wf": dWf, "gate": dgate}
    for name in args:
        for _ in range(2):
            dirn = rng.standard_normal(args[name].shape)
            plus = dict(args)
            minus = dict(args)
            plus[name] = args[name] + h * dirn
            minus[name] = args[name] - h * dirn
            fd = (_loss_c_gated(plus["q"], plus["k"], plus["v"], plus["Wf"], plus["gate"], dy, W, C, m, T_max, sel, lam)
                  - _loss_c_gated(minus["q"], minus["k"], minus["v"], minus["Wf"], minus["gate"], dy, W, C, m, T_max,
                                  sel, lam)) / (2 * h)
            an = float((grads[name] * dirn).sum())
            assert an == pytest.approx(fd, rel=1e-6, abs=1e-7), name


def test_open_gate_gradient_is_the_ungated_gradient():
    # sigmoid(60) rounds to 1 in fp64: the gated layer is the ungated one, and the
    # gate's own gradient (sigmoid' ~ e^-60) vanishes
    cfg = FD_CASES[1]
    q, k, v, Wf, dy, sel, lam = _random_case(41, *cfg)
    W, C = cfg[6], cfg[7]
    ref_g = grad.layer_grad(q, k, v, Wf, W, C, sel, dy)
    got = grad.layer_grad(q, k, v, Wf, W, C, sel, dy, gate=np.full(q.shape, 60.0))
    for a, b in zip(ref_g[:5], got[:5]):
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(a).max())
    assert np.abs(got[6]).max() <= 1e-20 * np.abs(got[1]).max()


def test_softmax_reduction_matches_scaled_dot_product_attention():
    # lambda = 0 and W >= N: no linear keys, every earlier key in the window
    B, Hq, Hkv, N, d, df = 1, 4, 2, 17, 8, 8
    q, k, v, Wf, dy, _, _ = _random_case(3, B, Hq, Hkv, N, d, df, 32, 4, 32, 2)
    sel = np.full((B, Hkv, 2, 0), -1)
    _, dq, dk, dv, dWf, _ = grad.layer_grad(q, k, v, Wf, 32, 4, sel, dy)
    G = Hq // Hkv
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(v, requires_grad=True)
    ke = kt.repeat_interleave(G, dim=1)
    ve = vt.repeat_interleave(G, dim=1)
    yt = torch.nn.functional.scaled_dot_product_attention(qt, ke, ve, is_causal=True)
    (yt * torch.tensor(dy)).sum().backward()
    assert np.abs(dq - qt.grad.numpy()).max() <= 1e-12 * np.abs(dq).max()
    assert np.abs(dk - kt.grad.numpy()).max() <= 1e-12 * np.abs(dk).max()
    assert np.abs(dv - vt.grad.numpy()).max() <= 1e-12 * np.abs(dv).max()
    assert np.all(dWf == 0.0)


def test_row_max_override_moves_only_the_stabiliser_gradient():
    # row 3 has two equal maximal softmax logits (keys 2 and 3) and two linear keys: the
    # gradient of c moves from one key to the other, y does not change
    q = np.ones((1, 1, 4, 1))
    k = np.array([0.5, 1.0, 2.0, 2.0]).reshape(1, 1, 4, 1)
    v = np.array([1.0, 3.0, -2.0, 0.5]).reshape(1, 1, 4, 1)
    sel = np.full((1, 1, 1, 0), -1)
    dy = np.ones_like(q)
    y1, dq1, dk1, dv1, _, c1 = grad.layer_grad(q, k, v, np.zeros((1, 1)), 2, 4, sel, dy)
    assert c1[0, 0].tolist() == [0, 1, 2, 2]          # first maximal position
    cid = c1.copy()
    cid[0, 0, 3] = 3
    y2, dq2, dk2, dv2, _, c2 = grad.layer_grad(q, k, v, np.zeros((1, 1)), 2, 4, sel, dy, cidx=cid)
    assert np.array_equal(y1, y2) and np.array_equal(dv1, dv2) and np.allclose(dq1, dq2, rtol=0, atol=1e-15)
    moved = dk1[0, 0, 2, 0] - dk2[0, 0, 2, 0]
    assert abs(moved) > 1e-3
    assert dk2[0, 0, 3, 0] - dk1[0, 0, 3, 0] == pytest.approx(moved, rel=1e-12)
    assert dk1[0, 0, 0, 0] == dk2[0, 0, 0, 0] and dk1[0, 0, 1, 0] == dk2[0, 0, 1, 0]


def test_max_gaps_flags_equal_maxima():
    q = np.ones((1, 1, 4, 1))
    k = np.array([0.5, 1.0, 2.0, 2.0]).reshape(1, 1, 4, 1)
    gaps = grad.max_gaps(q, k, 2, 4, np.full((1, 1, 1, 0), -1))
    assert gaps[0, 0, 0] == np.inf           # one key
    assert gaps[0, 0, 1] == pytest.approx(0.5)
    assert gaps[0, 0, 2] == pytest.approx(1.0)
    assert gaps[0, 0, 3] == 0.0
