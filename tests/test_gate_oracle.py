"""Pins of the oracle's linear-branch gate (CPU only).

The pages say a gate raises the linear branch's rank ("STILL: Content-Aware
Intra-Layer Hybrid Attention for Efficient LLM Linearization", section
"NP-Map: Norm-Preserving Feature Map"; ablation: removing it costs 5.8
points) but its equation did not survive extraction.  The reading taken: a
per-channel sigmoid gate g_t = 1/(1+exp(-a_t)) on the linear branch's
numerator, the shared denominator ungated.  Pinned by a hand-worked example,
the g = 1 reduction to the ungated layer, the brute-force set definition with
random gates, and prefill == prefill + decode steps under a gate.
"""
import numpy as np
import pytest

from conftest import read_golden
from linear_attention_linearization_gb300 import inputs
from linear_attention_linearization_gb300.inputs import to_f64
from oracle import brute, ref


def hand_inputs():
    q = np.array([1.0, 2.0]).reshape(1, 1, 2, 1)
    k = np.array([3.0, -1.0]).reshape(1, 1, 2, 1)
    v = np.array([5.0, 7.0]).reshape(1, 1, 2, 1)
    return q, k, v, np.zeros((1, 1))


def test_hand_example():
    q, k, v, Wf = hand_inputs()
    for line in read_golden("gate_hand.txt"):
        _, a0, a1, y0, y1 = line.split()
        gate = np.array([float(a0), float(a1)]).reshape(1, 1, 2, 1)
        y, _, _ = ref.prefill(q, k, v, Wf, 1, 2, 1, 1, gate=gate)
        assert abs(y[0, 0, 0, 0] - float(y0)) < 1e-14
        assert abs(y[0, 0, 1, 0] - float(y1)) < 1e-14
        yb, _, _ = brute.prefill(q[0], k[0], v[0], Wf, 1, 2, 1, 1, gate=gate[0])
        assert abs(yb[0, 1, 0] - float(y1)) < 1e-14


CASES = [
    inputs.Workload("a", 1, 4, 2, 16, 70, 8, 16, 8 + 3 * 4, 4, 16),     # W < C
    inputs.Workload("b", 1, 2, 1, 16, 50, 12, 6, 12 + 2 * 5, 5, 8),     # W > C, d_f < d
    inputs.Workload("c", 1, 2, 2, 8, 41, 0, 8, 0, 3, 8),                # W = 0: linear only
    inputs.Workload("d", 1, 3, 3, 16, 37, 40, 16, 48, 2, 16),           # W > N: softmax only
]


def gate_for(w, rng, extreme=False):
    a = rng.standard_normal((w.B, w.Hq, w.N, w.d)) * 2.0
    if extreme:
        a[..., ::3] = 40.0
        a[..., 1::3] = -40.0
    return a


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_open_gate_is_the_ungated_layer(w):
    q, k, v, Wf = (to_f64(t) for t in inputs.make_inputs(w, seed=1))
    y0, _, _ = ref.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max)
    y1, _, _ = ref.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max, gate=np.full(q.shape, 40.0))
    assert np.abs(y1 - y0).max() <= 1e-13 * max(np.abs(y0).max(), 1.0)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("extreme", [False, True])
def test_streaming_oracle_equals_set_definition_with_gates(w, extreme):
    q, k, v, Wf = (to_f64(t) for t in inputs.make_inputs(w, seed=2))
    a = gate_for(w, np.random.default_rng(3), extreme)
    y, sc, _ = ref.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max, gate=a)
    yb, _, _ = brute.prefill(q[0], k[0], v[0], Wf, w.W, w.C, w.m, w.T_max, gate=a[0])
    assert np.abs(y[0] - yb).max() <= 1e-10 * max(np.abs(yb).max(), 1.0)
    if w.W > 0 and w.N > w.W:
        # the gate changes the output (the linear branch is not empty)
        y0, _, _ = ref.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max)
        assert np.abs(y - y0).max() > 1e-6


@pytest.mark.parametrize("w", CASES[:3], ids=lambda w: w.name)
def test_gated_prefill_then_decode_equals_gated_prefill(w):
    q, k, v, Wf = (to_f64(t) for t in inputs.make_inputs(w, seed=4))
    a = gate_for(w, np.random.default_rng(5))
    y_all, _, _ = ref.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max, gate=a)
    n0 = w.N // 2
    y0, _, st = ref.prefill(q[:, :, :n0], k[:, :, :n0], v[:, :, :n0], Wf, w.W, w.C, w.m, w.T_max,
                            gate=a[:, :, :n0])
    np.testing.assert_array_equal(y0, y_all[:, :, :n0])
    for t in range(n0, w.N):
        yt = ref.decode_step(st, q[:, :, t], k[:, :, t], v[:, :, t], Wf, w.W, w.C, w.m, w.T_max,
                             gate_t=a[:, :, t])
        np.testing.assert_array_equal(yt, y_all[:, :, t])
