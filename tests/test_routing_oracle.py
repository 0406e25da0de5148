"""Pins of the routing-metric oracle (the metrics of the routing comparison in
"STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
Linearization", section "Ablation Studies") against values fixed outside it:
published generator outputs, hand-derived offsets and norms, the Self-Saliency
closed form, and the brute-force set definition of the layer.
"""
import math

import numpy as np
import pytest

from oracle import brute, ref

from linear_attention_linearization_gb300 import inputs


def custom(B, Hq, Hkv, d, N, W, C, m, T_max, df):
    return inputs.Workload("case", B, Hq, Hkv, d, N, W, C, m, T_max, df)


def test_random_metric_reproduces_published_splitmix64_outputs():
    # SplitMix64 started at seed 0 (Steele, Lea, Flood 2014; the reference
    # implementation's first three outputs): 0xE220A8397B1DCDAF,
    # 0x6E789E6AA1B965F4, 0x06C45D188009454F; the score keeps the top 24 bits
    published = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    s = ref.metric_scores(np.zeros((1, 3, 4)), np.zeros((1, 3, 4)), 1, 3, 1, "random", seed=0)
    assert s.shape == (1, 3)
    assert s[0].tolist() == [(z >> 40) / 2.0 ** 24 for z in published]


def test_random_metric_counter_layout_and_range():
    # the flat index (b Hkv + g) N + t: sequence 1 continues where sequence 0 ends
    q = np.zeros((2, 5, 4))
    both = ref.metric_scores(q, np.zeros((2, 5, 4)), 1, 5, 1, "random", seed=7, unit0=0)
    second = ref.metric_scores(q[:1], np.zeros((1, 5, 4)), 1, 5, 1, "random", seed=7, unit0=1)
    np.testing.assert_array_equal(both[1], second[0])
    big = ref.metric_scores(np.zeros((1, 100000, 1)), np.zeros((1, 100000, 1)), 1, 64, 1, "random", seed=3)
    assert big.min() >= 0.0 and big.max() < 1.0
    assert abs(big.mean() - 0.5) < 0.005 and abs(big.var() - 1.0 / 12) < 0.002
    other = ref.metric_scores(np.zeros((1, 64, 1)), np.zeros((1, 64, 1)), 1, 64, 1, "random", seed=4)
    assert not np.array_equal(big[0, :64], other[0])


@pytest.mark.parametrize("C,lam,offsets", [
    (8, 3, [1, 4, 6]),            # floor(8/6), floor(24/6), floor(40/6)
    (256, 3, [42, 128, 213]),     # floor(256/6), floor(768/6), floor(1280/6)
    (64, 1, [32]),
    (10, 4, [1, 3, 6, 8]),        # floor(10/8), floor(30/8), floor(50/8), floor(70/8)
    (4, 4, [0, 1, 2, 3]),
    (4, 6, [0, 1, 2, 3]),         # lambda >= C keeps every offset
])
def test_uniform_metric_hand_offsets(C, lam, offsets):
    N = 3 * C
    s = ref.metric_scores(np.zeros((1, N, 2)), np.zeros((1, N, 2)), 1, C, lam, "uniform")
    want = np.zeros(N)
    for c in range(3):
        want[[c * C + o for o in offsets]] = 1.0
    np.testing.assert_array_equal(s[0], want)
    # the selection of the completed chunks is exactly those offsets
    sel = ref.select(s, C, lam, 3)
    for c in range(3):
        got = [int(x) - c * C for x in sel[0, c] if x >= 0]
        assert got == offsets[:lam]


def test_key_norm_and_qk_hand_values():
    k = np.array([[[3.0, 4.0], [1.0, 2.0]]])          # one kv head, two tokens, d = 2
    np.testing.assert_allclose(ref.metric_scores(np.zeros((1, 2, 2)), k, 1, 2, 1, "key_norm")[0],
                               [5.0, math.sqrt(5.0)])
    q = np.array([[[1.0, 2.0], [0.0, 1.0]], [[-1.0, 1.0], [2.0, 2.0]]])   # two query heads of the group
    s = ref.metric_scores(q, k, 1, 2, 1, "qk")[0]
    # token 0: (1*3 + 2*4 + (-3 + 4)) / sqrt(2) / 2; token 1: (0 + 2 + 2 + 4) / sqrt(2) / 2
    np.testing.assert_allclose(s, [12.0 / math.sqrt(2.0) / 2.0, 8.0 / math.sqrt(2.0) / 2.0])


def test_diagonal_metric_special_cases_and_closed_form():
    rng = np.random.default_rng(0)
    # token 0 attends only to itself; equal keys give every window key weight 1/n
    q = rng.standard_normal((1, 6, 4))
    k = np.tile(rng.standard_normal((1, 1, 4)), (1, 6, 1))
    s = ref.metric_scores(q, k, 3, 6, 1, "diagonal")[0]
    np.testing.assert_allclose(s, [1.0, 1 / 2, 1 / 3, 1 / 3, 1 / 3, 1 / 3], rtol=1e-12)
    # one head per group: the Self-Saliency Score is -log(1 - p + 1e-6) of this p
    q = rng.standard_normal((2, 40, 8))
    k = rng.standard_normal((2, 40, 8)) * 2.0
    p = ref.metric_scores(q, k, 7, 8, 2, "diagonal")
    _, sal = ref.scores(q, k, 7)
    np.testing.assert_allclose(-np.log(1.0 - p + 1e-6), sal, rtol=1e-9, atol=1e-12)
    # grouped heads: the mean of the per-head values
    q4 = rng.standard_normal((4, 30, 8))
    k2 = rng.standard_normal((2, 30, 8))
    pg = ref.metric_scores(q4, k2, 5, 8, 2, "diagonal")
    per = [ref.metric_scores(q4[h:h + 1], k2[h // 2:h // 2 + 1], 5, 8, 2, "diagonal")[0] for h in range(4)]
    np.testing.assert_allclose(pg, [(per[0] + per[1]) / 2, (per[2] + per[3]) / 2], rtol=1e-12)


@pytest.mark.parametrize("metric", ["diagonal", "qk", "key_norm", "uniform", "random"])
def test_routed_prefill_equals_set_definition(metric):
    # the streaming oracle run on the metric's selection against the brute-force
    # SA / LA sets with the same selection; W < C and a ragged tail
    w = custom(B=1, Hq=4, Hkv=2, d=16, N=70, W=6, C=16, m=6 + 2 * 4, T_max=4, df=16)
    q, k, v, Wf = (inputs.to_f64(t) for t in inputs.make_inputs(w, seed=5))
    y, sc, sel = ref.prefill_routed(q, k, v, Wf, w.W, w.C, w.m, w.T_max, metric, seed=11)
    yb, _, _ = brute.prefill(q[0], k[0], v[0], Wf, w.W, w.C, w.m, w.T_max, sel=sel[0])
    np.testing.assert_allclose(y[0], yb, rtol=1e-9, atol=1e-12)
    if metric == "uniform":   # lambda = 2 of C = 16: offsets 4 and 12 of every completed chunk
        for c in range(w.N // w.C):
            assert sel[0, :, c].tolist() == [[c * 16 + 4, c * 16 + 12]] * 2


def test_routed_prefill_with_self_saliency_is_the_prefill():
    w = custom(B=2, Hq=2, Hkv=1, d=16, N=50, W=4, C=8, m=4 + 2 * 6, T_max=6, df=16)
    q, k, v, Wf = (inputs.to_f64(t) for t in inputs.make_inputs(w, seed=2))
    y, sc, _ = ref.prefill_routed(q, k, v, Wf, w.W, w.C, w.m, w.T_max, "self_saliency")
    y0, sc0, _ = ref.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max)
    # the same layer; the given selection changes only the order of the folds
    np.testing.assert_allclose(y, y0, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(sc, sc0)
