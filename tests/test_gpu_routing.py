"""Parity of the routing metrics (section "Ablation Studies" of "STILL:
Content-Aware Intra-Layer Hybrid Attention for Efficient LLM Linearization",
routing metric comparison) on the CUDA path, through the C ABI, with the CPU
oracle.

Bars: uniform and random scores bit-exact (both are exact in fp32); diagonal
attention within 1e-4 relative (+1e-6) like the Self-Saliency Score; q.k and
the key norm within 1e-4 relative of the value plus 1e-5 of the largest
magnitude (fp32 sums of bf16 products); selections exact outside near ties;
the routed layer's output within 1e-2 max|y_ref|.
"""
import numpy as np
import pytest
import torch

from linear_attention_linearization_gb300 import inputs
from linear_attention_linearization_gb300.inputs import Workload, to_f64
from oracle import brute, ref

pytestmark = pytest.mark.gpu

DEV = "cuda"
OUT_TOL = 1e-2
METRICS = ["diagonal", "qk", "key_norm", "uniform", "random"]


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    from linear_attention_linearization_gb300 import build
    build.build()
    ref.build()


def still():
    from linear_attention_linearization_gb300 import still as s
    return s


def custom(B, Hq, Hkv, d, N, W, C, m, T_max, df=None):
    return Workload("case", B, Hq, Hkv, d, N, W, C, m, T_max, df or d)


CASES = {
    "tiny": inputs.WORKLOADS["tiny_prefill_n512"],
    "1b_4k": inputs.WORKLOADS["llama32_1b_layer_prefill_4k"],
    "g4_d128_ragged": custom(2, 8, 2, 128, 515, 24, 40, 24 + 5 * 6, 6),
    "g3_general": custom(1, 6, 2, 64, 301, 20, 32, 20 + 4 * 4, 4),   # G = 3: the CUDA-core score kernel
}


def check_scores(metric, got, want):
    if metric in ("uniform", "random"):
        np.testing.assert_array_equal(got, want)
    else:
        assert (np.abs(got - want) <= score_tol(metric, want)).all()


def oracle_scores(q, k, w, metric, seed):
    qa, ka = to_f64(q), to_f64(k)
    return np.stack([ref.metric_scores(qa[b], ka[b], w.W, w.C, w.lam, metric, seed, b * w.Hkv)
                     for b in range(w.B)])


@pytest.mark.parametrize("metric", METRICS)
@pytest.mark.parametrize("case", list(CASES))
def test_metric_scores(case, metric):
    w = CASES[case]
    q, k, _, _ = inputs.make_inputs(w, seed=3)
    sc = still().score_metric(q.to(DEV), k.to(DEV), w.W, w.C, w.m, w.T_max, metric, seed=123)
    check_scores(metric, sc.cpu().double().numpy(), oracle_scores(q, k, w, metric, 123))


def test_metric_scores_need_only_their_inputs():
    # position metrics read neither q nor k; the key norm reads k only
    w = CASES["tiny"]
    s = still()
    _, k, _, _ = inputs.make_inputs(w, seed=4)
    kw = dict(B=w.B, Hq=w.Hq, Hkv=w.Hkv, N=w.N, d=w.d)
    for metric in ("uniform", "random"):
        sc = s.score_metric(None, None, w.W, w.C, w.m, w.T_max, metric, seed=9, **kw).cpu().double().numpy()
        check_scores(metric, sc, oracle_scores(torch.zeros(w.B, w.Hq, w.N, w.d), k, w, metric, 9))
    sc = s.score_metric(None, k.to(DEV), w.W, w.C, w.m, w.T_max, "key_norm", Hq=w.Hq).cpu().double().numpy()
    check_scores("key_norm", sc, oracle_scores(torch.zeros(w.B, w.Hq, w.N, w.d), k, w, "key_norm", 0))


def score_tol(metric, want):
    if metric in ("uniform", "random"):
        return 0.0
    if metric == "diagonal":
        return 1e-4 * np.abs(want) + 1e-6
    return 1e-4 * np.abs(want) + 1e-5 * np.abs(want).max()


def check_selection(sel_gpu, scores_ref, w, metric):
    """Where the GPU's set differs from the oracle's, it must still be a valid
    top-lambda under the oracle scores within the scores' tolerance (exact for
    the metrics whose scores are exact).  Returns the number of such chunks."""
    n_diff = 0
    for b in range(w.B):
        sel_ref = brute.select(scores_ref[b], w.C, w.lam, w.T_max)
        tol = np.broadcast_to(score_tol(metric, scores_ref[b]), scores_ref[b].shape)
        for g, c in np.argwhere((sel_gpu[b] != sel_ref).any(axis=-1)):
            assert metric not in ("uniform", "random"), f"exact metric selection differs: b={b} g={g} c={c}"
            chunk = scores_ref[b, g, c * w.C:(c + 1) * w.C]
            ctol = tol[g, c * w.C:(c + 1) * w.C].max()
            picked = sel_gpu[b, g, c] - c * w.C
            assert chunk[picked].min() >= np.delete(chunk, picked).max() - 2 * ctol
            n_diff += 1
    return n_diff


@pytest.mark.parametrize("metric", METRICS)
@pytest.mark.parametrize("case", ["tiny", "1b_4k", "g4_d128_ragged", "g3_general"])
def test_prefill_routed(case, metric):
    w = CASES[case]
    s = still()
    q, k, v, Wf = inputs.make_inputs(w, seed=6)
    out, sel = s.prefill_routed(*(t.to(DEV) for t in (q, k, v, Wf)), w.W, w.C, w.m, w.T_max, metric, seed=77)
    torch.cuda.synchronize()
    sel_g = sel.cpu().numpy()
    qa, ka, va, Wa = (to_f64(t) for t in (q, k, v, Wf))
    y_ref, sc_ref, sel_ref = ref.prefill_routed(qa, ka, va, Wa, w.W, w.C, w.m, w.T_max, metric, seed=77)
    if w.lam > 0 and check_selection(sel_g, sc_ref, w, metric):
        y_ref, _, _ = ref.prefill_routed(qa, ka, va, Wa, w.W, w.C, w.m, w.T_max, metric, seed=77, sel=sel_g)
    y = to_f64(out)
    err = np.abs(y - y_ref).max()
    assert err <= OUT_TOL * np.abs(y_ref).max(), (err, np.abs(y_ref).max())


def test_prefill_routed_by_self_saliency_is_the_prefill():
    w = CASES["1b_4k"]
    s = still()
    args = [t.to(DEV) for t in inputs.make_inputs(w, seed=8)]
    out0, sel0 = s.prefill(*args, w.W, w.C, w.m, w.T_max)
    out1, sel1 = s.prefill_routed(*args, w.W, w.C, w.m, w.T_max, "self_saliency")
    assert torch.equal(out0, out1) and torch.equal(sel0, sel1)


def test_metric_scores_16k_layer():
    """The 16K Llama-3-8B-shaped layer, as the benchmark runs it: the per-token
    metrics over every token, diagonal attention on sampled 32-token tiles (each
    with the W - 1 keys before it, so that the oracle's windows are complete)."""
    w = inputs.WORKLOADS["llama3_8b_layer_prefill_16k"]
    q, k, _, _ = inputs.make_inputs(w, seed=0, device=DEV)
    s = still()
    qa_full, ka_full = q.cpu(), k.cpu()
    qa64, ka64 = to_f64(qa_full[0]), to_f64(ka_full[0])
    for metric in ("qk", "key_norm", "uniform", "random"):
        sc = s.score_metric(q, k, w.W, w.C, w.m, w.T_max, metric, seed=5).cpu().double().numpy()
        check_scores(metric, sc[0], ref.metric_scores(qa64, ka64, w.W, w.C, w.lam, metric, 5, 0))
    del qa64, ka64
    sc = s.score_metric(q, k, w.W, w.C, w.m, w.T_max, "diagonal").cpu().double().numpy()
    rng = np.random.default_rng(1)
    for t0 in [0, 32, 8192, w.N - 32] + [int(x) * 32 for x in rng.integers(2, w.N // 32 - 1, 4)]:
        lo = max(0, t0 - w.W + 1)
        qa = to_f64(qa_full[0, :, lo:t0 + 32])
        ka = to_f64(ka_full[0, :, lo:t0 + 32])
        want = ref.metric_scores(qa, ka, w.W, w.C, w.lam, "diagonal")[:, t0 - lo:]
        check_scores("diagonal", sc[0, :, t0:t0 + 32], want)
