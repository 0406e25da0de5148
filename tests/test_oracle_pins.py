"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Neither oracle (C streaming recurrence, NumPy set definition) is trusted on its
own: each test below checks one of them against a hand-worked example, a closed
form, a textbook routine, an invariant or the other oracle on tiny inputs.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

from conftest import read_golden
from oracle import brute, ref

rng = np.random.default_rng(1234)


def rand_case(B, Hq, Hkv, N, d, df, scale=1.0):
    q = rng.standard_normal((B, Hq, N, d)) * scale
    k = rng.standard_normal((B, Hkv, N, d)) * scale
    v = rng.standard_normal((B, Hkv, N, d))
    Wf = rng.standard_normal((d, df)) / np.sqrt(d)
    return q, k, v, Wf


# --------------------------------------------------------------------------
# Self-Saliency score
# --------------------------------------------------------------------------

def test_score_closed_form_is_kl_of_window_distributions():
    """KL(a^nodiag || a^diag) written out from the two window distributions
    equals -log(1-p); the oracle's regularised score is within eps/(1-p)."""
    Hq = Hkv = 1
    N, d, W = 40, 8, 6
    q, k, _, _ = rand_case(1, Hq, Hkv, N, d, 4)
    hs, _ = ref.scores(q[0], k[0], W)
    hs_b = brute.head_scores(q[0], k[0], W)
    for t in range(1, N):
        lo = max(0, t - W + 1)
        s = k[0, 0, lo:t + 1] @ q[0, 0, t] / math.sqrt(d)
        a_diag = np.exp(s) / np.exp(s).sum()
        a_nod = np.exp(s[:-1]) / np.exp(s[:-1]).sum()
        kl = float(np.sum(a_nod * np.log(a_nod / a_diag[:-1])))
        one_minus_p = 1.0 - a_diag[-1]
        assert kl == pytest.approx(-math.log(one_minus_p), rel=1e-9, abs=1e-12)
        bound = 1e-6 / one_minus_p * 1.01 + 1e-12
        assert abs(hs[0, t] - kl) <= bound
        assert abs(hs_b[0, t] - kl) <= bound


def test_score_first_token_has_only_itself():
    q, k, _, _ = rand_case(1, 2, 1, 10, 8, 8)
    hs, s = ref.scores(q[0], k[0], 4)
    assert hs[:, 0] == pytest.approx(-math.log(1e-6), rel=1e-14)
    assert s[0, 0] == pytest.approx(13.815510557964274, rel=1e-14)


def test_proposition1_score_is_monotone_in_self_probability():
    """Proposition 1 (section "Theoretical Guarantee: Local-Global
    Consistency"): raising the self logit raises the score."""
    N, d, W = 24, 8, 5
    q, k, _, _ = rand_case(1, 1, 1, N, d, 8)
    t = 17
    base = ref.scores(q[0], k[0], W)[1][0, t]
    prev = base
    for step in range(1, 6):
        k2 = k.copy()
        k2[0, 0, t] += 0.1 * step * q[0, 0, t]       # raises s_tt only in row t
        cur = ref.scores(q[0], k2[0], W)[1][0, t]
        assert cur > prev
        prev = cur


def test_group_score_is_mean_over_query_heads():
    q, k, _, _ = rand_case(1, 4, 1, 30, 8, 8)
    hs, s = ref.scores(q[0], k[0], 7)
    np.testing.assert_allclose(s[0], hs.mean(axis=0), rtol=1e-13)


@pytest.mark.parametrize("name", ["A", "B"])
def test_hand_example_scores_and_outputs(name):
    lines = read_golden("hand_examples.txt")
    cases, cur = {}, None
    for ln in lines:
        tok = ln.split()
        if tok[0] == "case":
            cur = cases.setdefault(tok[1], {"hdr": list(map(int, tok[2:])), "y": {}, "score": {}})
        elif tok[0] in ("q", "k", "v"):
            cur[tok[0]] = np.array(list(map(float, tok[1:])))
        else:
            cur[tok[0]][int(tok[1])] = eval(" ".join(tok[2:]), {"math": math})
    c = cases[name]
    N, d, W, C, m, T_max = c["hdr"]
    q = c["q"].reshape(1, 1, N, 1)
    k = c["k"].reshape(1, 1, N, 1)
    v = c["v"].reshape(1, 1, N, 1)
    Wf = np.zeros((1, 1))
    y, sc, _ = ref.prefill(q, k, v, Wf, W, C, m, T_max)
    yb, scb, _ = brute.prefill(q[0], k[0], v[0], Wf, W, C, m, T_max)
    for t, val in c["y"].items():
        assert y[0, 0, t, 0] == pytest.approx(val, rel=1e-13)
        assert yb[0, t, 0] == pytest.approx(val, rel=1e-13)
    for t, val in c["score"].items():
        assert sc[0, 0, t] == pytest.approx(val, rel=1e-12)
        assert scb[0, t] == pytest.approx(val, rel=1e-12)


# --------------------------------------------------------------------------
# Selection
# --------------------------------------------------------------------------

def test_hand_selection_with_distinct_scores():
    lines = read_golden("select_w2_c4.txt")
    kk = sel_exp = None
    sc_exp = {}
    for ln in lines:
        tok = ln.split()
        if tok[0] == "k":
            kk = np.array(list(map(float, tok[1:])))
        elif tok[0] == "sel":
            sel_exp = list(map(int, tok[1:]))
        elif tok[0] == "score":
            sc_exp[int(tok[1])] = eval(" ".join(tok[2:]), {"math": math})
    N = kk.size
    q = np.ones((1, 1, N, 1))
    k = kk.reshape(1, 1, N, 1)
    v = rng.standard_normal((1, 1, N, 1))
    W, C, m, T_max = 2, 4, 6, 2
    lam = ref.lam_of(m, W, T_max)
    assert lam == 2
    _, sc, st = ref.prefill(q, k, v, np.zeros((1, 1)), W, C, m, T_max)
    for t, val in sc_exp.items():
        assert sc[0, 0, t] == pytest.approx(val, rel=1e-12)
    sel_c = ref.select(sc[0], C, lam, T_max)
    sel_b = brute.select(brute.kv_scores(q[0], k[0], W), C, lam, T_max)
    assert sel_c.reshape(-1).tolist() == sel_exp
    assert sel_b.reshape(-1).tolist() == sel_exp
    # the streaming recurrence kept exactly these tokens in its budget slots
    kept = sorted(p for p in st.pos[0, 0, W:].tolist() if p >= 0)
    assert kept == sel_exp


def test_select_special_cases():
    s = rng.standard_normal((2, 40))
    assert ref.select(s, 8, 0, 5).size == 0
    allk = ref.select(s, 8, 8, 5)                    # lambda == C keeps every token
    assert allk[0, 2].tolist() == list(range(16, 24))
    over = ref.select(s, 4, 6, 10)                   # lambda > C: C tokens, -1 pad
    assert over[1, 3].tolist() == [12, 13, 14, 15, -1, -1]
    tie = ref.select(np.zeros((1, 16)), 8, 3, 2)     # exact ties: lower positions
    assert tie[0].tolist() == [[0, 1, 2], [8, 9, 10]]
    part = ref.select(s, 16, 2, 5)                   # the partial chunk 2 keeps nothing
    assert part[0, 2].tolist() == [-1, -1]
    cap = ref.select(s, 8, 2, 3)                     # T_max caps the chunks kept
    assert cap.shape == (2, 3, 2) and (cap >= 0).all()


def test_select_matches_brute_sort():
    for _ in range(20):
        Hkv, C = 3, int(rng.integers(1, 12))
        N = int(rng.integers(1, 80))
        lam = int(rng.integers(0, C + 2))
        T_max = int(rng.integers(1, 12))
        s = np.round(rng.standard_normal((Hkv, N)), 1)   # rounding makes ties common
        a = ref.select(s, C, lam, T_max)
        b = brute.select(s, C, lam, T_max)
        assert a.tolist() == b.tolist()


# --------------------------------------------------------------------------
# Routing table and the two oracles against each other
# --------------------------------------------------------------------------

def _golden_routing():
    lines = read_golden("routing_w1_c2.txt")
    sel = list(map(int, lines[0].split()[1:]))
    table = {}
    for ln in lines[1:]:
        t, rest = ln.split(":")
        sa, la = rest.split("|")
        table[int(t)] = (sorted(map(int, sa.split())), sorted(map(int, la.split())))
    return sel, table


def test_routing_table_hand_derived():
    sel, table = _golden_routing()
    N, W, C, m, T_max = 8, 1, 2, 3, 2
    lam = brute.lam_of(m, W, T_max)
    assert lam == 1
    scores = np.full((1, N), -math.log(1e-6))
    bsel = brute.select(scores, C, lam, T_max)
    assert [x for x in bsel.reshape(-1).tolist() if x >= 0] == sel
    sa, la = brute.route_masks(brute.kept_mask(bsel, N)[0], N, W, C)
    for t, (sa_t, la_t) in table.items():
        assert np.flatnonzero(sa[t]).tolist() == sa_t
        assert np.flatnonzero(la[t]).tolist() == la_t

    # Read the sets back from the streaming oracle's outputs: v_j = e_j.
    d = N
    v = np.eye(N).reshape(1, 1, N, d)
    # (1) q = 0: every softmax key weighs 1 and phi(q) = 0 -> y = mean of SA values
    q = np.zeros((1, 1, N, d))
    k = rng.standard_normal((1, 1, N, d))
    y, _, _ = ref.prefill(q, k, v, np.zeros((d, 4)), W, C, m, T_max)
    for t, (sa_t, _) in table.items():
        exp = np.zeros(d)
        exp[sa_t] = 1.0 / len(sa_t)
        np.testing.assert_allclose(y[0, 0, t], exp, atol=1e-14)
    # (2) q orthogonal to all keys (softmax weights 1) and huge norms: linear
    #     weights ||q|| ||k|| = 1e6 dominate -> y ~ mean of LA values
    q = np.zeros((1, 1, N, d)); q[..., 1] = 1000.0
    k = np.zeros((1, 1, N, d)); k[..., 0] = 1000.0
    y, _, _ = ref.prefill(q, k, v, np.zeros((d, 4)), W, C, m, T_max)
    for t, (sa_t, la_t) in table.items():
        if not la_t:
            continue
        exp = np.zeros(d)
        exp[la_t] = 1.0 / len(la_t)
        np.testing.assert_allclose(y[0, 0, t], exp, atol=1e-5)


CASES = [
    # B, Hq, Hkv, N, d, df, W, C, m, T_max
    (1, 2, 2, 40, 8, 8, 4, 8, 12, 4),      # W < C
    (1, 4, 2, 50, 8, 6, 3, 8, 12, 3),      # d_f != d, GQA
    (2, 2, 1, 64, 4, 4, 8, 4, 20, 6),      # W > C
    (1, 2, 2, 33, 8, 8, 4, 4, 12, 4),      # W == C, ragged tail
    (1, 2, 1, 37, 8, 8, 5, 8, 13, 2),      # T_max cap reached early
    (1, 2, 2, 64, 8, 8, 10, 4, 30, 5),
    (1, 1, 1, 20, 4, 4, 1, 3, 7, 3),       # W = 1, ties everywhere
    (1, 2, 2, 48, 8, 8, 6, 8, 62, 7),      # lambda = 8 = C: whole chunks kept
]


@pytest.mark.parametrize("case", CASES)
def test_stream_equals_set_definition(case):
    B, Hq, Hkv, N, d, df, W, C, m, T_max = case
    q, k, v, Wf = rand_case(B, Hq, Hkv, N, d, df)
    y, sc, st = ref.prefill(q, k, v, Wf, W, C, m, T_max)
    for b in range(B):
        yb, scb, selb = brute.prefill(q[b], k[b], v[b], Wf, W, C, m, T_max)
        np.testing.assert_allclose(y[b], yb, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(sc[b], scb, rtol=1e-12, atol=1e-12)
        # the permanent slots of finished chunks hold exactly the selection
        lam = brute.lam_of(m, W, T_max)
        for g in range(Hkv):
            for c in range(min(N // C, T_max)):
                slots = st.pos[b, g, W + c * lam: W + (c + 1) * lam].tolist()
                want = [x for x in selb[g, c].tolist() if x >= 0]
                assert sorted(x for x in slots if x >= 0) == want
        # rows at any N: the per-row evaluator agrees with the full matrix form
        picks = [(h, t) for h in range(Hq) for t in (0, N // 2, N - 1)]
        rows = brute.rows(q[b], k[b], v[b], Wf, W, C, selb, picks)
        for i, (h, t) in enumerate(picks):
            np.testing.assert_allclose(rows[i], yb[h, t], rtol=1e-10, atol=1e-12)


def test_random_routing_fuzz():
    for _ in range(12):
        Hkv = int(rng.integers(1, 3))
        G = int(rng.integers(1, 3))
        N = int(rng.integers(1, 60))
        W = int(rng.integers(1, 12))
        C = int(rng.integers(1, 12))
        T_max = int(rng.integers(1, 8))
        m = W + int(rng.integers(0, 3 * T_max))
        d = 4
        q, k, v, Wf = rand_case(1, G * Hkv, Hkv, N, d, 3)
        y, _, _ = ref.prefill(q, k, v, Wf, W, C, m, T_max)
        yb, _, _ = brute.prefill(q[0], k[0], v[0], Wf, W, C, m, T_max)
        np.testing.assert_allclose(y[0], yb, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------------------
# Reductions to textbook attention
# --------------------------------------------------------------------------

def _causal_softmax(q, k, v):
    N, d = q.shape
    s = q @ k.T / np.sqrt(d)
    s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
    return sp_softmax(s, axis=1) @ v


@pytest.mark.parametrize("m_extra,T_max", [(0, 4), (12, 4)])
def test_reduction_causal_softmax(m_extra, T_max):
    """W >= N: every key stays in the window, with or without a selection
    budget, so the layer is causal softmax attention."""
    N, d = 30, 8
    q, k, v, Wf = rand_case(1, 4, 2, N, d, 8)
    W = N + 2
    y, _, _ = ref.prefill(q, k, v, Wf, W, 8, W + m_extra, T_max)
    yb, _, _ = brute.prefill(q[0], k[0], v[0], Wf, W, 8, W + m_extra, T_max)
    for h in range(4):
        exp = _causal_softmax(q[0, h], k[0, h // 2], v[0, h // 2])
        np.testing.assert_allclose(y[0, h], exp, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(yb[h], exp, rtol=1e-10, atol=1e-12)


def _np_map_textbook(x, Wf):
    u = sp_softmax(x @ Wf, axis=-1)
    return np.linalg.norm(x, axis=-1, keepdims=True) * u / np.linalg.norm(u, axis=-1, keepdims=True)


def test_reduction_causal_linear():
    """W = 0 and lambda = 0: pure causal linear attention with phi."""
    N, d, df = 25, 8, 6
    q, k, v, Wf = rand_case(1, 2, 1, N, d, df)
    y, _, _ = ref.prefill(q, k, v, Wf, 0, 4, 0, 3)
    yb, _, _ = brute.prefill(q[0], k[0], v[0], Wf, 0, 4, 0, 3)
    pk = _np_map_textbook(k[0, 0], Wf)
    Scum = np.cumsum(pk[:, :, None] * v[0, 0][:, None, :], axis=0)
    zcum = np.cumsum(pk, axis=0)
    for h in range(2):
        pq = _np_map_textbook(q[0, h], Wf)
        exp = np.einsum("tf,tfd->td", pq, Scum) / np.einsum("tf,tf->t", pq, zcum)[:, None]
        np.testing.assert_allclose(y[0, h], exp, rtol=1e-10)
        np.testing.assert_allclose(yb[h], exp, rtol=1e-10)


# --------------------------------------------------------------------------
# NP-Map
# --------------------------------------------------------------------------

def test_npmap_invariants():
    d, df = 8, 6
    x = rng.standard_normal((50, d)) * rng.lognormal(0, 0.5, (50, 1))
    Wf = rng.standard_normal((d, df)) / np.sqrt(d)
    for f in (ref.npmap, brute.npmap):
        phi = f(x, Wf)
        assert phi.shape == (50, df)
        assert (phi >= 0).all()
        np.testing.assert_allclose(np.linalg.norm(phi, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
        assert np.all(f(np.zeros((1, d)), Wf) == 0)
        # Wf = 0: uniform direction
        np.testing.assert_allclose(f(x, np.zeros((d, df))),
                                   np.linalg.norm(x, axis=1, keepdims=True) / np.sqrt(df) * np.ones((1, df)),
                                   rtol=1e-12)
        # the softmax runs over the feature axis: a rank-one a 1^T added to Wf
        # shifts every logit of a row equally and changes nothing
        a = rng.standard_normal((d, 1))
        np.testing.assert_allclose(f(x, Wf + a @ np.ones((1, df))), phi, rtol=1e-10)
        # permuting feature columns permutes phi
        perm = rng.permutation(df)
        np.testing.assert_allclose(f(x, Wf[:, perm]), phi[:, perm], rtol=1e-12)
        # scaling x scales the norm and sharpens the direction toward the arg-max
        big = f(x[:1] * 1e3, Wf)
        j = int(np.argmax(x[:1] @ Wf))
        assert big[0, j] == pytest.approx(np.linalg.norm(x[0]) * 1e3, rel=1e-6)
    np.testing.assert_allclose(ref.npmap(x, Wf), _np_map_textbook(x, Wf), rtol=1e-12)


# --------------------------------------------------------------------------
# Prefill / decode unification and the recurrent state
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", [(2, 4, 2, 45, 8, 8, 4, 8, 16, 3), (1, 2, 2, 40, 8, 8, 9, 4, 21, 4),
                                  (1, 2, 1, 30, 8, 8, 0, 4, 0, 2)])
def test_prefill_then_decode_equals_longer_prefill(case):
    B, Hq, Hkv, N, d, df, W, C, m, T_max = case
    q, k, v, Wf = rand_case(B, Hq, Hkv, N, d, df)
    y_all, _, st_all = ref.prefill(q, k, v, Wf, W, C, m, T_max)
    for N0 in (0, 1, N // 3, N - 1):
        if N0 == 0:
            st = ref.State(B, Hkv, d, df, C, m)
        else:
            _, _, st = ref.prefill(q[:, :, :N0], k[:, :, :N0], v[:, :, :N0], Wf, W, C, m, T_max)
        for t in range(N0, N):
            yt = ref.decode_step(st, q[:, :, t], k[:, :, t], v[:, :, t], Wf, W, C, m, T_max)
            np.testing.assert_array_equal(yt, y_all[:, :, t])
        for name in ("K", "V", "pos", "cnt", "ssc", "S", "z", "ring", "t"):
            np.testing.assert_array_equal(getattr(st, name), getattr(st_all, name))


@pytest.mark.parametrize("case", CASES[:6])
def test_state_matches_definition(case):
    """After N tokens: S, z sum exactly the tokens that left the window and do
    not sit in a budget slot; the window ring holds the last W tokens; at most
    m softmax slots are in use; candidates belong to the unfinished chunk."""
    B, Hq, Hkv, N, d, df, W, C, m, T_max = case
    q, k, v, Wf = rand_case(B, Hq, Hkv, N, d, df)
    _, sc, st = ref.prefill(q, k, v, Wf, W, C, m, T_max)
    lam = brute.lam_of(m, W, T_max)
    for b in range(B):
        for g in range(Hkv):
            pos = st.pos[b, g]
            assert (pos >= 0).sum() <= m
            ring = sorted(p for p in pos[:W].tolist() if p >= 0)
            assert ring == list(range(max(0, N - W), N))
            slotted = set(p for p in pos[W:].tolist() if p >= 0)
            folded = [j for j in range(N - W) if j not in slotted]
            phk = brute.npmap(k[b, g], Wf)
            S = sum((np.outer(phk[j], v[b, g, j]) for j in folded), np.zeros((df, d)))
            np.testing.assert_allclose(st.S[b, g], S, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(st.z[b, g], phk[folded].sum(0) if folded else 0, rtol=1e-11)
            cur = N // C
            if N % C and cur < T_max and lam > 0:
                part = np.arange(cur * C, N)
                sp = sc[b, g, part]
                order = np.lexsort((part, -sp))[:lam]
                top = set(part[order].tolist())
                cands = set(p for p in pos[W + cur * lam: W + (cur + 1) * lam].tolist() if p >= 0)
                assert cands == set(j for j in top if j <= N - 1 - W)
