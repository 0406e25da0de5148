"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars: selected index sets exact (chunks whose lambda-th and (lambda+1)-th
oracle scores differ by < 1e-5 relative are near-ties: reported, and compared
using the GPU's selection); outputs max|err| <= 1e-2 * max|y_ref|; scores
within 1e-4 relative (+1e-6 absolute); NP-Map within 1e-4 relative of its norm.
"""
from dataclasses import replace as dataclass_replace

import numpy as np
import pytest
import torch

from linear_attention_linearization_gb300 import inputs
from linear_attention_linearization_gb300.inputs import Workload, to_f64
from conftest import record_parity
from oracle import brute, ref

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
DEV = "cuda"
U_BF16 = 2.0 ** -8      # unit roundoff of bf16: 8 significant bits, round to nearest
U_F32 = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    from linear_attention_linearization_gb300 import build
    build.build()
    ref.build()


def still():
    from linear_attention_linearization_gb300 import still as s
    return s


def custom(B, Hq, Hkv, d, N, W, C, m, T_max, df=None, dist="dirnorm", outlier=0.0):
    return Workload("case", B, Hq, Hkv, d, N, W, C, m, T_max, df or d, dist, outlier)


def check_selection(sel_gpu, scores_ref, w):
    """Exact set equality, except on near-tie chunks, where the GPU's set must
    still be a valid top-lambda under the oracle scores.  Returns (near-tie
    chunks of the oracle, chunks whose selection differs -- all near ties)."""
    lam = w.lam
    B = sel_gpu.shape[0]
    n_diff = n_ties = 0
    for b in range(B):
        sel_ref = brute.select(scores_ref[b], w.C, lam, w.T_max)
        ties = set(brute.near_ties(scores_ref[b], w.C, lam, w.T_max))
        n_ties += len(ties)
        diff = np.argwhere((sel_gpu[b] != sel_ref).any(axis=-1))
        for g, c in diff:
            assert (g, c) in ties, f"selection differs outside a near tie: b={b} g={g} c={c}"
            chunk = scores_ref[b, g, c * w.C:(c + 1) * w.C]
            picked = sel_gpu[b, g, c] - c * w.C
            worst_in = chunk[picked].min()
            best_out = np.delete(chunk, picked).max()
            assert worst_in >= best_out - 1e-5 * abs(best_out)
            n_diff += 1
    return n_ties, n_diff


def prefill_checked(s, w, qd, kd, vd, Wd, st=None):
    """still_prefill with a caller workspace; its device status word must read 0."""
    ws = torch.empty(s.workspace_size(qd, kd, Wd, w.W, w.C, w.m, w.T_max), dtype=torch.uint8, device=DEV)
    out, sel = s.prefill(qd, kd, vd, Wd, w.W, w.C, w.m, w.T_max, workspace=ws, export_state=st)
    assert s.workspace_status(ws) == 0, "a prefill kernel reported an error in the status word"
    return out, sel


def run_prefill_case(w, seed=0, state=False, name=None):
    s = still()
    q, k, v, Wf = inputs.make_inputs(w, seed=seed)
    qd, kd, vd, Wd = (t.to(DEV) for t in (q, k, v, Wf))
    st = s.DecodeState(w.B, w.Hkv, w.d, w.df, w.C, w.m) if state else None
    out, sel = prefill_checked(s, w, qd, kd, vd, Wd, st)
    torch.cuda.synchronize()
    qa, ka, va, Wa = (to_f64(t) for t in (q, k, v, Wf))
    y_ref, sc_ref, st_ref = ref.prefill(qa, ka, va, Wa, w.W, w.C, w.m, w.T_max)
    sel_g = sel.cpu().numpy()
    n_diff = n_ties = 0
    if w.lam > 0 and w.W >= 1:
        n_ties, n_diff = check_selection(sel_g, sc_ref, w)
        if n_diff:
            y_ref, sc_ref, st_ref = ref.prefill(qa, ka, va, Wa, w.W, w.C, w.m, w.T_max, sel_override=sel_g)
    y = to_f64(out)
    err = np.abs(y - y_ref).max()
    rel = err / max(np.abs(y_ref).max(), 1e-300)
    record_parity(name or f"B{w.B}_Hq{w.Hq}_Hkv{w.Hkv}_d{w.d}_df{w.df}_N{w.N}_W{w.W}_C{w.C}_lam{w.lam}",
                  max_err_rel=float(rel), near_tie_chunks=n_ties, sel_differs_in_ties=n_diff,
                  sel_exact_outside_ties=True)
    assert err <= OUT_TOL * np.abs(y_ref).max(), (err, np.abs(y_ref).max())
    return dict(out=y, y_ref=y_ref, sel=sel_g, sc_ref=sc_ref, st=st, st_ref=st_ref, n_diff=n_diff, err=err,
                inputs=(q, k, v, Wf))


# --------------------------------------------------------------------------
# a3: NP-Map
# --------------------------------------------------------------------------

@pytest.mark.parametrize("d,df", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_npmap_parity(d, df):
    w = custom(1, 4, 4, d, 300, 8, 8, 8, 1, df=df)
    q, _, _, Wf = inputs.make_inputs(w, seed=3)
    phi = still().npmap(q.to(DEV), Wf.to(DEV))
    exp = ref.npmap(to_f64(q).reshape(-1, d), to_f64(Wf)).reshape(phi.shape)
    got = phi.double().cpu().numpy()
    nrm = np.linalg.norm(to_f64(q), axis=-1, keepdims=True)
    assert (np.abs(got - exp) <= 1e-4 * nrm + 1e-6).all()
    assert (got >= 0).all()


# --------------------------------------------------------------------------
# a1 / a2: score and select
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny_prefill_n512", "llama32_1b_layer_prefill_4k"])
def test_score_and_select_parity(name):
    w = inputs.WORKLOADS[name]
    q, k, _, _ = inputs.make_inputs(w, seed=1)
    s = still()
    sc = s.score(q.to(DEV), k.to(DEV), w.W).cpu().double().numpy()
    qa, ka = to_f64(q), to_f64(k)
    for b in range(w.B):
        _, sr = ref.scores(qa[b], ka[b], w.W)
        assert (np.abs(sc[b] - sr) <= 1e-4 * np.abs(sr) + 1e-6).all()
    # selection on identical fp32 inputs is integer work: bit-exact
    sc32 = torch.from_numpy(sc.astype(np.float32))
    sel = s.select(sc32.to(DEV), w.Hq, w.d, w.W, w.C, w.m, w.T_max).cpu().numpy()
    for b in range(w.B):
        exp = ref.select(sc32[b].double().numpy(), w.C, w.lam, w.T_max)
        np.testing.assert_array_equal(sel[b], exp)


def test_select_ties_and_special_cases():
    s = still()
    sc = torch.zeros((2, 3, 100), dtype=torch.float32)
    sc[0, 1, 40:60] = 1.0
    sel = s.select(sc.to(DEV), 3, 64, 4, 20, 4 + 3 * 6, 6).cpu().numpy()   # lambda = 3
    assert sel[0, 0, 0].tolist() == [0, 1, 2]
    assert sel[0, 1, 2].tolist() == [40, 41, 42]
    assert (sel[:, :, 5] == -1).all()                                      # chunk 5 absent (N=100)
    sel = s.select(sc.to(DEV), 3, 64, 4, 8, 4 + 10 * 3, 3).cpu().numpy()   # lambda = 10 > C = 8
    assert sel[1, 2, 1].tolist() == list(range(8, 16)) + [-1, -1]
    r = np.random.default_rng(0).standard_normal((1, 2, 1000)).astype(np.float32)
    sel = s.select(torch.from_numpy(r).to(DEV), 2, 64, 64, 100, 64 + 7 * 10, 10).cpu().numpy()
    np.testing.assert_array_equal(sel[0], ref.select(r[0].astype(np.float64), 100, 7, 10))


# --------------------------------------------------------------------------
# a1-a5: full prefill
# --------------------------------------------------------------------------

EDGE = [
    custom(1, 2, 2, 64, 1, 64, 64, 128, 8),             # one token
    custom(1, 2, 2, 64, 37, 64, 64, 128, 8),            # N < W, ragged
    custom(1, 4, 2, 64, 300, 16, 32, 40, 8),            # W < C, candidates in the tail
    custom(2, 8, 2, 128, 515, 24, 40, 24 + 5 * 6, 6),   # ragged everything, B = 2, G = 4
    custom(1, 2, 1, 64, 400, 600, 64, 700, 4),          # W >= N: causal softmax
    custom(1, 2, 2, 64, 333, 0, 16, 0, 4),              # W = 0, lambda = 0: causal linear
    custom(1, 2, 2, 64, 260, 8, 4, 8 + 6 * 12, 12),     # lambda = 6 > C = 4: whole chunks kept
    custom(1, 4, 4, 64, 257, 32, 64, 32 + 2 * 3, 3),    # T_max reached early
    custom(1, 4, 1, 64, 200, 16, 16, 16, 4, df=128),    # lambda = 0, d_f != d
    custom(1, 3, 3, 128, 190, 20, 48, 20 + 4 * 4, 4, df=64, dist="iid"),
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: f"N{w.N}_W{w.W}_C{w.C}_lam{w.lam}_d{w.d}_df{w.df}")
def test_prefill_edge_cases(w):
    run_prefill_case(w, seed=7)


def test_prefill_empty_sequence():
    s = still()
    w = custom(1, 2, 2, 64, 0, 8, 8, 16, 1)
    q = torch.zeros((1, 2, 0, 64), dtype=torch.bfloat16, device=DEV)
    out, sel = s.prefill(q, q, q, torch.zeros((64, 64), device=DEV), w.W, w.C, w.m, w.T_max)
    assert out.numel() == 0 and (sel.cpu() == -1).all()


@pytest.mark.parametrize("name", ["tiny_prefill_n512", "llama32_1b_layer_prefill_4k",
                                  "train_b8_n1k_chunk_parallel"])
def test_prefill_workloads(name):
    run_prefill_case(inputs.WORKLOADS[name], seed=2, name=name)


def test_prefill_16k_full_layer():
    """The full 16K layer in the launch configuration the benchmark times:
    every score, the selection, every output element and the exported decode
    state against the fp64 oracle run over the whole layer."""
    w = inputs.WORKLOADS["llama3_8b_layer_prefill_16k"]
    s = still()
    q, k, v, Wf = inputs.make_inputs(w, seed=0)
    qd, kd, vd, Wd = (t.to(DEV) for t in (q, k, v, Wf))
    st = s.DecodeState(w.B, w.Hkv, w.d, w.df, w.C, w.m)
    out, sel = prefill_checked(s, w, qd, kd, vd, Wd, st)
    sc_gpu = s.score(qd, kd, w.W).cpu().double().numpy()
    qa, ka, va, Wa = (to_f64(t) for t in (q, k, v, Wf))
    y_ref, sc_ref, st_ref = ref.prefill(qa, ka, va, Wa, w.W, w.C, w.m, w.T_max)
    assert (np.abs(sc_gpu - sc_ref) <= 1e-4 * np.abs(sc_ref) + 1e-6).all()
    sel_g = sel.cpu().numpy()
    n_ties, n_diff = check_selection(sel_g, sc_ref, w)
    if n_diff:
        y_ref, sc_ref, st_ref = ref.prefill(qa, ka, va, Wa, w.W, w.C, w.m, w.T_max, sel_override=sel_g)
    y = to_f64(out)
    err = np.abs(y - y_ref).max()
    record_parity("llama3_8b_layer_prefill_16k (every element)", max_err_rel=float(err / np.abs(y_ref).max()),
                  near_tie_chunks=n_ties, sel_differs_in_ties=n_diff, sel_exact_outside_ties=True)
    assert err <= OUT_TOL * np.abs(y_ref).max()
    compare_state(st, st_ref, w, ka, va, Wa, pre_state=st_ref)


# --------------------------------------------------------------------------
# a6: decode step and the prefill -> decode hand-over
# --------------------------------------------------------------------------

def state_sets(pos, W, lam, T_max):
    """Per slot group (window, then each chunk's kept range): set of positions."""
    out = [frozenset(p for p in pos[:W].tolist() if p >= 0)]
    for c in range(T_max):
        grp = pos[W + c * lam: W + (c + 1) * lam].tolist() if lam > 0 else []
        out.append(frozenset(p for p in grp if p >= 0))
    return out


def folded_mask(pos, t):
    """Tokens 0..t-1 that sit in no slot of the state: the ones in (S, z)."""
    f = np.ones(t, dtype=bool)
    p = pos[pos >= 0]
    f[p[p < t]] = False
    return f


def state_tolerance(kg, vg, Wf, folded, pre_folded):
    """Per-element bound on |S_gpu - S_oracle| and |z_gpu - z_oracle| for one
    (sequence, kv head), derived from the declared rounding of the two paths:

    * keys folded by the GPU prefill (pre_folded) enter through NP-Map
      features computed from U = k Wf with Wf rounded to bf16 (a tensor-core
      operand), then rounded to bf16 themselves.  The effect of the rounded Wf
      is computed exactly here: phi~ = the oracle's NP-Map fed bf16(Wf), and
      |S~ - S_ref| with S~ = sum phi~ v^T is part of the bound.  The bf16
      rounding of each phi~ element is an independent error of at most
      u = 2^-8 relative (half an ulp of 8 significant bits; uniform, variance
      at most (u phi~)^2 / 3); their sum over the folded keys is bounded by 6
      standard deviations.
    * keys folded by the decode step use fp32 features from the fp32 Wf.
    * fp32 accumulation of the sums: 8 u32 sqrt(n) max|S|.
    Returns (tol_S [d_f, d], tol_z [d_f], S_model, z_model) where the model
    sums are the exact fp64 sums the bound is centred on."""
    n = int(folded.sum())
    if n == 0:
        return 0.0, 0.0, None, None
    phi = ref.npmap(kg, Wf)
    wf_b = to_f64(torch.from_numpy(Wf).to(torch.float32).to(torch.bfloat16))
    phi_t = np.where(pre_folded[:, None], ref.npmap(kg, wf_b), phi)
    F = folded
    S_ref = phi[F].T @ vg[F]
    z_ref = phi[F].sum(axis=0)
    S_mod = phi_t[F].T @ vg[F]
    z_mod = phi_t[F].sum(axis=0)
    Fp = F & pre_folded
    sig_S = U_BF16 * np.sqrt((phi_t[Fp] ** 2).T @ (vg[Fp] ** 2) / 3.0)
    sig_z = U_BF16 * np.sqrt((phi_t[Fp] ** 2).sum(axis=0) / 3.0)
    acc = 8 * U_F32 * np.sqrt(n)
    tol_S = np.abs(S_mod - S_ref) + 6 * sig_S + acc * np.abs(S_ref).max()
    tol_z = np.abs(z_mod - z_ref) + 6 * sig_z + acc * np.abs(z_ref).max()
    return tol_S, tol_z, S_ref, z_ref


def compare_state(st, st_ref, w, ka, va, Wa, pre_state=None):
    """Slots bit-exact by position; (S, z) within state_tolerance of the oracle.
    ka, va: fp64 keys/values of every token absorbed so far; pre_state: the
    oracle state at the hand-over from a GPU prefill (None: all decode steps)."""
    pos = st.slot_pos.cpu().numpy()
    K = to_f64(st.K)
    S = st.S.cpu().double().numpy()
    z = st.z.cpu().double().numpy()
    T = int(st_ref.t[0])
    for b in range(w.B):
        for g in range(w.Hkv):
            assert state_sets(pos[b, g], w.W, w.lam, w.T_max) == state_sets(st_ref.pos[b, g], w.W, w.lam, w.T_max)
            for sl in range(w.m):
                p = pos[b, g, sl]
                if p < 0:
                    continue
                rs = int(np.flatnonzero(st_ref.pos[b, g] == p)[0])
                np.testing.assert_array_equal(K[b, g, sl], st_ref.K[b, g, rs])
            F = folded_mask(st_ref.pos[b, g], T)
            if pre_state is None:
                pre = np.zeros(T, dtype=bool)
            else:
                t0 = int(pre_state.t[b])
                pre = np.zeros(T, dtype=bool)
                pre[:t0] = folded_mask(pre_state.pos[b, g], t0)
            tol_S, tol_z, S_chk, z_chk = state_tolerance(ka[b, g, :T], va[b, g, :T], Wa, F, pre)
            if S_chk is None:
                assert np.abs(S[b, g]).max() == 0 and np.abs(z[b, g]).max() == 0
                continue
            # the folded set read off the oracle's slots reproduces the oracle's own sums
            assert np.abs(S_chk - st_ref.S[b, g]).max() <= 1e-9 * np.abs(st_ref.S[b, g]).max()
            assert (np.abs(S[b, g] - st_ref.S[b, g]) <= tol_S).all()
            assert (np.abs(z[b, g] - st_ref.z[b, g]) <= tol_z).all()
    assert (st.t.cpu().numpy() == st_ref.t[:, None]).all()


DEC = [
    custom(2, 4, 2, 64, 300, 16, 32, 16 + 3 * 8, 8),      # W < C: candidates, T_max reached
    custom(1, 2, 2, 64, 150, 8, 8, 8 + 2 * 20, 20),       # W == C
    custom(1, 2, 1, 128, 120, 20, 6, 20 + 1 * 30, 30),    # W > C
    custom(1, 2, 2, 64, 90, 0, 8, 0, 3),                  # W = 0: linear only
]


@pytest.mark.parametrize("w", DEC, ids=lambda w: f"W{w.W}_C{w.C}_lam{w.lam}")
def test_decode_from_empty_state_equals_prefill(w):
    s = still()
    q, k, v, Wf = inputs.make_inputs(w, seed=11)
    st = s.DecodeState(w.B, w.Hkv, w.d, w.df, w.C, w.m)
    s.decode_state_init(st, w.Hq, w.W, w.C, w.m, w.T_max)
    Wd = Wf.to(DEV)
    ys = []
    for t in range(w.N):
        qt, kt, vt = (x[:, :, t].contiguous().to(DEV) for x in (q, k, v))
        ys.append(s.decode_step(st, qt, kt, vt, Wd, w.W, w.C, w.m, w.T_max))
    y = torch.stack(ys, dim=2)
    qa, ka, va, Wa = (to_f64(x) for x in (q, k, v, Wf))
    y_ref, _, st_ref = ref.prefill(qa, ka, va, Wa, w.W, w.C, w.m, w.T_max)
    err = np.abs(to_f64(y) - y_ref).max()
    record_parity(f"decode_from_empty_W{w.W}_C{w.C}_lam{w.lam}", max_err_rel=float(err / np.abs(y_ref).max()))
    assert err <= OUT_TOL * np.abs(y_ref).max()
    assert st.read_status() == 0
    compare_state(st, st_ref, w, ka, va, Wa)


# the last case: 48 sequences x 8 kv heads = 384 units of the decode kernel,
# more than one wave of its CTAs, at the 16K layer's head shape
@pytest.mark.parametrize("w", DEC[:3] + [custom(1, 4, 2, 64, 301, 16, 32, 16 + 3 * 8, 8),
                                         custom(48, 32, 8, 128, 300, 16, 32, 16 + 3 * 10, 10)],
                         ids=lambda w: f"B{w.B}_N{w.N}_W{w.W}_C{w.C}")
def test_prefill_export_then_decode(w):
    r = run_prefill_case(w, seed=4, state=True)
    _, k, v, Wf = r["inputs"]
    Wa = to_f64(Wf)
    st, st_ref = r["st"], r["st_ref"]
    at_export = st_ref.copy()
    compare_state(st, st_ref, w, to_f64(k), to_f64(v), Wa, pre_state=at_export)
    s = still()
    q2, k2, v2, _ = inputs.make_inputs(w, seed=5, N=70)
    err = 0.0
    for t in range(q2.shape[2]):
        qt, kt, vt = (x[:, :, t].contiguous() for x in (q2, k2, v2))
        yt = s.decode_step(st, qt.to(DEV), kt.to(DEV), vt.to(DEV), Wf.to(DEV), w.W, w.C, w.m, w.T_max)
        yr = ref.decode_step(st_ref, to_f64(qt), to_f64(kt), to_f64(vt), Wa, w.W, w.C, w.m, w.T_max)
        e = np.abs(to_f64(yt) - yr).max() / np.abs(yr).max()
        err = max(err, e)
        assert e <= OUT_TOL
    record_parity(f"prefill_export_then_70_decode_steps_N{w.N}_W{w.W}_C{w.C}", max_err_rel=float(err))
    ka = np.concatenate([to_f64(k), to_f64(k2)], axis=2)
    va = np.concatenate([to_f64(v), to_f64(v2)], axis=2)
    compare_state(st, st_ref, w, ka, va, Wa, pre_state=at_export)


def test_decode_step_16k_batch128():
    """The decode workload: 128 sequences whose cache and state come from the
    prefill of 16K seeded tokens, one new token each.  Sixteen sequences
    spread over the batch are checked against the oracle's prefill + decode
    step (outputs, and the whole decode state for four of them)."""
    w = inputs.WORKLOADS["llama31_8b_decode_b128_ctx16k"]
    s = still()
    q, k, v, Wf = inputs.make_inputs(w, seed=3, device=DEV)
    st = s.DecodeState(w.B, w.Hkv, w.d, w.df, w.C, w.m)
    _, sel = prefill_checked(s, w, q, k, v, Wf, st)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(99)
    qt = torch.randn((w.B, w.Hq, w.d), generator=gen, device=DEV).to(torch.bfloat16)
    kt = torch.randn((w.B, w.Hkv, w.d), generator=gen, device=DEV).to(torch.bfloat16)
    vt = torch.randn((w.B, w.Hkv, w.d), generator=gen, device=DEV).to(torch.bfloat16)
    yt = s.decode_step(st, qt, kt, vt, Wf, w.W, w.C, w.m, w.T_max)
    torch.cuda.synchronize()
    assert st.read_status() == 0
    # valid softmax slots: 64 window + 3 per chunk for 64 chunks
    assert int((st.slot_pos[0, 0] >= 0).sum()) == w.W + w.lam * w.T_max
    Wa = to_f64(Wf)
    idx = list(range(0, w.B, w.B // 16))
    n_ties = n_diff = 0
    worst = 0.0
    for pair in range(0, len(idx), 2):          # two sequences per oracle call (fp64 inputs: ~1 GB each)
        ii = idx[pair:pair + 2]
        qa, ka, va = (to_f64(x[ii]) for x in (q, k, v))
        sel_b = sel[ii].cpu().numpy()
        _, sc_ref, st_ref = ref.prefill(qa, ka, va, Wa, w.W, w.C, w.m, w.T_max, sel_override=sel_b)
        nt, nd = check_selection(sel_b, sc_ref, w)
        n_ties += nt
        n_diff += nd
        at_export = st_ref.copy()
        yr = ref.decode_step(st_ref, to_f64(qt[ii]), to_f64(kt[ii]), to_f64(vt[ii]), Wa, w.W, w.C, w.m, w.T_max)
        err = np.abs(to_f64(yt[ii]) - yr).max(axis=(1, 2)) / np.abs(yr).max(axis=(1, 2))
        worst = max(worst, float(err.max()))
        assert (err <= OUT_TOL).all(), err
        if pair % 8 == 0:
            # the whole decode state of this pair: slot by slot, (S, z) within the derived bound
            ka1 = np.concatenate([ka, to_f64(kt[ii])[:, :, None]], axis=2)
            va1 = np.concatenate([va, to_f64(vt[ii])[:, :, None]], axis=2)
            gsub = _StateView(st, ii)
            compare_state(gsub, st_ref, dataclass_replace(w, B=len(ii)), ka1, va1, Wa, pre_state=at_export)
    record_parity("llama31_8b_decode_b128_ctx16k (16 of 128 sequences)", max_err_rel=worst,
                  near_tie_chunks=n_ties, sel_differs_in_ties=n_diff, sel_exact_outside_ties=True)


class _StateView:
    """The decode-state tensors of some sequences of a DecodeState."""

    def __init__(self, st, seqs):
        for name in ("K", "slot_pos", "S", "z", "t"):
            setattr(self, name, getattr(st, name)[seqs])


def test_prefill_repeated_calls_stable():
    """Many prefills of alternating shapes in one process, each compared with
    the oracle: a race between the warps that share a row (which show up only
    under some interleavings) or a dependence on what an earlier call left in
    reused device memory fails here even when a single call passes."""
    s = still()
    cases = [custom(1, 4, 2, 64, 301, 16, 32, 16 + 3 * 8, 8), custom(1, 2, 1, 128, 120, 20, 6, 20 + 1 * 30, 30),
             custom(2, 8, 2, 128, 260, 64, 64, 64 + 2 * 4, 4)]
    prepared = []
    for w in cases:
        q, k, v, Wf = inputs.make_inputs(w, seed=4)
        y_ref, _, _ = ref.prefill(*(to_f64(t) for t in (q, k, v, Wf)), w.W, w.C, w.m, w.T_max)
        prepared.append((w, tuple(t.to(DEV) for t in (q, k, v, Wf)), y_ref))
    for rep in range(24):
        for w, (qd, kd, vd, Wd), y_ref in prepared:
            st = s.DecodeState(w.B, w.Hkv, w.d, w.df, w.C, w.m) if rep % 2 else None
            out, _ = s.prefill(qd, kd, vd, Wd, w.W, w.C, w.m, w.T_max, export_state=st)
            torch.cuda.synchronize()
            err = np.abs(to_f64(out) - y_ref).max()
            assert err <= OUT_TOL * np.abs(y_ref).max(), (rep, w.N, err)


@pytest.mark.parametrize("name", ["tiny_prefill_n512", "llama32_1b_layer_prefill_4k",
                                  "llama3_8b_layer_prefill_16k", "train_b8_n1k_chunk_parallel"])
def test_every_prefill_workload_takes_the_tensor_core_kernels(name):
    """The kernels a workload's prefill launches, by the library's timer names:
    the tensor-core score and attention kernels, never the CUDA-core fallbacks."""
    w = inputs.WORKLOADS[name]
    s = still()
    q, k, v, Wf = (t.to(DEV) for t in inputs.make_inputs(w, seed=1))
    s.timing_read()
    s.timing_enable(True)
    try:
        s.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max)
        torch.cuda.synchronize()
    finally:
        s.timing_enable(False)
    names = set(s.timing_read())
    assert "hybrid_attn" in names and "hybrid_attn_general" not in names, names
    assert "score" in names and "features_linstate" in names, names
