"""Brute-force NumPy oracle: the STILL layer written out from its set definition.

TEST INFRASTRUCTURE ONLY -- nothing in the product path imports this module.
It shares no code with the C streaming oracle (``still_ref.c``) nor with the
CUDA library; both are checked against it.

Sources ("STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
Linearization", besthub.dev; roboind.com write-up "STILL: Selecting Tokens for
Intra-Layer Hybrid Attention to Linearize LLMs"):

* Self-Saliency Score -- section "Self-Saliency Score: Predicting Future Utility
  from Local Context": a^diag / a^nodiag over the token's causal window of W
  keys (its own key included in a^diag).  Closed form fixed by this library:
  Score = -log(1 - p + 1e-6), p the self probability of a^diag.  For grouped
  query heads the kv-head score is the mean over the group's query heads.
* Routing -- sections "Content-Aware Routing with Fixed Budget" and "Delayed
  Chunk-Level Selection ...": lambda = floor((m - W) / T_max); each completed
  chunk c < T_max keeps its top-lambda tokens (ties to the lower position).
  A kept token of chunk c is a softmax key for queries of later chunks only
  (selection runs when the next chunk begins).
* For query t:  SA(t) = {t-W < j <= t} U {j kept, chunk(j) < chunk(t), j <= t-W}
                LA(t) = {j <= t-W} minus SA(t)
* NP-Map -- section "NP-Map: Norm-Preserving Feature Map":
  phi(x) = ||x|| u / ||u||, u = softmax(x Wf) over the feature axis.
* Output: y = (sum_SA e^{s-c} v + sum_LA (phi(q).phi(k)) v) /
              (sum_SA e^{s-c} + sum_LA phi(q).phi(k)),  c = max_SA s.
  The linear sums are written out key by key here (no recurrent state).

Every array is float64; inputs are the bf16 values upcast exactly.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def lam_of(m: int, W: int, T_max: int) -> int:
    """lambda = floor((m - W) / T_max)."""
    if T_max < 1 or W < 0 or m < W:
        raise ValueError("invalid budget")
    return (m - W) // T_max


def npmap(x: np.ndarray, Wf: np.ndarray) -> np.ndarray:
    """NP-Map of the rows of x [..., d] with Wf [d, df]."""
    logits = x @ Wf
    logits = logits - logits.max(axis=-1, keepdims=True)
    u = np.exp(logits)
    u = u / u.sum(axis=-1, keepdims=True)
    nx = np.linalg.norm(x, axis=-1, keepdims=True)
    return nx * u / np.linalg.norm(u, axis=-1, keepdims=True)


def head_scores(q: np.ndarray, k: np.ndarray, W: int) -> np.ndarray:
    """Per-query-head Self-Saliency scores [Hq, N] for one sequence.

    q [Hq, N, d], k [Hkv, N, d].  Works at any N: the window logits are built
    offset by offset (offset 0 = the token itself)."""
    Hq, N, d = q.shape
    G = Hq // k.shape[0]
    out = np.empty((Hq, N))
    nw = min(W, N)
    for h in range(Hq):
        kk = k[h // G]
        s = np.full((N, nw), -np.inf)
        for o in range(nw):
            s[o:, o] = np.einsum("td,td->t", q[h, o:], kk[: N - o]) / np.sqrt(d)
        a_diag = np.exp(s - s.max(axis=1, keepdims=True))
        a_diag /= a_diag.sum(axis=1, keepdims=True)
        one_minus_p = a_diag[:, 1:].sum(axis=1)          # mass of the other keys
        out[h] = -np.log(one_minus_p + EPS)
    return out


def kv_scores(q: np.ndarray, k: np.ndarray, W: int) -> np.ndarray:
    """kv-head scores [Hkv, N]: mean of the per-head scores over each group."""
    hs = head_scores(q, k, W)
    Hkv = k.shape[0]
    return hs.reshape(Hkv, -1, hs.shape[-1]).mean(axis=1)


def select(scores: np.ndarray, C: int, lam: int, T_max: int) -> np.ndarray:
    """Top-lambda per completed chunk c < T_max: [Hkv, T_max, lam], -1 padded."""
    Hkv, N = scores.shape
    sel = np.full((Hkv, T_max, max(lam, 0)), -1, dtype=np.int64)
    if lam <= 0:
        return sel
    for g in range(Hkv):
        for c in range(min(N // C, T_max)):
            idx = np.arange(c * C, (c + 1) * C)
            sc = scores[g, idx]
            order = np.lexsort((idx, -sc))      # score descending, position ascending
            keep = np.sort(idx[order[: min(lam, C)]])
            sel[g, c, : keep.size] = keep
    return sel


def near_ties(scores: np.ndarray, C: int, lam: int, T_max: int, rel: float = 1e-5):
    """Chunks whose lambda-th and (lambda+1)-th scores differ by < rel (relative)."""
    Hkv, N = scores.shape
    out = []
    if lam <= 0:
        return out
    for g in range(Hkv):
        for c in range(min(N // C, T_max)):
            if lam >= C:
                continue
            sc = np.sort(scores[g, c * C:(c + 1) * C])[::-1]
            a, b = sc[lam - 1], sc[lam]
            if abs(a - b) <= rel * max(abs(a), abs(b), 1e-30):
                out.append((g, c))
    return out


def kept_mask(sel: np.ndarray, N: int) -> np.ndarray:
    """Boolean [Hkv, N]: token j was kept by its chunk."""
    Hkv = sel.shape[0]
    kept = np.zeros((Hkv, N), dtype=bool)
    for g in range(Hkv):
        s = sel[g].reshape(-1)
        kept[g, s[s >= 0]] = True
    return kept


def route_masks(kept_g: np.ndarray, N: int, W: int, C: int):
    """SA and LA masks [N(query), N(key)] of one kv head from the set rules."""
    t = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    window = (j <= t) & (j > t - W)
    old = j <= t - W
    sa = window | (kept_g[None, :] & (j // C < t // C) & old)
    la = old & ~sa
    return sa, la


def prefill(q, k, v, Wf, W, C, m, T_max, sel=None, gate=None):
    """Full output [Hq, N, d] of one sequence; O(N^2), tiny inputs only.
    gate (optional [Hq, N, d]): pre-activations of the linear branch's gate,
    y = (softmax numerator + sigmoid(gate) * linear numerator) / (both denominators).

    Returns (y, kv scores, sel)."""
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    lam = lam_of(m, W, T_max)
    scores = kv_scores(q, k, W) if W >= 1 else np.zeros((Hkv, N))
    if sel is None:
        sel = select(scores, C, lam, T_max)
    kept = kept_mask(sel, N)
    y = np.zeros_like(q)
    for g in range(Hkv):
        sa, la = route_masks(kept[g], N, W, C)
        phk = npmap(k[g], Wf)
        for h in range(g * G, (g + 1) * G):
            s = q[h] @ k[g].T / np.sqrt(d)
            s_sa = np.where(sa, s, -np.inf)
            c = s_sa.max(axis=1, keepdims=True)
            c = np.where(np.isfinite(c), c, 0.0)
            e = np.where(sa, np.exp(s_sa - c), 0.0)
            a = np.where(la, npmap(q[h], Wf) @ phk.T, 0.0)
            den = (e + a).sum(axis=1, keepdims=True)
            g_h = 1.0 / (1.0 + np.exp(-gate[h])) if gate is not None else 1.0
            num = e @ v[g] + g_h * (a @ v[g])
            y[h] = np.where(den != 0, num / np.where(den != 0, den, 1.0), 0.0)
    return y, scores, sel


def rows(q, k, v, Wf, W, C, sel, picks):
    """Output rows y[h, t] for the (h, t) pairs in `picks`, at any N.

    Each row is formed from the set definition with explicit sums over its
    softmax and linear keys.  Returns [len(picks), d]."""
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    kept = kept_mask(sel, N)
    phk_cache = {}
    out = np.zeros((len(picks), d))
    for i, (h, t) in enumerate(picks):
        g = h // G
        if g not in phk_cache:
            phk_cache[g] = npmap(k[g], Wf)
        j = np.arange(t + 1)
        window = j > t - W
        old = j <= t - W
        sa = window | (kept[g, : t + 1] & (j // C < t // C) & old)
        la = old & ~sa
        s = (k[g, j[sa]] @ q[h, t]) / np.sqrt(d)
        num = np.zeros(d)
        den = 0.0
        if s.size:
            e = np.exp(s - s.max())
            num += e @ v[g, j[sa]]
            den += e.sum()
        if la.any():
            a = phk_cache[g][j[la]] @ npmap(q[h, t][None], Wf)[0]
            num += a @ v[g, j[la]]
            den += a.sum()
        out[i] = num / den if den != 0 else 0.0
    return out
