"""Gradient oracle of the STILL layer with the routing held fixed.

TEST INFRASTRUCTURE ONLY -- nothing in the product path imports this module.
It shares no code with the CUDA library; the masks come from ``brute`` (the
set definition), the arithmetic is plain PyTorch in float64 on the CPU.

What it computes: the exact derivative of the layer output of "STILL:
Content-Aware Intra-Layer Hybrid Attention for Efficient LLM Linearization"
(sections "Content-Aware Routing with Fixed Budget", "NP-Map: Norm-Preserving
Feature Map"),

    y_t = (sum_SA e^{s_tj - c_t} v_j + sum_LA (phi(q_t).phi(k_j)) v_j)
          / (sum_SA e^{s_tj - c_t} + sum_LA phi(q_t).phi(k_j)),
    s_tj = q_t.k_j / sqrt(d),  c_t = max_{j in SA(t)} s_tj,
    phi(x) = ||x|| u / ||u||,  u = softmax(x Wf),

with respect to q, k, v and Wf (and, for the gated layer, the gate's
pre-activations), for an upstream gradient dy, with the kept
set (the selection) held fixed: the selection is a discrete choice made from
the scores, and the training path of the pages' "Experiments" section trains
through the layer with the routing given.  The stabiliser c_t is part of the
output (the linear terms are not scaled by it), so its gradient is part of
the derivative: it reaches the logit that attains the row maximum.  Where
several logits attain it the lowest key position takes it (the one the row
keeps after a first-maximum scan), or the position a caller passes in
``cidx`` -- the GPU reports its own choice, and near-equal maxima are
compared with that choice.

The gated layer (section "NP-Map: Norm-Preserving Feature Map": a gate raises
the linear branch's rank; its equation is lost, and the reading taken is a
per-channel sigmoid gate on the linear numerator) is

    y_t = (sum_SA e^{s_tj - c_t} v_j + sigmoid(a_t) * sum_LA (phi(q_t).phi(k_j)) v_j)
          / (sum_SA e^{s_tj - c_t} + sum_LA phi(q_t).phi(k_j)),

a_t of the layout of q_t, the denominator ungated.

The derivative is taken by reverse-mode automatic differentiation of the
forward written out below (a library primitive); the tests pin it against
central differences of the independent C streaming oracle, against the
softmax-attention gradient of torch's scaled_dot_product_attention where the
layer reduces to it, and against hand-derived values.
"""
from __future__ import annotations

import numpy as np
import torch

from . import brute


def _npmap_t(x: torch.Tensor, Wf: torch.Tensor) -> torch.Tensor:
    """NP-Map of the rows of x [..., d]: ||x|| u / ||u||, u = softmax(x Wf)."""
    u = torch.softmax(x @ Wf, dim=-1)
    return torch.linalg.vector_norm(x, dim=-1, keepdim=True) * u / torch.linalg.vector_norm(u, dim=-1, keepdim=True)


def _group_forward(qg, kg, vg, Wf, sa, la, cidx_g, gate_g=None):
    """Outputs [G, N, d] of the G query heads of one kv head, and the row-max
    positions used for c ([G, N], -1 where SA(t) is empty).  gate_g: the
    gate's pre-activations [G, N, d] of the gated layer, or None."""
    G, N, d = qg.shape
    s = qg @ kg.T / np.sqrt(d)                                     # [G, N, N]
    sa_t = torch.as_tensor(sa)[None].expand(G, N, N)
    la_t = torch.as_tensor(la)[None].expand(G, N, N)
    has = sa_t.any(dim=-1)                                          # [G, N]
    if cidx_g is None:
        masked = torch.where(sa_t, s.detach(), torch.full_like(s, -np.inf))
        idx = torch.argmax(masked, dim=-1)                          # first maximal position
        idx = torch.where(has, idx, torch.full_like(idx, -1))
    else:
        idx = torch.as_tensor(np.asarray(cidx_g, dtype=np.int64))
    c = torch.where(has, s.gather(-1, idx.clamp(min=0)[..., None])[..., 0], torch.zeros_like(s[..., 0]))
    # masked entries take the exponent 0 so that no inf enters the graph
    arg = torch.where(sa_t, s - c[..., None], torch.zeros_like(s))
    e = torch.where(sa_t, torch.exp(arg), torch.zeros_like(s))
    phq = _npmap_t(qg, Wf)                                          # [G, N, df]
    phk = _npmap_t(kg, Wf)                                          # [N, df]
    a = torch.where(la_t, phq @ phk.T, torch.zeros_like(s))
    if gate_g is None:
        num = (e + a) @ vg
    else:
        num = e @ vg + torch.sigmoid(gate_g) * (a @ vg)
    den = (e + a).sum(dim=-1, keepdim=True)
    nz = den != 0
    y = torch.where(nz, num / torch.where(nz, den, torch.ones_like(den)), torch.zeros_like(num))
    return y, idx


def layer_grad(q, k, v, Wf, W, C, sel, dy, cidx=None, gate=None):
    """Gradients of sum(dy * y) for one layer call.

    q [B, Hq, N, d], k, v [B, Hkv, N, d], Wf [d, df], sel [B, Hkv, T_max, lam]
    (the kept positions, -1 padded), dy [B, Hq, N, d]; cidx (optional)
    [B, Hq, N] row-max positions to use for c; gate (optional) [B, Hq, N, d]
    the pre-activations of the gated layer.
    Returns (y, dq, dk, dv, dWf, cidx) as float64 / int64 numpy arrays, and
    dgate [B, Hq, N, d] after them when gate is given."""
    q, k, v, Wf, dy = (np.asarray(a, dtype=np.float64) for a in (q, k, v, Wf, dy))
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    y = np.zeros_like(q)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dWf = np.zeros_like(Wf)
    cid = np.full((B, Hq, N), -1, dtype=np.int64)
    gated = gate is not None
    if gated:
        gate = np.asarray(gate, dtype=np.float64)
        dgate = np.zeros_like(gate)
    Wf_t = torch.tensor(Wf, requires_grad=True)
    for b in range(B):
        kept = brute.kept_mask(np.asarray(sel[b]), N)
        for g in range(Hkv):
            sa, la = brute.route_masks(kept[g], N, W, C)
            hs = slice(g * G, (g + 1) * G)
            qg = torch.tensor(q[b, hs], requires_grad=True)
            kg = torch.tensor(k[b, g], requires_grad=True)
            vg = torch.tensor(v[b, g], requires_grad=True)
            ag = torch.tensor(gate[b, hs], requires_grad=True) if gated else None
            yg, idx = _group_forward(qg, kg, vg, Wf_t, sa, la, None if cidx is None else cidx[b, hs], ag)
            loss = (yg * torch.tensor(dy[b, hs])).sum()
            loss.backward()
            y[b, hs] = yg.detach().numpy()
            dq[b, hs] = qg.grad.numpy()
            dk[b, g] = kg.grad.numpy()
            dv[b, g] = vg.grad.numpy()
            cid[b, hs] = idx.numpy()
            if gated:
                dgate[b, hs] = ag.grad.numpy()
    dWf[...] = Wf_t.grad.numpy() if Wf_t.grad is not None else 0.0
    if gated:
        return y, dq, dk, dv, dWf, cid, dgate
    return y, dq, dk, dv, dWf, cid


def max_gaps(q, k, W, C, sel):
    """Per row, the gap between the largest and the second largest logit over
    SA(t) (inf where SA(t) has one key or none): rows whose gap is below the
    logits' rounding can take c from either position.  Returns [B, Hq, N]."""
    q, k = (np.asarray(a, dtype=np.float64) for a in (q, k))
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.full((B, Hq, N), np.inf)
    for b in range(B):
        kept = brute.kept_mask(np.asarray(sel[b]), N)
        for g in range(Hkv):
            sa, _ = brute.route_masks(kept[g], N, W, C)
            for h in range(g * G, (g + 1) * G):
                s = np.where(sa, q[b, h] @ k[b, g].T / np.sqrt(d), -np.inf)
                top2 = -np.sort(-s, axis=-1)[:, :2]
                ok = np.isfinite(top2[:, 1])
                out[b, h, ok] = top2[ok, 0] - top2[ok, 1]
    return out
