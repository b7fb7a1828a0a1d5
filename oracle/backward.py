"""Backward of the KVM prefill at fixed fold decisions: plain PyTorch fp64 autograd.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: the tests and the
benchmark's CPU baseline call it; the CUDA library never does.

The pages say the layer trains chunk-parallel ("Key-Value Means", technical
summary, Contributions and Significance) but say nothing about the gradient of
the winner-take-all assignment.  Reading taken here: the fold's discrete
decisions -- the slot each merged token joins, which tokens the surprise
selection appends, which tokens found the sink slots -- are constants taken
from the forward pass; the gradient flows through everything continuous:

* the attention (one softmax over the state rows and the RoPE window; Core
  mechanism 4), with RoPE as the linear map it is;
* the just-in-time read of the state (Core mechanism 2 and 4): key rows
  LayerNorm(sum_k / count) with the rotary dims zeroed, value rows
  rho * sum_v / |sum_v| (or sum_v / count in the no-value-norm ablation);
* the gate-weighted sums sum_k = sum g_t k_t, sum_v = sum g_t v_t of each
  slot's members (Core mechanism 2: the gate modulates what is absorbed), and
  the read radius rho = |v| of the token that founded the slot (Core
  mechanism 3).

Counts are integers and carry no gradient; the cosine that made the
decisions carries none either (it only chose).

``forward_fixed`` restates the prefill of one (batch, head) row with torch
operations and the given decisions; the tests pin it to the C oracle's
forward (same outputs) and its gradient to central finite differences, both
of this function and of the full method (which re-decides) where no decision
is near a tie.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import MERGED, APPENDED, SINK  # noqa: F401  (kinds of the debug record)


def _rope_tables(cfg, N: int):
    half = cfg.rope_dims // 2
    pos = torch.arange(N, dtype=torch.float64)
    i = torch.arange(half, dtype=torch.float64)
    inv = torch.tensor(cfg.rope_theta, dtype=torch.float64) ** (-2.0 * i / max(cfg.rope_dims, 1))
    ang = pos[:, None] * inv[None, :]
    return torch.cos(ang), torch.sin(ang)


def _rotate(x, cos, sin, r: int):
    """Rotate-half RoPE on dims [0, r) of rows x [n, d] at the positions of cos/sin."""
    if r == 0:
        return x
    half = r // 2
    a, b = x[:, :half], x[:, half:r]
    return torch.cat([a * cos - b * sin, b * cos + a * sin, x[:, r:]], dim=1)


def _read_view(cfg, sk, sv, cnt, rho):
    """Read rows of n slots: keys LayerNorm(sk / cnt) with dims [0, r) zeroed,
    values rho * unit(sv) (ablation: sv / cnt)."""
    d, r = cfg.head_dim, cfg.rope_dims
    x = sk / cnt[:, None]
    mu = x.mean(dim=1, keepdim=True)
    var = ((x - mu) ** 2).mean(dim=1, keepdim=True)
    kh = (x - mu) / torch.sqrt(var + cfg.ln_eps)
    mask = torch.ones(d, dtype=torch.float64)
    mask[:r] = 0.0
    kh = kh * mask
    if cfg.no_value_norm:
        vh = sv / cnt[:, None]
    else:
        nv = torch.sqrt((sv * sv).sum(dim=1, keepdim=True))
        vh = rho[:, None] * sv / nv
    return kh, vh


def forward_fixed(cfg, q, k, v, g, assign, kind):
    """Prefill of one row with the given decisions.

    q, k, v: torch fp64 [N, d]; g: [N]; assign, kind: int arrays [E, C] of the
    fold events (slot and kind of every folded token).  Returns out [N, d].
    Event e folds tokens e*C .. e*C + C - 1: founders (sinks, appended tokens)
    set their new slot's sums, count 1 and radius |v|; merged tokens then add
    g*k and g*v to their slot in position order.  Chunk c attends to the state
    after event c - W/C - 1 (none before) and to tokens (c - W/C)*C .. p.
    """
    N, d = q.shape
    C, Wc, r = cfg.chunk, cfg.window // cfg.chunk, cfg.rope_dims
    E = int(np.asarray(assign).shape[0]) if np.asarray(assign).size else 0
    cos, sin = _rope_tables(cfg, N)
    qr = _rotate(q, cos, sin, r)
    kr = _rotate(k, cos, sin, r)
    scale = 1.0 / math.sqrt(d)
    # slot state as python lists of row tensors (functional updates keep autograd simple)
    sk, sv, cnt, rho = [], [], [], []
    views = []  # (kh, vh) after every event
    assign = np.asarray(assign)
    kind = np.asarray(kind)
    for e in range(E):
        base = e * C
        for i in range(C):
            if kind[e, i] in (APPENDED, SINK):
                j, t = int(assign[e, i]), base + i
                while len(sk) <= j:
                    sk.append(None), sv.append(None), cnt.append(0), rho.append(None)
                sk[j] = g[t] * k[t]
                sv[j] = g[t] * v[t]
                cnt[j] = 1
                rho[j] = torch.sqrt((v[t] * v[t]).sum())
        for i in range(C):
            if kind[e, i] == MERGED:
                j, t = int(assign[e, i]), base + i
                sk[j] = sk[j] + g[t] * k[t]
                sv[j] = sv[j] + g[t] * v[t]
                cnt[j] += 1
        n = len(sk)
        kh, vh = _read_view(cfg, torch.stack(sk[:n]), torch.stack(sv[:n]),
                            torch.tensor(cnt[:n], dtype=torch.float64), torch.stack(rho[:n]))
        views.append((kh, vh))
    outs = []
    nchunks = -(-N // C)
    for c in range(nchunks):
        p0, p1 = c * C, min(N, (c + 1) * C)
        ws = max(0, (c - Wc) * C)
        qc = q[p0:p1]
        s_win = (qr[p0:p1] @ kr[ws:p1].T) * scale
        pos_q = torch.arange(p0, p1)[:, None]
        pos_k = torch.arange(ws, p1)[None, :]
        s_win = s_win.masked_fill(pos_k > pos_q, float("-inf"))
        e = c - Wc - 1
        if e >= 0:
            kh, vh = views[e]
            s_st = (qc @ kh.T) * scale
            s = torch.cat([s_st, s_win], dim=1)
            vals = torch.cat([vh, v[ws:p1]], dim=0)
        else:
            s, vals = s_win, v[ws:p1]
        outs.append(torch.softmax(s, dim=1) @ vals)
    return torch.cat(outs, dim=0)


def backward(cfg, q, k, v, g, assign, kind, dout):
    """Gradients (dq, dk, dv, dg) of sum(out * dout) for one row at fixed
    decisions; numpy fp64 in and out."""
    t = [torch.tensor(np.asarray(x, dtype=np.float64), requires_grad=True) for x in (q, k, v, g)]
    out = forward_fixed(cfg, *t, assign, kind)
    (out * torch.tensor(np.asarray(dout, dtype=np.float64))).sum().backward()
    # an input the output does not depend on (the gate before the first fold) has no grad
    return tuple(x.grad.numpy() if x.grad is not None else np.zeros(x.shape) for x in t)


def forward_fixed_np(cfg, q, k, v, g, assign, kind):
    """forward_fixed on numpy fp64 inputs (no gradient)."""
    with torch.no_grad():
        t = [torch.tensor(np.asarray(x, dtype=np.float64)) for x in (q, k, v, g)]
        return forward_fixed(cfg, *t, assign, kind).numpy()


__all__ = ["forward_fixed", "forward_fixed_np", "backward"]
