"""Independent brute-force restatement of the KVM layer forward for tiny inputs.

Used only to pin the C oracle.  It is written differently on purpose:
vectorised numpy cosine matrices, ``np.lexsort`` for the surprise selection,
``torch.nn.functional.layer_norm`` for the state keys, complex-number RoPE and
``torch.softmax`` for the attention, so that a slip in one formulation does
not repeat in the other.  Sources: "Key-Value Means" (gist.science technical
summary, Core mechanisms 1-5).
"""
from __future__ import annotations

import math

import numpy as np
import torch


def cap_of(t, S, sched, M, coef, expo):
    if sched == 0:
        return M
    return S if t <= 0 else S + math.ceil(coef * t ** expo)


def rope_complex(x, pos, r, theta):
    """RoPE as a complex rotation of the pairs (i, i + r/2), i < r/2."""
    x = np.asarray(x, dtype=np.float64)
    h = r // 2
    z = x[..., :h] + 1j * x[..., h:r]
    freq = theta ** (-np.arange(h) * 2.0 / r)
    z = z * np.exp(1j * np.asarray(pos, dtype=np.float64)[..., None] * freq)
    out = x.copy()
    out[..., :h] = z.real
    out[..., h:r] = z.imag
    return out


def ln(x, eps):
    t = torch.as_tensor(np.asarray(x, dtype=np.float64))
    return torch.nn.functional.layer_norm(t, (t.shape[-1],), eps=eps).numpy()


def cos_matrix(a, b):
    na = np.linalg.norm(a, axis=-1, keepdims=True)
    nb = np.linalg.norm(b, axis=-1, keepdims=True)
    num = a @ b.T
    den = na * nb.T
    with np.errstate(invalid="ignore", divide="ignore"):
        c = np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)
    return c


class BFState:
    def __init__(self):
        self.sk, self.sv, self.cnt, self.rho = [], [], [], []
        self.t = 0

    @property
    def n(self):
        return len(self.sk)


class NoMergeTarget(ValueError):
    """A token must merge but the state has no mergeable slot (possible only
    when merge targets are restricted to the slots before the chunk's appends)."""


def bf_fold(st: BFState, first_pos, k, v, g, *, S, sched, M, coef, expo, eps, C,
            r=0, pre_append=False, nope_only=False):
    """One fold event.  Alternative readings: ``pre_append`` restricts merge
    targets to the slots that existed before this chunk's appends;
    ``nope_only`` takes the cosine over the non-rotary dims [r, d) only."""
    lo_dim = r if nope_only else 0
    idx = np.arange(first_pos, first_pos + C)
    assign = np.full(C, -1)
    kind = np.full(C, -1)
    for i in range(C):
        if idx[i] < S:
            st.sk.append(g[i] * k[i]); st.sv.append(g[i] * v[i]); st.cnt.append(1)
            st.rho.append(float(np.linalg.norm(v[i])))
            assign[i] = st.n - 1; kind[i] = 2
    cand = np.array([i for i in range(C) if idx[i] >= S], dtype=np.int64)
    st.t += C
    n0 = st.n
    if n0 > S and cand.size:
        kh = ln(np.array(st.sk[S:]) / np.array(st.cnt[S:])[:, None], eps)
        m = cos_matrix(k[cand][:, lo_dim:], kh[:, lo_dim:]).max(axis=1)
    else:
        m = np.full(cand.size, -np.inf)
    a = int(np.clip(cap_of(st.t, S, sched, M, coef, expo) - n0, 0, cand.size))
    order = np.lexsort((cand, m))          # by m, then by position
    chosen = np.sort(cand[order[:a]])
    for i in chosen:
        st.sk.append(g[i] * k[i]); st.sv.append(g[i] * v[i]); st.cnt.append(1)
        st.rho.append(float(np.linalg.norm(v[i])))
        assign[i] = st.n - 1; kind[i] = 1
    rest = np.array([i for i in cand if i not in set(chosen.tolist())], dtype=np.int64)
    if rest.size:
        hi = n0 if pre_append else st.n
        if hi <= S:
            raise NoMergeTarget(f"event at position {first_pos}: no slot to merge into")
        kh = ln(np.array(st.sk[S:hi]) / np.array(st.cnt[S:hi])[:, None], eps)
        # first maximum = lowest index
        tgt = np.argmax(cos_matrix(k[rest][:, lo_dim:], kh[:, lo_dim:]), axis=1) + S
        for i, j in zip(rest, tgt):
            assign[i] = j; kind[i] = 0
        for i, j in zip(rest, tgt):
            st.sk[j] = st.sk[j] + g[i] * k[i]
            st.sv[j] = st.sv[j] + g[i] * v[i]
            st.cnt[j] += 1
    return assign, kind


def bf_view(st: BFState, r, eps, no_vnorm=False):
    if st.n == 0:
        return np.zeros((0, 0)), np.zeros((0, 0))
    kh = ln(np.array(st.sk) / np.array(st.cnt)[:, None], eps)
    kh[:, :r] = 0.0
    sv = np.array(st.sv)
    if no_vnorm:  # ablation without the value-length normalisation: the member mean
        return kh, sv / np.array(st.cnt, dtype=np.float64)[:, None]
    nv = np.linalg.norm(sv, axis=1, keepdims=True)
    vh = np.where(nv > 0, np.array(st.rho)[:, None] * sv / np.where(nv > 0, nv, 1.0), 0.0)
    return kh, vh


def bf_prefill(q, k, v, g, *, C, W, S, r, sched=0, M=32, coef=4.0, expo=0.5, eps=1e-5,
               theta=10000.0, pre_append=False, nope_only=False, no_vnorm=False):
    """One head: q, k, v [N, d] float64, g [N]. Returns out [N, d], state, assignments."""
    q, k, v, g = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g))
    N, d = q.shape
    st = BFState()
    out = np.zeros((N, d))
    events = []
    pos = np.arange(N)
    qr = rope_complex(q, pos, r, theta)
    kr = rope_complex(k, pos, r, theta)
    for c in range(-(-N // C)):
        if c >= W // C + 1:
            e = c - W // C - 1
            sl = slice(e * C, (e + 1) * C)
            events.append(bf_fold(st, e * C, k[sl], v[sl], g[sl], S=S, sched=sched, M=M,
                                  coef=coef, expo=expo, eps=eps, C=C, r=r,
                                  pre_append=pre_append, nope_only=nope_only))
        kh, vh = bf_view(st, r, eps, no_vnorm)
        ws = max(0, (c - W // C) * C)
        for p in range(c * C, min(N, (c + 1) * C)):
            s_state = (q[p] @ kh.T) if st.n else np.zeros(0)
            s_win = kr[ws:p + 1] @ qr[p]
            s = torch.as_tensor(np.concatenate([s_state, s_win]) / math.sqrt(d))
            w = torch.softmax(s, dim=0).numpy()
            vals = np.concatenate([vh.reshape(-1, d), v[ws:p + 1]], axis=0)
            out[p] = w @ vals
    return out, st, events
