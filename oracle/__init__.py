"""Plain fp64 CPU oracle for the Key-Value Means (KVM) layer forward.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline are the only callers.  The CUDA library never imports, links or runs
anything here, and nothing here imports the CUDA library.

The arithmetic lives in ``kvm_oracle.c`` (plain C, fp64, naive loops, one
step at a time as the method states it).  This module compiles it with gcc,
loads it with ctypes and adds the decode-step composition, which is plain
bookkeeping of which tokens sit in the window.

Page title of every source cited: "Key-Value Means".  "KVM summary" is the
gist.science technical summary, "KVM abstract" the chatpaper.ai abstract.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvm_oracle.c")
_LIB = os.path.join(_HERE, "libkvm_oracle.so")

MERGED, APPENDED, SINK = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/libkvm_oracle.so (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("head_dim", ctypes.c_int32), ("rope_dims", ctypes.c_int32),
        ("rope_theta", ctypes.c_double), ("chunk", ctypes.c_int32),
        ("window", ctypes.c_int32), ("n_sinks", ctypes.c_int32),
        ("sched", ctypes.c_int32), ("max_slots", ctypes.c_int32),
        ("coef", ctypes.c_double), ("expo", ctypes.c_double),
        ("ln_eps", ctypes.c_double), ("merge_pre_append", ctypes.c_int32),
        ("cos_nope_only", ctypes.c_int32), ("no_value_norm", ctypes.c_int32),
    ]


@dataclass
class OracleConfig:
    """Layer hyper-parameters as the pages' problem statement lists them
    (KVM summary, Methodology and Core mechanisms 1-5)."""
    head_dim: int = 64
    rope_dims: int = 32
    rope_theta: float = 10000.0
    chunk: int = 128
    window: int = 512
    n_sinks: int = 16
    sched: int = 0            # 0 fixed (cap = max_slots), 1 power law
    max_slots: int = 256
    coef: float = 4.0
    expo: float = 0.5
    ln_eps: float = 1e-5
    merge_pre_append: int = 0
    cos_nope_only: int = 0
    no_value_norm: int = 0    # ablation: read value = sum_v / count

    def c(self) -> _Cfg:
        return _Cfg(self.head_dim, self.rope_dims, self.rope_theta, self.chunk, self.window,
                    self.n_sinks, self.sched, self.max_slots, self.coef, self.expo,
                    self.ln_eps, self.merge_pre_append, self.cos_nope_only, self.no_value_norm)


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64, I32 = ctypes.c_int64, ctypes.c_int32
        _lib.kvo_capacity.restype = I64
        _lib.kvo_capacity.argtypes = [P, I64]
        _lib.kvo_fold_event.restype = ctypes.c_int
        _lib.kvo_fold_event.argtypes = [P, P, P, P, P, P, P, I64, P, P, P, P, P, P, P, P]
        _lib.kvo_state_view.restype = None
        _lib.kvo_state_view.argtypes = [P, I64, P, P, P, P, P, P]
        _lib.kvo_attend_query.restype = None
        _lib.kvo_attend_query.argtypes = [P, I64, P, P, P, I64, I64, P, P, P]
        _lib.kvo_rope_rows.restype = None
        _lib.kvo_rope_rows.argtypes = [P, I64, I64, P, P]
        _lib.kvo_prefill_head.restype = ctypes.c_int
        _lib.kvo_prefill.restype = ctypes.c_int
        _lib.kvo_prefill.argtypes = [P, I64, I64, P, P, P, P, P, P, P, P, P, P, P, I64,
                                     P, P, P, P, P, ctypes.c_int]
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def capacity(cfg: OracleConfig, t: int) -> int:
    """Slot capacity after t overflowed tokens (KVM summary, Core mechanism 3)."""
    c = cfg.c()
    return int(lib().kvo_capacity(ctypes.byref(c), int(t)))


class OracleState:
    """State of one (batch, head): raw sums, integer counts, read radii, slot
    count n and overflowed-token count t (KVM summary, lay part 'smart merge')."""

    def __init__(self, cfg: OracleConfig):
        M, d = cfg.max_slots, cfg.head_dim
        self.n = 0
        self.t = 0
        self.sum_k = np.zeros((M, d))
        self.sum_v = np.zeros((M, d))
        self.count = np.zeros(M, dtype=np.int64)
        self.rho = np.zeros(M)

    def copy(self) -> "OracleState":
        s = OracleState.__new__(OracleState)
        s.n, s.t = self.n, self.t
        s.sum_k, s.sum_v = self.sum_k.copy(), self.sum_v.copy()
        s.count, s.rho = self.count.copy(), self.rho.copy()
        return s


class OracleError(RuntimeError):
    pass


def fold_event(cfg: OracleConfig, st: OracleState, first_pos: int, k, v, g):
    """Fold one chunk of overflowed tokens into ``st`` (in place).

    Returns a dict with per-token ``assign`` (slot), ``kind`` (0 merged,
    1 appended, 2 sink), ``max_sim`` (surprise score), ``gap`` (top-2 gap of
    the final argmax) and the event's ``sel_margin``.
    """
    C = cfg.chunk
    k, v, g = _f64(k), _f64(v), _f64(g)
    assert k.shape == (C, cfg.head_dim) and v.shape == k.shape and g.shape == (C,)
    n = ctypes.c_int64(st.n)
    t = ctypes.c_int64(st.t)
    assign = np.full(C, -1, dtype=np.int32)
    kind = np.full(C, -1, dtype=np.int32)
    max_sim = np.zeros(C)
    gap = np.zeros(C)
    sel = ctypes.c_double(0.0)
    c = cfg.c()
    rc = lib().kvo_fold_event(ctypes.byref(c), ctypes.byref(n), ctypes.byref(t),
                              _p(st.sum_k), _p(st.sum_v), _p(st.count), _p(st.rho),
                              int(first_pos), _p(k), _p(v), _p(g),
                              _p(assign), _p(kind), _p(max_sim), _p(gap), ctypes.byref(sel))
    if rc != 0:
        raise OracleError(f"kvo_fold_event failed with status {rc}")
    st.n, st.t = int(n.value), int(t.value)
    return dict(assign=assign, kind=kind, max_sim=max_sim, gap=gap, sel_margin=sel.value)


def state_view(cfg: OracleConfig, st: OracleState):
    """Just-in-time read view: keys LayerNorm(sum_k/count) with the RoPE dims
    zeroed, values rho * unit(sum_v) (KVM summary, Core mechanisms 2 and 4)."""
    n, d = st.n, cfg.head_dim
    kv = np.zeros((max(n, 1), d))
    vv = np.zeros((max(n, 1), d))
    c = cfg.c()
    lib().kvo_state_view(ctypes.byref(c), n, _p(st.sum_k), _p(st.sum_v), _p(st.count),
                         _p(st.rho), _p(kv), _p(vv))
    return kv[:n], vv[:n]


def attend_query(cfg: OracleConfig, key_view, val_view, q, p: int, wk, wv, w_first_pos: int):
    """One query at position p over the state view and a window of tokens at
    positions w_first_pos.. (one softmax; KVM summary, Core mechanism 4)."""
    d = cfg.head_dim
    key_view, val_view = _f64(key_view).reshape(-1, d), _f64(val_view).reshape(-1, d)
    wk, wv, q = _f64(wk).reshape(-1, d), _f64(wv).reshape(-1, d), _f64(q)
    out = np.zeros(d)
    c = cfg.c()
    wk_rot = np.zeros_like(wk)
    lib().kvo_rope_rows(ctypes.byref(c), wk.shape[0], int(w_first_pos), _p(wk), _p(wk_rot))
    lib().kvo_attend_query(ctypes.byref(c), key_view.shape[0], _p(key_view), _p(val_view),
                           _p(q), int(p), wk.shape[0], _p(wk_rot), _p(wv), _p(out))
    return out


def n_events(cfg: OracleConfig, N: int) -> int:
    """Fold events a prefill of N tokens performs: chunk c >= W/C + 1 folds chunk
    c - W/C - 1 before it runs."""
    nchunks = -(-N // cfg.chunk)
    return max(0, nchunks - cfg.window // cfg.chunk - 1)


def prefill(cfg: OracleConfig, q, k, v, g, threads: int | None = None, max_events: int | None = None):
    """Chunked prefill of [H, N, d] independent heads from an empty state.

    q, k, v: [H, N, d]; g: [H, N].  Returns (out [H,N,d], states list, debug dict).
    """
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    H, N, d = q.shape
    assert d == cfg.head_dim and k.shape == q.shape and v.shape == q.shape and g.shape == (H, N)
    M, C = cfg.max_slots, cfg.chunk
    E = n_events(cfg, N) if max_events is None else max_events
    out = np.zeros((H, N, d))
    n = np.zeros(H, dtype=np.int64)
    t = np.zeros(H, dtype=np.int64)
    sum_k = np.zeros((H, M, d))
    sum_v = np.zeros((H, M, d))
    count = np.zeros((H, M), dtype=np.int64)
    rho = np.zeros((H, M))
    Ea = max(E, 1)
    assign = np.full((H, Ea, C), -1, dtype=np.int32)
    kind = np.full((H, Ea, C), -1, dtype=np.int32)
    max_sim = np.zeros((H, Ea, C))
    gap = np.zeros((H, Ea, C))
    sel = np.zeros((H, Ea))
    if threads is None:
        threads = len(os.sched_getaffinity(0))
    c = cfg.c()
    rc = lib().kvo_prefill(ctypes.byref(c), H, N, _p(q), _p(k), _p(v), _p(g), _p(out),
                           _p(n), _p(t), _p(sum_k), _p(sum_v), _p(count), _p(rho), E,
                           _p(assign), _p(kind), _p(max_sim), _p(gap), _p(sel), int(threads))
    if rc != 0:
        raise OracleError(f"kvo_prefill failed with status {rc}")
    states = []
    for h in range(H):
        s = OracleState.__new__(OracleState)
        s.n, s.t = int(n[h]), int(t[h])
        s.sum_k, s.sum_v, s.count, s.rho = sum_k[h], sum_v[h], count[h], rho[h]
        states.append(s)
    dbg = dict(assign=assign[:, :E], kind=kind[:, :E], max_sim=max_sim[:, :E], gap=gap[:, :E],
               sel_margin=sel[:, :E])
    return out, states, dbg


class OracleDecoder:
    """Decode of one (batch, head), one token per step (KVM summary, Core
    mechanism 1: a block that leaves the window is folded before the query
    that no longer sees it).

    The window is kept as a plain list of the unfolded tokens in position
    order.  At position p = c*C (first token of chunk c) with c >= W/C + 1,
    the oldest C tokens (chunk c - W/C - 1) are folded first.
    """

    def __init__(self, cfg: OracleConfig, state: OracleState, pos: int, wk, wv, wg):
        self.cfg = cfg
        self.st = state
        self.pos = int(pos)
        self.wk = [np.asarray(x, dtype=np.float64) for x in _f64(wk).reshape(-1, cfg.head_dim)]
        self.wv = [np.asarray(x, dtype=np.float64) for x in _f64(wv).reshape(-1, cfg.head_dim)]
        self.wg = [float(x) for x in _f64(wg).reshape(-1)]
        self.last_fold = None

    def step(self, q, k, v, g):
        cfg, C = self.cfg, self.cfg.chunk
        p = self.pos
        c, r = divmod(p, C)
        self.last_fold = None
        if r == 0 and c >= cfg.window // C + 1:
            first = (c - cfg.window // C - 1) * C
            w_first = p - len(self.wk)
            if w_first != first or len(self.wk) != cfg.window + C:
                raise OracleError("window does not hold the chunk that overflows")
            self.last_fold = fold_event(cfg, self.st, first, np.stack(self.wk[:C]),
                                        np.stack(self.wv[:C]), np.array(self.wg[:C]))
            del self.wk[:C], self.wv[:C], self.wg[:C]
        self.wk.append(_f64(k))
        self.wv.append(_f64(v))
        self.wg.append(float(g))
        kv, vv = state_view(cfg, self.st)
        w_first = p - len(self.wk) + 1
        out = attend_query(cfg, kv, vv, q, p, np.stack(self.wk), np.stack(self.wv), w_first)
        self.pos += 1
        return out


__all__ = ["OracleConfig", "OracleState", "OracleDecoder", "OracleError", "capacity",
           "fold_event", "state_view", "attend_query", "prefill", "n_events", "build",
           "MERGED", "APPENDED", "SINK"]


# ------------------------------------------------------------- whole layer
#
# The layer around the KVM attention (KVM summary, Methodology: queries, keys,
# values and a data-dependent merge gate are projections of the layer input;
# the heads are projected back).  Weight layouts follow the linear layer's
# [out_features, in_features] convention: w_in rows are q of heads 0..H-1 (64
# rows per head), then k, then v, then one merge-gate row per head; w_out is
# [d_model, H * 64] over head-major features.  Plain fp64 matrix products.

def bf16_round(a):
    """Round float64 values to the nearest bf16 value (8 significant bits, ties to
    even), exactly, returned as float64 (normal range)."""
    a = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(a)                        # a = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)


def layer_project_in(x, w_in, H: int, d: int = 64):
    """q, k, v [B, H, N, d] and gate = sigmoid(logit) [B, H, N] from x [B, N, d_model]."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w_in, dtype=np.float64)
    B, N, _ = x.shape
    z = x @ w.T                               # [B, N, 3*H*d + H]
    Hd = H * d
    heads = lambda part: part.reshape(B, N, H, d).transpose(0, 2, 1, 3)
    q, k, v = heads(z[..., :Hd]), heads(z[..., Hd:2 * Hd]), heads(z[..., 2 * Hd:3 * Hd])
    gate = 1.0 / (1.0 + np.exp(-z[..., 3 * Hd:3 * Hd + H])).transpose(0, 2, 1)
    return q, k, v, gate


def layer_project_out(o, w_out):
    """y [B, N, d_model] from the attention output o [B, H, N, d]."""
    o = np.asarray(o, dtype=np.float64)
    B, H, N, d = o.shape
    flat = o.transpose(0, 2, 1, 3).reshape(B, N, H * d)
    return flat @ np.asarray(w_out, dtype=np.float64).T


def layer_forward(cfg: OracleConfig, x, w_in, w_out, H: int, threads: int | None = None):
    """Whole-layer forward.  The projected q, k, v are rounded to bf16 before the
    attention: they are bf16 tensors between the layer's operations, and the
    fold's winner-take-all decisions are taken on those values."""
    q, k, v, gate = layer_project_in(x, w_in, H, cfg.head_dim)
    B, _, N, d = q.shape
    q, k, v = bf16_round(q), bf16_round(k), bf16_round(v)
    o = np.empty_like(q)
    dbgs = []
    for b in range(B):
        out, _, dbg = prefill(cfg, q[b], k[b], v[b], gate[b], threads=threads)
        o[b] = out
        dbgs.append(dbg)
    return layer_project_out(o, w_out), (q, k, v, gate, o), dbgs
