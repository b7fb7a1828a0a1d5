"""Pins of the backward oracle (oracle/backward.py), CPU only.

The backward is the gradient of the prefill at fixed fold decisions (the
reading stated in oracle/backward.py).  Pinned by:
* its forward restatement equals the C oracle's forward (independent code:
  same outputs to rounding, given the C oracle's decisions);
* directional central finite differences of that forward;
* central finite differences of the full method (the C oracle, which decides
  again) where the perturbation changes no decision;
* a textbook reduction: before the first fold the layer is causal softmax
  attention with partial RoPE, so the gradient equals torch's SDPA gradient;
* an invariance: a slot founded by one token that never takes a merge reads
  LayerNorm(g k) and rho * unit(g v), which do not depend on g (up to the
  LayerNorm epsilon), so such tokens (the sinks) get no gate gradient.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import backward as ob

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _cfg(**kw):
    base = dict(head_dim=64, rope_dims=32, chunk=16, window=32, n_sinks=4, max_slots=24)
    base.update(kw)
    return oracle.OracleConfig(**base)


def _inputs(N, seed=0, rep=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((N, 64))
    k = rng.standard_normal((N, 64))
    v = rng.standard_normal((N, 64))
    g = 1.0 / (1.0 + np.exp(-rng.standard_normal(N)))
    if rep:  # some keys repeat earlier ones, so slots take several members
        for t in range(8, N, 7):
            k[t] = k[t - 5] + 0.05 * rng.standard_normal(64)
    return q, k, v, g


def _decisions(cfg, q, k, v, g):
    out, _, dbg = oracle.prefill(cfg, q[None], k[None], v[None], g[None], threads=1)
    return out[0], dbg["assign"][0], dbg["kind"][0], dbg


CASES = [
    ("fixed", dict()),
    ("sqrt", dict(sched=1, max_slots=64, coef=2.0, expo=0.5)),
    ("novnorm", dict(no_value_norm=1)),
    ("nosinks", dict(n_sinks=0)),
    ("norope", dict(rope_dims=0)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_fixed_decision_forward_equals_the_oracle(name, kw):
    cfg = _cfg(**kw)
    q, k, v, g = _inputs(200, seed=1)
    out, assign, kind, _ = _decisions(cfg, q, k, v, g)
    assert assign.shape[0] == oracle.n_events(cfg, 200) > 5
    got = ob.forward_fixed_np(cfg, q, k, v, g, assign, kind)
    np.testing.assert_allclose(got, out, rtol=0, atol=1e-11)


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_gradient_matches_finite_differences(name, kw):
    cfg = _cfg(**kw)
    q, k, v, g = _inputs(160, seed=2)
    _, assign, kind, _ = _decisions(cfg, q, k, v, g)
    rng = np.random.default_rng(3)
    dout = rng.standard_normal(q.shape)
    grads = ob.backward(cfg, q, k, v, g, assign, kind, dout)
    x0 = [q, k, v, g]
    eps = 1e-6
    for trial in range(3):
        u = [rng.standard_normal(x.shape) for x in x0]
        lp = (ob.forward_fixed_np(cfg, *[x + eps * du for x, du in zip(x0, u)], assign, kind) * dout).sum()
        lm = (ob.forward_fixed_np(cfg, *[x - eps * du for x, du in zip(x0, u)], assign, kind) * dout).sum()
        fd = (lp - lm) / (2 * eps)
        an = sum((gr * du).sum() for gr, du in zip(grads, u))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (trial, fd, an)


def test_gradient_of_the_full_method_where_no_decision_moves():
    """The C oracle decides again on the perturbed inputs; where it decides the
    same (no near tie within the perturbation), its finite difference equals
    the fixed-decision gradient."""
    cfg = _cfg()
    q, k, v, g = _inputs(160, seed=4)
    out, assign, kind, dbg = _decisions(cfg, q, k, v, g)
    rng = np.random.default_rng(5)
    dout = rng.standard_normal(q.shape)
    grads = ob.backward(cfg, q, k, v, g, assign, kind, dout)
    eps = 1e-7
    checked = 0
    for trial in range(4):
        u = [rng.standard_normal(x.shape) for x in (q, k, v, g)]
        xp = [x + eps * du for x, du in zip((q, k, v, g), u)]
        xm = [x - eps * du for x, du in zip((q, k, v, g), u)]
        op, ap, kp, _ = _decisions(cfg, *xp)
        om, am, km, _ = _decisions(cfg, *xm)
        if not (np.array_equal(ap, assign) and np.array_equal(am, assign) and
                np.array_equal(kp, kind) and np.array_equal(km, kind)):
            continue
        fd = ((op - om) * dout).sum() / (2 * eps)
        an = sum((gr * du).sum() for gr, du in zip(grads, u))
        assert abs(fd - an) <= 1e-5 * max(1.0, abs(an)), (trial, fd, an)
        checked += 1
    assert checked >= 2


def test_before_the_first_fold_the_gradient_is_that_of_causal_rope_attention():
    cfg = _cfg(chunk=16, window=64)
    N = 64  # (W/C + 1) chunks: no fold event yet
    q, k, v, g = _inputs(N, seed=6)
    rng = np.random.default_rng(7)
    dout = rng.standard_normal(q.shape)
    assign = np.zeros((0, 16), np.int32)
    grads = ob.backward(cfg, q, k, v, g, assign, assign, dout)
    # independent textbook form: complex-number RoPE on pairs (i, i + r/2) and torch SDPA
    r, half = 32, 16
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    pos = torch.arange(N, dtype=torch.float64)
    ang = pos[:, None] * (10000.0 ** (-torch.arange(half, dtype=torch.float64) * 2 / r))[None]
    rot = torch.polar(torch.ones_like(ang), ang)

    def rope(x):
        z = torch.complex(x[:, :half], x[:, half:r]) * rot
        return torch.cat([z.real, z.imag, x[:, r:]], dim=1)

    o = torch.nn.functional.scaled_dot_product_attention(rope(tq)[None], rope(tk)[None], tv[None],
                                                         is_causal=True)[0]
    (o * torch.tensor(dout)).sum().backward()
    for mine, ref in zip(grads[:3], (tq.grad, tk.grad, tv.grad)):
        np.testing.assert_allclose(mine, ref.numpy(), rtol=0, atol=1e-12)
    assert np.all(grads[3] == 0.0)  # no fold: the gate is never used


def test_sinks_get_no_gate_gradient():
    """Sink slots take no merges: their read rows do not depend on the gate."""
    cfg = _cfg(n_sinks=4)
    q, k, v, g = _inputs(160, seed=8)
    _, assign, kind, _ = _decisions(cfg, q, k, v, g)
    rng = np.random.default_rng(9)
    dout = rng.standard_normal(q.shape)
    dq, dk, dv, dg = ob.backward(cfg, q, k, v, g, assign, kind, dout)
    merged = np.zeros(160, bool)
    merged[: assign.size][np.asarray(kind).reshape(-1) == oracle.MERGED] = True
    typical = np.abs(dg[merged]).max()
    assert typical > 1e-3
    # LayerNorm's epsilon (1e-5) leaves a trace of g in the key row: far below a merged token's
    assert np.abs(dg[:4]).max() <= 1e-3 * typical
    # sinks still get key and value gradients through their read rows
    assert np.abs(dk[:4]).max() > 0 and np.abs(dv[:4]).max() > 0
