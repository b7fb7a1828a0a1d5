"""Numerical assumptions of the GPU design, checked on the CPU.

The on-chip fold chain computes the winner-take-all cosines on bf16 tensor
cores: chunk keys are exactly bf16, and each slot's unit direction u (fp32) is
split into two bf16 terms hi + lo, so S = k.hi + k.lo with fp32 accumulation.
The parity tests exempt tokens whose top-2 cosine gap is below 1e-5; that is
sound only if the split's cosine error stays well below it.  Cosine rule:
"Key-Value Means" (gist.science technical summary, Core mechanism 2).
"""
import numpy as np
import torch


def test_two_term_bf16_split_keeps_the_cosine_well_below_the_tie_threshold():
    rng = np.random.default_rng(0)
    n, d = 8192, 64
    k = torch.from_numpy(rng.standard_normal((n, d))).bfloat16().float()
    # centred slot sums of widely varying magnitude (the mean of a slot's members)
    c = rng.standard_normal((n, d)) * rng.uniform(0.05, 80.0, (n, 1))
    c -= c.mean(axis=1, keepdims=True)
    u64 = c / np.linalg.norm(c, axis=1, keepdims=True)
    u = torch.from_numpy(u64).float()
    hi = u.bfloat16().float()
    lo = (u - hi).bfloat16().float()
    approx = (k * hi).sum(1) + (k * lo).sum(1)          # fp32 products and sums
    exact = (k.double() * torch.from_numpy(u64)).sum(1)
    err = ((approx.double() - exact) / k.double().norm(dim=1)).abs()
    assert float(err.max()) < 2e-6
    # a single bf16 term would not do: its error is far above the threshold
    one = ((k * hi).sum(1).double() - exact) / k.double().norm(dim=1)
    assert float(one.abs().max()) > 1e-4


def _lazy_online_softmax(scores, values, tau, block=64):
    """The tensor-core attention's per-row softmax: blocks of keys, a running
    maximum that is raised only when a block exceeds it by more than tau (log2
    units), unnormalised P = 2^(s - m) in [0, 2^tau], O and l rescaled when it is."""
    m_used, l = -np.inf, np.float32(0)
    o = np.zeros(values.shape[1], np.float32)
    pmax = 0.0
    for b0 in range(0, len(scores), block):
        s = scores[b0:b0 + block].astype(np.float32)
        mblk = float(s.max())
        alpha = np.float32(1)
        if mblk > m_used:
            if m_used == -np.inf:
                m_used = mblk
            elif mblk > m_used + tau:
                alpha = np.float32(np.exp2(m_used - mblk))
                m_used = mblk
        p = np.exp2(s - np.float32(m_used)).astype(np.float32)
        pmax = max(pmax, float(p.max()))
        l = l * alpha + p.sum(dtype=np.float32)
        o = o * alpha + (p[:, None] * values[b0:b0 + block]).sum(0, dtype=np.float32)
    return o / l, pmax


def test_lazy_rescaling_is_exact_softmax_and_bounds_p():
    """Raising the running maximum only by more than 2^8 changes nothing but
    rounding, and keeps every unnormalised probability within [0, 2^8]."""
    rng = np.random.default_rng(1)
    for trial in range(40):
        n = int(rng.integers(1, 900))
        # log2-scaled scores with drifting level, the case that triggers rescales
        s = (rng.standard_normal(n) * rng.uniform(0.1, 6.0) + np.linspace(0, rng.uniform(-20, 40), n))
        v = rng.standard_normal((n, 8))
        w = np.exp2(s - s.max())
        exact = (w[:, None] * v).sum(0) / w.sum()
        got, pmax = _lazy_online_softmax(s, v.astype(np.float32), tau=8.0)
        np.testing.assert_allclose(got, exact, rtol=0, atol=2e-5 * np.abs(v).max())
        assert pmax <= 2.0 ** 8 * (1 + 1e-6)


def test_decode_butterfly_leaves_key_i_on_lane_i():
    """The decode kernel's transpose-reduce of per-lane partial dot products (32
    lanes x 32 keys): at offsets 16, 8, 4, 2, 1 each lane keeps the half of its
    live entries on its side of the offset bit and adds its partner's other
    half; afterwards lane i holds the full sum for key i.  Emulated lane by lane
    with distinct integer partials, so any index slip shows."""
    rng = np.random.default_rng(2)
    part = rng.integers(-1000, 1000, size=(32, 32))  # [lane, key]
    v = part.copy()
    off, w = 16, 32
    while off >= 1:
        nv = v.copy()
        for lane in range(32):
            partner = lane ^ off
            up, pup = (lane & off) != 0, (partner & off) != 0
            for i in range(w // 2):
                keep = v[lane, i + w // 2] if up else v[lane, i]
                recv = v[partner, i] if pup else v[partner, i + w // 2]
                nv[lane, i] = keep + recv
        v = nv
        off, w = off >> 1, w >> 1
    np.testing.assert_array_equal(v[:, 0], part.sum(axis=0))

