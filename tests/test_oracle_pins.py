"""Pins of the fp64 CPU oracle against facts that do not come from the oracle.

Each test names what fixes its expected value: a textbook routine the special
case reduces to, a closed form, an invariant the pages state, a hand-worked
example, or an independent brute-force restatement on tiny inputs.  Sources:
"Key-Value Means" (gist.science technical summary, Core mechanisms 1-5).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from bruteforce import NoMergeTarget, bf_prefill, ln, rope_complex
from compressed_kv_state_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(seed, N, d, gate=True):
    rng = np.random.default_rng(seed)
    q, k, v = rng.standard_normal((3, N, d))
    g = 1.0 / (1.0 + np.exp(-rng.standard_normal(N))) if gate else np.ones(N)
    return q, k, v, g


def _run(cfg, q, k, v, g):
    out, states, dbg = oracle.prefill(cfg, q[None], k[None], v[None], g[None], threads=1)
    return out[0], states[0], {key: val[0] for key, val in dbg.items()}


# ---------------------------------------------------------------- textbook

@pytest.mark.parametrize("N", [1, 5, 37, 64])
def test_no_state_reduces_to_causal_attention_with_partial_rope(N):
    """Window >= N: nothing ever overflows, so the layer is plain causal
    softmax attention with RoPE on the first r dims (KVM summary, Core
    mechanisms 1 and 4).  Reference: torch SDPA on complex-rotated q, k."""
    d, r = 16, 8
    cfg = oracle.OracleConfig(head_dim=d, rope_dims=r, chunk=8, window=64, n_sinks=2, max_slots=8)
    q, k, v, g = _inputs(1, N, d)
    out, st, _ = _run(cfg, q, k, v, g)
    pos = np.arange(N)
    qr = torch.as_tensor(rope_complex(q, pos, r, 1e4))[None, None]
    kr = torch.as_tensor(rope_complex(k, pos, r, 1e4))[None, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qr, kr, torch.as_tensor(v)[None, None], is_causal=True)[0, 0].numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    assert st.n == 0 and st.t == 0


def test_rope_relative_position():
    """RoPE scores depend only on the position difference (property of the
    rotation, independent of either implementation)."""
    d, r = 16, 16
    cfg = oracle.OracleConfig(head_dim=d, rope_dims=r, chunk=4, window=64, n_sinks=1, max_slots=4)
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((3, d))
    # one query over one window key: output = v regardless, so check scores via two keys
    k2 = rng.standard_normal(d)
    outs = []
    for shift in (0, 7, 1000):
        o = oracle.attend_query(cfg, np.zeros((0, d)), np.zeros((0, d)), q, 5 + shift,
                                np.stack([k, k2]), np.stack([v, -v]), 2 + shift)
        outs.append(o)
    np.testing.assert_allclose(outs[0], outs[1], atol=1e-9)
    np.testing.assert_allclose(outs[0], outs[2], atol=1e-9)


# -------------------------------------------------------------- closed form

@pytest.mark.parametrize("r", [0, 8, 16])
@pytest.mark.parametrize("N,C,W,S", [(70, 8, 16, 3), (64, 4, 8, 1), (33, 8, 8, 0), (41, 8, 0, 2)])
def test_every_token_appended_closed_form(N, C, W, S, r):
    """Capacity >= N: every overflowed token founds its own slot (count 1),
    so the state read is keys LN(g k) with the RoPE dims zeroed and values
    rho * unit(g v) = v (g > 0).  The layer output is then one softmax over
    [tokens before the window, keyed by LN(g k) against the unrotated query]
    and [the window, RoPE on both sides] (KVM summary, Core mechanisms 2-4).
    Also at the degenerate settings: no window (W = 0: a chunk sees itself and
    the state), no rotary dims (r = 0) and all dims rotary (r = d: the state
    keys are all zero, so every state row scores 0)."""
    d = 16
    cfg = oracle.OracleConfig(head_dim=d, rope_dims=r, chunk=C, window=W, n_sinks=S,
                              max_slots=max(N, S + 1))
    q, k, v, g = _inputs(2, N, d)
    out, st, dbg = _run(cfg, q, k, v, g)
    pos = np.arange(N)
    qr, kr = rope_complex(q, pos, r, 1e4), rope_complex(k, pos, r, 1e4)
    state_keys = ln(g[:, None] * k, 1e-5)
    state_keys[:, :r] = 0.0
    exp = np.zeros_like(out)
    for p in range(N):
        c = p // C
        ws = max(0, (c - W // C) * C)
        n_state = ws if c >= W // C + 1 else 0
        s = np.concatenate([state_keys[:n_state] @ q[p], kr[ws:p + 1] @ qr[p]]) / math.sqrt(d)
        w = torch.softmax(torch.as_tensor(s), 0).numpy()
        exp[p] = w @ np.concatenate([v[:n_state], v[ws:p + 1]])
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-11)
    folded = oracle.n_events(cfg, N) * C
    assert st.n == folded and st.t == folded
    assert (st.count[:folded] == 1).all()
    np.testing.assert_allclose(st.sum_k[:folded], g[:folded, None] * k[:folded], atol=0)


# ---------------------------------------------------------------- invariants

def _random_run(seed=5, N=600, sched=1, M=64, C=16, W=32, S=4, d=16, r=8, dup=0.3, coef=2.0,
                expo=0.5):
    rng = np.random.default_rng(seed)
    q, k, v, g = _inputs(seed, N, d)
    for t in range(1, N):               # some near-duplicate keys so merges happen
        if rng.random() < dup:
            k[t] = k[rng.integers(0, t)] + 0.1 * rng.standard_normal(d)
    cfg = oracle.OracleConfig(head_dim=d, rope_dims=r, chunk=C, window=W, n_sinks=S,
                              sched=sched, max_slots=M, coef=coef, expo=expo)
    return cfg, (q, k, v, g), _run(cfg, q, k, v, g)


@pytest.mark.parametrize("sched,M", [(0, 24), (1, 64)])
def test_read_radius_preserved(sched, M):
    """||value view_i|| = rho_i = ||founding value|| for every slot (KVM
    summary, Core mechanism 2: values renormalised to the read radius fixed
    at slot creation)."""
    cfg, (q, k, v, g), (_, st, dbg) = _random_run(sched=sched, M=M)
    kv, vv = oracle.state_view(cfg, st)
    np.testing.assert_allclose(np.linalg.norm(vv, axis=1), st.rho[:st.n], rtol=1e-12)
    founders = {}
    for e in range(dbg["assign"].shape[0]):
        for i in range(cfg.chunk):
            if dbg["kind"][e, i] in (oracle.APPENDED, oracle.SINK):
                founders[int(dbg["assign"][e, i])] = e * cfg.chunk + i
    assert sorted(founders) == list(range(st.n))
    for j, tok in founders.items():
        assert st.rho[j] == pytest.approx(np.linalg.norm(v[tok]), rel=1e-15)
    # the attention key view is zero on the rotary dims (Core mechanism 4)
    assert (kv[:, :cfg.rope_dims] == 0).all()


@pytest.mark.parametrize("sched,M", [(0, 24), (1, 64), (1, 200)])
def test_slots_founded_once_in_order_before_their_merges(sched, M):
    """Every slot is founded exactly once (a sink or an appended token), the
    founders of an event take the next slot numbers (new slots are appended
    after the existing ones: KVM summary, Core mechanism 3), and no token
    merges into a slot in an event before the one that founds it (a merge
    joins an existing slot: Core mechanism 2).  The replay of a slot's history
    (founder first, then its merged tokens in order) relies on this."""
    cfg, _, (_, st, dbg) = _random_run(sched=sched, M=M)
    A, K = dbg["assign"], dbg["kind"]
    founded_at = {}
    n = 0
    for e in range(A.shape[0]):
        new = sorted(int(A[e, i]) for i in range(cfg.chunk) if K[e, i] in (oracle.APPENDED, oracle.SINK))
        assert new == list(range(n, n + len(new))), f"event {e}: founders {new} after {n} slots"
        for j in new:
            founded_at[j] = e
        n += len(new)
        for i in range(cfg.chunk):
            if K[e, i] == oracle.MERGED:
                j = int(A[e, i])
                assert j in founded_at and founded_at[j] <= e, f"event {e}: token {i} merges into slot {j} before it exists"
    assert n == st.n


@pytest.mark.parametrize("sched,M,coef,expo", [(0, 24, 2.0, 0.5), (1, 64, 2.0, 0.5),
                                                (1, 128, 1.0, 0.75), (1, 80, 8.0, 0.25),
                                                (1, 200, 0.3, 1.0)])
def test_counts_sums_and_growth(sched, M, coef, expo):
    """Counts sum to the number of overflowed tokens; the slot count follows
    the schedule: after each fold n = min(cap(t), n_before + candidates) and
    never exceeds cap(t); sums equal the gate-weighted sum of their members
    (KVM summary, Core mechanisms 2 and 3; lay part 'smart merge').  Power-law
    growth with other exponents and coefficients than the sqrt schedule
    (Core mechanism 3 names power-law growth in general)."""
    cfg, (q, k, v, g), (_, st, dbg) = _random_run(sched=sched, M=M, coef=coef, expo=expo)
    E = dbg["assign"].shape[0]
    C, S = cfg.chunk, cfg.n_sinks
    assert st.t == E * C
    assert int(st.count[:st.n].sum()) == st.t
    n = 0
    for e in range(E):
        kinds = dbg["kind"][e]
        n_sinks_here = int((kinds == oracle.SINK).sum())
        ncand = C - n_sinks_here
        n0 = n + n_sinks_here
        cap = oracle.capacity(cfg, (e + 1) * C)
        n_new = n0 + int((kinds == oracle.APPENDED).sum())
        assert n_new == min(max(cap, n0), n0 + ncand)
        assert n_new <= max(cap, S)
        n = n_new
    assert n == st.n
    members_k = np.zeros((cfg.max_slots, cfg.head_dim))
    members_v = np.zeros_like(members_k)
    cnt = np.zeros(cfg.max_slots, dtype=np.int64)
    for e in range(E):
        for i in range(C):
            tok = e * C + i
            j = dbg["assign"][e, i]
            members_k[j] += g[tok] * k[tok]
            members_v[j] += g[tok] * v[tok]
            cnt[j] += 1
    np.testing.assert_array_equal(cnt, st.count)
    np.testing.assert_allclose(st.sum_k, members_k, atol=1e-12)
    np.testing.assert_allclose(st.sum_v, members_v, atol=1e-12)


@pytest.mark.parametrize("coef,expo", [(4.0, 0.5), (1.0, 0.75), (8.0, 0.25), (0.3, 1.0), (2.5, 0.6)])
def test_power_law_capacity_closed_form(coef, expo):
    """cap(t) = S + ceil(coef * t^expo) for t > 0 and S at t = 0 (power-law
    growth, KVM summary Core mechanism 3), checked against exact rational
    arithmetic where t^expo is rational, else against math.pow."""
    import fractions
    import math
    S = 16
    cfg = oracle.OracleConfig(n_sinks=S, sched=1, max_slots=10**6, coef=coef, expo=expo)
    assert oracle.capacity(cfg, 0) == S
    for t in (1, 2, 3, 16, 100, 127, 128, 1000, 7552, 64256):
        want = S + math.ceil(coef * math.pow(t, expo))
        if expo == 1.0:
            want = S + math.ceil(fractions.Fraction(coef) * t)
        assert oracle.capacity(cfg, t) == want, (t, oracle.capacity(cfg, t), want)
    # monotone in t
    caps = [oracle.capacity(cfg, t) for t in range(0, 3000, 7)]
    assert all(b >= a for a, b in zip(caps, caps[1:]))


@pytest.mark.parametrize("sched,M", [(0, 24), (1, 64)])
def test_no_value_norm_ablation_reads_member_means(sched, M):
    """Ablation of the value-length normalisation (KVM summary, Experimental
    results, ablation studies): the fold decisions and sums are unchanged, the
    read value becomes sum_v / count (the gate-weighted member mean), the read
    key is unchanged, and the outputs differ from the normalised read."""
    cfg, (q, k, v, g), (out, st, dbg) = _random_run(sched=sched, M=M)
    cfg_a = oracle.OracleConfig(**{**cfg.__dict__, "no_value_norm": 1})
    out_a, st_a, dbg_a = _run(cfg_a, q, k, v, g)
    np.testing.assert_array_equal(dbg_a["assign"], dbg["assign"])
    np.testing.assert_array_equal(dbg_a["kind"], dbg["kind"])
    np.testing.assert_array_equal(st_a.count, st.count)
    np.testing.assert_array_equal(st_a.sum_v, st.sum_v)
    kv, vv = oracle.state_view(cfg, st)
    kv_a, vv_a = oracle.state_view(cfg_a, st_a)
    np.testing.assert_array_equal(kv_a, kv)
    n = st.n
    np.testing.assert_allclose(vv_a, st.sum_v[:n] / st.count[:n, None], rtol=0, atol=1e-15)
    # members of each slot, gate-weighted, averaged over the count
    mem = np.zeros((M, cfg.head_dim))
    for e in range(dbg["assign"].shape[0]):
        for i in range(cfg.chunk):
            mem[dbg["assign"][e, i]] += g[e * cfg.chunk + i] * v[e * cfg.chunk + i]
    np.testing.assert_allclose(vv_a, mem[:n] / st.count[:n, None], atol=1e-12)
    assert np.abs(out_a - out).max() > 1e-3


def test_workload_slot_literals_match_schedule():
    """The sqrt workloads' max_slots literals equal the schedule's capacity
    after their last fold (16 + ceil(4 sqrt(t)))."""
    for w in (wl.SQRT_8K, wl.LONG_64K):
        cfg = oracle.OracleConfig(chunk=w.chunk, window=w.window, n_sinks=w.n_sinks,
                                  sched=1, max_slots=10**6, coef=w.coef, expo=w.expo)
        assert oracle.capacity(cfg, oracle.n_events(cfg, w.N) * w.chunk) == w.max_slots
    assert wl.SQRT_8K.max_slots == 364 and wl.LONG_64K.max_slots == 1030


def test_sinks_protected():
    """Sink rows (the first S overflowed tokens) are never merged into: their
    counts stay 1 and their value view is exactly their token's value (KVM
    summary, Core mechanism 5)."""
    cfg, (q, k, v, g), (_, st, dbg) = _random_run(sched=0, M=24, S=4)
    S = cfg.n_sinks
    merged_targets = dbg["assign"][dbg["kind"] == oracle.MERGED]
    assert (merged_targets >= S).all()
    assert (st.count[:S] == 1).all()
    _, vv = oracle.state_view(cfg, st)
    np.testing.assert_allclose(vv[:S], v[:S], atol=1e-12)


@pytest.mark.parametrize("alpha,beta", [(3.7, 1.0), (0.25, 1.0), (1.0, 0.3), (2.0, 5.0)])
def test_assignments_invariant_to_positive_rescaling(alpha, beta):
    """Cosine against LayerNorm'd means only sees directions (centred), so
    assignments do not change when every key is scaled by alpha > 0 or every
    gate by beta > 0."""
    cfg, (q, k, v, g), (_, st, dbg) = _random_run(sched=1, M=64)
    _, st2, dbg2 = _run(cfg, q, alpha * k, v, beta * g)
    np.testing.assert_array_equal(dbg["assign"], dbg2["assign"])
    np.testing.assert_array_equal(dbg["kind"], dbg2["kind"])


# ------------------------------------------------------------- hand example

def test_hand_worked_fold():
    """Hand-derived fold outcome (tests/golden/fold_hand_example.json)."""
    G = json.load(open(os.path.join(GOLDEN, "fold_hand_example.json")))
    c = G["config"]
    cfg = oracle.OracleConfig(head_dim=c["head_dim"], rope_dims=c["rope_dims"], chunk=c["chunk"],
                              window=c["window"], n_sinks=c["n_sinks"], sched=c["sched"],
                              max_slots=c["max_slots"], ln_eps=c["ln_eps"])
    k, v, g = np.array(G["k"], float), np.array(G["v"], float), np.array(G["g"], float)
    q = np.zeros_like(k)
    _, st, dbg = _run(cfg, q, k, v, g)
    E = G["expect"]
    assert st.n == E["n_slots"] and st.t == E["t"]
    np.testing.assert_array_equal(dbg["assign"], np.array(E["assign"]))
    np.testing.assert_array_equal(dbg["kind"], np.array(E["kind"]))
    np.testing.assert_array_equal(st.count[:st.n], E["count"])
    np.testing.assert_allclose(st.sum_k[:st.n], E["sum_k"], atol=0)
    np.testing.assert_allclose(st.sum_v[:st.n], E["sum_v"], atol=0)
    np.testing.assert_allclose(st.rho[:st.n], E["rho"], atol=0)
    kv, vv = oracle.state_view(cfg, st)
    np.testing.assert_allclose(vv[1], E["val_view_slot1"], atol=1e-12)
    np.testing.assert_allclose(kv[2], E["key_view_slot2"], atol=1e-8)


def test_hand_worked_merge_into_slot_appended_by_the_same_event():
    """Hand-derived fold (tests/golden/fold_post_append_example.json): a token
    merges into the slot its own chunk just appended; surprise scores, sums,
    counts, read radii, read views and every output row."""
    G = json.load(open(os.path.join(GOLDEN, "fold_post_append_example.json")))
    c = G["config"]
    cfg = oracle.OracleConfig(head_dim=c["head_dim"], rope_dims=c["rope_dims"], chunk=c["chunk"],
                              window=c["window"], n_sinks=c["n_sinks"], sched=c["sched"],
                              max_slots=c["max_slots"], ln_eps=c["ln_eps"])
    k, v, g = np.array(G["k"], float), np.array(G["v"], float), np.array(G["g"], float)
    out, st, dbg = _run(cfg, np.zeros_like(k), k, v, g)
    E = G["expect"]
    assert st.n == E["n_slots"] and st.t == E["t"]
    np.testing.assert_array_equal(dbg["assign"], np.array(E["assign"]))
    np.testing.assert_array_equal(dbg["kind"], np.array(E["kind"]))
    np.testing.assert_allclose(dbg["max_sim"][1], E["max_sim_event1"], rtol=0, atol=1e-12)
    assert np.isneginf(dbg["max_sim"][0]).all()
    np.testing.assert_array_equal(st.count[:st.n], E["count"])
    np.testing.assert_allclose(st.sum_k[:st.n], E["sum_k"], atol=0)
    np.testing.assert_allclose(st.sum_v[:st.n], E["sum_v"], atol=0)
    np.testing.assert_allclose(st.rho[:st.n], E["rho"], atol=0)
    kv, vv = oracle.state_view(cfg, st)
    np.testing.assert_allclose(vv[2], E["val_view_slot2"], atol=1e-12)
    np.testing.assert_allclose(kv[2], E["key_view_slot2"], atol=1e-12)
    np.testing.assert_allclose(out, np.array(E["out"]), rtol=0, atol=1e-12)
    # the alternative reading (merge targets before the appends) sends token 2 to
    # slot 0 (tie between slots 0 and 1 at -0.2887, lowest index)
    alt = oracle.OracleConfig(head_dim=c["head_dim"], rope_dims=c["rope_dims"], chunk=c["chunk"],
                              window=c["window"], n_sinks=c["n_sinks"], sched=c["sched"],
                              max_slots=c["max_slots"], ln_eps=c["ln_eps"], merge_pre_append=1)
    _, _, dbg_alt = _run(alt, np.zeros_like(k), k, v, g)
    assert dbg_alt["assign"][1].tolist() == [0, 2]
    # the no-value-norm ablation reads the member mean: slot 2 = (0,0,1,6)/2, slots 0
    # and 1 = their single members' gate-weighted values; decisions unchanged
    abl = oracle.OracleConfig(head_dim=c["head_dim"], rope_dims=c["rope_dims"], chunk=c["chunk"],
                              window=c["window"], n_sinks=c["n_sinks"], sched=c["sched"],
                              max_slots=c["max_slots"], ln_eps=c["ln_eps"], no_value_norm=1)
    out_a, st_a, dbg_a = _run(abl, np.zeros_like(k), k, v, g)
    np.testing.assert_array_equal(dbg_a["assign"], np.array(E["assign"]))
    np.testing.assert_allclose(oracle.state_view(abl, st_a)[1][2], [0, 0, 0.5, 3.0], atol=1e-15)
    np.testing.assert_allclose(out_a[6], np.array([3, 3, 2.5, 4]) / 6, atol=1e-15)
    np.testing.assert_allclose(out_a[7], np.array([3, 4, 2.5, 5]) / 7, atol=1e-15)


def test_hand_worked_attention():
    """Hand-derived outputs of every position (tests/golden/attention_hand_example.json):
    window extent, fold timing, the state's read view and the single softmax."""
    G = json.load(open(os.path.join(GOLDEN, "attention_hand_example.json")))
    c = G["config"]
    cfg = oracle.OracleConfig(head_dim=c["head_dim"], rope_dims=c["rope_dims"], chunk=c["chunk"],
                              window=c["window"], n_sinks=c["n_sinks"], sched=c["sched"],
                              max_slots=c["max_slots"], ln_eps=c["ln_eps"], rope_theta=c["rope_theta"])
    q, k, v, g = (np.array(G[x], float) for x in ("q", "k", "v", "g"))
    out, _, _ = _run(cfg, q, k, v, g)
    np.testing.assert_allclose(out, np.array(G["expect_out"]), rtol=0, atol=1e-12)


def test_ties_go_to_lowest_index_and_lowest_position():
    """Surprise ties append the lower positions; argmax ties go to the lowest
    slot index."""
    d = 8
    cfg = oracle.OracleConfig(head_dim=d, rope_dims=4, chunk=4, window=4, n_sinks=1, max_slots=3)
    st = oracle.OracleState(cfg)
    rng = np.random.default_rng(0)
    base = rng.standard_normal(d)
    k = np.stack([rng.standard_normal(d), base, base, base + 0.01 * rng.standard_normal(d)])
    v = rng.standard_normal((4, d))
    g = np.ones(4)
    r = oracle.fold_event(cfg, st, 0, k, v, g)
    # token 0 founds the sink; tokens 1..3 all have m = -inf (no mergeable slot):
    # a = min(3 - 1, 3) = 2, so the lower positions 1 and 2 are appended
    assert list(r["kind"]) == [oracle.SINK, oracle.APPENDED, oracle.APPENDED, oracle.MERGED]
    # slots 1 and 2 have identical keys; token 3 ties between them -> slot 1
    assert list(r["assign"]) == [0, 1, 2, 1]
    assert r["gap"][3] == 0.0


def test_most_surprising_token_is_appended():
    """Tokens that copy existing slot keys score high; the one orthogonal
    token has the lowest max-similarity and is the one appended (KVM summary,
    Core mechanism 3)."""
    d = 8
    cfg = oracle.OracleConfig(head_dim=d, rope_dims=4, chunk=4, window=4, n_sinks=0, max_slots=5)
    st = oracle.OracleState(cfg)
    rng = np.random.default_rng(1)
    keys = rng.standard_normal((4, d))
    r0 = oracle.fold_event(cfg, st, 0, keys, rng.standard_normal((4, d)), np.ones(4))
    assert st.n == 4 and list(r0["kind"]) == [oracle.APPENDED] * 4
    odd = np.zeros(d); odd[0], odd[1] = 1.0, -1.0       # centred direction orthogonal-ish
    chunk = np.stack([keys[2], odd, keys[0], keys[3]])
    r1 = oracle.fold_event(cfg, st, 4, chunk, rng.standard_normal((4, d)), np.ones(4))
    mins = np.argmin(r1["max_sim"])
    assert mins == 1 and list(r1["kind"]) == [0, 1, 0, 0]
    assert list(r1["assign"]) == [2, 4, 0, 3]
    # a copy of slot key x scores cos(x, x - mean(x)) = ||x - mean(x)|| / ||x||
    x = keys[2]
    assert r1["max_sim"][0] == pytest.approx(np.linalg.norm(x - x.mean()) / np.linalg.norm(x),
                                             abs=1e-12)


# ---------------------------------------------------------- brute force

TINY = [
    dict(N=96, C=8, W=16, S=2, r=4, d=8, sched=0, M=12),
    dict(N=101, C=8, W=8, S=3, r=8, d=16, sched=1, M=40),
    dict(N=64, C=4, W=8, S=0, r=4, d=8, sched=0, M=6),
    dict(N=130, C=16, W=32, S=16, r=8, d=16, sched=1, M=64),
    dict(N=7, C=4, W=4, S=1, r=2, d=4, sched=0, M=3),
    dict(N=120, C=8, W=16, S=2, r=4, d=8, sched=1, M=60, coef=1.0, expo=0.75),
    dict(N=200, C=8, W=24, S=4, r=8, d=16, sched=0, M=8),
]


@pytest.mark.parametrize("case", TINY)
@pytest.mark.parametrize("seed", [0, 1])
def test_oracle_matches_bruteforce(case, seed):
    """The C oracle agrees with the independent numpy/torch restatement:
    assignments exactly, outputs and state to rounding."""
    c = dict(case)
    rng = np.random.default_rng(100 + seed)
    q, k, v, g = _inputs(seed + 10, c["N"], c["d"])
    for t in range(1, c["N"]):
        if rng.random() < 0.25:
            k[t] = k[rng.integers(0, t)] + 0.2 * rng.standard_normal(c["d"])
    coef, expo = c.get("coef", 2.0), c.get("expo", 0.5)
    cfg = oracle.OracleConfig(head_dim=c["d"], rope_dims=c["r"], chunk=c["C"], window=c["W"],
                              n_sinks=c["S"], sched=c["sched"], max_slots=c["M"], coef=coef,
                              expo=expo)
    out, st, dbg = _run(cfg, q, k, v, g)
    bout, bst, bev = bf_prefill(q, k, v, g, C=c["C"], W=c["W"], S=c["S"], r=c["r"],
                                sched=c["sched"], M=c["M"], coef=coef, expo=expo)
    assert len(bev) == dbg["assign"].shape[0]
    for e, (a, kd) in enumerate(bev):
        np.testing.assert_array_equal(dbg["assign"][e], a)
        np.testing.assert_array_equal(dbg["kind"][e], kd)
    np.testing.assert_allclose(out, bout, rtol=0, atol=1e-10)
    assert st.n == bst.n and st.t == bst.t
    if bst.n:
        np.testing.assert_allclose(st.sum_k[:st.n], np.array(bst.sk), atol=1e-12)
        np.testing.assert_allclose(st.sum_v[:st.n], np.array(bst.sv), atol=1e-12)
        np.testing.assert_array_equal(st.count[:st.n], bst.cnt)
        np.testing.assert_allclose(st.rho[:st.n], bst.rho, rtol=1e-14)


VARIANTS = [
    dict(merge_pre_append=1),
    dict(cos_nope_only=1),
    dict(no_value_norm=1),
    dict(merge_pre_append=1, cos_nope_only=1, no_value_norm=1),
]


@pytest.mark.parametrize("case", TINY)
@pytest.mark.parametrize("var", VARIANTS)
def test_alternative_readings_match_bruteforce(case, var):
    """The oracle's alternative readings (merge targets before the chunk's
    appends, cosine over the non-rotary dims only) and the no-value-norm
    ablation agree with the brute force.  Where the pre-append reading leaves a
    token without any slot to merge into, both sides refuse the input."""
    c = dict(case)
    rng = np.random.default_rng(7)
    q, k, v, g = _inputs(21, c["N"], c["d"])
    for t in range(1, c["N"]):
        if rng.random() < 0.25:
            k[t] = k[rng.integers(0, t)] + 0.2 * rng.standard_normal(c["d"])
    coef, expo = c.get("coef", 2.0), c.get("expo", 0.5)
    cfg = oracle.OracleConfig(head_dim=c["d"], rope_dims=c["r"], chunk=c["C"], window=c["W"],
                              n_sinks=c["S"], sched=c["sched"], max_slots=c["M"], coef=coef,
                              expo=expo, **var)
    kw = dict(C=c["C"], W=c["W"], S=c["S"], r=c["r"], sched=c["sched"], M=c["M"], coef=coef,
              expo=expo, pre_append=bool(var.get("merge_pre_append")),
              nope_only=bool(var.get("cos_nope_only")), no_vnorm=bool(var.get("no_value_norm")))
    try:
        bout, bst, bev = bf_prefill(q, k, v, g, **kw)
    except NoMergeTarget:
        with pytest.raises(oracle.OracleError):
            _run(cfg, q, k, v, g)
        return
    out, st, dbg = _run(cfg, q, k, v, g)
    assert len(bev) == dbg["assign"].shape[0]
    for e, (a, kd) in enumerate(bev):
        np.testing.assert_array_equal(dbg["assign"][e], a)
        np.testing.assert_array_equal(dbg["kind"][e], kd)
    np.testing.assert_allclose(out, bout, rtol=0, atol=1e-10)
    assert st.n == bst.n and st.t == bst.t
    if bst.n:
        np.testing.assert_array_equal(st.count[:st.n], bst.cnt)
        np.testing.assert_allclose(st.sum_k[:st.n], np.array(bst.sk), atol=1e-12)


def test_alternative_readings_change_decisions():
    """Each alternative reading decides differently from the main one on some
    input, so the pins above would notice a flag that the oracle ignores."""
    # sqrt growth: every event appends a few slots and merges the rest
    c = dict(N=400, C=8, W=8, S=2, r=8, d=16, sched=1, M=200)
    q, k, v, g = _inputs(5, c["N"], c["d"])
    base = dict(head_dim=c["d"], rope_dims=c["r"], chunk=c["C"], window=c["W"], n_sinks=c["S"],
                sched=c["sched"], max_slots=c["M"])
    _, _, d0 = _run(oracle.OracleConfig(**base), q, k, v, g)
    for var in (dict(merge_pre_append=1), dict(cos_nope_only=1)):
        _, _, d1 = _run(oracle.OracleConfig(**base, **var), q, k, v, g)
        assert (d1["assign"] != d0["assign"]).any(), var
    o0, _, _ = _run(oracle.OracleConfig(**base), q, k, v, g)
    o1, _, _ = _run(oracle.OracleConfig(**base, no_value_norm=1), q, k, v, g)
    assert np.abs(o1 - o0).max() > 1e-3


def test_empty_prefill():
    cfg = oracle.OracleConfig(head_dim=8, rope_dims=4, chunk=4, window=4, n_sinks=1, max_slots=4)
    out, st, dbg = oracle.prefill(cfg, np.zeros((1, 0, 8)), np.zeros((1, 0, 8)),
                                  np.zeros((1, 0, 8)), np.zeros((1, 0)), threads=1)
    assert out.shape == (1, 0, 8) and st[0].n == 0 and st[0].t == 0


def test_capacity_error():
    """A fixed capacity above max_slots cannot happen; a power-law schedule
    that outgrows max_slots is reported as an error, not clamped."""
    cfg = oracle.OracleConfig(head_dim=8, rope_dims=4, chunk=4, window=4, n_sinks=1, sched=1,
                              max_slots=4, coef=4.0)
    q, k, v, g = _inputs(0, 64, 8)
    with pytest.raises(oracle.OracleError):
        _run(cfg, q, k, v, g)


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("N0,steps", [(40, 30), (64, 20), (3, 50)])
def test_decode_equals_prefill_rows(N0, steps):
    """Decoding token by token from a prefill of N0 tokens gives the same
    outputs as the last rows of one prefill of N0 + steps tokens (chunked
    recurrence: KVM summary, Core mechanism 1; KVM abstract)."""
    d, r, C, W = 8, 4, 4, 8
    cfg = oracle.OracleConfig(head_dim=d, rope_dims=r, chunk=C, window=W, n_sinks=2, sched=1,
                              max_slots=64, coef=2.0)
    N = N0 + steps
    q, k, v, g = _inputs(7, N, d)
    full, _, _ = _run(cfg, q, k, v, g)
    _, st, _ = _run(cfg, q[:N0], k[:N0], v[:N0], g[:N0])
    F = oracle.n_events(cfg, N0) * C
    dec = oracle.OracleDecoder(cfg, st, N0, k[F:N0], v[F:N0], g[F:N0])
    outs = [dec.step(q[p], k[p], v[p], g[p]) for p in range(N0, N)]
    np.testing.assert_allclose(np.stack(outs), full[N0:], rtol=0, atol=1e-12)


# ------------------------------------------------------------ whole layer

def test_bf16_round_ties_to_even_and_matches_torch():
    """The oracle's bf16 rounding (8 significant bits, ties to even) against hand
    values and torch's float32 -> bfloat16 conversion."""
    import torch
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 3 * 2 ** -9, -3.0, 0.0, 2.0 ** -20 * 1.5])
    want = np.array([1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -3.0, 0.0, 2.0 ** -20 * 1.5])
    np.testing.assert_array_equal(oracle.bf16_round(x), want)
    r = np.random.default_rng(3).standard_normal(20000).astype(np.float32) * 7
    ref = torch.from_numpy(r).bfloat16().double().numpy()
    np.testing.assert_array_equal(oracle.bf16_round(r.astype(np.float64)), ref)


def test_layer_projections_index_convention_bruteforce():
    """Projection layouts by explicit loops: q/k/v of head h, dim x are rows
    h*64+x of the q, k, v blocks of w_in; the gate of head h is the sigmoid of
    row 3*H*64+h; y[n, j] sums o[h, n, x] * w_out[j, h*64+x] (KVM summary,
    Methodology: per-head projections of the layer input, heads projected back)."""
    rng = np.random.default_rng(11)
    B, N, H, d, dm = 2, 3, 2, 64, 5
    x = rng.standard_normal((B, N, dm))
    w_in = rng.standard_normal((3 * H * d + H, dm))
    w_out = rng.standard_normal((dm, H * d))
    q, k, v, g = oracle.layer_project_in(x, w_in, H, d)
    for b in range(B):
        for n in range(N):
            for h in range(H):
                for part, arr in ((0, q), (1, k), (2, v)):
                    for xx in (0, 17, 63):
                        row = part * H * d + h * d + xx
                        want = sum(x[b, n, i] * w_in[row, i] for i in range(dm))
                        assert arr[b, h, n, xx] == pytest.approx(want, abs=1e-12)
                logit = sum(x[b, n, i] * w_in[3 * H * d + h, i] for i in range(dm))
                assert g[b, h, n] == pytest.approx(1.0 / (1.0 + np.exp(-logit)), abs=1e-14)
    o = rng.standard_normal((B, H, N, d))
    y = oracle.layer_project_out(o, w_out)
    for b in range(B):
        for n in range(N):
            for j in range(dm):
                want = sum(o[b, h, n, xx] * w_out[j, h * d + xx] for h in range(H) for xx in range(d))
                assert y[b, n, j] == pytest.approx(want, abs=1e-10)


def test_layer_with_identity_projections_reduces_to_the_attention():
    """With w_in = [I; I; I; 0] (q = k = v = the head slices of x, gate logit 0 so
    the gate is 1/2) and w_out = I, the whole layer is the pinned KVM attention
    on those inputs, heads laid out back along the features."""
    H, d, N = 2, 64, 700
    dm = H * d
    cfg = oracle.OracleConfig(head_dim=d, rope_dims=32, chunk=64, window=128, n_sinks=4,
                              max_slots=24)
    rng = np.random.default_rng(5)
    x = oracle.bf16_round(rng.standard_normal((1, N, dm)))
    eye = np.eye(dm)
    w_in = np.concatenate([eye, eye, eye, np.zeros((H, dm))])
    y, (q, k, v, gate, o), _ = oracle.layer_forward(cfg, x, w_in, eye, H)
    xh = x[0].reshape(N, H, d).transpose(1, 0, 2)
    np.testing.assert_array_equal(q[0], xh)
    np.testing.assert_array_equal(gate, 0.5)
    out, _, _ = oracle.prefill(cfg, xh, xh, xh, np.full((H, N), 0.5))
    np.testing.assert_allclose(y[0], out.transpose(1, 0, 2).reshape(N, dm), rtol=0, atol=1e-12)


@pytest.mark.parametrize("w,n_tokens", [
    (wl.TINY_FP32, None),
    (wl.FIXED_8K, 2048),
    (wl.SQRT_8K, 2048),
    (wl.LONG_64K, 3072),
], ids=lambda x: getattr(x, "name", str(x)))
def test_oracle_matches_bruteforce_on_the_workload_shapes(w, n_tokens):
    """The brute force and the C oracle on the workloads' own shapes and key
    structure (head dim 64, RoPE on 32 dims, their chunk, window, sinks and
    schedule; the large ones truncated to their first tokens, one head each):
    assignments exactly, outputs and sums to rounding."""
    N = w.N if n_tokens is None else n_tokens
    q, k, v, g = wl.prefill_inputs(w.with_(B=1, H=min(w.H, 2)))
    heads = range(q.shape[1]) if n_tokens is None else [0]
    cfg = oracle.OracleConfig(head_dim=w.d, rope_dims=w.rope_dims, chunk=w.chunk, window=w.window,
                              n_sinks=w.n_sinks, sched=w.sched, max_slots=w.max_slots,
                              coef=w.coef, expo=w.expo)
    for h in heads:
        qh, kh, vh = (x[0, h, :N].astype(np.float64) for x in (q, k, v))
        gh = g[0, h, :N].astype(np.float64)
        out, st, dbg = _run(cfg, qh, kh, vh, gh)
        bout, bst, bev = bf_prefill(qh, kh, vh, gh, C=w.chunk, W=w.window, S=w.n_sinks, r=w.rope_dims,
                                    sched=w.sched, M=w.max_slots, coef=w.coef, expo=w.expo)
        assert len(bev) == dbg["assign"].shape[0] > 0
        for e, (a, kd) in enumerate(bev):
            np.testing.assert_array_equal(dbg["assign"][e], a)
            np.testing.assert_array_equal(dbg["kind"][e], kd)
        np.testing.assert_allclose(out, bout, rtol=0, atol=1e-9)
        assert st.n == bst.n
        np.testing.assert_allclose(st.sum_k[:st.n], np.array(bst.sk), atol=1e-9)
        np.testing.assert_array_equal(st.count[:st.n], bst.cnt)


def test_oracle_decoder_matches_bruteforce_on_the_decode_sweep_shape():
    """Decode from an imported state (the decode sweep's shape: head dim 64, RoPE
    on 32 dims, W 512, C 128, 16 sinks, a full fixed state of 256 slots), over 130
    steps that cross two chunk boundaries: the oracle's decoder against a brute
    force built from the independent restatement (fold, read view, complex RoPE,
    torch softmax)."""
    from bruteforce import BFState, bf_fold, bf_view
    from compressed_kv_state_gb300.workloads import DecodeWorkload, decode_inputs
    dw = DecodeWorkload("dec_pin", B=1, H=1, n_slots=256, steps=130)
    state, (wk, wv, wg), (q, k, v, g) = decode_inputs(dw)
    d, r, C, W, S, n = dw.d, dw.rope_dims, dw.chunk, dw.window, dw.n_sinks, dw.n_slots
    cfg = oracle.OracleConfig(head_dim=d, rope_dims=r, chunk=C, window=W, n_sinks=S, sched=0,
                              max_slots=n)
    ost = oracle.OracleState(cfg)
    ost.n, ost.t = n, state["t"]
    ost.sum_k[:n] = state["sum_k"][0, 0]
    ost.sum_v[:n] = state["sum_v"][0, 0]
    ost.count[:n] = state["counts"][0, 0]
    ost.rho[:n] = state["rho"][0, 0]
    dec = oracle.OracleDecoder(cfg, ost, state["pos"], wk[0, 0], wv[0, 0], wg[0, 0])

    bst = BFState()
    bst.sk = [np.array(x, np.float64) for x in state["sum_k"][0, 0]]
    bst.sv = [np.array(x, np.float64) for x in state["sum_v"][0, 0]]
    bst.cnt = [int(x) for x in state["counts"][0, 0]]
    bst.rho = [float(x) for x in state["rho"][0, 0]]
    bst.t = state["t"]
    win_k = [np.array(x, np.float64) for x in wk[0, 0]]
    win_v = [np.array(x, np.float64) for x in wv[0, 0]]
    win_g = [float(x) for x in wg[0, 0]]
    pos = state["pos"]
    for s in range(dw.steps):
        p = pos + s
        c = p // C
        if p % C == 0 and c >= W // C + 1:
            first = (c - W // C - 1) * C
            bf_fold(bst, first, np.stack(win_k[:C]), np.stack(win_v[:C]), np.array(win_g[:C]),
                    S=S, sched=0, M=n, coef=4.0, expo=0.5, eps=1e-5, C=C, r=r)
            del win_k[:C], win_v[:C], win_g[:C]
        qs, ks, vs, gs = (np.array(x[s, 0, 0], np.float64) for x in (q, k, v, g))
        win_k.append(ks)
        win_v.append(vs)
        win_g.append(float(gs))
        kh, vh = bf_view(bst, r, 1e-5)
        w_first = p - len(win_k) + 1
        assert w_first == max(0, (c - W // C) * C)
        pos_w = np.arange(w_first, p + 1)
        kr = rope_complex(np.stack(win_k), pos_w, r, 1e4)
        qr = rope_complex(qs[None], np.array([p]), r, 1e4)[0]
        sc = np.concatenate([kh @ qs, kr @ qr]) / math.sqrt(d)
        wts = torch.softmax(torch.as_tensor(sc), 0).numpy()
        want = wts @ np.concatenate([vh, np.stack(win_v)])
        got = dec.step(q[s, 0, 0], k[s, 0, 0], v[s, 0, 0], g[s, 0, 0])
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-10, err_msg=f"step {s}")
    assert dec.st.n == len(bst.sk) == n
    np.testing.assert_array_equal(dec.st.count[:n], bst.cnt)
