"""Shared helpers of the GPU parity tests: build a layer for a workload, run
the CUDA path through the C ABI, run the oracle on the same inputs, and
compare fold events with the near-tie accounting.

Tolerances: slot assignments, kinds and counts are compared exactly; a token
whose oracle top-2 cosine gap is below NEAR_TIE (or an event whose surprise
selection margin is below it) is exempt, counted and reported.  Outputs and
state sums: max-abs error TOL_BF16 for bf16 inputs, TOL_FP32 for fp32.
"""
from __future__ import annotations

import numpy as np

import oracle

NEAR_TIE = 1e-5
TOL_BF16 = 2e-2
TOL_FP32 = 1e-4


def oracle_cfg(w) -> oracle.OracleConfig:
    return oracle.OracleConfig(head_dim=w.d, rope_dims=w.rope_dims, rope_theta=w.rope_theta,
                               chunk=w.chunk, window=w.window, n_sinks=w.n_sinks, sched=w.sched,
                               max_slots=w.max_slots, coef=w.coef, expo=w.expo, ln_eps=w.ln_eps,
                               no_value_norm=int(w.flags & 1))


def tol_of(w) -> float:
    return TOL_FP32 if w.dtype == "fp32" else TOL_BF16


def make_layer(w, max_tokens=None):
    from compressed_kv_state_gb300 import kvm
    cfg = kvm.make_config(batch=w.B, heads=w.H, head_dim=w.d, rope_dims=w.rope_dims,
                          rope_theta=w.rope_theta, chunk=w.chunk, window=w.window,
                          n_sinks=w.n_sinks, sched=w.sched, max_slots=w.max_slots, coef=w.coef,
                          expo=w.expo, ln_eps=w.ln_eps,
                          dtype=kvm.KVM_BF16 if w.dtype == "bf16" else kvm.KVM_FP32,
                          max_tokens=max_tokens or max(w.N, 1), flags=w.flags)
    return kvm.KvmLayer(cfg)


def to_dev(a, w):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if w.dtype == "bf16" and a.dtype == np.float32 and a.ndim == 4:
        t = t.to(torch.bfloat16)
    return t.cuda()


def gpu_prefill(layer, w, q, k, v, g, n_tokens=None, debug=True):
    """Run kvm_prefill on the first n_tokens tokens; returns (out, dbg, state) as numpy."""
    import torch
    from compressed_kv_state_gb300 import kvm
    N = w.N if n_tokens is None else n_tokens
    sl = (slice(None), slice(None), slice(0, N))
    dq, dk, dv = (to_dev(np.ascontiguousarray(x[sl]), w) for x in (q, k, v))
    dg = torch.from_numpy(np.ascontiguousarray(g[sl])).cuda()
    E = oracle.n_events(oracle_cfg(w), N)
    dbg = None
    bufs = {}
    if debug and E > 0:
        shp = (w.B, w.H, E, w.chunk)
        bufs = dict(assign=torch.full(shp, -7, dtype=torch.int32, device="cuda"),
                    kind=torch.full(shp, -7, dtype=torch.int32, device="cuda"),
                    max_sim=torch.zeros(shp, device="cuda"), gap=torch.zeros(shp, device="cuda"))
        dbg = kvm.kvm_debug(bufs["assign"].data_ptr(), bufs["kind"].data_ptr(),
                            bufs["max_sim"].data_ptr(), bufs["gap"].data_ptr(), E)
    out = layer.prefill(dq, dk, dv, dg, dbg=dbg)
    st = layer.export_state()
    layer.sync()
    torch.cuda.synchronize()
    res_dbg = {key: val.cpu().numpy() for key, val in bufs.items()}
    state = {key: (val.float().cpu().numpy() if hasattr(val, "cpu") else val)
             for key, val in st.items()}
    return out.float().cpu().numpy(), res_dbg, state


def state_to_oracle(w, state, b, h) -> oracle.OracleState:
    """The GPU's exported state of one (b, h) as an oracle state (fp32 -> fp64 exactly)."""
    s = oracle.OracleState(oracle_cfg(w))
    n = int(state["n_slots"])
    s.n, s.t = n, int(state["n_overflow"])
    s.sum_k[:n] = state["sum_k"][b, h, :n]
    s.sum_v[:n] = state["sum_v"][b, h, :n]
    s.count[:n] = state["counts"][b, h, :n].astype(np.int64)
    s.rho[:n] = state["rho"][b, h, :n]
    return s


def compare_chain(gpu_dbg, ora_dbg, head_index, b, h):
    """Compare one head's fold events, GPU vs oracle, from event 0.

    Returns (first_divergent_event or None, n_exempt).  Raises AssertionError
    on a mismatch that is not a near tie.
    """
    ga, gk = gpu_dbg["assign"][b, h], gpu_dbg["kind"][b, h]
    oa, ok = ora_dbg["assign"][head_index], ora_dbg["kind"][head_index]
    og, osel = ora_dbg["gap"][head_index], ora_dbg["sel_margin"][head_index]
    E = oa.shape[0]
    for e in range(E):
        bad = (ga[e] != oa[e]) | (gk[e] != ok[e])
        if not bad.any():
            continue
        toks = np.nonzero(bad)[0]
        exempt = osel[e] < NEAR_TIE or all(ok[e, t] == oracle.MERGED and og[e, t] < NEAR_TIE
                                           for t in toks)
        assert exempt, (f"(b={b}, h={h}) event {e}: tokens {toks.tolist()} differ: gpu assign "
                        f"{ga[e, toks].tolist()} kind {gk[e, toks].tolist()}, oracle assign "
                        f"{oa[e, toks].tolist()} kind {ok[e, toks].tolist()} gap "
                        f"{og[e, toks].tolist()} sel_margin {osel[e]}")
        return e, len(toks)
    return None, 0


def compare_event_teacher_forced(w, st_before, first_pos, k, v, g, gpu_assign, gpu_kind):
    """Run the oracle's fold on the GPU's own state; compare one event.

    Returns (oracle result dict, n_exempt)."""
    ocfg = oracle_cfg(w)
    r = oracle.fold_event(ocfg, st_before, first_pos, k, v, g)
    bad = (gpu_assign != r["assign"]) | (gpu_kind != r["kind"])
    n_ex = 0
    if bad.any():
        toks = np.nonzero(bad)[0]
        exempt = r["sel_margin"] < NEAR_TIE or all(
            r["kind"][t] == oracle.MERGED and r["gap"][t] < NEAR_TIE for t in toks)
        assert exempt, (f"event at {first_pos}: tokens {toks.tolist()} gpu {gpu_assign[toks].tolist()}"
                        f"/{gpu_kind[toks].tolist()} oracle {r['assign'][toks].tolist()}/"
                        f"{r['kind'][toks].tolist()} gaps {r['gap'][toks].tolist()}")
        n_ex = len(toks)
    return r, n_ex


def chain_with_resync(w, layer, inputs, dbg, heads, max_resyncs=None):
    """Compare every fold event of the sampled heads' chains, GPU against the
    oracle, event by event.  The oracle folds from its own state; where the two
    disagree (which must be a near tie, else AssertionError), the oracle's state
    is replaced by the GPU's exported state after that event, so a near-tie flip
    cannot cascade and every later event is still checked exactly.

    Returns {(b, h): dict(first_divergent_event, exempt_events, exempt_tokens)}.
    """
    q, k, v, g = inputs
    ocfg = oracle_cfg(w)
    C, Wc = w.chunk, w.window // w.chunk
    E = oracle.n_events(ocfg, w.N)
    if max_resyncs is None:
        max_resyncs = max(2, E // 10)
    gpu_states = {}

    def gpu_state_after(e):
        if e not in gpu_states:
            _, _, st = gpu_prefill(layer, w, q, k, v, g, n_tokens=min(w.N, (e + Wc + 2) * C),
                                   debug=False)
            gpu_states[e] = st
        return gpu_states[e]

    res = {}
    for b, h in heads:
        st = oracle.OracleState(ocfg)
        first, ex_events, ex_tokens = None, 0, 0
        for e in range(E):
            sl = slice(e * C, (e + 1) * C)
            r = oracle.fold_event(ocfg, st, e * C, k[b, h, sl], v[b, h, sl], g[b, h, sl])
            ga, gk = dbg["assign"][b, h, e], dbg["kind"][b, h, e]
            bad = (ga != r["assign"]) | (gk != r["kind"])
            if not bad.any():
                continue
            toks = np.nonzero(bad)[0]
            exempt = r["sel_margin"] < NEAR_TIE or all(
                r["kind"][t] == oracle.MERGED and r["gap"][t] < NEAR_TIE for t in toks)
            assert exempt, (f"(b={b}, h={h}) event {e}: tokens {toks.tolist()} gpu "
                            f"{ga[toks].tolist()}/{gk[toks].tolist()} oracle "
                            f"{r['assign'][toks].tolist()}/{r['kind'][toks].tolist()} gaps "
                            f"{r['gap'][toks].tolist()} sel_margin {r['sel_margin']}")
            first = e if first is None else first
            ex_events += 1
            ex_tokens += len(toks)
            assert ex_events <= max_resyncs, f"(b={b}, h={h}): more than {max_resyncs} near-tie events"
            st = state_to_oracle(w, gpu_state_after(e), b, h)
        res[(b, h)] = dict(first_divergent_event=first, exempt_events=ex_events,
                           exempt_tokens=ex_tokens)
    return res


# ------------------------------------------------------------ near-tie report
#
# The parity tests record, per workload, how many tokens and events were exempt
# as near ties and where the first divergence fell; the session writes them to
# tests/reports/near_ties.json (the GPU run regenerates it).

REPORT = {}


def report_near_ties(workload: str, entry: dict):
    REPORT.setdefault(workload, []).append(entry)
