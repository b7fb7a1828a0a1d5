"""Overlapped prefill (fold segments on one SM partition, the attention of
ready chunks on the other, the rest on every SM) against the sequential
prefill and the oracle.

The overlapped path runs the same kernels with the same per-tile arithmetic,
so its outputs and final state must equal the sequential prefill's bit for
bit; the sequential prefill with a debug record is checked against the oracle
elsewhere, and here the overlapped outputs of sampled heads are also compared
with the oracle directly (rows before the first event with an oracle near tie).
"""
import os

import numpy as np
import pytest

import oracle
from compressed_kv_state_gb300 import workloads as wl
from kvm_testlib import NEAR_TIE, gpu_prefill, make_layer, oracle_cfg, tol_of

pytestmark = pytest.mark.gpu

MID = wl.Workload("fixed_B2H3N4096_C128W512", B=2, H=3, N=4096, chunk=128, window=512,
                  n_sinks=16, max_slots=256, keys="repeat5")
RAGGED = wl.Workload("fixed_B1H4N3000_C128W256_ragged", B=1, H=4, N=3000, chunk=128, window=256,
                     n_sinks=16, max_slots=96, keys="repeat5")
# the streamed-state fold (more than 256 slots; chunks of 256 tokens) in the overlapped prefill
BIG = wl.Workload("big_fixed300_B1H2N6000_C128W256", B=1, H=2, N=6000, chunk=128, window=256,
                  n_sinks=16, max_slots=300, keys="repeat5")
BIG256 = wl.Workload("big_fixed600_C256_B2H1N9000_W512", B=2, H=1, N=9000, chunk=256, window=512,
                     n_sinks=16, max_slots=600, keys="repeat5")


# Under a CUDA injection library (a profiler or tracer) the library makes no SM
# partition and every prefill runs sequentially.
PROFILED = bool(os.environ.get("CUDA_INJECTION64_PATH"))


def _overlap_ran(used, want=None):
    if PROFILED:
        assert used == 0, "the overlap must stay off under an injection library"
        return
    assert used > 0, "overlapped prefill did not run (no SM partition?)"
    if want is not None:
        assert used == want


def _run(w, inputs, segs, debug=False):
    from compressed_kv_state_gb300 import kvm
    layer = make_layer(w)
    kvm.kvm_layer_set_overlap(layer.handle, segs)
    out, dbg, state = gpu_prefill(layer, w, *inputs, debug=debug)
    used = kvm.kvm_layer_get_overlap(layer.handle)
    layer.close()
    return out, dbg, state, used


def _same_state(a, b):
    for key in ("n_slots", "n_overflow", "pos"):
        assert a[key] == b[key], key
    for key in ("sum_k", "sum_v", "counts", "rho"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    # ring rows that hold a token (positions n_overflow .. pos-1); the others are
    # unspecified on export (whatever the workspace held)
    L = a["ring_g"].shape[-1]
    rows = np.arange(a["n_overflow"], a["pos"]) % L
    for key in ("ring_k", "ring_v", "ring_g"):
        np.testing.assert_array_equal(a[key][:, :, rows], b[key][:, :, rows], err_msg=key)


@pytest.mark.parametrize("w", [MID, RAGGED, wl.FIXED_8K, BIG, BIG256, wl.SQRT_8K, wl.LONG_64K],
                         ids=lambda w: w.name)
def test_overlapped_equals_sequential(w):
    inputs = wl.prefill_inputs(w)
    E = oracle.n_events(oracle_cfg(w), w.N)
    out_d, _, st_d, used_d = _run(w, inputs, 0, debug=True)
    out_s, _, st_s, used_s = _run(w, inputs, 0)
    assert used_d == 0 and used_s == 0
    # the debug record changes nothing
    np.testing.assert_array_equal(out_d, out_s)
    _same_state(st_d, st_s)
    for segs in (-1, 1, 3, 16):
        out_o, _, st_o, used = _run(w, inputs, segs)
        _overlap_ran(used, min(segs, E) if segs > 0 else None)
        np.testing.assert_array_equal(out_o, out_s, err_msg=f"segments={segs}")
        _same_state(st_o, st_s)


@pytest.mark.parametrize("w", [MID, wl.FIXED_8K, BIG256], ids=lambda w: w.name)
def test_overlapped_outputs_match_oracle(w):
    """Sampled heads of the overlapped prefill (the benchmark's launch
    configuration at full size) against the oracle."""
    inputs = wl.prefill_inputs(w)
    q, k, v, g = inputs
    out, _, _, used = _run(w, inputs, -1)
    _overlap_ran(used)
    hs = [(0, 0), (w.B - 1, w.H - 1)]
    ocfg = oracle_cfg(w)
    oout, _, odbg = oracle.prefill(ocfg, np.stack([q[b, h] for b, h in hs]),
                                   np.stack([k[b, h] for b, h in hs]),
                                   np.stack([v[b, h] for b, h in hs]),
                                   np.stack([g[b, h] for b, h in hs]))
    Wc = w.window // w.chunk
    tol = tol_of(w)
    for i, (b, h) in enumerate(hs):
        # rows whose state comes only from events without an oracle near tie
        near = [e for e in range(odbg["gap"].shape[1])
                if odbg["sel_margin"][i, e] < NEAR_TIE or
                (np.asarray(odbg["kind"][i, e]) == oracle.MERGED).any() and
                odbg["gap"][i, e][np.asarray(odbg["kind"][i, e]) == oracle.MERGED].min() < NEAR_TIE]
        rows = w.N if not near else min(w.N, (near[0] + Wc + 1) * w.chunk)
        assert rows >= min(w.N, (Wc + 2) * w.chunk)
        err = np.abs(out[b, h, :rows] - oout[i, :rows]).max()
        assert err <= tol, f"(b={b}, h={h}) max-abs error {err} over {rows} rows"
