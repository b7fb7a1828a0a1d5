"""kvm_prefill_noalloc: the prefill entry point for callers that may not
allocate device memory (for instance a plugin inside a host framework that
owns all device memory through its own pool, or a latency-critical loop that
cannot take an allocation's device synchronisation).  Its scratch is the
library's static device array instead of a caller workspace; its output must
match the ordinary kvm_prefill on the same inputs.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

from kvm_testlib import TOL_BF16, TOL_FP32

pytestmark = pytest.mark.gpu


def _both(w):
    import torch
    from compressed_kv_state_gb300 import kvm
    from compressed_kv_state_gb300 import workloads as wl
    q, k, v, g = wl.prefill_inputs(w)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dq, dk, dv = (torch.from_numpy(x).cuda().to(dt) for x in (q, k, v))
    dg = torch.from_numpy(g).cuda()
    cfg = kvm.make_config(batch=w.B, heads=w.H, rope_dims=w.rope_dims, chunk=w.chunk,
                          window=w.window, n_sinks=w.n_sinks, sched=w.sched, max_slots=w.max_slots,
                          dtype=kvm.KVM_BF16 if w.dtype == "bf16" else kvm.KVM_FP32,
                          max_tokens=w.N)
    layer = kvm.KvmLayer(cfg)                       # ordinary entry point, caller workspace
    ref = layer.prefill(dq, dk, dv, dg)
    layer.sync()
    out = torch.full_like(ref, float("nan"))
    kvm.kvm_prefill_noalloc(cfg, dq, dk, dv, dg, w.N, out)
    torch.cuda.synchronize()
    return ref.float().cpu().numpy(), out.float().cpu().numpy()


def test_noalloc_matches_prefill_on_two_calls_in_a_row():
    from compressed_kv_state_gb300 import workloads as wl
    first = wl.Workload("noalloc_bf16_B2H3N1500", B=2, H=3, N=1500, chunk=128, window=256,
                        n_sinks=16, max_slots=96, keys="repeat5")
    # the second call is smaller and uses another kernel path: it must not see
    # anything the first call left in the shared static scratch
    second = wl.Workload("noalloc_fp32_B1H2N700", B=1, H=2, N=700, chunk=64, window=128,
                         n_sinks=8, max_slots=40, dtype="fp32", keys="repeat5")
    for w, tol in ((first, TOL_BF16), (second, TOL_FP32)):
        ref, out = _both(w)
        assert np.isfinite(out).all()
        err = float(np.abs(ref - out).max())
        assert err <= tol, f"{w.name}: max-abs difference {err} > {tol}"


def test_noalloc_rejects_calls_beyond_its_static_scratch():
    from compressed_kv_state_gb300 import kvm
    cfg = kvm.make_config(batch=8, heads=12, max_tokens=8192)
    with pytest.raises(kvm.KvmError) as ei:
        kvm.kvm_prefill_noalloc(cfg, None, None, None, None, 8192, None)
    assert ei.value.status == kvm.KVM_ERR_WORKSPACE
    assert "KVM_NOALLOC_SCRATCH_BYTES" in str(ei.value)
