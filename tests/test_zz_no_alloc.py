"""kvm_prefill_noalloc: the prefill entry point for callers that may not
allocate device memory (for instance a plugin inside a host framework that
owns all device memory through its own pool, or a latency-critical loop that
cannot take an allocation's device synchronisation).  Its scratch is the
library's static device array instead of a caller workspace; it runs the same
kernels on the same tables as the ordinary kvm_prefill, so its output must
equal kvm_prefill's bit for bit, and a call must not change the device's
allocated or free memory.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _cfg(w):
    from compressed_kv_state_gb300 import kvm
    return kvm.make_config(batch=w.B, heads=w.H, rope_dims=w.rope_dims, chunk=w.chunk,
                           window=w.window, n_sinks=w.n_sinks, sched=w.sched, max_slots=w.max_slots,
                           dtype=kvm.KVM_BF16 if w.dtype == "bf16" else kvm.KVM_FP32,
                           max_tokens=w.N)


def _inputs(w):
    import torch
    from compressed_kv_state_gb300 import workloads as wl
    q, k, v, g = wl.prefill_inputs(w)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dq, dk, dv = (torch.from_numpy(x).cuda().to(dt) for x in (q, k, v))
    return dq, dk, dv, torch.from_numpy(g).cuda()


def _both(w):
    import torch
    from compressed_kv_state_gb300 import kvm
    dq, dk, dv, dg = _inputs(w)
    cfg = _cfg(w)
    layer = kvm.KvmLayer(cfg)                       # ordinary entry point, caller workspace
    ref = layer.prefill(dq, dk, dv, dg)
    layer.sync()
    out = torch.full_like(ref, float("nan"))
    kvm.kvm_prefill_noalloc(cfg, dq, dk, dv, dg, w.N, out)
    torch.cuda.synchronize()
    return ref.cpu(), out.cpu()


def test_noalloc_matches_prefill_on_two_calls_in_a_row():
    import torch
    from compressed_kv_state_gb300 import workloads as wl
    first = wl.Workload("noalloc_bf16_B2H3N1500", B=2, H=3, N=1500, chunk=128, window=256,
                        n_sinks=16, max_slots=96, keys="repeat5")
    # the second call is smaller and uses another kernel path: it must not see
    # anything the first call left in the shared static scratch
    second = wl.Workload("noalloc_fp32_B1H2N700", B=1, H=2, N=700, chunk=64, window=128,
                         n_sinks=8, max_slots=40, dtype="fp32", keys="repeat5")
    for w in (first, second):
        ref, out = _both(w)
        assert torch.isfinite(out.float()).all()
        # same kernels, same tables: identical bit for bit
        assert torch.equal(ref.view(torch.int16 if w.dtype == "bf16" else torch.int32),
                           out.view(torch.int16 if w.dtype == "bf16" else torch.int32)), \
            f"{w.name}: max-abs difference {float((ref.float() - out.float()).abs().max())}"


def test_noalloc_call_allocates_nothing():
    """After a first call (which may load the library's device code and with it the
    static array), a second identical call leaves torch's allocated bytes and the
    device's free bytes unchanged."""
    import torch
    from compressed_kv_state_gb300 import kvm
    from compressed_kv_state_gb300 import workloads as wl
    w = wl.Workload("noalloc_mem_B1H4N2048", B=1, H=4, N=2048, chunk=128, window=256,
                    n_sinks=16, max_slots=64, keys="repeat5")
    dq, dk, dv, dg = _inputs(w)
    cfg = _cfg(w)
    out = torch.empty_like(dq)
    kvm.kvm_prefill_noalloc(cfg, dq, dk, dv, dg, w.N, out)
    torch.cuda.synchronize()
    first = out.clone()
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    kvm.kvm_prefill_noalloc(cfg, dq, dk, dv, dg, w.N, out)
    torch.cuda.synchronize()
    alloc1, free1 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    assert alloc1 == alloc0, (alloc0, alloc1)
    assert free1 == free0, (free0, free1)
    assert torch.equal(first, out)


def test_noalloc_rejects_calls_beyond_its_static_scratch():
    from compressed_kv_state_gb300 import kvm
    cfg = kvm.make_config(batch=8, heads=12, max_tokens=8192)
    with pytest.raises(kvm.KvmError) as ei:
        kvm.kvm_prefill_noalloc(cfg, None, None, None, None, 8192, None, check=False)
    assert ei.value.status == kvm.KVM_ERR_WORKSPACE
    assert "KVM_NOALLOC_SCRATCH_BYTES" in str(ei.value)


def test_noalloc_rejects_host_buffers_before_enqueuing():
    """Pointers that are not device memory of the current device are refused by the
    library itself (checked with cudaPointerGetAttributes, nothing enqueued)."""
    import torch
    from compressed_kv_state_gb300 import kvm
    from compressed_kv_state_gb300 import workloads as wl
    w = wl.Workload("noalloc_host_B1H2N300", B=1, H=2, N=300, chunk=64, window=128, n_sinks=4,
                    max_slots=24)
    dq, dk, dv, dg = _inputs(w)
    host_out = torch.zeros(dq.shape, dtype=dq.dtype)          # pageable host memory
    with pytest.raises(kvm.KvmError) as ei:
        kvm.kvm_prefill_noalloc(_cfg(w), dq, dk, dv, dg, w.N, host_out, check=False)
    assert ei.value.status == kvm.KVM_ERR_INVALID_ARG
    assert "out" in str(ei.value)
    assert not host_out.any()
    torch.cuda.synchronize()
