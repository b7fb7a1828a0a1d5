"""Failure detection on the GPU without a fault: a bounded device-side wait
that is made to run out (the fold chain waits for a chunk copy that is never
issued) must be reported as KVM_ERR_TIMEOUT by kvm_layer_sync, and the same
context must then run a normal prefill correctly."""
import numpy as np
import pytest

import oracle
from compressed_kv_state_gb300 import workloads as wl
from kvm_testlib import gpu_prefill, make_layer, oracle_cfg, tol_of

pytestmark = pytest.mark.gpu


def test_bounded_wait_expiry_is_reported_and_the_context_survives():
    import torch
    from compressed_kv_state_gb300 import kvm
    w = wl.Workload("stall", B=1, H=2, N=600, chunk=64, window=128, n_sinks=4, max_slots=24,
                    keys="repeat5")
    q, k, v, g = wl.prefill_inputs(w)
    layer = make_layer(w)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().bfloat16()
    dbg = kvm.kvm_debug(None, None, None, None, 0, 1)
    layer.prefill(dev(q), dev(k), dev(v), torch.from_numpy(g).cuda(), dbg=dbg)
    with pytest.raises(kvm.KvmError) as ei:
        layer.sync()
    assert ei.value.status == kvm.KVM_ERR_TIMEOUT
    layer.sync()  # the status word was cleared
    out, _, _ = gpu_prefill(layer, w, q, k, v, g, debug=False)
    ref, _, _ = oracle.prefill(oracle_cfg(w), q[0], k[0], v[0], g[0])
    assert np.abs(out[0] - ref).max() <= tol_of(w)
