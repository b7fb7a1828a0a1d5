"""GPU backward of the prefill (kvm_prefill_backward) against the fp64 oracle.

Both sides take the fold decisions the GPU forward recorded (the backward's
reading: decisions are constants), so near ties cannot make them differ.  The
oracle (oracle/backward.py, pinned on the CPU) differentiates the restated
prefill in fp64 on the exact bf16/fp32 input values.  Chunks that are multiples of
64 run the tiled kernels, others the row-per-warp kernels; both are covered.  Tolerance: the GPU reads
its state through bf16 read rows and rotates in bf16 for bf16 layers, so every
gradient is compared against its own scale: max |gpu - oracle| <= TOL x
max |oracle|, TOL 3e-2 (bf16) / 1e-4 (fp32); and the relative Frobenius error
<= TOL / 3.
"""
import numpy as np
import pytest

import oracle
from oracle import backward as ob
from compressed_kv_state_gb300 import workloads as wl
from kvm_testlib import make_layer, oracle_cfg

pytestmark = pytest.mark.gpu

CASES = [
    wl.Workload("bwd_fixed_B1H2N1200_C128W256", B=1, H=2, N=1200, chunk=128, window=256,
                n_sinks=16, max_slots=48, keys="repeat5"),
    wl.Workload("bwd_fp32_B1H2N700_C64W128", B=1, H=2, N=700, chunk=64, window=128, n_sinks=8,
                max_slots=40, keys="repeat5", dtype="fp32"),
    wl.Workload("bwd_sqrt_B2H1N1500_C128W256", B=2, H=1, N=1500, chunk=128, window=256,
                n_sinks=16, sched=1, max_slots=160, coef=4.0, keys="neardup20"),
    wl.Workload("bwd_C256_B1H1N2000_W512", B=1, H=1, N=2000, chunk=256, window=512, n_sinks=16,
                max_slots=300, keys="repeat5"),
    wl.Workload("bwd_novnorm_B1H2N1000_C64W128", B=1, H=2, N=1000, chunk=64, window=128,
                n_sinks=8, max_slots=40, keys="repeat5", flags=1),
    wl.Workload("bwd_norope_fp32_B1H1N600_C64W128", B=1, H=1, N=600, chunk=64, window=128,
                n_sinks=4, max_slots=24, keys="plain", dtype="fp32", rope_dims=0),
    # chunks that are not a multiple of 64 take the row-per-warp kernels
    wl.Workload("bwd_C32_B1H2N500_W64", B=1, H=2, N=500, chunk=32, window=64, n_sinks=4,
                max_slots=32, keys="repeat5"),
    wl.Workload("bwd_C32_fp32_B1H1N400_W96", B=1, H=1, N=400, chunk=32, window=96, n_sinks=4,
                max_slots=24, keys="repeat5", dtype="fp32"),
    # no fold event yet (N <= W + C): window attention only, no member lists or sweep
    wl.Workload("bwd_E0_B1H2N170_C64W128", B=1, H=2, N=170, chunk=64, window=128, n_sinks=4,
                max_slots=16, keys="repeat5"),
    wl.Workload("bwd_E0_B1H1N250_C128W128", B=1, H=1, N=250, chunk=128, window=128, n_sinks=4,
                max_slots=16, keys="repeat5"),
]


def _run(w):
    import torch
    from compressed_kv_state_gb300 import kvm
    q, k, v, g = wl.prefill_inputs(w)
    rng = np.random.default_rng(11)
    dout = rng.standard_normal(q.shape).astype(np.float32)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    tq, tk, tv, tdo = (dev(x).to(dt) for x in (q, k, v, dout))
    tg = dev(g)
    layer = make_layer(w)
    E = oracle.n_events(oracle_cfg(w), w.N)
    shp = (w.B, w.H, E, w.chunk)
    bufs = dict(assign=torch.full(shp, -7, dtype=torch.int32, device="cuda"),
                kind=torch.full(shp, -7, dtype=torch.int32, device="cuda"),
                max_sim=torch.zeros(shp, device="cuda"), gap=torch.zeros(shp, device="cuda"))
    rec = kvm.kvm_debug(bufs["assign"].data_ptr(), bufs["kind"].data_ptr(), bufs["max_sim"].data_ptr(),
                        bufs["gap"].data_ptr(), E)
    out = layer.prefill(tq, tk, tv, tg, dbg=rec)
    grads = layer.prefill_backward(tq, tk, tv, tg, out, tdo, rec)
    layer.sync()
    torch.cuda.synchronize()
    exact = [x.double().cpu().numpy() for x in (tq, tk, tv, tdo)]  # the values the GPU saw
    res = dict(grads=[x.cpu().numpy().astype(np.float64) for x in grads],
               assign=bufs["assign"].cpu().numpy(), kind=bufs["kind"].cpu().numpy(),
               q=exact[0], k=exact[1], v=exact[2], g=g.astype(np.float64), dout=exact[3])
    layer.close()
    return res


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_backward_matches_the_oracle(w):
    r = _run(w)
    cfg = oracle_cfg(w)
    tol = 1e-4 if w.dtype == "fp32" else 3e-2
    for b in range(w.B):
        for h in range(w.H):
            ref = ob.backward(cfg, r["q"][b, h], r["k"][b, h], r["v"][b, h], r["g"][b, h],
                              r["assign"][b, h], r["kind"][b, h], r["dout"][b, h])
            for name, mine, want in zip(("dq", "dk", "dv", "dgate"), (x[b, h] for x in r["grads"]), ref):
                assert np.isfinite(mine).all(), name
                scale = np.abs(want).max()
                err = np.abs(mine - want).max()
                fro = np.linalg.norm(mine - want) / max(np.linalg.norm(want), 1e-30)
                assert err <= tol * scale, f"(b={b}, h={h}) {name}: max err {err:.3g} vs scale {scale:.3g}"
                assert fro <= tol / 3, f"(b={b}, h={h}) {name}: relative Frobenius error {fro:.3g}"


def test_backward_full_size_sampled_heads():
    """The fixed-state 8k workload (B8 H12 N8192, 59 fold events per row): every head
    on the GPU, two heads against the oracle."""
    w = wl.FIXED_8K
    r = _run(w)
    cfg = oracle_cfg(w)
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        ref = ob.backward(cfg, r["q"][b, h], r["k"][b, h], r["v"][b, h], r["g"][b, h],
                          r["assign"][b, h], r["kind"][b, h], r["dout"][b, h])
        for name, mine, want in zip(("dq", "dk", "dv", "dgate"), (x[b, h] for x in r["grads"]), ref):
            scale = np.abs(want).max()
            err = np.abs(mine - want).max()
            fro = np.linalg.norm(mine - want) / max(np.linalg.norm(want), 1e-30)
            assert err <= 3e-2 * scale, f"(b={b}, h={h}) {name}: max err {err:.3g} vs scale {scale:.3g}"
            assert fro <= 1e-2, f"(b={b}, h={h}) {name}: relative Frobenius error {fro:.3g}"
    for x in r["grads"]:
        assert np.isfinite(x).all()


def test_backward_refuses_a_mismatched_call():
    import torch
    from compressed_kv_state_gb300 import kvm
    w = CASES[0]
    q, k, v, g = wl.prefill_inputs(w)
    layer = make_layer(w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().bfloat16()
    tq, tk, tv = t(q), t(k), t(v)
    tg = torch.from_numpy(g).cuda()
    out = layer.prefill(tq, tk, tv, tg)
    # no record of the fold decisions
    with pytest.raises(kvm.KvmError):
        layer.prefill_backward(tq, tk, tv, tg, out, out, None)
    # a prefill of another length ran last
    layer.prefill(tq[:, :, :900].contiguous(), tk[:, :, :900].contiguous(), tv[:, :, :900].contiguous(),
                  tg[:, :, :900].contiguous())
    E = oracle.n_events(oracle_cfg(w), w.N)
    a = torch.zeros((w.B, w.H, E, w.chunk), dtype=torch.int32, device="cuda")
    rec = kvm.kvm_debug(a.data_ptr(), a.data_ptr(), None, None, E)
    with pytest.raises(kvm.KvmError):
        layer.prefill_backward(tq, tk, tv, tg, out, out, rec)
    layer.close()
