"""Whole-layer forward (kvm_layer_forward): the tensor-core projections around
the KVM attention, checked stage by stage against the oracle, each stage fed
the GPU's own output of the previous stage (the bf16 projections decide the
fold's winner-take-all, so the oracle takes those decisions on the same values):

  1. q, k, v (bf16) and gate (fp32) against the fp64 input projection;
  2. the attention output against the oracle's prefill on the GPU's q, k, v,
     gate (rows before the first event with an oracle near tie);
  3. y against the fp64 output projection of the GPU's attention output.

Tolerances: bf16 tensors max-abs 2e-2 (values of order one), gates 1e-5.
"""
import numpy as np
import pytest

import oracle
from compressed_kv_state_gb300 import workloads as wl
from kvm_testlib import NEAR_TIE, TOL_BF16, oracle_cfg

pytestmark = pytest.mark.gpu

CASES = [
    # small: two K blocks, a partial last column tile (the two gate columns)
    (wl.Workload("layer_B2H2N1024_dm128", B=2, H=2, N=1024, chunk=128, window=256, n_sinks=16,
                 max_slots=64), 128),
    # ragged token count, three heads, K = 192
    (wl.Workload("layer_B1H3N1500_dm192", B=1, H=3, N=1500, chunk=128, window=256, n_sinks=16,
                 max_slots=96), 192),
]
FULL = (wl.Workload("layer_B8H12N8192_dm768", B=8, H=12, N=8192), 768)


def _run(w, d_model):
    import torch
    from compressed_kv_state_gb300 import kvm
    from kvm_testlib import make_layer
    x, w_in, w_out = wl.layer_inputs(w, d_model)
    layer = make_layer(w)
    dev = torch.device("cuda")
    tx = torch.from_numpy(x).to(dev).bfloat16()
    tin = torch.from_numpy(w_in).to(dev).bfloat16()
    tout = torch.from_numpy(w_out).to(dev).bfloat16()
    y, inter = layer.forward(tx, tin, tout)
    layer.sync()
    torch.cuda.synchronize()
    got = {k: v.float().cpu().numpy().astype(np.float64) for k, v in inter.items()}
    return x, w_in, w_out, y.float().cpu().numpy().astype(np.float64), got


def _near_rows(w, odbg, i):
    Wc = w.window // w.chunk
    near = [e for e in range(odbg["gap"].shape[1])
            if odbg["sel_margin"][i, e] < NEAR_TIE or
            ((odbg["kind"][i, e] == oracle.MERGED).any() and
             odbg["gap"][i, e][odbg["kind"][i, e] == oracle.MERGED].min() < NEAR_TIE)]
    return w.N if not near else min(w.N, (near[0] + Wc + 1) * w.chunk)


def _check(w, d_model, heads=None, tokens=None):
    x, w_in, w_out, y, got = _run(w, d_model)
    H = w.H
    # stage 1: input projection (sampled tokens at full size)
    sel = slice(None) if tokens is None else tokens
    q, k, v, gate = oracle.layer_project_in(x[:, sel], w_in, H)
    for name, ref in (("q", q), ("k", k), ("v", v)):
        err = np.abs(got[name][:, :, sel] - ref).max()
        assert err <= TOL_BF16, f"{name} max-abs error {err}"
    gerr = np.abs(got["gate"][:, :, sel] - gate).max()
    assert gerr <= 1e-5, f"gate max-abs error {gerr}"
    # stage 2: attention on the GPU's own projections
    hs = heads if heads is not None else [(b, h) for b in range(w.B) for h in range(H)]
    cfg = oracle_cfg(w)
    oo, _, odbg = oracle.prefill(cfg, np.stack([got["q"][b, h] for b, h in hs]),
                                 np.stack([got["k"][b, h] for b, h in hs]),
                                 np.stack([got["v"][b, h] for b, h in hs]),
                                 np.stack([got["gate"][b, h] for b, h in hs]))
    for i, (b, h) in enumerate(hs):
        rows = _near_rows(w, odbg, i)
        assert rows >= min(w.N, (w.window // w.chunk + 2) * w.chunk)
        err = np.abs(got["o"][b, h, :rows] - oo[i, :rows]).max()
        assert err <= TOL_BF16, f"(b={b}, h={h}) attention max-abs error {err} over {rows} rows"
    # stage 3: output projection of the GPU's attention output
    yref = oracle.layer_project_out(got["o"][:, :, sel], w_out)
    err = np.abs(y[:, sel] - yref).max()
    assert err <= TOL_BF16, f"y max-abs error {err}"


@pytest.mark.parametrize("w,d_model", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_layer_forward_stages(w, d_model):
    _check(w, d_model)


def test_layer_forward_full_size_sampled():
    """The 8k fixed-state workload as a whole layer (d_model 768, 12 heads):
    projections on sampled tokens, attention on two sampled heads."""
    w, d_model = FULL
    rng = np.random.default_rng(0)
    tokens = np.sort(rng.choice(w.N, size=96, replace=False))
    _check(w, d_model, heads=[(0, 0), (w.B - 1, w.H - 1)], tokens=tokens)


def test_layer_forward_rejects_bad_arguments():
    import torch
    from compressed_kv_state_gb300 import kvm
    from kvm_testlib import make_layer
    w = CASES[0][0]
    layer = make_layer(w)
    x = torch.zeros((w.B, w.N, 100), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvm.KvmError):
        kvm.kvm_forward_scratch_bytes(layer.cfg, 100, w.N)  # d_model not a multiple of 64
    wf = make_layer(w.with_(dtype="fp32"))
    x = torch.zeros((w.B, w.N, 128), dtype=torch.bfloat16, device="cuda")
    w_in = torch.zeros((3 * w.H * 64 + w.H, 128), dtype=torch.bfloat16, device="cuda")
    w_out = torch.zeros((128, w.H * 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvm.KvmError):
        wf.forward(x, w_in, w_out)  # fp32 layer
