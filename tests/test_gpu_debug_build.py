"""The KVM_DEBUG build (lib/libkvm_debug.so): device-side checks of data-dependent
indices and of imported state latch the layer's status word (kvm_layer_sync then
reports KVM_ERR_DEVICE) instead of reading out of range, and a valid call gives
the same output as the normal build.  The binding loads one library per process,
so the debug library runs in a child process (selected by KVM_LIBRARY)."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
from compressed_kv_state_gb300 import kvm
from compressed_kv_state_gb300 import workloads as wl
assert kvm.LIB_PATH.endswith(LIBNAME), kvm.LIB_PATH
w = wl.Workload("dbg_B1H2N1000", B=1, H=2, N=1000, chunk=128, window=256, n_sinks=16,
                max_slots=48, keys="repeat5")
q, k, v, g = wl.prefill_inputs(w)
cfg = kvm.make_config(batch=1, heads=2, chunk=128, window=256, n_sinks=16, max_slots=48,
                      max_tokens=1100)
layer = kvm.KvmLayer(cfg)
dev = lambda a: torch.from_numpy(a).cuda()
out = layer.prefill(dev(q).bfloat16(), dev(k).bfloat16(), dev(v).bfloat16(), dev(g))
layer.sync()  # a valid prefill latches nothing
np.save(OUT, out.float().cpu().numpy())
st = layer.export_state()
st["counts"][0, 0, 3] = 0  # an invalid imported state: a slot with no members
layer.import_state(st)
try:
    layer.sync()
    print("STATUS 0")
except kvm.KvmError as e:
    print("STATUS", e.status)
"""


def _run(tmp_path, lib, tag):
    out = tmp_path / f"{tag}.npy"
    env = dict(os.environ)
    if lib:
        env["KVM_LIBRARY"] = lib
    else:
        env.pop("KVM_LIBRARY", None)
    head = f"ROOT = {ROOT!r}\nOUT = {str(out)!r}\nLIBNAME = {os.path.basename(lib or 'libkvm.so')!r}\n"
    r = subprocess.run([sys.executable, "-c", head + SCRIPT], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    status = int(r.stdout.strip().splitlines()[-1].split()[1])
    return np.load(out), status


def test_debug_build_latches_bad_state_and_matches_the_normal_build(tmp_path):
    from compressed_kv_state_gb300 import build
    from compressed_kv_state_gb300 import kvm
    dbg_lib = build.build(debug=True)
    out_dbg, st_dbg = _run(tmp_path, dbg_lib, "debug")
    out_rel, st_rel = _run(tmp_path, None, "release")
    assert st_dbg == kvm.KVM_ERR_DEVICE          # the zero-count slot was caught on the device
    assert st_rel == kvm.KVM_OK                  # the normal build has no such check
    np.testing.assert_array_equal(out_dbg, out_rel)
