"""C ABI checks that need no GPU: the library loads, exports every function
include/kvm.h declares, and validates configurations on the host."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvm():
    from compressed_kv_state_gb300 import build
    build.build()
    from compressed_kv_state_gb300 import kvm as mod
    return mod


def _declared(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvm_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(kvm):
    names = _declared("kvm.h")
    assert "kvm_prefill" in names and "kvm_decode_step" in names
    lib = ctypes.CDLL(kvm.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_headers_cover_the_boundary():
    for f in os.listdir(os.path.join(ROOT, "include")):
        assert f.endswith(".h")
    names = _declared("kvm.h")
    for n in ("kvm_workspace_bytes", "kvm_layer_create", "kvm_prefill", "kvm_decode_step",
              "kvm_state_export", "kvm_state_import", "kvm_layer_sync", "kvm_last_error",
              "kvm_layer_destroy"):
        assert n in names


def test_struct_sizes_match_header(kvm):
    # 16 four-byte fields, no padding
    assert ctypes.sizeof(kvm.kvm_config) == 64
    assert ctypes.sizeof(kvm.kvm_state_bufs) == 7 * 8 + 3 * 8
    assert ctypes.sizeof(kvm.kvm_debug) == 5 * 8 + 8  # + int32 test hook, padded


def test_binding_argument_counts_match_the_header(kvm):
    """Each function the binding declares takes as many arguments as its
    prototype in include/kvm.h."""
    text = open(os.path.join(ROOT, "include", "kvm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    protos = dict(re.findall(r"\b(kvm_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S))
    lib = kvm.lib
    checked = 0
    for name, args in protos.items():
        argtypes = getattr(lib, name).argtypes
        if argtypes is None:
            continue
        n = 0 if args.strip() in ("", "void") else args.count(",") + 1
        assert len(argtypes) == n, (name, n, len(argtypes))
        checked += 1
    assert checked >= 15


def test_struct_layouts_match_the_c_compiler(kvm, tmp_path):
    """Every field offset and struct size of the ctypes binding equals what a C
    compiler makes of include/kvm.h (gcc, this host's ABI)."""
    structs = {"kvm_config": kvm.kvm_config, "kvm_state_bufs": kvm.kvm_state_bufs,
               "kvm_debug": kvm.kvm_debug, "kvm_timing": kvm.kvm_timing}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "kvm.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for fname, _ in cls._fields_:
            lines.append(f'printf("{name} {fname} %zu\\n", offsetof({name}, {fname}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    import subprocess
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for name, cls in structs.items():
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for fname, _ in cls._fields_:
            assert got[(name, fname)] == getattr(cls, fname).offset, (name, fname)


@pytest.mark.parametrize("field,value,msg", [
    ("head_dim", 32, "head_dim"),
    ("chunk", 24, "chunk"),
    ("chunk", 512, "chunk"),
    ("window", 100, "window"),
    ("n_sinks", 200, "n_sinks"),
    ("max_slots", 16, "max_slots"),
    ("rope_dims", 3, "rope_dims"),
    ("dtype", 9, "dtype"),
    ("sched", 5, "schedule"),
    ("batch", 0, "batch"),
    ("max_tokens", 0, "max_tokens"),
    ("flags", 2, "flags"),
])
def test_invalid_configs_rejected(kvm, field, value, msg):
    cfg = kvm.make_config(batch=1, heads=2)
    setattr(cfg, field, value)
    assert kvm.lib.kvm_workspace_bytes(ctypes.byref(cfg)) == 0
    assert msg in kvm.kvm_last_error(None)


def test_power_schedule_needs_positive_coef(kvm):
    cfg = kvm.make_config(batch=1, heads=1, sched=kvm.KVM_SCHED_POWER, coef=0.0)
    assert kvm.lib.kvm_workspace_bytes(ctypes.byref(cfg)) == 0


def test_workspace_size_grows_with_slots_and_tokens(kvm):
    a = kvm.kvm_workspace_bytes(kvm.make_config(batch=8, heads=12))
    b = kvm.kvm_workspace_bytes(kvm.make_config(batch=8, heads=12, max_slots=512))
    c = kvm.kvm_workspace_bytes(kvm.make_config(batch=8, heads=12, max_tokens=16384))
    assert 0 < a < b and a < c
    assert a % 256 == 0


def test_null_handles_are_rejected(kvm):
    assert kvm.lib.kvm_prefill(None, None, None, None, None, 0, None, None, None) == \
        kvm.KVM_ERR_INVALID_ARG
    assert kvm.lib.kvm_layer_sync(None) == kvm.KVM_ERR_INVALID_ARG
    out = ctypes.c_void_p()
    cfg = kvm.make_config(batch=1, heads=1)
    assert kvm.lib.kvm_layer_create(ctypes.byref(cfg), None, 0, ctypes.byref(out)) == \
        kvm.KVM_ERR_WORKSPACE
    assert out.value is None


def test_forward_scratch_bytes_validates_and_sizes(kvm):
    cfg = kvm.make_config(batch=2, heads=3, max_tokens=1000)
    rows = 2 * 3 * 700
    al = lambda n: (n + 255) // 256 * 256
    want = 4 * al(rows * 64 * 2) + al(rows * 4)
    assert kvm.lib.kvm_forward_scratch_bytes(ctypes.byref(cfg), 128, 700) == want
    for d_model, n in ((100, 700), (0, 700), (128, 0), (128, 1001)):
        assert kvm.lib.kvm_forward_scratch_bytes(ctypes.byref(cfg), d_model, n) == 0
    cfg32 = kvm.make_config(batch=2, heads=3, max_tokens=1000, dtype=kvm.KVM_FP32)
    assert kvm.lib.kvm_forward_scratch_bytes(ctypes.byref(cfg32), 128, 700) == 0


def test_overlap_and_forward_entry_points_reject_null_layers(kvm):
    assert kvm.lib.kvm_layer_set_overlap(None, 3) == kvm.KVM_ERR_INVALID_ARG
    n = ctypes.c_int32(5)
    assert kvm.lib.kvm_layer_get_overlap(None, ctypes.byref(n)) == kvm.KVM_ERR_INVALID_ARG
    assert kvm.lib.kvm_layer_forward(None, 128, None, None, None, 1, None, None, 0, None) == \
        kvm.KVM_ERR_INVALID_ARG


def test_state_buffers_are_checked_before_the_library_copies_them(kvm):
    """The binding rejects state tensors whose size, type or layout differs from
    what kvm_state_export / kvm_state_import copy (fixed byte counts)."""
    import torch
    cfg = kvm.make_config(batch=2, heads=3, chunk=64, window=128, max_slots=40)
    spec = kvm.state_spec(cfg)
    assert spec["sum_k"][0] == (2, 3, 40, 64) and spec["ring_k"][0] == (2, 3, 192, 64)
    assert spec["ring_k"][1] == torch.bfloat16 and spec["counts"][1] == torch.int32
    good = {n: torch.zeros(s, dtype=d) for n, (s, d) in spec.items()}
    kvm.check_state_tensors(cfg, good, require_cuda=False)
    bad_cases = [
        ("sum_k", torch.zeros(2, 3, 39, 64)),                         # too few slots
        ("counts", torch.zeros(2, 3, 40, dtype=torch.int64)),          # wrong type
        ("ring_k", torch.zeros(2, 3, 64, 192, dtype=torch.bfloat16).transpose(2, 3)),  # strided
    ]
    for name, t in bad_cases:
        with pytest.raises(ValueError):
            kvm.check_state_tensors(cfg, dict(good, **{name: t}), require_cuda=False)
    with pytest.raises(ValueError):
        kvm.check_state_tensors(cfg, {k: v for k, v in good.items() if k != "rho"}, require_cuda=False)
    with pytest.raises(ValueError):
        kvm.check_state_tensors(cfg, good)  # CPU tensors where device memory is required


def test_noalloc_tensors_are_checked_before_the_library_is_called(kvm, monkeypatch):
    """kvm_prefill_noalloc's binding rejects tensors of the wrong shape, type, layout
    or device (and n_tokens beyond them) with ValueError before calling the library."""
    import torch
    calls = []
    monkeypatch.setattr(kvm, "lib", type("L", (), {"kvm_prefill_noalloc": lambda *a: calls.append(a) or 0})())
    cfg = kvm.make_config(batch=1, heads=2, chunk=64, window=128, max_slots=24, max_tokens=300)
    shp = (1, 2, 300, 64)
    q, k, v, out = (torch.zeros(shp, dtype=torch.bfloat16) for _ in range(4))
    g = torch.zeros(shp[:3])
    cases = [
        dict(q=torch.zeros(1, 2, 299, 64, dtype=torch.bfloat16)),        # wrong shape
        dict(k=torch.zeros(shp)),                                        # wrong dtype
        dict(v=torch.zeros(1, 2, 64, 300, dtype=torch.bfloat16).transpose(2, 3)),  # strided
        dict(gate=torch.zeros(shp[:3], dtype=torch.bfloat16)),           # gate not fp32
        dict(n_tokens=301),                                              # beyond the tensors
        dict(),                                                          # CPU tensors
    ]
    for bad in cases:
        a = dict(q=q, k=k, v=v, gate=g, n_tokens=300, out=out)
        a.update(bad)
        with pytest.raises(ValueError):
            kvm.kvm_prefill_noalloc(cfg, a["q"], a["k"], a["v"], a["gate"], a["n_tokens"], a["out"])
    assert not calls


def test_backward_tensors_are_checked_before_the_library_is_called(kvm, monkeypatch):
    """kvm_prefill_backward's binding (given the layer's config) rejects inputs, output
    gradients or scratch of the wrong shape, type, layout or device with ValueError
    before calling the library."""
    import torch
    calls = []
    monkeypatch.setattr(kvm, "lib", type("L", (), {"kvm_prefill_backward": lambda *a: calls.append(a) or 0})())
    cfg = kvm.make_config(batch=1, heads=2, chunk=64, window=128, max_slots=24, max_tokens=300)
    shp = (1, 2, 300, 64)
    q, k, v, out, dout = (torch.zeros(shp, dtype=torch.bfloat16) for _ in range(5))
    g = torch.zeros(shp[:3])
    dq, dk, dv = (torch.zeros(shp) for _ in range(3))
    dg = torch.zeros(shp[:3])
    scratch = torch.zeros(1024, dtype=torch.uint8)
    cases = [
        dict(dout=torch.zeros(1, 2, 299, 64, dtype=torch.bfloat16)),     # dout shape
        dict(dq=torch.zeros(shp, dtype=torch.bfloat16)),                 # gradient not fp32
        dict(dk=torch.zeros(1, 2, 64, 300).transpose(2, 3)),             # strided
        dict(dgate=torch.zeros(1, 2, 301)),                              # dgate shape
        dict(q=torch.zeros(1, 2, 300, 32, dtype=torch.bfloat16)),        # input shape
        dict(n_tokens=301),                                              # beyond the tensors
        dict(),                                                          # CPU tensors
    ]
    for bad in cases:
        a = dict(q=q, k=k, v=v, gate=g, out=out, dout=dout, n_tokens=300, dq=dq, dk=dk, dv=dv, dgate=dg)
        a.update(bad)
        with pytest.raises(ValueError):
            kvm.kvm_prefill_backward(None, a["q"], a["k"], a["v"], a["gate"], a["out"], a["dout"], None,
                                     a["n_tokens"], a["dq"], a["dk"], a["dv"], a["dgate"], scratch, cfg=cfg)
    assert not calls


def test_binding_fails_loudly_without_the_library(tmp_path):
    """No fallback: importing the binding without libkvm.so raises (run in a fresh
    interpreter against a copy of the package whose library is absent)."""
    import shutil
    import subprocess
    import sys
    pkg = os.path.join(ROOT, "compressed_kv_state_gb300")
    dst = tmp_path / "compressed_kv_state_gb300"
    shutil.copytree(pkg, dst, ignore=shutil.ignore_patterns("lib", "__pycache__", "csrc"))
    r = subprocess.run([sys.executable, "-c", "import compressed_kv_state_gb300.kvm"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "libkvm.so not built" in r.stderr
