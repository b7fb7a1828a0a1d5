"""Thin ctypes binding of libkvm.so (include/kvm.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions keep the C names; tensors are torch CUDA tensors (torch is
used for device memory and streams only).  There is no fallback: if the
library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVM_LIBRARY selects another build of the same library (the KVM_DEBUG variant,
# lib/libkvm_debug.so, with device-side checks); default: lib/libkvm.so
LIB_PATH = os.environ.get("KVM_LIBRARY") or os.path.join(_HERE, "lib", "libkvm.so")

KVM_OK, KVM_ERR_INVALID_ARG, KVM_ERR_UNSUPPORTED, KVM_ERR_CAPACITY = 0, 1, 2, 3
KVM_ERR_WORKSPACE, KVM_ERR_CUDA, KVM_ERR_TIMEOUT, KVM_ERR_DEVICE = 4, 5, 6, 7
KVM_BF16, KVM_FP32 = 0, 1
KVM_SCHED_FIXED, KVM_SCHED_POWER = 0, 1
KVM_FLAG_NO_VALUE_NORM = 1
STATUS_NAMES = {0: "KVM_OK", 1: "KVM_ERR_INVALID_ARG", 2: "KVM_ERR_UNSUPPORTED",
                3: "KVM_ERR_CAPACITY", 4: "KVM_ERR_WORKSPACE", 5: "KVM_ERR_CUDA",
                6: "KVM_ERR_TIMEOUT", 7: "KVM_ERR_DEVICE"}


class kvm_config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("rope_dims", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("chunk", ctypes.c_int32),
                ("window", ctypes.c_int32), ("n_sinks", ctypes.c_int32),
                ("sched", ctypes.c_int32), ("max_slots", ctypes.c_int32),
                ("coef", ctypes.c_float), ("expo", ctypes.c_float),
                ("ln_eps", ctypes.c_float), ("dtype", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("flags", ctypes.c_int32)]


class kvm_state_bufs(ctypes.Structure):
    _fields_ = [("sum_k", ctypes.c_void_p), ("sum_v", ctypes.c_void_p),
                ("counts", ctypes.c_void_p), ("rho", ctypes.c_void_p),
                ("ring_k", ctypes.c_void_p), ("ring_v", ctypes.c_void_p),
                ("ring_g", ctypes.c_void_p), ("n_slots", ctypes.c_int64),
                ("n_overflow", ctypes.c_int64), ("pos", ctypes.c_int64)]


class kvm_debug(ctypes.Structure):
    _fields_ = [("assign", ctypes.c_void_p), ("kind", ctypes.c_void_p),
                ("max_sim", ctypes.c_void_p), ("gap", ctypes.c_void_p),
                ("max_events", ctypes.c_int64), ("test_stall", ctypes.c_int32)]


class kvm_timing(ctypes.Structure):
    _fields_ = [("fold_ms", ctypes.c_double), ("attn_ms", ctypes.c_double),
                ("decode_ms", ctypes.c_double), ("other_ms", ctypes.c_double),
                ("fold_launches", ctypes.c_int64), ("attn_launches", ctypes.c_int64),
                ("decode_launches", ctypes.c_int64), ("other_launches", ctypes.c_int64),
                ("kernels", ctypes.c_int64), ("proj_ms", ctypes.c_double),
                ("proj_launches", ctypes.c_int64)]


class KvmError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libkvm.so not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    lib.kvm_workspace_bytes.restype = ctypes.c_size_t
    lib.kvm_workspace_bytes.argtypes = [P]
    lib.kvm_layer_create.restype = ctypes.c_int
    lib.kvm_layer_create.argtypes = [P, P, ctypes.c_size_t, ctypes.POINTER(P)]
    lib.kvm_prefill.restype = ctypes.c_int
    lib.kvm_prefill.argtypes = [P, P, P, P, P, I64, P, P, P]
    lib.kvm_decode_step.restype = ctypes.c_int
    lib.kvm_decode_step.argtypes = [P, P, P, P, P, P, P]
    lib.kvm_state_export.restype = ctypes.c_int
    lib.kvm_state_export.argtypes = [P, P, P]
    lib.kvm_state_import.restype = ctypes.c_int
    lib.kvm_state_import.argtypes = [P, P, P]
    lib.kvm_layer_sync.restype = ctypes.c_int
    lib.kvm_layer_sync.argtypes = [P]
    lib.kvm_last_error.restype = ctypes.c_char_p
    lib.kvm_last_error.argtypes = [P]
    lib.kvm_layer_set_timing.restype = ctypes.c_int
    lib.kvm_layer_set_timing.argtypes = [P, ctypes.c_int]
    lib.kvm_layer_get_timing.restype = ctypes.c_int
    lib.kvm_layer_get_timing.argtypes = [P, P]
    lib.kvm_forward_scratch_bytes.restype = ctypes.c_size_t
    lib.kvm_forward_scratch_bytes.argtypes = [P, ctypes.c_int32, I64]
    lib.kvm_layer_forward.restype = ctypes.c_int
    lib.kvm_layer_forward.argtypes = [P, ctypes.c_int32, P, P, P, I64, P, P, ctypes.c_size_t, P]
    lib.kvm_layer_set_overlap.restype = ctypes.c_int
    lib.kvm_layer_set_overlap.argtypes = [P, ctypes.c_int32]
    lib.kvm_layer_get_overlap.restype = ctypes.c_int
    lib.kvm_layer_get_overlap.argtypes = [P, P]
    lib.kvm_prefill_noalloc.restype = ctypes.c_int
    lib.kvm_prefill_noalloc.argtypes = [P, P, P, P, P, I64, P, P]
    lib.kvm_backward_scratch_bytes.restype = ctypes.c_size_t
    lib.kvm_backward_scratch_bytes.argtypes = [P, I64]
    lib.kvm_prefill_backward.restype = ctypes.c_int
    lib.kvm_prefill_backward.argtypes = [P, P, P, P, P, P, P, P, I64, P, P, P, P, P, ctypes.c_size_t, P]
    lib.kvm_layer_destroy.restype = None
    lib.kvm_layer_destroy.argtypes = [P]
    return lib


lib = _load()


def _check(status: int, layer=None):
    if status != KVM_OK:
        raise KvmError(status, kvm_last_error(layer))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream))


# ------------------------------------------------------------- C entry points

def kvm_workspace_bytes(cfg: kvm_config) -> int:
    n = lib.kvm_workspace_bytes(ctypes.byref(cfg))
    if n == 0:
        raise KvmError(KVM_ERR_INVALID_ARG, kvm_last_error(None))
    return int(n)


def kvm_layer_create(cfg: kvm_config, workspace) -> ctypes.c_void_p:
    out = ctypes.c_void_p()
    st = lib.kvm_layer_create(ctypes.byref(cfg), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), ctypes.byref(out))
    _check(st, None)
    return out


def kvm_prefill(layer, q, k, v, gate, n_tokens: int, out, stream=None, dbg: kvm_debug | None = None):
    st = lib.kvm_prefill(layer, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), int(n_tokens), _ptr(out),
                         _stream(stream), ctypes.byref(dbg) if dbg is not None else None)
    _check(st, layer)


def kvm_decode_step(layer, q, k, v, gate, out, stream=None):
    st = lib.kvm_decode_step(layer, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out),
                             _stream(stream))
    _check(st, layer)


def kvm_state_export(layer, dst: kvm_state_bufs, stream=None):
    _check(lib.kvm_state_export(layer, ctypes.byref(dst), _stream(stream)), layer)


def kvm_state_import(layer, src: kvm_state_bufs, stream=None):
    _check(lib.kvm_state_import(layer, ctypes.byref(src), _stream(stream)), layer)


def kvm_layer_sync(layer):
    _check(lib.kvm_layer_sync(layer), layer)


def kvm_layer_set_timing(layer, enable: bool):
    _check(lib.kvm_layer_set_timing(layer, 1 if enable else 0), layer)


def kvm_layer_get_timing(layer) -> dict:
    t = kvm_timing()
    _check(lib.kvm_layer_get_timing(layer, ctypes.byref(t)), layer)
    return {name: getattr(t, name) for name, _ in kvm_timing._fields_}


def kvm_forward_scratch_bytes(cfg: kvm_config, d_model: int, n_tokens: int) -> int:
    n = lib.kvm_forward_scratch_bytes(ctypes.byref(cfg), int(d_model), int(n_tokens))
    if n == 0:
        raise KvmError(KVM_ERR_INVALID_ARG, kvm_last_error(None))
    return n


def kvm_layer_forward(layer, d_model: int, x, w_in, w_out, n_tokens: int, y, scratch, stream=None):
    """Whole-layer forward: projections (tensor cores) around the KVM attention."""
    st = lib.kvm_layer_forward(layer, int(d_model), _ptr(x), _ptr(w_in), _ptr(w_out), int(n_tokens), _ptr(y),
                               _ptr(scratch), int(scratch.numel() * scratch.element_size()), _stream(stream))
    _check(st, layer)


def kvm_layer_set_overlap(layer, segments: int):
    """0: sequential prefill; n > 0: n fold segments overlapped with attention; < 0: automatic."""
    _check(lib.kvm_layer_set_overlap(layer, int(segments)), layer)


def kvm_layer_get_overlap(layer) -> int:
    """Fold segments of the layer's last prefill (0: it ran sequentially)."""
    n = ctypes.c_int32(0)
    _check(lib.kvm_layer_get_overlap(layer, ctypes.byref(n)), layer)
    return n.value


KVM_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def check_prefill_tensors(cfg: kvm_config, q, k, v, gate, n_tokens: int, out) -> None:
    """Raise ValueError unless q, k, v, out are contiguous [B, H, n_tokens, d] tensors
    of the config's dtype and gate a contiguous fp32 [B, H, n_tokens] tensor, all on
    the current CUDA device: the library reads and writes n_tokens rows through
    these pointers."""
    import torch
    io = torch.bfloat16 if cfg.dtype == KVM_BF16 else torch.float32
    n_tokens = int(n_tokens)
    shp = (cfg.batch, cfg.heads, n_tokens, cfg.head_dim)
    cur = torch.cuda.current_device() if torch.cuda.is_available() else None
    for name, t, want, dt in (("q", q, shp, io), ("k", k, shp, io), ("v", v, shp, io),
                              ("gate", gate, shp[:3], torch.float32), ("out", out, shp, io)):
        if t is None or not hasattr(t, "data_ptr"):
            raise ValueError(f"{name} must be a tensor")
        if tuple(t.shape) != want or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name}: expected contiguous {dt} {want}, got {t.dtype} "
                             f"{tuple(t.shape)}")
        if not t.is_cuda or t.device.index != cur:
            raise ValueError(f"{name} must be on the current CUDA device (cuda:{cur})")


def kvm_prefill_noalloc(cfg: kvm_config, q, k, v, gate, n_tokens: int, out, stream=None,
                        check: bool = True):
    """One-shot prefill with no allocation (scratch in the library's static device array).
    The tensors are checked first (check=False passes raw pointers through, for
    the library's own argument validation)."""
    if check:
        check_prefill_tensors(cfg, q, k, v, gate, n_tokens, out)
    st = lib.kvm_prefill_noalloc(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(gate),
                                 int(n_tokens), _ptr(out), _stream(stream))
    _check(st, None)


def kvm_backward_scratch_bytes(cfg: kvm_config, n_tokens: int) -> int:
    n = lib.kvm_backward_scratch_bytes(ctypes.byref(cfg), int(n_tokens))
    if n == 0:
        raise KvmError(KVM_ERR_INVALID_ARG, kvm_last_error(None))
    return n


def check_backward_tensors(cfg: kvm_config, q, k, v, gate, out, dout, n_tokens: int, dq, dk, dv, dgate,
                           scratch) -> None:
    """Raise ValueError unless the inputs are what check_prefill_tensors wants, dout is
    shaped like out, dq / dk / dv are contiguous fp32 [B, H, n_tokens, d], dgate contiguous
    fp32 [B, H, n_tokens] and scratch a contiguous tensor, all on the current CUDA device
    (the library reads and writes n_tokens rows through these pointers; it checks the
    scratch size itself)."""
    import torch
    check_prefill_tensors(cfg, q, k, v, gate, n_tokens, out)
    n_tokens = int(n_tokens)
    io = torch.bfloat16 if cfg.dtype == KVM_BF16 else torch.float32
    shp = (cfg.batch, cfg.heads, n_tokens, cfg.head_dim)
    cur = torch.cuda.current_device() if torch.cuda.is_available() else None
    for name, t, want, dt in (("dout", dout, shp, io), ("dq", dq, shp, torch.float32),
                              ("dk", dk, shp, torch.float32), ("dv", dv, shp, torch.float32),
                              ("dgate", dgate, shp[:3], torch.float32), ("scratch", scratch, None, None)):
        if t is None or not hasattr(t, "data_ptr"):
            raise ValueError(f"{name} must be a tensor")
        if not t.is_contiguous() or (want is not None and (tuple(t.shape) != want or t.dtype != dt)):
            raise ValueError(f"{name}: expected contiguous {dt} {want}, got {t.dtype} {tuple(t.shape)}")
        if not t.is_cuda or t.device.index != cur:
            raise ValueError(f"{name} must be on the current CUDA device (cuda:{cur})")


def kvm_prefill_backward(layer, q, k, v, gate, out, dout, record: kvm_debug | None, n_tokens: int,
                         dq, dk, dv, dgate, scratch, stream=None, cfg: kvm_config | None = None):
    """Backward of the layer's last prefill at its fold decisions (fp32 gradients).  With
    cfg (the layer's config) every tensor is checked first (check_backward_tensors).  The
    record's assign / kind arrays must hold [B, H, max_events, chunk] int32 each."""
    if cfg is not None:
        check_backward_tensors(cfg, q, k, v, gate, out, dout, n_tokens, dq, dk, dv, dgate, scratch)
    st = lib.kvm_prefill_backward(layer, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out), _ptr(dout),
                                  ctypes.byref(record) if record is not None else None, int(n_tokens),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dgate), _ptr(scratch),
                                  int(scratch.numel() * scratch.element_size()), _stream(stream))
    _check(st, layer)


def kvm_last_error(layer) -> str:
    return lib.kvm_last_error(layer).decode()


def kvm_layer_destroy(layer):
    lib.kvm_layer_destroy(layer)


# --------------------------------------------------------- convenience owner

def make_config(*, batch, heads, head_dim=64, rope_dims=32, rope_theta=10000.0, chunk=128,
                window=512, n_sinks=16, sched=KVM_SCHED_FIXED, max_slots=256, coef=4.0, expo=0.5,
                ln_eps=1e-5, dtype=KVM_BF16, max_tokens=8192, flags=0) -> kvm_config:
    return kvm_config(batch, heads, head_dim, rope_dims, rope_theta, chunk, window, n_sinks, sched,
                      max_slots, coef, expo, ln_eps, dtype, max_tokens, flags)


def state_spec(cfg: kvm_config) -> dict:
    """Shape and torch dtype of every state buffer of kvm_state_bufs (include/kvm.h)."""
    import torch
    B, H, M, d, L = cfg.batch, cfg.heads, cfg.max_slots, cfg.head_dim, cfg.window + cfg.chunk
    io = torch.bfloat16 if cfg.dtype == KVM_BF16 else torch.float32
    return dict(sum_k=((B, H, M, d), torch.float32), sum_v=((B, H, M, d), torch.float32),
                counts=((B, H, M), torch.int32), rho=((B, H, M), torch.float32),
                ring_k=((B, H, L, d), io), ring_v=((B, H, L, d), io), ring_g=((B, H, L), torch.float32))


def check_state_tensors(cfg: kvm_config, t: dict, require_cuda: bool = True) -> None:
    """Raise ValueError unless t holds every state buffer with the layer's shape and
    dtype, contiguous (and on a CUDA device): the library copies fixed byte counts
    from and to these pointers."""
    for name, (shape, dtype) in state_spec(cfg).items():
        x = t.get(name)
        if x is None or not hasattr(x, "data_ptr"):
            raise ValueError(f"state buffer {name!r} missing")
        if tuple(x.shape) != shape or x.dtype != dtype or not x.is_contiguous():
            raise ValueError(f"state buffer {name!r}: expected contiguous {dtype} {shape}, got "
                             f"{x.dtype} {tuple(x.shape)}")
        if require_cuda and not x.is_cuda:
            raise ValueError(f"state buffer {name!r} must be on a CUDA device")


class KvmLayer:
    """Owns one layer handle and its device workspace (a torch uint8 tensor)."""

    def __init__(self, cfg: kvm_config, device="cuda"):
        import torch
        self.cfg = cfg
        self.ws = torch.empty(kvm_workspace_bytes(cfg), dtype=torch.uint8, device=device)
        self.handle = kvm_layer_create(cfg, self.ws)
        self.io_dtype = torch.bfloat16 if cfg.dtype == KVM_BF16 else torch.float32

    def _io(self, t, shape, dtype=None):
        import torch
        dtype = dtype or self.io_dtype
        if t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != tuple(shape) or not t.is_cuda:
            raise ValueError(f"expected contiguous CUDA {dtype} tensor of shape {shape}, got "
                             f"{t.dtype} {tuple(t.shape)}")
        return t

    def prefill(self, q, k, v, gate, out=None, stream=None, dbg: kvm_debug | None = None):
        import torch
        c = self.cfg
        N = q.shape[2]
        shp = (c.batch, c.heads, N, c.head_dim)
        for t in (q, k, v):
            self._io(t, shp)
        self._io(gate, shp[:3], torch.float32)
        if out is None:
            out = torch.empty(shp, dtype=self.io_dtype, device=q.device)
        self._io(out, shp)
        kvm_prefill(self.handle, q, k, v, gate, N, out, stream, dbg)
        return out

    def prefill_backward(self, q, k, v, gate, out, dout, record: kvm_debug | None, stream=None):
        """Gradients (dq, dk, dv, dgate; fp32) of the last prefill of these inputs, at its
        fold decisions (record: the kvm_debug that prefill filled)."""
        import torch
        c = self.cfg
        N = q.shape[2]
        shp = (c.batch, c.heads, N, c.head_dim)
        for t in (q, k, v, out, dout):
            self._io(t, shp)
        self._io(gate, shp[:3], torch.float32)
        dev = q.device
        dq, dk, dv = (torch.empty(shp, dtype=torch.float32, device=dev) for _ in range(3))
        dg = torch.empty(shp[:3], dtype=torch.float32, device=dev)
        scratch = torch.empty(kvm_backward_scratch_bytes(c, N), dtype=torch.uint8, device=dev)
        kvm_prefill_backward(self.handle, q, k, v, gate, out, dout, record, N, dq, dk, dv, dg, scratch, stream,
                             cfg=c)
        return dq, dk, dv, dg

    def decode_step(self, q, k, v, gate, out=None, stream=None):
        import torch
        c = self.cfg
        shp = (c.batch, c.heads, c.head_dim)
        for t in (q, k, v):
            self._io(t, shp)
        self._io(gate, shp[:2], torch.float32)
        if out is None:
            out = torch.empty(shp, dtype=self.io_dtype, device=q.device)
        self._io(out, shp)
        kvm_decode_step(self.handle, q, k, v, gate, out, stream)
        return out

    def state_buffers(self, device="cuda"):
        """Fresh caller-owned tensors shaped for export/import."""
        import torch
        return {name: torch.zeros(shape, dtype=dtype, device=device)
                for name, (shape, dtype) in state_spec(self.cfg).items()}

    @staticmethod
    def _bufs(t, n_slots=0, n_overflow=0, pos=0) -> kvm_state_bufs:
        return kvm_state_bufs(t["sum_k"].data_ptr(), t["sum_v"].data_ptr(), t["counts"].data_ptr(),
                              t["rho"].data_ptr(), t["ring_k"].data_ptr(), t["ring_v"].data_ptr(),
                              t["ring_g"].data_ptr(), n_slots, n_overflow, pos)

    def export_state(self, stream=None):
        t = self.state_buffers(self.ws.device)
        check_state_tensors(self.cfg, t)
        b = self._bufs(t)
        kvm_state_export(self.handle, b, stream)
        t.update(n_slots=b.n_slots, n_overflow=b.n_overflow, pos=b.pos)
        return t

    def import_state(self, t, stream=None):
        check_state_tensors(self.cfg, t)
        b = self._bufs(t, t["n_slots"], t["n_overflow"], t["pos"])
        kvm_state_import(self.handle, b, stream)

    def forward(self, x, w_in, w_out, stream=None):
        """Whole-layer forward of x [B, N, d_model] bf16; returns y and the
        scratch views q, k, v, o [B, H, N, 64] bf16 and gate [B, H, N] fp32."""
        import torch
        c = self.cfg
        B, N, d_model = x.shape
        for t, shp in ((x, (c.batch, N, d_model)), (w_in, (3 * c.heads * 64 + c.heads, d_model)),
                       (w_out, (d_model, c.heads * 64))):
            self._io(t, shp, torch.bfloat16)
        nbytes = kvm_forward_scratch_bytes(c, d_model, N)
        scratch = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
        y = torch.empty((c.batch, N, d_model), dtype=torch.bfloat16, device=x.device)
        kvm_layer_forward(self.handle, d_model, x, w_in, w_out, N, y, scratch, stream)
        rows = c.batch * c.heads * N
        al = lambda n: (n + 255) // 256 * 256
        off, parts = 0, {}
        for name, nb in (("q", rows * 128), ("k", rows * 128), ("v", rows * 128), ("o", rows * 128),
                         ("gate", rows * 4)):
            parts[name] = scratch[off:off + nb]
            off = al(off + nb)
        shp = (c.batch, c.heads, N, 64)
        inter = {n: parts[n].view(torch.bfloat16).view(shp) for n in ("q", "k", "v", "o")}
        inter["gate"] = parts["gate"].view(torch.float32).view(c.batch, c.heads, N)
        return y, inter

    def sync(self):
        kvm_layer_sync(self.handle)

    def close(self):
        if getattr(self, "handle", None) is not None:
            kvm_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
