"""GB300 (sm_103a) large-chunk TTT-KVB layer and chunked linear attention.

Thin ctypes binding over the C ABI in ``include/ttt.h``: every step of the
computation runs in the library's CUDA kernels; this module only marshals
arguments (device pointers of torch tensors, the current CUDA stream) and
allocates outputs and workspace with torch.  There is no CPU fallback: if the
shared library is missing or cannot load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

APPLY_THEN_UPDATE = 0
BLOCK_CAUSAL = 1
BIDIRECTIONAL = 2
STRIDED = 3

TTT_F32 = 0
TTT_BF16 = 1

MUON_COEF = (3.4445, -4.7750, 2.0315)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libttt_gb300.so")

# Every symbol the public headers declare.
EXPORTED = (
    "ttt_status_string", "ttt_layer_workspace_size", "ttt_layer_forward",
    "linattn_workspace_size", "linattn_chunked_forward", "ttt_device_status",
    "ttt_set_wait_limit_ns", "ttt_selftest_gemm", "ttt_launch_count", "ttt_profile_start",
    "ttt_profile_stop", "linattn_chunked_forward_noalloc", "ttt_layer_host_workspace_size",
    "ttt_layer_forward_host", "ttt_selftest_withhold_release", "linattn_rule_workspace_size",
    "linattn_chunked_forward_rule",
)


class ProfileEntry(ctypes.Structure):
    """Mirror of ``ttt_profile_entry``."""
    _fields_ = [("name", ctypes.c_char * 32), ("kernel", ctypes.c_char * 32),
                ("launches", ctypes.c_int), ("ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double),
                ("sm_ms", ctypes.c_double)]


FORM_AUTO = 0
FORM_RECURRENT = 1
FORM_PARALLEL = 2


class UpdateRule(ctypes.Structure):
    """Mirror of ``ttt_update_rule``."""
    _fields_ = [("l2norm", ctypes.c_int), ("muon_steps", ctypes.c_int),
                ("momentum_beta", ctypes.c_float), ("ns_a", ctypes.c_float),
                ("ns_b", ctypes.c_float), ("ns_c", ctypes.c_float),
                ("last_layer_only", ctypes.c_int), ("inner_steps", ctypes.c_int),
                ("form", ctypes.c_int)]


class LinattnRule(ctypes.Structure):
    """Mirror of ``linattn_rule``."""
    _fields_ = [("alpha", ctypes.c_void_p), ("lr", ctypes.c_void_p), ("M0", ctypes.c_void_p),
                ("M_final", ctypes.c_void_p), ("muon_steps", ctypes.c_int),
                ("ns_a", ctypes.c_float), ("ns_b", ctypes.c_float), ("ns_c", ctypes.c_float)]


def update_rule(l2norm=True, muon_steps=0, momentum_beta=0.0, ns_coef=MUON_COEF,
                last_layer_only=False, inner_steps=1, form=FORM_AUTO) -> UpdateRule:
    a, b, c = ns_coef
    return UpdateRule(int(bool(l2norm)), int(muon_steps), float(momentum_beta),
                      float(a), float(b), float(c), int(bool(last_layer_only)),
                      int(inner_steps), int(form))


class TTTError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} (status {code})")
        self.code = code


_lib = None


def _declare(lib):
    vp, i, sz, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    lib.ttt_status_string.restype = ctypes.c_char_p
    lib.ttt_status_string.argtypes = [i]
    lib.ttt_layer_workspace_size.restype = sz
    lib.ttt_layer_workspace_size.argtypes = [i, i, i, i, i, i, i, i, ctypes.POINTER(UpdateRule)]
    lib.ttt_layer_forward.restype = i
    lib.ttt_layer_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i,
                                      vp, ctypes.POINTER(UpdateRule), vp, vp, vp, vp, vp, vp,
                                      sz, vp]
    lib.ttt_layer_host_workspace_size.restype = sz
    lib.ttt_layer_host_workspace_size.argtypes = [i, i, i, i, i, i, i, i,
                                                  ctypes.POINTER(UpdateRule), i]
    lib.ttt_layer_forward_host.restype = i
    lib.ttt_layer_forward_host.argtypes = lib.ttt_layer_forward.argtypes
    lib.linattn_workspace_size.restype = sz
    lib.linattn_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
    lib.linattn_chunked_forward.restype = i
    lib.linattn_chunked_forward.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, vp,
                                            vp, vp, vp, sz, vp]
    lib.linattn_rule_workspace_size.restype = sz
    lib.linattn_rule_workspace_size.argtypes = [i, i, i, i, i, i, i, i,
                                                ctypes.POINTER(LinattnRule)]
    lib.linattn_chunked_forward_rule.restype = i
    lib.linattn_chunked_forward_rule.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, vp,
                                                 ctypes.POINTER(LinattnRule), vp, vp, vp, sz, vp]
    lib.ttt_device_status.restype = i
    lib.ttt_device_status.argtypes = [vp]
    lib.ttt_set_wait_limit_ns.restype = None
    lib.ttt_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.ttt_selftest_gemm.restype = i
    lib.ttt_selftest_gemm.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, i, vp]
    lib.linattn_chunked_forward_noalloc.restype = i
    lib.linattn_chunked_forward_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i,
                                                    vp, vp, vp, vp]
    lib.ttt_selftest_withhold_release.restype = None
    lib.ttt_selftest_withhold_release.argtypes = [i]
    lib.ttt_launch_count.restype = ctypes.c_ulonglong
    lib.ttt_launch_count.argtypes = []
    lib.ttt_profile_start.restype = None
    lib.ttt_profile_start.argtypes = []
    lib.ttt_profile_stop.restype = i
    lib.ttt_profile_stop.argtypes = [ctypes.POINTER(ProfileEntry), i]
    return lib


def library():
    """Loads the shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library not built: {LIB_PATH} is missing "
                "(run chunked_linear_attention_gb300._build.build())")
        _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def status_string(code: int) -> str:
    return library().ttt_status_string(int(code)).decode()


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the CUDA path must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _io_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return TTT_BF16
    if t.dtype == torch.float32:
        return TTT_F32
    raise ValueError(f"unsupported I/O dtype {t.dtype}")


def _flags(update_chunks, n_chunks):
    if update_chunks is None:
        return None, None
    if len(update_chunks) != n_chunks:
        raise ValueError(f"update_chunks needs {n_chunks} flags, got {len(update_chunks)}")
    arr = (ctypes.c_ubyte * n_chunks)(*[1 if x else 0 for x in update_chunks])
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise TTTError(rc, what)


def layer_workspace_size(B, H, N, d_h, m_h, chunk, io_dtype, mask_mode, rule: UpdateRule) -> int:
    return library().ttt_layer_workspace_size(B, H, N, d_h, m_h, chunk, io_dtype, mask_mode,
                                              ctypes.byref(rule))


def ttt_layer_forward(q, k, v, eta, W1, W2, W3, chunk: int, mask_mode: int,
                      rule: Optional[UpdateRule] = None,
                      update_chunks: Optional[Sequence[int]] = None,
                      momentum: Optional[torch.Tensor] = None,
                      out: Optional[torch.Tensor] = None,
                      W_final: Optional[Sequence[torch.Tensor]] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None):
    """LaCT TTT layer forward (see ``ttt_layer_forward`` in include/ttt.h).

    q, k, v: [B, H, N, d] CUDA tensors (bf16 or fp32); eta [B, H, N] fp32;
    W1, W3 [H, m, d] or [B, H, m, d]; W2 [H, d, m] or [B, H, d, m], fp32.
    Returns (out, W1_final, W2_final, W3_final).  Asynchronous on the current
    stream (or ``stream``).
    """
    lib = library()
    rule = update_rule() if rule is None else rule
    B, H, N, d = q.shape
    m = W1.shape[-2]
    io = _io_dtype(q)
    w_per_batch = 1 if W1.dim() == 4 else 0
    dev = q.device
    if out is None:
        out = torch.empty_like(q)
    if W_final is None:
        W_final = (torch.empty((B, H, m, d), device=dev, dtype=torch.float32),
                   torch.empty((B, H, d, m), device=dev, dtype=torch.float32),
                   torch.empty((B, H, m, d), device=dev, dtype=torch.float32))
    ws_bytes = lib.ttt_layer_workspace_size(B, H, N, d, m, chunk, io, mask_mode, ctypes.byref(rule))
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    keep, fl = _flags(update_chunks, N // chunk if chunk > 0 else 0)
    rc = lib.ttt_layer_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(eta), _ptr(W1), _ptr(W2), _ptr(W3),
                               w_per_batch, B, H, N, d, m, chunk, io, mask_mode, fl,
                               ctypes.byref(rule), _ptr(out), _ptr(W_final[0]), _ptr(W_final[1]),
                               _ptr(W_final[2]), _ptr(momentum), _ptr(workspace),
                               0 if workspace is None else workspace.numel(), _stream(stream))
    del keep
    _check(rc, "ttt_layer_forward")
    return out, W_final[0], W_final[1], W_final[2]


def _hptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("tensors passed to the host-buffer call must be in host memory")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    if not t.is_pinned():
        raise ValueError("host tensors must be page-locked (tensor.pin_memory())")
    return ctypes.c_void_p(t.data_ptr())


def layer_host_workspace_size(B, H, N, d_h, m_h, chunk, io_dtype, mask_mode, rule: UpdateRule,
                              w_per_batch: int = 0) -> int:
    return library().ttt_layer_host_workspace_size(B, H, N, d_h, m_h, chunk, io_dtype, mask_mode,
                                                   ctypes.byref(rule), int(w_per_batch))


def ttt_layer_forward_host(q, k, v, eta, W1, W2, W3, chunk: int, mask_mode: int,
                           rule: Optional[UpdateRule] = None,
                           update_chunks: Optional[Sequence[int]] = None,
                           momentum: Optional[torch.Tensor] = None,
                           out: Optional[torch.Tensor] = None,
                           W_final: Optional[Sequence[torch.Tensor]] = None,
                           workspace: Optional[torch.Tensor] = None, stream=None, device=None):
    """LaCT TTT layer forward on page-locked HOST tensors (see
    ``ttt_layer_forward_host`` in include/ttt.h): the same shapes as
    ``ttt_layer_forward``; chunk transfers overlap the kernels.  ``workspace``
    (a CUDA uint8 tensor) and ``stream`` select the device (else ``device`` or
    the current one).  Returns (out, W1_final, W2_final, W3_final) host
    tensors, complete once ``stream`` reaches this point.
    """
    lib = library()
    rule = update_rule() if rule is None else rule
    B, H, N, d = q.shape
    m = W1.shape[-2]
    io = _io_dtype(q)
    w_per_batch = 1 if W1.dim() == 4 else 0
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if W_final is None:
        W_final = (torch.empty((B, H, m, d), dtype=torch.float32, pin_memory=True),
                   torch.empty((B, H, d, m), dtype=torch.float32, pin_memory=True),
                   torch.empty((B, H, m, d), dtype=torch.float32, pin_memory=True))
    dev = workspace.device if workspace is not None else torch.device(
        "cuda", torch.cuda.current_device() if device is None else torch.device(device).index)
    ws_bytes = lib.ttt_layer_host_workspace_size(B, H, N, d, m, chunk, io, mask_mode,
                                                 ctypes.byref(rule), w_per_batch)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    keep, fl = _flags(update_chunks, N // chunk if chunk > 0 else 0)
    with torch.cuda.device(dev):
        rc = lib.ttt_layer_forward_host(
            _hptr(q), _hptr(k), _hptr(v), _hptr(eta), _hptr(W1), _hptr(W2), _hptr(W3),
            w_per_batch, B, H, N, d, m, chunk, io, mask_mode, fl, ctypes.byref(rule), _hptr(out),
            _hptr(W_final[0]), _hptr(W_final[1]), _hptr(W_final[2]), _hptr(momentum),
            _ptr(workspace), 0 if workspace is None else workspace.numel(), _stream(stream))
    del keep
    _check(rc, "ttt_layer_forward_host")
    return out, W_final[0], W_final[1], W_final[2]


def linattn_workspace_size(B, H, N, d_k, d_v, chunk, io_dtype, mask_mode) -> int:
    return library().linattn_workspace_size(B, H, N, d_k, d_v, chunk, io_dtype, mask_mode)


def linattn_chunked_forward(q, k, v, eta, chunk: int, mask_mode: int,
                            S0: Optional[torch.Tensor] = None,
                            update_chunks: Optional[Sequence[int]] = None,
                            out: Optional[torch.Tensor] = None,
                            S_final: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None, stream=None):
    """Chunked linear attention (see ``linattn_chunked_forward`` in include/ttt.h).

    Returns (out [B, H, N, d_v], S_final [B, H, d_v, d_k] fp32).
    """
    lib = library()
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    io = _io_dtype(q)
    dev = q.device
    if out is None:
        out = torch.empty((B, H, N, dv), device=dev, dtype=q.dtype)
    if S_final is None:
        S_final = torch.empty((B, H, dv, dk), device=dev, dtype=torch.float32)
    ws_bytes = lib.linattn_workspace_size(B, H, N, dk, dv, chunk, io, mask_mode)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    keep, fl = _flags(update_chunks, N // chunk if chunk > 0 else 0)
    rc = lib.linattn_chunked_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(eta), _ptr(S0), B, H, N, dk,
                                     dv, chunk, io, mask_mode, fl, _ptr(out), _ptr(S_final),
                                     _ptr(workspace), 0 if workspace is None else workspace.numel(),
                                     _stream(stream))
    del keep
    _check(rc, "linattn_chunked_forward")
    return out, S_final


def linattn_rule(alpha=None, lr=None, M0=None, M_final=None, muon_steps=0,
                 ns_coef=MUON_COEF) -> LinattnRule:
    """The ``linattn_rule`` struct from CUDA tensors (or None)."""
    a, b, c = ns_coef
    return LinattnRule(_ptr(alpha), _ptr(lr), _ptr(M0), _ptr(M_final), int(muon_steps),
                       float(a), float(b), float(c))


def linattn_chunked_forward_rule(q, k, v, eta, chunk: int, mask_mode: int,
                                 S0: Optional[torch.Tensor] = None,
                                 update_chunks: Optional[Sequence[int]] = None,
                                 alpha: Optional[torch.Tensor] = None,
                                 lr: Optional[torch.Tensor] = None,
                                 M0: Optional[torch.Tensor] = None,
                                 M_final=None, muon_steps: int = 0, ns_coef=MUON_COEF,
                                 out: Optional[torch.Tensor] = None,
                                 S_final: Optional[torch.Tensor] = None,
                                 workspace: Optional[torch.Tensor] = None, stream=None):
    """Chunked linear attention with momentum, per-chunk learning rates and
    Muon of the momentum (see ``linattn_chunked_forward_rule`` in
    include/ttt.h).  alpha, lr: [B, H, N / chunk] fp32 CUDA tensors or None;
    M0 [B, H, d_v, d_k] or None; M_final: a tensor to write, True to allocate
    one, or None.  Returns (out, S_final, M_final or None)."""
    lib = library()
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    io = _io_dtype(q)
    dev = q.device
    if out is None:
        out = torch.empty((B, H, N, dv), device=dev, dtype=q.dtype)
    if S_final is None:
        S_final = torch.empty((B, H, dv, dk), device=dev, dtype=torch.float32)
    if M_final is True:
        M_final = torch.empty((B, H, dv, dk), device=dev, dtype=torch.float32)
    rule = linattn_rule(alpha, lr, M0, M_final, muon_steps, ns_coef)
    ws_bytes = lib.linattn_rule_workspace_size(B, H, N, dk, dv, chunk, io, mask_mode,
                                               ctypes.byref(rule))
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    keep, fl = _flags(update_chunks, N // chunk if chunk > 0 else 0)
    rc = lib.linattn_chunked_forward_rule(_ptr(q), _ptr(k), _ptr(v), _ptr(eta), _ptr(S0), B, H,
                                          N, dk, dv, chunk, io, mask_mode, fl, ctypes.byref(rule),
                                          _ptr(out), _ptr(S_final), _ptr(workspace),
                                          0 if workspace is None else workspace.numel(),
                                          _stream(stream))
    del keep
    _check(rc, "linattn_chunked_forward_rule")
    return out, S_final, M_final


def linattn_chunked_forward_noalloc(q, k, v, eta, chunk: int, mask_mode: int,
                                    S0: Optional[torch.Tensor] = None,
                                    update_chunks: Optional[Sequence[int]] = None,
                                    out: Optional[torch.Tensor] = None,
                                    S_final: Optional[torch.Tensor] = None, stream=None):
    """Chunked linear attention whose scratch is the library's fixed 16 MiB
    device array instead of a workspace (see
    ``linattn_chunked_forward_noalloc`` in include/ttt.h).  Output tensors are
    still the caller's (allocated here with torch when not given)."""
    lib = library()
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if out is None:
        out = torch.empty((B, H, N, dv), device=dev, dtype=q.dtype)
    if S_final is None:
        S_final = torch.empty((B, H, dv, dk), device=dev, dtype=torch.float32)
    keep, fl = _flags(update_chunks, N // chunk if chunk > 0 else 0)
    # the library looks up its scratch array on the CURRENT device: make it
    # the tensors' device for the call
    with torch.cuda.device(dev):
        rc = lib.linattn_chunked_forward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(eta), _ptr(S0),
                                                 B, H, N, dk, dv, chunk, _io_dtype(q), mask_mode,
                                                 fl, _ptr(out), _ptr(S_final),
                                                 _stream(stream))
    del keep
    _check(rc, "linattn_chunked_forward_noalloc")
    return out, S_final


def device_status(stream=None) -> int:
    """Synchronises the stream; returns and clears the device status word."""
    return library().ttt_device_status(_stream(stream))


def launch_count() -> int:
    """Kernels the library has launched in this process."""
    return int(library().ttt_launch_count())


def profile_start():
    library().ttt_profile_start()


def profile_stop():
    """Per launch kind: dict(name, kernel, launches, ms, flops, bytes, sm_ms)."""
    arr = (ProfileEntry * 32)()
    n = library().ttt_profile_stop(arr, 32)
    if n < 0:
        raise TTTError(n, "ttt_profile_stop")
    return [dict(name=e.name.decode(), kernel=e.kernel.decode(), launches=e.launches, ms=e.ms,
                 flops=e.flops, bytes=e.bytes, sm_ms=e.sm_ms) for e in arr[:n]]


def set_wait_limit_ns(ns: int):
    library().ttt_set_wait_limit_ns(int(ns))


def selftest_withhold_release(bh: int):
    """Test hook: from the next linear-attention call on, batch-head ``bh``'s
    state items never report completion, so the items waiting for them run
    into their bounded waits (-1 turns it off).  See include/ttt_selftest.h."""
    library().ttt_selftest_withhold_release(int(bh))


def selftest_gemm(A, B, a_mn_major: bool, b_mn_major: bool, tile_n: int = 128, stream=None):
    """fp32 D = A * B through the library's GEMM building block (self-test).

    A: [Z, M, K] (or [Z, K, M] when a_mn_major); B: [Z, N, K] (or [Z, K, N]).
    """
    lib = library()
    Z = A.shape[0]
    if a_mn_major:
        K, M = A.shape[1], A.shape[2]
    else:
        M, K = A.shape[1], A.shape[2]
    N = B.shape[2] if b_mn_major else B.shape[1]
    D = torch.empty((Z, M, N), device=A.device, dtype=torch.float32)
    rc = lib.ttt_selftest_gemm(_ptr(A), _ptr(B), _ptr(D), Z, M, N, K, int(a_mn_major),
                               int(b_mn_major), _io_dtype(A), tile_n, _stream(stream))
    _check(rc, "ttt_selftest_gemm")
    return D
