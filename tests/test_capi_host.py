"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every symbol the public headers declare, and rejects bad
arguments on the host with the documented status codes before touching the
device."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

TTT_OK, TTT_ERR_NULL, TTT_ERR_SHAPE, TTT_ERR_ALIGN = 0, -1, -2, -3
TTT_ERR_UNSUPPORTED, TTT_ERR_WORKSPACE, TTT_ERR_CUDA, TTT_ERR_ARG = -4, -5, -6, -8
TTT_ERR_PAGEABLE = -9


@pytest.fixture(scope="module")
def cla():
    from chunked_linear_attention_gb300 import _build
    _build.build()
    import chunked_linear_attention_gb300 as m
    m.library()
    return m


def header_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M):
            if m.group(1) not in ("if", "typedef"):
                names.append(m.group(1))
    return sorted(set(names))


def test_exports_every_declared_symbol(cla):
    names = header_functions()
    assert "ttt_layer_forward" in names and "linattn_chunked_forward" in names
    lib = ctypes.CDLL(cla.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(names) == set(cla.EXPORTED)


def test_status_strings(cla):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, -9):
        s = cla.status_string(code)
        assert s and s != "unknown status"
    assert cla.status_string(12345) == "unknown status"


def fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def call_layer(cla, B=1, H=1, N=256, d=64, m=64, chunk=128, io=1, mode=0, flags=None,
               rule=None, ws_bytes=None, nulls=(), align_off=0, w_per_batch=0):
    lib = cla.library()
    rule = cla.update_rule() if rule is None else rule
    need = lib.ttt_layer_workspace_size(B, H, N, d, m, chunk, io, mode, ctypes.byref(rule))
    ws = need if ws_bytes is None else ws_bytes
    ptrs = [fake(0x100000 * (i + 1) + (align_off if i == 0 else 0)) for i in range(12)]
    for i in nulls:
        ptrs[i] = None
    q, k, v, eta, W1, W2, W3, out, F1, F2, F3, ws_ptr = ptrs
    return lib.ttt_layer_forward(q, k, v, eta, W1, W2, W3, w_per_batch, B, H, N, d, m, chunk, io,
                                 mode, flags, ctypes.byref(rule), out, F1, F2, F3, None, ws_ptr,
                                 ws, None)


def test_layer_rejects_bad_arguments(cla):
    assert call_layer(cla, nulls=(0,)) == TTT_ERR_NULL
    assert call_layer(cla, nulls=(8,)) == TTT_ERR_NULL
    assert call_layer(cla, N=300, chunk=128) == TTT_ERR_SHAPE
    assert call_layer(cla, B=0) == TTT_ERR_SHAPE
    assert call_layer(cla, mode=2, N=256, chunk=128) == TTT_ERR_SHAPE   # bidirectional: one chunk
    assert call_layer(cla, mode=7) == TTT_ERR_ARG
    assert call_layer(cla, io=5) == TTT_ERR_ARG
    assert call_layer(cla, mode=3, flags=None) == TTT_ERR_NULL          # strided needs flags
    assert call_layer(cla, d=100) == TTT_ERR_UNSUPPORTED                # bf16 needs multiples of 64
    assert call_layer(cla, chunk=64, N=256) == TTT_ERR_UNSUPPORTED      # bf16 chunk multiple of 128
    assert call_layer(cla, d=2048, m=64) == TTT_ERR_UNSUPPORTED
    assert call_layer(cla, align_off=8) == TTT_ERR_ALIGN
    assert call_layer(cla, ws_bytes=16) == TTT_ERR_WORKSPACE
    assert call_layer(cla, nulls=(11,)) == TTT_ERR_WORKSPACE
    assert call_layer(cla, w_per_batch=3) == TTT_ERR_ARG
    bad = cla.update_rule(muon_steps=-1)
    assert call_layer(cla, rule=bad) == TTT_ERR_ARG
    bad = cla.update_rule(momentum_beta=float("nan"))
    assert call_layer(cla, rule=bad) == TTT_ERR_ARG


def test_workspace_sizes(cla):
    lib = cla.library()
    r0 = cla.update_rule()
    r1 = cla.update_rule(muon_steps=5, momentum_beta=0.9)
    a = lib.ttt_layer_workspace_size(2, 4, 32768, 384, 384, 2048, 1, 0, ctypes.byref(r0))
    b = lib.ttt_layer_workspace_size(2, 4, 32768, 384, 384, 2048, 1, 0, ctypes.byref(r1))
    assert 0 < a < b
    assert lib.ttt_layer_workspace_size(2, 4, 1000, 384, 384, 2048, 1, 0, ctypes.byref(r0)) == 0
    assert lib.linattn_workspace_size(4, 4, 8192, 128, 128, 2048, 1, 1) > 0
    assert lib.linattn_workspace_size(4, 4, 8192, 100, 128, 2048, 1, 1) == 0


def test_linattn_rejects_bad_arguments(cla):
    lib = cla.library()

    def call(N=1024, dk=128, dv=128, chunk=256, io=1, mode=1, flags=None, nulls=(), ws=None):
        need = lib.linattn_workspace_size(1, 1, N, dk, dv, chunk, io, mode)
        ptrs = [fake(0x100000 * (i + 1)) for i in range(8)]
        for i in nulls:
            ptrs[i] = None
        q, k, v, eta, S0, out, Sf, wsp = ptrs
        return lib.linattn_chunked_forward(q, k, v, eta, S0, 1, 1, N, dk, dv, chunk, io, mode,
                                           flags, out, Sf, wsp, need if ws is None else ws, None)

    assert call(nulls=(0,)) == TTT_ERR_NULL
    assert call(N=1000) == TTT_ERR_SHAPE
    assert call(dk=96) == TTT_ERR_UNSUPPORTED
    assert call(mode=3) == TTT_ERR_NULL
    assert call(ws=8) == TTT_ERR_WORKSPACE


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_reports_cuda_error(cla):
    # arguments are valid, so the call reaches the runtime, which finds no GPU
    assert call_layer(cla) == TTT_ERR_CUDA


def test_binding_refuses_cpu_tensors(cla):
    q = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16)
    eta = torch.zeros(1, 1, 256)
    W1 = torch.zeros(1, 64, 64)
    with pytest.raises((ValueError, RuntimeError)):
        cla.ttt_layer_forward(q, q, q, eta, W1, W1, W1, 128, cla.APPLY_THEN_UPDATE,
                              W_final=(W1, W1, W1), workspace=torch.zeros(16, dtype=torch.uint8))


def call_layer_host(cla, B=1, H=1, N=256, d=64, m=64, chunk=128, io=1, mode=0, flags=None,
                    nulls=(), ws_bytes=None, w_per_batch=0):
    lib = cla.library()
    rule = cla.update_rule()
    need = lib.ttt_layer_host_workspace_size(B, H, N, d, m, chunk, io, mode, ctypes.byref(rule),
                                             w_per_batch)
    ptrs = [fake(0x100000 * (i + 1)) for i in range(12)]
    for i in nulls:
        ptrs[i] = None
    q, k, v, eta, W1, W2, W3, out, F1, F2, F3, ws_ptr = ptrs
    return lib.ttt_layer_forward_host(q, k, v, eta, W1, W2, W3, w_per_batch, B, H, N, d, m, chunk,
                                      io, mode, flags, ctypes.byref(rule), out, F1, F2, F3, None,
                                      ws_ptr, need if ws_bytes is None else ws_bytes, None)


def test_layer_host_call_checks_arguments_and_page_locking(cla):
    assert call_layer_host(cla, nulls=(0,)) == TTT_ERR_NULL
    assert call_layer_host(cla, N=300) == TTT_ERR_SHAPE
    assert call_layer_host(cla, d=100) == TTT_ERR_UNSUPPORTED
    assert call_layer_host(cla, w_per_batch=2) == TTT_ERR_ARG
    assert call_layer_host(cla, mode=3) == TTT_ERR_NULL
    # valid sizes, but these host addresses are not page-locked allocations
    assert call_layer_host(cla) == TTT_ERR_PAGEABLE


def test_layer_host_workspace_adds_device_staging(cla):
    lib = cla.library()
    r = cla.update_rule(muon_steps=5, momentum_beta=0.9)
    B, H, N, d, m = 2, 4, 4096, 384, 384
    dev = lib.ttt_layer_workspace_size(B, H, N, d, m, 2048, 1, 0, ctypes.byref(r))
    host = lib.ttt_layer_host_workspace_size(B, H, N, d, m, 2048, 1, 0, ctypes.byref(r), 0)
    act = B * H * N * d * 2
    # q, k, v and out staging at least
    assert host >= dev + 4 * act
    assert lib.ttt_layer_host_workspace_size(B, H, N, d, m, 2048, 1, 0, ctypes.byref(r), 5) == 0


def test_host_binding_refuses_device_or_pageable_tensors(cla):
    q = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16)
    eta = torch.zeros(1, 1, 256)
    W1 = torch.zeros(1, 64, 64)
    with pytest.raises((ValueError, RuntimeError)):
        cla.ttt_layer_forward_host(q, q, q, eta, W1, W1, W1, 128, cla.APPLY_THEN_UPDATE,
                                   out=q, W_final=(W1, W1, W1),
                                   workspace=torch.zeros(16, dtype=torch.uint8))
