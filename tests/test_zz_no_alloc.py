"""The allocation-free linear-attention entry point against the regular one.

linattn_chunked_forward_noalloc serves callers that cannot call cudaMalloc
(and so cannot provide a workspace): its scratch is a fixed 16 MiB device
array inside the library.  This file runs last so that a failure here, in a
run that stops at the first failure, comes after every other test.
"""
import ctypes

import pytest
import torch

import workloads as W
from tests.gpu_util import assert_status_ok, f64, lib, rel_l2

pytestmark = pytest.mark.gpu

BF16_REL_L2 = 2e-2
DEV = "cuda:0"


def _raw_call(cla, q, k, v, eta, wl, out, S):
    """One call straight through the C ABI (ctypes), on the current stream."""
    c = cla.library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return c.linattn_chunked_forward_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(eta.data_ptr()), None, wl.B, wl.H, wl.N,
        wl.d_k, wl.d_v, wl.chunk, cla.TTT_BF16, wl.mode, None, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(S.data_ptr()), stream)


def test_noalloc_matches_workspace_call_twice():
    cla = lib()
    cases = [
        W.LinattnWorkload("noalloc-a", B=2, H=2, N=2048, d_k=128, d_v=128, chunk=512,
                          mode=W.BLOCK_CAUSAL, seed=3),
        W.LinattnWorkload("noalloc-b", B=1, H=4, N=1024, d_k=128, d_v=64, chunk=256,
                          mode=W.APPLY_THEN_UPDATE, seed=4),
    ]
    for wl in cases:   # two calls in a row, the second on stale scratch
        need = cla.linattn_workspace_size(wl.B, wl.H, wl.N, wl.d_k, wl.d_v, wl.chunk,
                                          cla.TTT_BF16, wl.mode)
        assert 0 < need <= 16 << 20
        q, k, v, eta, _ = [t.to(DEV) if t is not None else None for t in W.linattn_inputs(wl)]
        ref_o, ref_S = cla.linattn_chunked_forward(q, k, v, eta, wl.chunk, wl.mode)
        out = torch.empty_like(ref_o)
        S = torch.empty_like(ref_S)
        rc = _raw_call(cla, q, k, v, eta, wl, out, S)
        assert rc == 0, cla.status_string(rc)
        torch.cuda.synchronize()
        assert_status_ok(cla)
        assert rel_l2(f64(out), f64(ref_o)) <= BF16_REL_L2
        assert rel_l2(f64(S), f64(ref_S)) <= BF16_REL_L2


def test_noalloc_rejects_problems_beyond_its_scratch():
    cla = lib()
    wl = W.LINATTN_C2   # needs ~69 MB of scratch, more than the 16 MiB array
    need = cla.linattn_workspace_size(wl.B, wl.H, wl.N, wl.d_k, wl.d_v, wl.chunk, cla.TTT_BF16,
                                      wl.mode)
    assert need > 16 << 20
    q = torch.zeros((wl.B, wl.H, wl.N, wl.d_k), device=DEV, dtype=torch.bfloat16)
    eta = torch.zeros((wl.B, wl.H, wl.N), device=DEV)
    out = torch.empty_like(q)
    S = torch.empty((wl.B, wl.H, wl.d_v, wl.d_k), device=DEV)
    assert _raw_call(cla, q, q, q, eta, wl, out, S) == -5   # TTT_ERR_WORKSPACE
