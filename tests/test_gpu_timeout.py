"""A bounded wait that runs out, on the GPU, without a fault.

Every wait in the kernels gives up after a limit (ttt_set_wait_limit_ns),
records TTT_ERR_TIMEOUT in the device status word and lets the kernel end.
Here the one-launch linear-attention kernel is told (test hook) that one
batch-head's partial-state items never report completion; the items waiting
for them give up after 1 ms, before issuing any copy.  The host then reads
TTT_ERR_TIMEOUT, and the next regular call on the same context matches the
oracle.
"""
import dataclasses

import pytest
import torch

import workloads as W
from oracle import ttt_oracle as O
from tests.gpu_util import assert_status_ok, f64, lib, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TTT_ERR_TIMEOUT = -7


def test_withheld_release_times_out_and_next_call_is_correct():
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=1, H=2, N=1024, chunk=256)
    q, k, v, eta, _ = [t.to(DEV) if t is not None else None for t in W.linattn_inputs(wl)]
    assert_status_ok(cla)
    cla.set_wait_limit_ns(1_000_000)
    cla.selftest_withhold_release(1)
    try:
        cla.linattn_chunked_forward(q, k, v, eta, wl.chunk, wl.mode)
        status = cla.device_status()
    finally:
        cla.selftest_withhold_release(-1)
        cla.set_wait_limit_ns(200_000_000)
    assert status == TTT_ERR_TIMEOUT
    assert cla.device_status() == 0          # read and cleared
    o, S = cla.linattn_chunked_forward(q, k, v, eta, wl.chunk, wl.mode)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    ro, rS = O.linattn_chunked_forward(f64(q), f64(k), f64(v), f64(eta), None, wl.chunk, wl.mode)
    assert rel_l2(f64(o), ro) <= 2e-2
    assert rel_l2(f64(S), rS) <= 2e-2
