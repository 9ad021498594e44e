"""The kernels' bounded waits give up, report and leave the context usable.

moe_test_wait_timeout runs the grouped GEMMs' own wait routine on a barrier that
nothing completes: one warp with a 1 ms limit, one with the kernels' usual 1 s.
The first gives up and records its bit; the second must leave on the CTA's abort
word (well before its own second). The device error word reads MOE_ERR_TIMEOUT
with that bit once, then MOE_OK; a layer run afterwards is unchanged.
"""
import ctypes
import time

import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe
from routed_fp8_expert_gb300 import _lib

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ERR_WAIT_SELFTEST = 0x40


def _error_word():
    lib = moe.load()
    detail = ctypes.c_uint32(0)
    st = lib.moe_check_device_error(ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream),
                                    ctypes.byref(detail))
    return st, detail.value


def _toy_layer():
    inp = S.gen_moe_inputs(S.TOY, seed=3, device="cpu")
    return moe.layer_forward(inp.x.to(DEV), inp.w_gate.to(DEV), inp.bias.to(DEV), inp.experts.to(DEV),
                             moe.cfg_of(S.TOY))


def test_bounded_wait_gives_up_reports_and_recovers():
    y0 = _toy_layer()
    torch.cuda.synchronize()
    assert _error_word() == (_lib.MOE_OK, 0)
    t0 = time.perf_counter()
    moe.test_wait_timeout(1_000_000, DEV)           # 1 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert dt < 0.5, f"the self-test took {dt:.3f} s: the second warp did not leave on the abort word"
    assert _error_word() == (_lib.MOE_ERR_TIMEOUT, ERR_WAIT_SELFTEST)
    assert b"bounded wait" in moe.load().moe_last_error_string()
    assert _error_word() == (_lib.MOE_OK, 0)         # read and cleared
    y1 = _toy_layer()
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    assert _error_word() == (_lib.MOE_OK, 0)


def test_wait_limit_out_of_range_is_rejected():
    lib = moe.load()
    st = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    assert lib.moe_test_wait_timeout(999, st) == _lib.MOE_ERR_ARG
    assert lib.moe_test_wait_timeout(2_000_000_000, st) == _lib.MOE_ERR_ARG
    assert lib.moe_last_launch_count() == 0
