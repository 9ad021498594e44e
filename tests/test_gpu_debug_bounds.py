"""The bounds-checked build (-DMOE_DEBUG_BOUNDS, libmoe_fp8_debug.so).

Valid inputs give exactly the product library's outputs and no error bits. Bad
indices, which only this build may be given, are recorded (bit 0x80 of the
device error word) and their accesses skipped: a routed position far past the
permuted rows and a negative one in the combine; an expert id past E in the
permutation. The debug library runs in a subprocess of its own."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe
from routed_fp8_expert_gb300 import _lib

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ERR_BAD_INDEX = 0x80
HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounds_checked_build(tmp_path):
    out = tmp_path / "dbg.npz"
    r = subprocess.run([sys.executable, os.path.join(HERE, "_debug_bounds_run.py"), str(out)],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    res = np.load(out)
    for name, shape in (("toy", S.TOY), ("wide", S.MoEShape("dbg_wide", T=300, d=512, E=16, topk=4, H=256))):
        inp = S.gen_moe_inputs(shape, seed=5, device=DEV)
        y = moe.layer_forward(inp.x, inp.w_gate, inp.bias, inp.experts, moe.cfg_of(shape))
        torch.cuda.synchronize()
        assert np.array_equal(res[f"y_{name}"], y.float().cpu().numpy()), name
        assert tuple(res[f"err_{name}"]) == (_lib.MOE_OK, 0), name
    assert tuple(res["err_skip"]) == (_lib.MOE_OK, 0)
    assert tuple(res["err_bad_combine"]) == (_lib.MOE_ERR_INDEX, ERR_BAD_INDEX)
    assert bool(res["combine_same"])
    assert tuple(res["err_bad_id"]) == (_lib.MOE_ERR_INDEX, ERR_BAD_INDEX)
    assert int(res["bad_id_offsets_last"]) == S.TOY.T * S.TOY.topk - 1
