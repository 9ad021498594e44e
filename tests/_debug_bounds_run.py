"""Run in a subprocess by test_gpu_debug_bounds.py: the bounds-checked library
(libmoe_fp8_debug.so) alone in this process. Writes its results to argv[1] (npz)."""
import ctypes
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import moe_synth as S  # noqa: E402
import routed_fp8_expert_gb300._lib as L  # noqa: E402
from routed_fp8_expert_gb300 import build  # noqa: E402

L.LIB_PATH = build.build(debug_bounds=True)
import routed_fp8_expert_gb300 as moe  # noqa: E402

DEV = "cuda:0"


def error_word():
    detail = ctypes.c_uint32(0)
    st = moe.load().moe_check_device_error(ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream),
                                           ctypes.byref(detail))
    return st, detail.value


def main(out_path):
    res = {}
    # valid inputs: the toy layer and the wide toy layer, no error bits
    for name, shape in (("toy", S.TOY), ("wide", S.MoEShape("dbg_wide", T=300, d=512, E=16, topk=4, H=256))):
        inp = S.gen_moe_inputs(shape, seed=5, device=DEV)
        y = moe.layer_forward(inp.x, inp.w_gate, inp.bias, inp.experts, moe.cfg_of(shape))
        torch.cuda.synchronize()
        res[f"y_{name}"] = y.float().cpu().numpy()
        res[f"err_{name}"] = np.array(error_word())
    # a bad routed position in the combine: recorded, and the slot skipped
    shape = S.TOY
    cfg = moe.cfg_of(shape)
    T, k, d = shape.T, shape.topk, shape.d
    R = (k + shape.n_shared) * T
    g = torch.Generator(device=DEV).manual_seed(9)
    o = torch.randn((R, d), generator=g, device=DEV).to(torch.bfloat16)
    w = torch.rand((T, k), generator=g, device=DEV)
    inv = torch.arange(T * k, device=DEV, dtype=torch.int32).view(T, k)
    bad = inv.clone()
    bad[3, 2] = 100_000_000
    bad[7, 0] = -5
    skip = inv.clone()
    skip[3, 2] = -1
    skip[7, 0] = -1
    y_skip = moe.combine(o, w, skip, cfg, T)
    torch.cuda.synchronize()
    res["err_skip"] = np.array(error_word())
    y_bad = moe.combine(o, w, bad, cfg, T)
    torch.cuda.synchronize()
    res["err_bad_combine"] = np.array(error_word())
    res["combine_same"] = np.array(bool(torch.equal(y_bad, y_skip)))
    # an expert id past E in the permutation: recorded, the assignment ignored
    idx = torch.stack([torch.randperm(shape.E, generator=torch.Generator().manual_seed(t))[:k]
                       for t in range(T)]).to(torch.int32).to(DEV)
    xq, sx = moe.quant_fp8_1x128(torch.randn((T, d), device=DEV))
    torch.cuda.synchronize()
    error_word()
    bad_idx = idx.clone()
    bad_idx[5, 1] = shape.E + 5
    out = moe.permute(bad_idx, xq, sx, cfg)
    torch.cuda.synchronize()
    res["err_bad_id"] = np.array(error_word())
    res["bad_id_offsets_last"] = np.array(int(out[0][-1].item()))
    np.savez(out_path, **res)


if __name__ == "__main__":
    main(sys.argv[1])
