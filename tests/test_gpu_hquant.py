"""The fused gate/up epilogue's own outputs against the oracle: the 1x128 scales of
h = silu(g) * u and its e4m3 codes.

The GPU forms h in fp32 from fp32 accumulators; the oracle forms it in fp64 and
rounds to fp32. Both then quantise in fp32 (amax / 448, IEEE division, nearest-even
e4m3). So the scales agree to the fp32 rounding of h, and a code may differ only
where h / s lies next to an e4m3 rounding midpoint; everywhere else the codes must
be identical. Both the swap-AB kernel (about 9 rows per expert) and the token-major
256-row kernel (about 100 rows per expert, several 128-token tiles) are covered,
with all-zero token rows, whose groups quantise to scale 0 and codes 0.
"""
import numpy as np
import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe
from oracle import moe_oracle as O
from _hmargin import clear_of_midpoint, quotients

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

def _run(shape, seed, zero_tokens=()):
    inp = S.gen_moe_inputs(shape, seed=seed)
    x = inp.x.clone()
    x[list(zero_tokens)] = 0
    cfg = moe.cfg_of(shape)
    T, k = shape.T, shape.topk
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(shape.E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ex = inp.experts.to(DEV)
    xq, sx = moe.quant_fp8_1x128(x.to(DEV))
    offsets, st, _, xqp, sxp = moe.permute(torch.from_numpy(idx).to(DEV), xq, sx, cfg)
    hq, hs = moe.expert_gateup_fp8(xqp, sxp, offsets, ex, cfg, T)
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    hq, hs = hq.cpu().numpy(), hs.cpu().numpy().T          # hs -> [rows, H/128]
    xq_c, sx_c = xq.cpu().numpy(), sx.cpu().numpy()
    offs, st = offsets.cpu().numpy(), st.cpu().numpy()
    w13, w13s = inp.experts.w13.numpy(), inp.experts.w13_s.numpy()
    groups = [(e, np.arange(offs[e], offs[e + 1]), st[offs[e]:offs[e + 1]]) for e in range(shape.E)]
    groups += [(shape.E + s, k * T + s * T + np.arange(T), np.arange(T)) for s in range(shape.n_shared)]
    n_codes = n_diff = 0
    for e, rows, toks in groups:
        if rows.size == 0:
            continue
        h_ref = O.swiglu_h(xq_c[toks], sx_c[toks], w13[e, 0], w13s[e, 0], w13[e, 1], w13s[e, 1])
        q_ref, s_ref = O.quantize_1x128(h_ref)
        q, s = hq[rows], hs[rows]
        # scales: zero exactly where the oracle's group is all zero, else within the
        # fp32 rounding of h
        np.testing.assert_array_equal(s == 0, s_ref == 0, err_msg=f"expert {e}: zero groups")
        nz = s_ref != 0
        np.testing.assert_allclose(s[nz], s_ref[nz], rtol=1e-5, err_msg=f"expert {e}: scales")
        # codes: identical wherever the oracle's quotient h / s is clear of an e4m3
        # rounding midpoint; next to one, the neighbouring code on the same side of zero
        clear = clear_of_midpoint(quotients(h_ref, s_ref).astype(np.float64))
        diff = q != q_ref
        assert not (diff & clear).any(), f"expert {e}: {int((diff & clear).sum())} codes differ away from a midpoint"
        mag, mag_ref = (q & 0x7F).astype(int), (q_ref & 0x7F).astype(int)
        assert (np.abs(mag - mag_ref)[diff] <= 1).all(), f"expert {e}: codes more than one step apart"
        same_sign = ((q ^ q_ref) & 0x80) == 0
        assert (same_sign | (mag == 0) | (mag_ref == 0))[diff].all(), f"expert {e}: code sign"
        n_codes += q.size
        n_diff += int(diff.sum())
    assert n_diff <= 1e-3 * n_codes, f"{n_diff} of {n_codes} codes differ"
    return n_codes


def test_swap_ab_gateup_codes_and_scales():
    # about 9 rows per routed expert: the decode-regime kernel (32-token tiles)
    shape = S.MoEShape("hq_decode", T=37, d=1024, E=32, topk=8, H=384)
    assert _run(shape, seed=21, zero_tokens=(3, 17)) == 9 * 37 * 384


def test_token_major_gateup_codes_and_scales():
    # about 100 rows per routed expert and 400 shared rows: the 256-row token-major
    # kernel over several 128-token tiles, three feature blocks, a ragged last tile
    shape = S.MoEShape("hq_wide", T=400, d=512, E=32, topk=8, H=384)
    assert _run(shape, seed=22, zero_tokens=(0, 5, 399)) == 9 * 400 * 384
