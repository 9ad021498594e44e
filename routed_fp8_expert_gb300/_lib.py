"""ctypes binding of libmoe_fp8.so (include/moe_fp8.h).

Argument marshalling only: every function allocates its outputs with torch on
the inputs' device, passes raw device pointers and the current CUDA stream to
the C ABI, and raises on a non-zero status. There is no fallback: if the
library is missing or the tensors are not on a CUDA device, it raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_fp8.so")

MOE_OK, MOE_ERR_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_INDEX = 0, -1, -2, -3, -4, -5

_c_int, _c_size, _c_i64, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_int64, ctypes.c_void_p


class MoeCfg(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("E", ctypes.c_int), ("topk", ctypes.c_int), ("H", ctypes.c_int),
                ("n_shared", ctypes.c_int), ("route_scale", ctypes.c_float), ("w_tiled", ctypes.c_int)]


# name -> (restype, argtypes)
_SIGS = {
    "moe_permuted_rows": (_c_i64, [ctypes.POINTER(MoeCfg), _c_int]),
    "moe_workspace_bytes": (_c_size, [ctypes.POINTER(MoeCfg), _c_int]),
    "moe_quant_fp8_1x128": (_c_int, [_vp, _c_int, _c_i64, _c_int, _vp, _vp, _c_int, _vp]),
    "moe_pack_weights_fp8": (_c_int, [_vp, _c_i64, _c_int, _c_int, _vp, _vp]),
    "moe_route": (_c_int, [_vp, _vp, _vp, ctypes.POINTER(MoeCfg), _c_int, _vp, _vp, _vp, _vp, _c_size, _vp]),
    "moe_permute": (_c_int, [_vp, _vp, _vp, ctypes.POINTER(MoeCfg), _c_int, _vp, _vp, _vp, _vp, _vp, _vp,
                             _c_size, _vp]),
    "moe_quant_permute_fp8": (_c_int, [_vp, _vp, ctypes.POINTER(MoeCfg), _c_int, _vp, _vp, _vp, _vp, _vp, _vp,
                                       _c_size, _vp]),
    "moe_permute_noalloc": (_c_int, [_vp, _vp, _vp, ctypes.POINTER(MoeCfg), _c_int, _vp, _vp, _vp, _vp, _vp,
                                     _vp]),
    "moe_expert_gemm_fp8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.POINTER(MoeCfg), _c_int, _vp, _vp,
                                     _c_size, _vp]),
    "moe_expert_gateup_fp8": (_c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.POINTER(MoeCfg), _c_int, _vp, _vp, _vp,
                                       _c_size, _vp]),
    "moe_expert_down_fp8": (_c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.POINTER(MoeCfg), _c_int, _vp, _vp, _c_size,
                                     _vp]),
    "moe_combine": (_c_int, [_vp, _vp, _vp, ctypes.POINTER(MoeCfg), _c_int, _vp, _vp]),
    "moe_rmsnorm_quant_fp8": (_c_int, [_vp, _vp, ctypes.c_float, _c_int, _c_int, _vp, _vp, _vp, _c_int, _vp]),
    "moe_combine_residual_rmsnorm": (_c_int, [_vp, _vp, _vp, ctypes.POINTER(MoeCfg), _c_int, _vp, _vp,
                                              ctypes.c_float, _vp, _vp, _vp]),
    "moe_layer_forward": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.POINTER(MoeCfg), _c_int, _vp, _vp,
                                   _vp, _vp, _c_size, _vp]),
    "moe_block_ffn_forward": (_c_int, [_vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _vp,
                                       ctypes.POINTER(MoeCfg), _c_int, _vp, _vp, _vp, _vp, _vp, _vp, _c_size, _vp]),
    "dense_swiglu_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "dense_swiglu_fp8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _c_size, _vp]),
    "moe_check_device_error": (_c_int, [_vp, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_test_wait_timeout": (_c_int, [ctypes.c_uint64, _vp]),
    "moe_last_error_string": (ctypes.c_char_p, []),
    "moe_last_launch_count": (_c_int, []),
}

_lib = None


def load():
    """Load the library (built in-tree by routed_fp8_expert_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with routed_fp8_expert_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


class MoeError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"status {status}: {msg}")
        self.status = status


def _check(status):
    if status != MOE_OK:
        raise MoeError(status, load().moe_last_error_string().decode())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")


def cfg_of(shape, w_tiled: bool = False) -> MoeCfg:
    return MoeCfg(shape.d, shape.E, shape.topk, shape.H, shape.n_shared, shape.route_scale, int(w_tiled))


def pack_weights_fp8(w: torch.Tensor) -> torch.Tensor:
    """moe_pack_weights_fp8: e4m3 weights [..., rows, cols] (row-major, uint8) into
    the tiled layout [groups, rows/128, cols/128, 128, 128] (groups = the product of
    the leading dimensions); returned flat in w's shape."""
    _cuda(w)
    w = w.contiguous()
    rows, cols = w.shape[-2], w.shape[-1]
    groups = w.numel() // (rows * cols)
    out = torch.empty_like(w)
    _check(load().moe_pack_weights_fp8(_p(w), groups, rows, cols, _p(out), _stream(w.device)))
    return out


def permuted_rows(cfg: MoeCfg, T: int) -> int:
    return load().moe_permuted_rows(ctypes.byref(cfg), T)


def workspace_bytes(cfg: MoeCfg, T: int) -> int:
    return load().moe_workspace_bytes(ctypes.byref(cfg), T)


def workspace(cfg: MoeCfg, T: int, device) -> torch.Tensor:
    return torch.empty(max(1, workspace_bytes(cfg, T)), dtype=torch.uint8, device=device)


def last_launch_count() -> int:
    return load().moe_last_launch_count()


def quant_fp8_1x128(x: torch.Tensor, s_transposed: bool = False):
    """x [rows, cols] bf16 or fp32 -> (q uint8 [rows, cols], s fp32)."""
    _cuda(x)
    x = x.contiguous()
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    s = torch.empty(((cols // 128, rows) if s_transposed else (rows, cols // 128)), dtype=torch.float32,
                    device=x.device)
    _check(load().moe_quant_fp8_1x128(_p(x), int(x.dtype == torch.bfloat16), rows, cols, _p(q), _p(s),
                                      int(s_transposed), _stream(x.device)))
    return q, s


def route(x, w_gate, bias, cfg: MoeCfg, ws=None, want_scores=False):
    _cuda(x, w_gate, bias)
    T = x.shape[0]
    dev = x.device
    idx = torch.empty((T, cfg.topk), dtype=torch.int32, device=dev)
    w = torch.empty((T, cfg.topk), dtype=torch.float32, device=dev)
    scores = torch.empty((T, cfg.E), dtype=torch.float32, device=dev) if want_scores else None
    ws = workspace(cfg, T, dev) if ws is None else ws
    _check(load().moe_route(_p(x), _p(w_gate), _p(bias), ctypes.byref(cfg), T, _p(idx), _p(w), _p(scores),
                            _p(ws), ws.numel(), _stream(dev)))
    return idx, w, scores


def permute(topk_idx, xq, sx, cfg: MoeCfg, ws=None):
    _cuda(topk_idx, xq, sx)
    T = topk_idx.shape[0]
    dev = topk_idx.device
    R = permuted_rows(cfg, T)
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
    sorted_tok = torch.empty(T * cfg.topk, dtype=torch.int32, device=dev)
    inv_pos = torch.empty((T, cfg.topk), dtype=torch.int32, device=dev)
    xq_perm = torch.empty((R, cfg.d), dtype=torch.uint8, device=dev)
    sx_perm = torch.empty((cfg.d // 128, R), dtype=torch.float32, device=dev)
    ws = workspace(cfg, T, dev) if ws is None else ws
    _check(load().moe_permute(_p(topk_idx), _p(xq), _p(sx), ctypes.byref(cfg), T, _p(offsets), _p(sorted_tok),
                              _p(inv_pos), _p(xq_perm), _p(sx_perm), _p(ws), ws.numel(), _stream(dev)))
    return offsets, sorted_tok, inv_pos, xq_perm, sx_perm


def quant_permute_fp8(topk_idx, x, cfg: MoeCfg, ws=None):
    """moe_quant_permute_fp8: the 1x128 codes of bf16 x written straight to their
    permuted rows. Outputs as permute() of quant_fp8_1x128(x)."""
    _cuda(topk_idx, x)
    if x.dtype != torch.bfloat16:
        raise MoeError(MOE_ERR_ARG, "x must be bf16")
    T = topk_idx.shape[0]
    dev = topk_idx.device
    R = permuted_rows(cfg, T)
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
    sorted_tok = torch.empty(T * cfg.topk, dtype=torch.int32, device=dev)
    inv_pos = torch.empty((T, cfg.topk), dtype=torch.int32, device=dev)
    xq_perm = torch.empty((R, cfg.d), dtype=torch.uint8, device=dev)
    sx_perm = torch.empty((cfg.d // 128, R), dtype=torch.float32, device=dev)
    ws = workspace(cfg, T, dev) if ws is None else ws
    _check(load().moe_quant_permute_fp8(_p(topk_idx), _p(x), ctypes.byref(cfg), T, _p(offsets), _p(sorted_tok),
                                        _p(inv_pos), _p(xq_perm), _p(sx_perm), _p(ws), ws.numel(), _stream(dev)))
    return offsets, sorted_tok, inv_pos, xq_perm, sx_perm


def permute_noalloc(topk_idx, xq, sx, cfg: MoeCfg):
    """moe_permute_noalloc: the permutation without a workspace (the library's
    fixed device scratch; T <= 8192 and T * topk <= 65536). Outputs as permute()."""
    _cuda(topk_idx, xq, sx)
    T = topk_idx.shape[0]
    dev = topk_idx.device
    R = permuted_rows(cfg, T)
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
    sorted_tok = torch.empty(T * cfg.topk, dtype=torch.int32, device=dev)
    inv_pos = torch.empty((T, cfg.topk), dtype=torch.int32, device=dev)
    xq_perm = torch.empty((R, cfg.d), dtype=torch.uint8, device=dev)
    sx_perm = torch.empty((cfg.d // 128, R), dtype=torch.float32, device=dev)
    _check(load().moe_permute_noalloc(_p(topk_idx), _p(xq), _p(sx), ctypes.byref(cfg), T, _p(offsets),
                                      _p(sorted_tok), _p(inv_pos), _p(xq_perm), _p(sx_perm), _stream(dev)))
    return offsets, sorted_tok, inv_pos, xq_perm, sx_perm


def expert_gemm_fp8(xq_perm, sx_perm, offsets, experts, cfg: MoeCfg, T: int, ws=None):
    """Returns o bf16 [permuted_rows, d]."""
    _cuda(xq_perm, sx_perm, offsets, experts.w13)
    dev = xq_perm.device
    o = torch.empty((permuted_rows(cfg, T), cfg.d), dtype=torch.bfloat16, device=dev)
    ws = workspace(cfg, T, dev) if ws is None else ws
    _check(load().moe_expert_gemm_fp8(_p(xq_perm), _p(sx_perm), _p(offsets), _p(experts.w13), _p(experts.w13_s),
                                      _p(experts.w2), _p(experts.w2_s), ctypes.byref(cfg), T, _p(o), _p(ws),
                                      ws.numel(), _stream(dev)))
    return o


def expert_gateup_fp8(xq_perm, sx_perm, offsets, experts, cfg: MoeCfg, T: int, ws=None, hq=None, hs=None):
    """Returns (hq uint8 [permuted_rows, H], hs fp32 [H/128, permuted_rows])."""
    _cuda(xq_perm, sx_perm, offsets, experts.w13)
    dev = xq_perm.device
    R = permuted_rows(cfg, T)
    hq = torch.empty((R, cfg.H), dtype=torch.uint8, device=dev) if hq is None else hq
    hs = torch.empty((cfg.H // 128, R), dtype=torch.float32, device=dev) if hs is None else hs
    ws = workspace(cfg, T, dev) if ws is None else ws
    _check(load().moe_expert_gateup_fp8(_p(xq_perm), _p(sx_perm), _p(offsets), _p(experts.w13), _p(experts.w13_s),
                                        ctypes.byref(cfg), T, _p(hq), _p(hs), _p(ws), ws.numel(), _stream(dev)))
    return hq, hs


def expert_down_fp8(hq, hs, offsets, experts, cfg: MoeCfg, T: int, ws=None, o=None):
    """Returns o bf16 [permuted_rows, d]."""
    _cuda(hq, hs, offsets, experts.w2)
    dev = hq.device
    o = torch.empty((permuted_rows(cfg, T), cfg.d), dtype=torch.bfloat16, device=dev) if o is None else o
    ws = workspace(cfg, T, dev) if ws is None else ws
    _check(load().moe_expert_down_fp8(_p(hq), _p(hs), _p(offsets), _p(experts.w2), _p(experts.w2_s),
                                      ctypes.byref(cfg), T, _p(o), _p(ws), ws.numel(), _stream(dev)))
    return o


def combine(o, topk_w, inv_pos, cfg: MoeCfg, T: int):
    _cuda(o, topk_w, inv_pos)
    y = torch.empty((T, cfg.d), dtype=torch.bfloat16, device=o.device)
    _check(load().moe_combine(_p(o), _p(topk_w), _p(inv_pos), ctypes.byref(cfg), T, _p(y), _stream(o.device)))
    return y


RMS_NORM_EPS = 1e-6


def rmsnorm_quant_fp8(h, gamma, eps: float = RMS_NORM_EPS, write_y: bool = True, s_transposed: bool = False):
    """moe_rmsnorm_quant_fp8: h [rows, cols] bf16, gamma [cols] bf16 ->
    (y bf16 [rows, cols] or None, q uint8 [rows, cols], s fp32)."""
    _cuda(h, gamma)
    rows, cols = h.shape
    dev = h.device
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev) if write_y else None
    q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    s = torch.empty(((cols // 128, rows) if s_transposed else (rows, cols // 128)), dtype=torch.float32, device=dev)
    _check(load().moe_rmsnorm_quant_fp8(_p(h), _p(gamma), float(eps), rows, cols, _p(y) if y is not None else None,
                                        _p(q), _p(s), int(s_transposed), _stream(dev)))
    return y, q, s


def combine_residual_rmsnorm(o, topk_w, inv_pos, cfg: MoeCfg, T: int, residual, gamma=None,
                             eps: float = RMS_NORM_EPS):
    """moe_combine_residual_rmsnorm -> (h_out bf16 [T, d], x_next bf16 [T, d] or None)."""
    _cuda(o, topk_w, inv_pos, residual)
    dev = o.device
    h_out = torch.empty((T, cfg.d), dtype=torch.bfloat16, device=dev)
    x_next = torch.empty((T, cfg.d), dtype=torch.bfloat16, device=dev) if gamma is not None else None
    _check(load().moe_combine_residual_rmsnorm(_p(o), _p(topk_w), _p(inv_pos), ctypes.byref(cfg), T, _p(residual),
                                               _p(gamma) if gamma is not None else None, float(eps), _p(h_out),
                                               _p(x_next) if x_next is not None else None, _stream(dev)))
    return h_out, x_next


def layer_forward(x, w_gate, bias, experts, cfg: MoeCfg, ws=None, y=None, want_routing=False):
    """The whole MoE layer. Returns y bf16 [T, d] (and topk_idx, topk_w when want_routing)."""
    _cuda(x, w_gate, bias, experts.w13)
    T = x.shape[0]
    dev = x.device
    y = torch.empty((T, cfg.d), dtype=torch.bfloat16, device=dev) if y is None else y
    idx = torch.empty((T, cfg.topk), dtype=torch.int32, device=dev) if want_routing else None
    w = torch.empty((T, cfg.topk), dtype=torch.float32, device=dev) if want_routing else None
    ws = workspace(cfg, T, dev) if ws is None else ws
    _check(load().moe_layer_forward(_p(x), _p(w_gate), _p(bias), _p(experts.w13), _p(experts.w13_s),
                                    _p(experts.w2), _p(experts.w2_s), ctypes.byref(cfg), T, _p(y), _p(idx), _p(w),
                                    _p(ws), ws.numel(), _stream(dev)))
    return (y, idx, w) if want_routing else y


def block_ffn_forward(h, gamma_post, w_gate, bias, experts, cfg: MoeCfg, gamma_next=None,
                      eps: float = RMS_NORM_EPS, ws=None, h_out=None, x_next=None, want_routing=False):
    """moe_block_ffn_forward: RMSNorm_post(h) -> the MoE layer -> h + y -> RMSNorm_next.
    Returns (h_out, x_next or None) (and topk_idx, topk_w when want_routing)."""
    _cuda(h, gamma_post, w_gate, bias, experts.w13, gamma_next)
    T = h.shape[0]
    dev = h.device
    h_out = torch.empty((T, cfg.d), dtype=torch.bfloat16, device=dev) if h_out is None else h_out
    if gamma_next is not None and x_next is None:
        x_next = torch.empty((T, cfg.d), dtype=torch.bfloat16, device=dev)
    idx = torch.empty((T, cfg.topk), dtype=torch.int32, device=dev) if want_routing else None
    w = torch.empty((T, cfg.topk), dtype=torch.float32, device=dev) if want_routing else None
    ws = workspace(cfg, T, dev) if ws is None else ws
    _check(load().moe_block_ffn_forward(_p(h), _p(gamma_post), float(eps), _p(w_gate), _p(bias), _p(experts.w13),
                                        _p(experts.w13_s), _p(experts.w2), _p(experts.w2_s), ctypes.byref(cfg), T,
                                        _p(gamma_next), _p(h_out), _p(x_next if gamma_next is not None else None),
                                        _p(idx), _p(w), _p(ws), ws.numel(), _stream(dev)))
    x_out = x_next if gamma_next is not None else None
    return (h_out, x_out, idx, w) if want_routing else (h_out, x_out)


def dense_workspace(d, H, T, device):
    return torch.empty(max(1, load().dense_swiglu_workspace_bytes(d, H, T)), dtype=torch.uint8, device=device)


def dense_swiglu_fp8(x, w13, w13_s, w2, w2_s, ws=None, y=None):
    _cuda(x, w13, w2)
    T, d = x.shape
    H = w13.shape[1]
    dev = x.device
    y = torch.empty((T, d), dtype=torch.bfloat16, device=dev) if y is None else y
    ws = dense_workspace(d, H, T, dev) if ws is None else ws
    _check(load().dense_swiglu_fp8(_p(x), _p(w13), _p(w13_s), _p(w2), _p(w2_s), d, H, T, _p(y), _p(ws),
                                   ws.numel(), _stream(dev)))
    return y


def test_wait_timeout(limit_ns: int, device=None):
    """moe_test_wait_timeout: the bounded-wait self-test (see the header); raises on
    a bad limit. Read the result with check_device_error."""
    _check(load().moe_test_wait_timeout(int(limit_ns), _stream(device)))


def check_device_error(device=None):
    """Synchronise and read/clear the device error word; raises MoeError on a timeout."""
    detail = ctypes.c_uint32(0)
    _check(load().moe_check_device_error(_stream(device), ctypes.byref(detail)))
    return detail.value
