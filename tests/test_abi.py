"""The C ABI library: it builds, loads, exports every symbol the header declares,
and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

import routed_fp8_expert_gb300 as moe
from routed_fp8_expert_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_fp8.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_expert_gemm_fp8", "moe_combine", "moe_layer_forward",
              "dense_swiglu_fp8", "moe_quant_fp8_1x128", "moe_workspace_bytes"):
        assert n in names


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(_lib._SIGS), "binding misses a declared call"


def test_workspace_and_rows(lib):
    cfg = _lib.MoeCfg(7168, 384, 8, 2048, 1, 2.827)
    assert moe.permuted_rows(cfg, 256) == 9 * 256
    ws = moe.workspace_bytes(cfg, 256)
    # permuted activations, h and the bf16 expert outputs dominate
    assert ws > 9 * 256 * (7168 + 2048 + 2 * 7168)
    assert ws % 1024 == 0
    assert moe.workspace_bytes(cfg, 0) > 0
    bad = _lib.MoeCfg(7000, 384, 8, 2048, 1, 2.827)
    assert moe.workspace_bytes(bad, 256) == 0
    assert lib.dense_swiglu_workspace_bytes(7168, 18432, 8192) >= 8192 * (7168 + 18432)
    assert lib.dense_swiglu_workspace_bytes(7000, 18432, 8192) == 0


def _cfg(**kw):
    base = dict(d=1024, E=32, topk=8, H=256, n_shared=1, route_scale=2.827)
    base.update(kw)
    return _lib.MoeCfg(base["d"], base["E"], base["topk"], base["H"], base["n_shared"], base["route_scale"])


@pytest.mark.parametrize("kw,code", [
    (dict(d=1000), _lib.MOE_ERR_UNSUPPORTED),
    (dict(H=100), _lib.MOE_ERR_UNSUPPORTED),
    (dict(topk=0), _lib.MOE_ERR_UNSUPPORTED),
    (dict(topk=33, E=64), _lib.MOE_ERR_UNSUPPORTED),
    (dict(E=4), _lib.MOE_ERR_UNSUPPORTED),
    (dict(E=2048), _lib.MOE_ERR_UNSUPPORTED),
    (dict(n_shared=5), _lib.MOE_ERR_UNSUPPORTED),
    (dict(route_scale=float("inf")), _lib.MOE_ERR_ARG),
])
def test_bad_shapes_rejected_on_host(lib, kw, code):
    cfg = _cfg(**kw)
    fake = ctypes.c_void_p(0x1000)
    st = lib.moe_layer_forward(fake, fake, fake, fake, fake, fake, fake, ctypes.byref(cfg), 4, fake, None, None,
                               fake, 1 << 30, None)
    assert st == code
    assert lib.moe_last_error_string()


def test_null_and_misaligned_pointers_rejected(lib):
    cfg = _cfg()
    fake = ctypes.c_void_p(0x1000)
    assert lib.moe_route(None, fake, fake, ctypes.byref(cfg), 4, fake, fake, None, fake, 1 << 30, None) == _lib.MOE_ERR_ARG
    assert b"x is NULL" in lib.moe_last_error_string()
    odd = ctypes.c_void_p(0x1001)
    assert lib.moe_combine(odd, fake, fake, ctypes.byref(cfg), 4, fake, None) == _lib.MOE_ERR_ARG
    assert b"aligned" in lib.moe_last_error_string()
    assert lib.moe_layer_forward(fake, fake, fake, fake, fake, fake, fake, None, 4, fake, None, None, fake, 1 << 30,
                                 None) == _lib.MOE_ERR_ARG
    assert lib.moe_quant_fp8_1x128(fake, 1, 4, 100, fake, fake, 0, None) == _lib.MOE_ERR_UNSUPPORTED


def test_short_workspace_rejected(lib):
    cfg = _cfg()
    fake = ctypes.c_void_p(0x1000)
    st = lib.moe_layer_forward(fake, fake, fake, fake, fake, fake, fake, ctypes.byref(cfg), 64, fake, None, None,
                               fake, 1024, None)
    assert st == _lib.MOE_ERR_ARG and b"workspace" in lib.moe_last_error_string()


def test_negative_and_zero_tokens(lib):
    cfg = _cfg()
    fake = ctypes.c_void_p(0x1000)
    assert lib.moe_combine(fake, fake, fake, ctypes.byref(cfg), -1, fake, None) == _lib.MOE_ERR_ARG
    # T = 0 enqueues nothing and succeeds (no device is touched)
    assert lib.moe_layer_forward(None, None, None, None, None, None, None, ctypes.byref(cfg), 0, None, None, None,
                                 None, 0, None) == _lib.MOE_OK
    assert lib.moe_last_launch_count() == 0
    assert lib.dense_swiglu_fp8(None, None, None, None, None, 1024, 256, 0, None, None, 0, None) == _lib.MOE_OK
    assert lib.moe_quant_fp8_1x128(None, 1, 0, 128, None, None, 0, None) == _lib.MOE_OK


def test_plain_c_caller(lib, tmp_path):
    # the header compiles as C99 and a C program links against the library and calls
    # it: the host-side calls (sizes, argument checks) need no GPU
    src = tmp_path / "caller.c"
    src.write_text(r'''
#include <stdio.h>
#include "moe_fp8.h"
int main(void) {
    moe_cfg_t cfg = {7168, 384, 8, 2048, 1, 2.827f};
    printf("%lld %zu\n", (long long)moe_permuted_rows(&cfg, 256), moe_workspace_bytes(&cfg, 256));
    moe_cfg_t bad = {100, 384, 8, 2048, 1, 2.827f};   /* d not a multiple of 128 */
    printf("%d\n", moe_combine(NULL, NULL, NULL, &bad, 4, NULL, NULL));
    printf("%s\n", moe_last_error_string() ? "msg" : "none");
    return 0;
}
''')
    exe = tmp_path / "caller"
    libdir = os.path.dirname(_lib.LIB_PATH)
    import subprocess
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe),
                        "-L", libdir, "-lmoe_fp8", f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.split()
    cfg = _lib.MoeCfg(7168, 384, 8, 2048, 1, 2.827)
    assert int(lines[0]) == moe.permuted_rows(cfg, 256)
    assert int(lines[1]) == moe.workspace_bytes(cfg, 256)
    assert int(lines[2]) in (_lib.MOE_ERR_ARG, _lib.MOE_ERR_UNSUPPORTED)
    assert lines[3] == "msg"
