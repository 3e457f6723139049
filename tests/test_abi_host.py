"""The C-ABI library: it loads, exports every symbol include/moe.h declares,
and its host-side argument checks answer without a GPU (no CUDA call is made
before validation passes)."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_97_b300 import binding as B
from mixture_experts_layer_97_b300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return B.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z_0-9]+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["moe_route", "moe_permute", "moe_grouped_ffn", "moe_combine", "moe_forward"]:
        assert n in names
    assert set(names) == set(B.SIGNATURES), "binding signatures and header disagree"


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    for n in declared_functions():
        assert re.search(rf"\bT {n}\b", out), f"{n} not exported"


def test_version_and_status_strings(L):
    assert B.version() >= 100
    assert B.status_string(0) == "ok"
    assert "corrupt" in B.status_string(6)
    assert B.status_string(99) == "unknown status"


def S(**kw):
    base = dict(T=64, d=256, N=8, k=2, F=256, act="swiglu", dtype="bf16")
    base.update(kw)
    return B.shape(base["T"], base["d"], base["N"], base["k"], base["F"], base["act"], base["dtype"])


@pytest.mark.parametrize("kw,expect", [
    (dict(), B.MOE_OK),
    (dict(k=9), B.MOE_ERR_INVALID_ARG),
    (dict(k=0), B.MOE_ERR_INVALID_ARG),
    (dict(T=-1), B.MOE_ERR_INVALID_ARG),
    (dict(N=300, k=2), B.MOE_ERR_UNSUPPORTED),
    (dict(d=200), B.MOE_ERR_UNSUPPORTED),             # bf16 needs d % 128
    (dict(F=100), B.MOE_ERR_UNSUPPORTED),             # SwiGLU bf16 needs F % 64
    (dict(F=192, act="gelu_tanh"), B.MOE_ERR_UNSUPPORTED),   # GELU bf16 needs F % 128
    (dict(F=192), B.MOE_OK),
    (dict(d=12, F=7, dtype="f32"), B.MOE_OK),
    (dict(d=10, dtype="f32"), B.MOE_ERR_UNSUPPORTED),
    (dict(T=2 ** 30, k=2), B.MOE_ERR_UNSUPPORTED),     # T*k must stay below 2^31
    (dict(T=0), B.MOE_OK),
])
def test_shape_checks(L, kw, expect):
    assert B.check_shape(S(**kw)) == expect


def test_null_shape_is_invalid(L):
    assert L.moe_check_shape(None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_workspace_size(None) == 0


def test_workspace_sizes_cover_the_buffers(L):
    s = S(T=1000, d=512, N=16, k=4, F=768)
    A = 1000 * 4
    ws = B.workspace_size(s)
    assert ws >= 2 * A * 512 * 2 + A * 768 * 2 + 3 * A * 4
    assert B.grouped_ffn_workspace_size(s) >= A * 768 * 2
    assert B.permute_workspace_size(s) >= 16 * 4
    assert B.hostio_workspace_size(s) >= ws + 2 * 1000 * 512 * 2
    assert B.workspace_size(S(k=100)) == 0


def test_null_pointers_rejected_before_any_launch(L):
    s = S()
    st = L.moe_route(ctypes.byref(s), None, None, None, None, None, None)
    assert st == B.MOE_ERR_INVALID_ARG
    st = L.moe_forward(ctypes.byref(s), None, None, None, None, None, None, None, None, None, None, None, 0, None)
    assert st == B.MOE_ERR_INVALID_ARG
    bad = S(k=20)
    assert L.moe_combine(ctypes.byref(bad), None, None, None, None, None) == B.MOE_ERR_INVALID_ARG


def test_misaligned_pointer_rejected(L):
    s = S()
    p = ctypes.c_void_p(0x1000)
    q = ctypes.c_void_p(0x1004)        # not 16-byte aligned
    st = L.moe_route(ctypes.byref(s), q, p, None, p, p, None)
    assert st == B.MOE_ERR_INVALID_ARG


def test_small_workspace_rejected(L):
    s = S()
    p = ctypes.c_void_p(0x1000)
    need = B.workspace_size(s)
    st = L.moe_forward(ctypes.byref(s), p, p, None, p, p, p, p, None, None, None, p, need - 1, None)
    assert st == B.MOE_ERR_WORKSPACE
    st = L.moe_grouped_ffn(ctypes.byref(s), p, p, p, p, p, p, p, B.grouped_ffn_workspace_size(s) - 1, None)
    assert st == B.MOE_ERR_WORKSPACE
    # GELU takes no w_up
    g = S(act="gelu_tanh")
    st = L.moe_grouped_ffn(ctypes.byref(g), p, p, p, p, p, p, p, 1 << 40, None)
    assert st == B.MOE_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(L):
    import torch
    s = S(T=4, d=128, N=2, k=1, F=64)
    x = torch.zeros(4, 128, dtype=torch.bfloat16)
    with pytest.raises(RuntimeError, match="CUDA device"):
        B.route(s, x, x, None, x, x)


def test_tiling_policy_setter(L):
    assert B.get_ffn_tiling() == "auto"
    for m in ("rows", "tokens", "pairs", "rowpairs", "auto"):
        B.set_ffn_tiling(m)
        assert B.get_ffn_tiling() == m
    assert L.moe_set_ffn_tiling(7) == B.MOE_ERR_INVALID_ARG
    assert B.get_ffn_tiling() == "auto"


def test_pipelined_hostio_checks(L):
    s = S()
    p = ctypes.c_void_p(0x1000)
    need = B.hostio_pipelined_workspace_size(s)
    assert need >= B.workspace_size(s) + 4 * 64 * 256 * 2
    st = L.moe_forward_hostio_pipelined(ctypes.byref(s), p, p, None, p, p, p, p, p, need, 2, None, None, None)
    assert st == B.MOE_ERR_INVALID_ARG          # slot must be 0 or 1
    st = L.moe_forward_hostio_pipelined(ctypes.byref(s), p, p, None, p, p, p, p, p, need - 1, 0, None, None, None)
    assert st == B.MOE_ERR_WORKSPACE


def test_header_compiles_as_c99_and_links(L, tmp_path):
    """The boundary is plain C: a C99 program that includes only include/moe.h
    builds against libmoe_b300.so and calls the host-only entry points."""
    src = tmp_path / "use_moe.c"
    src.write_text(r"""
#include <stddef.h>
#include <stdio.h>
#include <string.h>
#include "moe.h"
int main(void) {
    moe_shape s = {4096, 4096, 8, 2, 14336, MOE_SWIGLU, MOE_BF16};
    moe_shape bad = s;
    bad.k = 9;
    if (moe_version() < 100) return 1;
    if (moe_check_shape(&s) != MOE_OK) return 2;
    if (moe_check_shape(&bad) != MOE_ERR_INVALID_ARG) return 3;
    if (moe_workspace_size(&s) == 0 || moe_workspace_size(&bad) != 0) return 4;
    if (strcmp(moe_status_string(MOE_OK), "ok") != 0) return 5;
    if (moe_route(&bad, NULL, NULL, NULL, NULL, NULL, NULL) != MOE_ERR_INVALID_ARG) return 6;
    printf("%zu %zu %zu %zu\n", moe_forward_hostio_pipelined_workspace_size(&s), sizeof(moe_options),
           offsetof(moe_options, use_tiling), offsetof(moe_options, ffn_tiling));
    return 0;
}
""")
    exe = tmp_path / "use_moe"
    libdir = os.path.dirname(B.LIB_PATH)
    import subprocess
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                           "-L", libdir, "-l:libmoe_b300.so", f"-Wl,-rpath,{libdir}", "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out
    ws, size, off_use, off_tiling = (int(v) for v in out.stdout.split())
    assert ws == B.hostio_pipelined_workspace_size(B.shape(4096, 4096, 8, 2, 14336, "swiglu", "bf16"))
    # the binding's options struct has the header's layout
    assert size == ctypes.sizeof(B.MoeOptions)
    assert off_use == B.MoeOptions.use_tiling.offset and off_tiling == B.MoeOptions.ffn_tiling.offset


def test_forward_ex_rejects_a_bad_per_call_tiling(L):
    s = S()
    p = ctypes.c_void_p(0x1000)
    o = B.MoeOptions(0, 0, 0.0, None, None, 1, 7)
    st = L.moe_forward_ex(ctypes.byref(s), ctypes.byref(o), p, p, None, p, p, p, p, None, None, None, p, 1 << 40,
                          None)
    assert st == B.MOE_ERR_INVALID_ARG
