"""ctypes binding of libmoe_b300.so (the C ABI in include/moe.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t, a non-OK status becomes ``MoEError``. Every
step of the layer runs in the library's kernels. There is no CPU fallback:
if the library is missing or a tensor is not on a CUDA device, calls raise.

Each function ``name`` wraps the C entry point ``moe_name`` with the same
arguments in the same order (a workspace tensor supplies both the pointer and
its byte size); the header documents meaning, layouts and errors.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_b300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_CORRUPT = 4, 5, 6
MOE_F32, MOE_BF16 = 0, 1
MOE_SWIGLU, MOE_GELU_TANH = 0, 1
TILING = {"auto": 0, "rows": 1, "tokens": 2, "pairs": 3, "rowpairs": 4}
ACT = {"swiglu": MOE_SWIGLU, "gelu_tanh": MOE_GELU_TANH}
DTYPE = {"f32": MOE_F32, "bf16": MOE_BF16}
TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}

# Every symbol the header declares, with its ctypes signature.
P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("N", ctypes.c_int32), ("k", ctypes.c_int32),
                ("d_ff", ctypes.c_int32), ("act", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class MoeOptions(ctypes.Structure):
    _fields_ = [("bias_mode", ctypes.c_int32), ("use_capacity", ctypes.c_int32), ("capacity_factor", ctypes.c_double),
                ("load_stats", ctypes.c_void_p), ("dropped", ctypes.c_void_p), ("use_tiling", ctypes.c_int32),
                ("ffn_tiling", ctypes.c_int32)]


SP = ctypes.POINTER(MoeShape)
OP = ctypes.POINTER(MoeOptions)
BIAS_MODES = {"logits": 0, "select": 1}


def load_stats_len(N: int) -> int:
    return 2 * N + 3
SIGNATURES = {
    "moe_route": (I32, [SP, P, P, P, P, P, P]),
    "moe_permute": (I32, [SP, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_grouped_ffn": (I32, [SP, P, P, P, P, P, P, P, SZ, P]),
    "moe_grouped_ffn_gather": (I32, [SP, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_permute_noalloc": (I32, [SP, P, P, P, P, P, P, P, P]),
    "moe_permute_capacity": (I32, [SP, P, P, ctypes.c_double, P, P, P, P, P, P, P, SZ, P]),
    "moe_forward_capacity": (I32, [SP, ctypes.c_double, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_route_ex": (I32, [SP, P, P, P, I32, P, P, P, P, SZ, P]),
    "moe_route_ex_workspace_size": (SZ, [SP]),
    "moe_forward_ex": (I32, [SP, OP, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_route_expert_choice": (I32, [SP, I64, P, P, P, P, P, P, P, P, P, P]),
    "moe_forward_expert_choice": (I32, [SP, I64, P, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_expert_choice_workspace_size": (SZ, [SP, I64]),
    "moe_gather_rows": (I32, [SP, P, I32, I64, P, P, P]),
    "moe_combine": (I32, [SP, P, P, P, P, P]),
    "moe_ep_regroup": (I32, [I32, I32, P, I64, I32, I32, P, P, P, P, P]),
    "moe_ep_ungroup": (I32, [I64, I32, I32, P, P, P, P]),
    "moe_forward": (I32, [SP, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_forward_hostio": (I32, [SP, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_forward_hostio_pipelined": (I32, [SP, P, P, P, P, P, P, P, P, SZ, I32, P, P, P]),
    "moe_forward_hostio_pipelined_workspace_size": (SZ, [SP]),
    "moe_workspace_size": (SZ, [SP]),
    "moe_forward_hostio_workspace_size": (SZ, [SP]),
    "moe_permute_workspace_size": (SZ, [SP]),
    "moe_grouped_ffn_workspace_size": (SZ, [SP]),
    "moe_check_shape": (I32, [SP]),
    "moe_get_error": (I32, [P]),
    "moe_selftest_bounded_wait": (I32, [I64, P]),
    "moe_status_string": (ctypes.c_char_p, [I32]),
    "moe_set_ffn_tiling": (I32, [ctypes.c_int]),
    "moe_get_ffn_tiling": (ctypes.c_int, []),
    "moe_version": (ctypes.c_int, []),
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib():
    """Open the library (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe_b300.so is not built ({LIB_PATH}); run "
                               "`python -m mixture_experts_layer_97_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(st: int) -> str:
    return lib().moe_status_string(st).decode()


def shape(T: int, d: int, N: int, k: int, F: int, act: str = "swiglu", dtype: str = "bf16") -> MoeShape:
    return MoeShape(T, d, N, k, F, ACT[act], DTYPE[dtype])


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise RuntimeError("MoE library tensors must live on a CUDA device (there is no CPU path)")
    if not t.is_contiguous():
        raise RuntimeError("MoE library tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _host_ptr(t: torch.Tensor):
    if t.is_cuda or not t.is_contiguous():
        raise RuntimeError("host buffer expected (contiguous CPU tensor, ideally pinned)")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(st: int, where: str):
    if st != MOE_OK:
        raise MoEError(st, where)


def check_shape(s: MoeShape) -> int:
    return lib().moe_check_shape(ctypes.byref(s))


def workspace_size(s: MoeShape) -> int:
    return lib().moe_workspace_size(ctypes.byref(s))


def hostio_workspace_size(s: MoeShape) -> int:
    return lib().moe_forward_hostio_workspace_size(ctypes.byref(s))


def permute_workspace_size(s: MoeShape) -> int:
    return lib().moe_permute_workspace_size(ctypes.byref(s))


def grouped_ffn_workspace_size(s: MoeShape) -> int:
    return lib().moe_grouped_ffn_workspace_size(ctypes.byref(s))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A caller-owned workspace buffer (the library itself never allocates)."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def route(s, x, w_g, bias, topk_idx, topk_w, stream=None):
    _check(lib().moe_route(ctypes.byref(s), _ptr(x), _ptr(w_g), _ptr(bias), _ptr(topk_idx), _ptr(topk_w),
                           _stream(stream)), "moe_route")


def permute(s, topk_idx, x, counts, offsets, perm, inv_perm, x_perm, ws, stream=None):
    _check(lib().moe_permute(ctypes.byref(s), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(offsets), _ptr(perm),
                             _ptr(inv_perm), _ptr(x_perm), _ptr(ws), ws.numel() if ws is not None else 0,
                             _stream(stream)), "moe_permute")


def permute_noalloc(s, topk_idx, x, counts, offsets, perm, inv_perm, x_perm, stream=None):
    """moe_permute with its scratch in the library's fixed device array (no workspace argument)."""
    _check(lib().moe_permute_noalloc(ctypes.byref(s), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(offsets),
                                     _ptr(perm), _ptr(inv_perm), _ptr(x_perm), _stream(stream)),
           "moe_permute_noalloc")


def route_ex_workspace_size(s) -> int:
    return lib().moe_route_ex_workspace_size(ctypes.byref(s))


def route_ex(s, x, w_g, bias, topk_idx, topk_w, bias_mode="logits", load_stats=None, ws=None, stream=None):
    _check(lib().moe_route_ex(ctypes.byref(s), _ptr(x), _ptr(w_g), _ptr(bias), BIAS_MODES[bias_mode], _ptr(topk_idx),
                              _ptr(topk_w), _ptr(load_stats), _ptr(ws), ws.numel() if ws is not None else 0,
                              _stream(stream)), "moe_route_ex")


def unpack_load_stats(t, N: int) -> dict:
    """The load_stats vector as named fields (host copy)."""
    v = t.detach().cpu().numpy().astype("float64")
    return dict(f=v[:N], P=v[N:2 * N], balance=float(v[2 * N]), entropy_bits=float(v[2 * N + 1]),
                top1=float(v[2 * N + 2]))


def forward_ex(s, x, w_g, bias, w_gate, w_up, w_down, out, ws, bias_mode="logits", capacity_factor=None,
               load_stats=None, dropped=None, topk_idx=None, topk_w=None, counts=None, ffn_tiling=None,
               stream=None):
    """ffn_tiling: None (the process-wide setting) or a key of TILING for this call only."""
    o = MoeOptions(BIAS_MODES[bias_mode], 0 if capacity_factor is None else 1,
                   0.0 if capacity_factor is None else float(capacity_factor),
                   None if load_stats is None else _ptr(load_stats).value,
                   None if dropped is None else _ptr(dropped).value,
                   0 if ffn_tiling is None else 1, 0 if ffn_tiling is None else TILING[ffn_tiling])
    _check(lib().moe_forward_ex(ctypes.byref(s), ctypes.byref(o), _ptr(x), _ptr(w_g), _ptr(bias), _ptr(w_gate),
                                _ptr(w_up), _ptr(w_down), _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(counts),
                                _ptr(ws), ws.numel(), _stream(stream)), "moe_forward_ex")


def gather_rows(s, inv, slots, rows, x, x_perm, stream=None):
    _check(lib().moe_gather_rows(ctypes.byref(s), _ptr(inv), int(slots), int(rows), _ptr(x), _ptr(x_perm),
                                 _stream(stream)), "moe_gather_rows")


def expert_choice_workspace_size(s, C: int) -> int:
    return lib().moe_expert_choice_workspace_size(ctypes.byref(s), int(C))


def route_expert_choice(s, C, x, w_g, bias, probs, perm, counts, offsets, inv, w, stream=None):
    _check(lib().moe_route_expert_choice(ctypes.byref(s), int(C), _ptr(x), _ptr(w_g), _ptr(bias), _ptr(probs),
                                         _ptr(perm), _ptr(counts), _ptr(offsets), _ptr(inv), _ptr(w),
                                         _stream(stream)), "moe_route_expert_choice")


def forward_expert_choice(s, C, x, w_g, bias, w_gate, w_up, w_down, out, ws, counts=None, stream=None):
    _check(lib().moe_forward_expert_choice(ctypes.byref(s), int(C), _ptr(x), _ptr(w_g), _ptr(bias), _ptr(w_gate),
                                           _ptr(w_up), _ptr(w_down), _ptr(out), _ptr(counts), _ptr(ws), ws.numel(),
                                           _stream(stream)), "moe_forward_expert_choice")


def permute_capacity(s, topk_idx, x, capacity_factor, counts, offsets, perm, inv_perm, x_perm, ws, dropped=None,
                     stream=None):
    _check(lib().moe_permute_capacity(ctypes.byref(s), _ptr(topk_idx), _ptr(x), float(capacity_factor), _ptr(counts),
                                      _ptr(offsets), _ptr(perm), _ptr(inv_perm), _ptr(x_perm), _ptr(dropped),
                                      _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)),
           "moe_permute_capacity")


def forward_capacity(s, capacity_factor, x, w_g, bias, w_gate, w_up, w_down, out, ws, topk_idx=None, topk_w=None,
                     counts=None, dropped=None, stream=None):
    _check(lib().moe_forward_capacity(ctypes.byref(s), float(capacity_factor), _ptr(x), _ptr(w_g), _ptr(bias),
                                      _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(out), _ptr(topk_idx),
                                      _ptr(topk_w), _ptr(counts), _ptr(dropped), _ptr(ws), ws.numel(),
                                      _stream(stream)), "moe_forward_capacity")


def grouped_ffn(s, x_perm, offsets, w_gate, w_up, w_down, y_perm, ws, stream=None):
    _check(lib().moe_grouped_ffn(ctypes.byref(s), _ptr(x_perm), _ptr(offsets), _ptr(w_gate), _ptr(w_up),
                                 _ptr(w_down), _ptr(y_perm), _ptr(ws), ws.numel() if ws is not None else 0,
                                 _stream(stream)), "moe_grouped_ffn")


def ep_regroup(G, E, recv_counts, recv_x, x_local, offsets_local, local_src, dtype, stream=None):
    """Received rows (source, local expert, source order) -> grouped by local expert."""
    rows, d = int(recv_x.shape[0]), int(recv_x.shape[1])
    _check(lib().moe_ep_regroup(int(G), int(E), _ptr(recv_counts), rows, d, DTYPE[dtype], _ptr(recv_x),
                                _ptr(x_local), _ptr(offsets_local), _ptr(local_src), _stream(stream)),
           "moe_ep_regroup")


def ep_ungroup(local_src, y_local, y_recv, dtype, stream=None):
    """y_recv[local_src[i]] = y_local[i]."""
    rows, d = int(y_local.shape[0]), int(y_local.shape[1])
    _check(lib().moe_ep_ungroup(rows, d, DTYPE[dtype], _ptr(local_src), _ptr(y_local), _ptr(y_recv),
                                _stream(stream)), "moe_ep_ungroup")


def grouped_ffn_gather(s, x, perm, offsets, w_gate, w_up, w_down, y_perm, ws, stream=None):
    _check(lib().moe_grouped_ffn_gather(ctypes.byref(s), _ptr(x), _ptr(perm), _ptr(offsets), _ptr(w_gate),
                                        _ptr(w_up), _ptr(w_down), _ptr(y_perm), _ptr(ws),
                                        ws.numel() if ws is not None else 0, _stream(stream)), "moe_grouped_ffn_gather")


def combine(s, y_perm, inv_perm, topk_w, out, stream=None):
    _check(lib().moe_combine(ctypes.byref(s), _ptr(y_perm), _ptr(inv_perm), _ptr(topk_w), _ptr(out),
                             _stream(stream)), "moe_combine")


def forward(s, x, w_g, bias, w_gate, w_up, w_down, out, ws, topk_idx=None, topk_w=None, counts=None, stream=None):
    _check(lib().moe_forward(ctypes.byref(s), _ptr(x), _ptr(w_g), _ptr(bias), _ptr(w_gate), _ptr(w_up),
                             _ptr(w_down), _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(ws),
                             ws.numel(), _stream(stream)), "moe_forward")


def hostio_pipelined_workspace_size(s) -> int:
    return lib().moe_forward_hostio_pipelined_workspace_size(ctypes.byref(s))


def forward_hostio_pipelined(s, x_host, w_g, bias, w_gate, w_up, w_down, out_host, ws, slot, compute_stream,
                             h2d_stream, d2h_stream):
    _check(lib().moe_forward_hostio_pipelined(ctypes.byref(s), _host_ptr(x_host), _ptr(w_g), _ptr(bias),
                                              _ptr(w_gate), _ptr(w_up), _ptr(w_down), _host_ptr(out_host),
                                              _ptr(ws), ws.numel(), int(slot), _stream(compute_stream),
                                              _stream(h2d_stream), _stream(d2h_stream)),
           "moe_forward_hostio_pipelined")


def forward_hostio(s, x_host, w_g, bias, w_gate, w_up, w_down, out_host, ws, stream=None):
    _check(lib().moe_forward_hostio(ctypes.byref(s), _host_ptr(x_host), _ptr(w_g), _ptr(bias), _ptr(w_gate),
                                    _ptr(w_up), _ptr(w_down), _host_ptr(out_host), _ptr(ws), ws.numel(),
                                    _stream(stream)), "moe_forward_hostio")


def get_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    return lib().moe_get_error(_stream(stream))


def selftest_bounded_wait(timeout_ns: int, stream=None):
    _check(lib().moe_selftest_bounded_wait(int(timeout_ns), _stream(stream)), "moe_selftest_bounded_wait")


def set_ffn_tiling(mode: str):
    """Choose the tensor-core tiling of the grouped GEMMs: "auto", "rows", "tokens" or "pairs"."""
    _check(lib().moe_set_ffn_tiling(TILING[mode]), "moe_set_ffn_tiling")


def get_ffn_tiling() -> str:
    return {v: k for k, v in TILING.items()}[lib().moe_get_ffn_tiling()]


def version() -> int:
    return lib().moe_version()
