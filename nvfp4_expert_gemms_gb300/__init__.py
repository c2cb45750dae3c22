"""Thin Python binding of libmoe_gb300.so (include/moe_gb300.h).

Argument marshalling only: every step of the forward pass runs in the library's CUDA
kernels.  torch supplies device memory and streams.  There is no fallback: if the
library cannot be loaded, every call raises.

Names mirror the C ABI: moe_packed_size, moe_pack_experts, moe_workspace_size,
moe_layer_forward, moe_workspace_size_host_io, moe_layer_forward_host,
moe_get_device_error, moe_status_string, moe_debug_route, moe_debug_dequant,
moe_debug_quant_act.
"""
from __future__ import annotations

import ctypes as C
import os

from . import _build

FMT_FP8 = 1
FMT_INT4 = 2
FMT_NVFP4_W4A16 = 3
FMT_NVFP4_W4A4 = 4
FMT_BF16 = 5
FMT_FP8_W8A8 = 6
FORMATS = {"fp8": FMT_FP8, "int4": FMT_INT4, "nvfp4_w4a16": FMT_NVFP4_W4A16, "nvfp4_w4a4": FMT_NVFP4_W4A4,
           "bf16": FMT_BF16, "fp8_w8a8": FMT_FP8_W8A8}

MOE_T_GU_A, MOE_T_GU_B, MOE_T_D_A, MOE_T_D_B, MOE_T_GU_GS, MOE_T_D_GS, MOE_T_GU_IMG, MOE_T_D_IMG = range(8)

EXPORTS = ("moe_packed_size", "moe_pack_experts", "moe_workspace_size", "moe_layer_forward",
           "moe_workspace_size_host_io", "moe_layer_forward_host", "moe_get_device_error", "moe_status_string",
           "moe_debug_route", "moe_debug_dequant", "moe_debug_quant_act", "moe_kernel_launch_count",
           "moe_time_next_step", "moe_layer_forward_static_act", "moe_calibrate_act_scales",
           "moe_debug_quant_act_static", "moe_debug_quant_act_fp8", "moe_debug_wait_timeout")


class PackedDesc(C.Structure):
    _fields_ = [("fmt", C.c_int32), ("E", C.c_int32), ("H", C.c_int32), ("I", C.c_int32),
                ("bytes", C.c_uint64), ("offset", C.c_uint64 * 8), ("size", C.c_uint64 * 8)]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {moe_status_string(status)} (status {status})")


_lib = None


def lib() -> C.CDLL:
    """Load the in-tree library (building it first when its sources are newer)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not _build.up_to_date():
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError("libmoe_gb300.so is missing and could not be built")
        L = C.CDLL(path)
        P, I32, SZ = C.c_void_p, C.c_int, C.c_size_t
        PD = C.POINTER(PackedDesc)
        for name in EXPORTS:
            getattr(L, name).restype = C.c_int
        L.moe_status_string.restype = C.c_char_p
        L.moe_status_string.argtypes = [I32]
        L.moe_packed_size.argtypes = [I32, I32, I32, I32, PD]
        L.moe_pack_experts.argtypes = [PD, P, P, P, P]
        L.moe_workspace_size.argtypes = [PD, I32, I32, C.POINTER(SZ)]
        L.moe_workspace_size_host_io.argtypes = [PD, I32, I32, C.POINTER(SZ)]
        L.moe_layer_forward.argtypes = [P, P, I32, PD, P, I32, P, P, SZ, P]
        L.moe_layer_forward_host.argtypes = [P, P, I32, PD, P, I32, P, P, SZ, P]
        L.moe_get_device_error.argtypes = [P, P, C.POINTER(C.c_int32)]
        L.moe_debug_route.argtypes = [P, I32, I32, I32, P, P, P, P, P, P, SZ, P]
        L.moe_debug_dequant.argtypes = [PD, P, I32, I32, P, P]
        L.moe_debug_quant_act.argtypes = [P, I32, I32, P, P, P, P]
        L.moe_debug_quant_act_static.argtypes = [P, I32, I32, P, P, P, P]
        L.moe_debug_quant_act_fp8.argtypes = [P, I32, I32, P, P, P]
        L.moe_debug_wait_timeout.argtypes = [P, P]
        L.moe_layer_forward_static_act.argtypes = [P, P, I32, PD, P, I32, P, P, P, SZ, P]
        L.moe_calibrate_act_scales.argtypes = [P, P, I32, PD, P, I32, P, P, SZ, P]
        L.moe_kernel_launch_count.restype = C.c_uint64
        L.moe_kernel_launch_count.argtypes = []
        L.moe_time_next_step.argtypes = [I32, P, P]
        _lib = L
    return _lib


def _check(st: int, where: str):
    if st != 0:
        raise MoEError(st, where)


def _stream(stream):
    import torch

    if stream is None:
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _ptr(t):
    return C.c_void_p(0 if t is None else t.data_ptr())


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def moe_packed_size(fmt, E: int, H: int, I: int) -> PackedDesc:
    d = PackedDesc()
    f = FORMATS[fmt] if isinstance(fmt, str) else int(fmt)
    _check(lib().moe_packed_size(f, E, H, I, C.byref(d)), "moe_packed_size")
    return d


def moe_pack_experts(desc: PackedDesc, w_gate_up, w_down, packed, stream=None):
    _check(lib().moe_pack_experts(C.byref(desc), _ptr(w_gate_up), _ptr(w_down), _ptr(packed), _stream(stream)),
           "moe_pack_experts")


def moe_workspace_size(desc: PackedDesc, T: int, top_k: int) -> int:
    n = C.c_size_t()
    _check(lib().moe_workspace_size(C.byref(desc), T, top_k, C.byref(n)), "moe_workspace_size")
    return n.value


def moe_workspace_size_host_io(desc: PackedDesc, T: int, top_k: int) -> int:
    n = C.c_size_t()
    _check(lib().moe_workspace_size_host_io(C.byref(desc), T, top_k, C.byref(n)), "moe_workspace_size_host_io")
    return n.value


def moe_layer_forward(x, router_logits, desc: PackedDesc, packed, top_k: int, out, workspace, stream=None):
    T = int(x.shape[0])
    _check(lib().moe_layer_forward(_ptr(x), _ptr(router_logits), T, C.byref(desc), _ptr(packed), top_k, _ptr(out),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_layer_forward")


def moe_layer_forward_static_act(x, router_logits, desc: PackedDesc, packed, top_k: int, act_gs, out, workspace,
                                 stream=None):
    """W4A4 with static activation scales act_gs (device f32 [2]: x's, then h's)."""
    T = int(x.shape[0])
    _check(lib().moe_layer_forward_static_act(_ptr(x), _ptr(router_logits), T, C.byref(desc), _ptr(packed), top_k,
                                              _ptr(act_gs), _ptr(out), _ptr(workspace),
                                              workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_layer_forward_static_act")


def moe_calibrate_act_scales(x, router_logits, desc: PackedDesc, packed, top_k: int, workspace, stream=None):
    """The static W4A4 activation scales of this batch: device f32 [2] (x's, then h's)."""
    import torch

    T = int(x.shape[0])
    act_gs = torch.empty(2, dtype=torch.float32, device=x.device)
    _check(lib().moe_calibrate_act_scales(_ptr(x), _ptr(router_logits), T, C.byref(desc), _ptr(packed), top_k,
                                          _ptr(act_gs), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _stream(stream)), "moe_calibrate_act_scales")
    return act_gs


def moe_layer_forward_host(x_host, logits_host, desc: PackedDesc, packed, top_k: int, out_host, workspace,
                           stream=None):
    T = int(x_host.shape[0])
    _check(lib().moe_layer_forward_host(_ptr(x_host), _ptr(logits_host), T, C.byref(desc), _ptr(packed), top_k,
                                        _ptr(out_host), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_layer_forward_host")


def moe_get_device_error(workspace, stream=None) -> int:
    code = C.c_int32()
    _check(lib().moe_get_device_error(_ptr(workspace), _stream(stream), C.byref(code)), "moe_get_device_error")
    return code.value


def moe_kernel_launch_count() -> int:
    return int(lib().moe_kernel_launch_count())


def moe_time_next_step(step: int, start_event=None, stop_event=None):
    """Record torch.cuda.Event pair around GEMM step `step` (0 gate/up, 1 down) of the next
    forward call made by this thread."""
    s = C.c_void_p(start_event.cuda_event if start_event is not None else 0)
    e = C.c_void_p(stop_event.cuda_event if stop_event is not None else 0)
    _check(lib().moe_time_next_step(step, s, e), "moe_time_next_step")


def moe_debug_route(router_logits, top_k: int, workspace, stream=None):
    """Returns (topk_idx, topk_w, offsets, perm, inv) as new device tensors."""
    import torch

    T, E = (int(s) for s in router_logits.shape)
    dev = router_logits.device
    idx = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    w = torch.empty((T, top_k), dtype=torch.float32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * top_k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * top_k, dtype=torch.int32, device=dev)
    _check(lib().moe_debug_route(_ptr(router_logits), T, E, top_k, _ptr(idx), _ptr(w), _ptr(off), _ptr(perm),
                                 _ptr(inv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)), "moe_debug_route")
    return idx, w, off, perm, inv


def moe_debug_dequant(desc: PackedDesc, packed, expert: int, which: int, stream=None):
    import torch

    N, K = (2 * desc.I, desc.H) if which == 0 else (desc.H, desc.I)
    out = torch.empty((N, K), dtype=torch.float32, device=packed.device)
    _check(lib().moe_debug_dequant(C.byref(desc), _ptr(packed), expert, which, _ptr(out), _stream(stream)),
           "moe_debug_dequant")
    return out


def moe_debug_quant_act_static(x, gs_static, stream=None):
    """NVFP4 codes and block scales of x's rows with one static global scale (device f32 [1])."""
    import torch

    T, H = (int(s) for s in x.shape)
    q = torch.empty((T, H // 2), dtype=torch.uint8, device=x.device)
    s = torch.empty((T, H // 16), dtype=torch.uint8, device=x.device)
    _check(lib().moe_debug_quant_act_static(_ptr(x), T, H, _ptr(gs_static), _ptr(q), _ptr(s), _stream(stream)),
           "moe_debug_quant_act_static")
    return q, s


def moe_debug_quant_act_fp8(x, stream=None):
    """E4M3 codes [T, H] and fp32 scale_inv [T, H/128] of x's rows, one scale per 1x128 group."""
    import torch

    T, H = (int(s) for s in x.shape)
    q = torch.empty((T, H), dtype=torch.uint8, device=x.device)
    s = torch.empty((T, H // 128), dtype=torch.float32, device=x.device)
    _check(lib().moe_debug_quant_act_fp8(_ptr(x), T, H, _ptr(q), _ptr(s), _stream(stream)), "moe_debug_quant_act_fp8")
    return q, s


def moe_debug_wait_timeout(workspace, stream=None):
    """Enqueue a device wait that runs out (about a second) and records MOE_ERR_DEVICE_TIMEOUT in
    the workspace's error word; read it with moe_get_device_error."""
    _check(lib().moe_debug_wait_timeout(_ptr(workspace), _stream(stream)), "moe_debug_wait_timeout")


def moe_debug_quant_act(x, stream=None):
    import torch

    T, H = (int(s) for s in x.shape)
    q = torch.empty((T, H // 2), dtype=torch.uint8, device=x.device)
    s = torch.empty((T, H // 16), dtype=torch.uint8, device=x.device)
    g = torch.empty(T, dtype=torch.float32, device=x.device)
    _check(lib().moe_debug_quant_act(_ptr(x), T, H, _ptr(q), _ptr(s), _ptr(g), _stream(stream)),
           "moe_debug_quant_act")
    return q, s, g


def packed_view(desc: PackedDesc, packed, which: int):
    """Canonical tensor `which` (MOE_T_*) of a packed buffer as a typed torch view (no copy)."""
    import torch

    E, H, I = desc.E, desc.H, desc.I
    o, n = int(desc.offset[which]), int(desc.size[which])
    raw = packed[o:o + n]
    fmt = desc.fmt
    gu = which in (MOE_T_GU_A, MOE_T_GU_B, MOE_T_GU_IMG)
    N, K = (2 * I, H) if gu else (H, I)
    if which in (MOE_T_GU_GS, MOE_T_D_GS):
        return raw.view(torch.float32)
    if which in (MOE_T_GU_IMG, MOE_T_D_IMG) and fmt == FMT_NVFP4_W4A16:  # the bf16 converter's weight image
        return raw.view(E, K // 128, N // 128, 9216)
    if which in (MOE_T_GU_IMG, MOE_T_D_IMG):  # tensor-core operand image (include/moe_gb300.h)
        return raw.view(E, N // 256 if gu else (N + 255) // 256, (K + 255) // 256, 36864)
    if fmt == FMT_BF16:
        return raw.view(torch.bfloat16).view(E, N, K)
    if fmt in (FMT_FP8, FMT_FP8_W8A8):
        return raw.view(E, N, K) if which in (MOE_T_GU_A, MOE_T_D_A) else raw.view(torch.float32).view(
            E, N // 128, K // 128)
    if fmt == FMT_INT4:
        return raw.view(torch.int32).view(E, K // 8, N) if which in (MOE_T_GU_A, MOE_T_D_A) else raw.view(
            torch.float16).view(E, K // 128, N)
    return raw.view(E, N, K // 2) if which in (MOE_T_GU_A, MOE_T_D_A) else raw.view(E, N, K // 16)


class MoELayer:
    """Convenience holder: packed experts of one layer plus a reusable workspace."""

    def __init__(self, fmt, w_gate_up, w_down, stream=None):
        import torch

        E, N2, H = (int(s) for s in w_gate_up.shape)
        self.desc = moe_packed_size(fmt, E, H, N2 // 2)
        self.packed = torch.empty(self.desc.bytes, dtype=torch.uint8, device=w_gate_up.device)
        moe_pack_experts(self.desc, w_gate_up.contiguous(), w_down.contiguous(), self.packed, stream)
        self.workspace = None

    def ensure_workspace(self, T: int, top_k: int, host_io: bool = False):
        import torch

        n = (moe_workspace_size_host_io if host_io else moe_workspace_size)(self.desc, T, top_k)
        if self.workspace is None or self.workspace.numel() < n:
            self.workspace = torch.empty(n, dtype=torch.uint8, device=self.packed.device)
        return self.workspace

    def forward(self, x, router_logits, top_k: int, out=None, stream=None):
        import torch

        if out is None:
            out = torch.empty_like(x)
        ws = self.ensure_workspace(int(x.shape[0]), top_k)
        moe_layer_forward(x, router_logits, self.desc, self.packed, top_k, out, ws, stream)
        return out
