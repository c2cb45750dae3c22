"""Python face of the CPU oracle (oracle/moe_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the CPU
baseline leg of bench.py -- never by the product package.  Every function here takes
and returns numpy arrays and calls the C oracle; no arithmetic of the method lives
in this file beyond reshaping.

Format ids: 1 = FP8 block-128 W8A16, 2 = INT4 g128 W4A16, 3 = NVFP4 W4A16, 4 = NVFP4 W4A4,
5 = BF16, 6 = FP8 block-128 weights with FP8 1x128-group activations (W8A8).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

FMT_FP8, FMT_INT4, FMT_NVFP4_W4A16, FMT_NVFP4_W4A4, FMT_BF16, FMT_FP8_W8A8 = 1, 2, 3, 4, 5, 6
FMT_IDS = {"fp8": 1, "int4": 2, "nvfp4_w4a16": 3, "nvfp4_w4a4": 4, "bf16": 5, "fp8_w8a8": 6}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc: fp32 steps stay single IEEE operations (no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
               "-fopenmp", "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        P = C.c_void_p
        L.orc_e4m3_decode.restype = C.c_double
        L.orc_e4m3_decode.argtypes = [C.c_uint8]
        L.orc_e4m3_encode.restype = C.c_uint8
        L.orc_e4m3_encode.argtypes = [C.c_float]
        L.orc_e2m1_decode.restype = C.c_double
        L.orc_e2m1_decode.argtypes = [C.c_uint8]
        L.orc_e2m1_encode.restype = C.c_uint8
        L.orc_e2m1_encode.argtypes = [C.c_float]
        L.orc_f16_encode.restype = C.c_uint16
        L.orc_f16_encode.argtypes = [C.c_double]
        L.orc_f16_decode.restype = C.c_double
        L.orc_f16_decode.argtypes = [C.c_uint16]
        L.orc_bf16_encode.restype = C.c_uint16
        L.orc_bf16_encode.argtypes = [C.c_double]
        for f in ("orc_pack_fp8", "orc_pack_int4", "orc_pack_nvfp4", "orc_dequant_fp8", "orc_dequant_int4",
                  "orc_quant_act_nvfp4", "orc_quant_act_nvfp4_static", "orc_quant_act_fp8",
                  "orc_dequant_act_fp8", "orc_route", "orc_permute"):
            getattr(L, f).restype = None
        L.orc_pack_fp8.argtypes = [P, C.c_int, C.c_int, P, P]
        L.orc_dequant_fp8.argtypes = [P, P, C.c_int, C.c_int, P]
        L.orc_pack_int4.argtypes = [P, C.c_int, C.c_int, P, P]
        L.orc_dequant_int4.argtypes = [P, P, C.c_int, C.c_int, P]
        L.orc_pack_nvfp4.argtypes = [P, C.c_int, C.c_int, P, P, P]
        L.orc_dequant_nvfp4.restype = None
        L.orc_dequant_nvfp4.argtypes = [P, P, C.c_float, C.c_int, C.c_int, P]
        L.orc_quant_act_nvfp4.argtypes = [P, C.c_int, C.c_int, P, P, P]
        L.orc_quant_act_nvfp4_static.argtypes = [P, C.c_int, C.c_int, C.c_float, P, P]
        L.orc_quant_act_fp8.argtypes = [P, C.c_int, C.c_int, P, P]
        L.orc_dequant_act_fp8.argtypes = [P, P, C.c_int, C.c_int, P]
        L.orc_route.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P]
        L.orc_permute.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P, P]
        L.orc_moe_layer.restype = C.c_int
        L.orc_moe_layer.argtypes = [C.c_int] * 6 + [P] * 8 + [P, C.c_int, C.c_int, C.c_int, P, P]
        L.orc_max_threads.restype = C.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(C.c_void_p)


# ---- scalar codecs ----------------------------------------------------------------------
def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def f16_encode(v: float) -> int:
    return lib().orc_f16_encode(float(v))


def f16_decode(h: int) -> float:
    return lib().orc_f16_decode(int(h))


def bf16_encode(v: float) -> int:
    return lib().orc_bf16_encode(float(v))


# ---- weight formats ---------------------------------------------------------------------
def pack_fp8(w_bf16: np.ndarray):
    """w [N, K] bf16 bits -> (codes u8 [N, K], scale_inv f32 [N/128, K/128])."""
    N, K = w_bf16.shape
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    codes = np.empty((N, K), np.uint8)
    sinv = np.empty((N // 128, K // 128), np.float32)
    lib().orc_pack_fp8(_p(w), N, K, _p(codes), _p(sinv))
    return codes, sinv


def dequant_fp8(codes, sinv):
    N, K = codes.shape
    out = np.empty((N, K), np.float32)
    lib().orc_dequant_fp8(_p(np.ascontiguousarray(codes)), _p(np.ascontiguousarray(sinv)), N, K, _p(out))
    return out


def pack_int4(w_bf16: np.ndarray):
    """w [N, K] -> (qweight int32 [K/8, N], scales fp16 bits uint16 [K/128, N])."""
    N, K = w_bf16.shape
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    qw = np.empty((K // 8, N), np.int32)
    sc = np.empty((K // 128, N), np.uint16)
    lib().orc_pack_int4(_p(w), N, K, _p(qw), _p(sc))
    return qw, sc


def dequant_int4(qweight, scales):
    K8, N = qweight.shape
    K = K8 * 8
    out = np.empty((N, K), np.float32)
    lib().orc_dequant_int4(_p(np.ascontiguousarray(qweight)), _p(np.ascontiguousarray(scales)), N, K, _p(out))
    return out


def pack_nvfp4(w_bf16: np.ndarray):
    """w [N, K] -> (packed u8 [N, K/2], block scales E4M3 codes u8 [N, K/16], global scale f32)."""
    N, K = w_bf16.shape
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    pk = np.empty((N, K // 2), np.uint8)
    sc = np.empty((N, K // 16), np.uint8)
    gs = np.zeros(1, np.float32)
    lib().orc_pack_nvfp4(_p(w), N, K, _p(pk), _p(sc), _p(gs))
    return pk, sc, np.float32(gs[0])


def dequant_nvfp4(packed, scales, gs):
    N, K2 = packed.shape
    K = K2 * 2
    out = np.empty((N, K), np.float32)
    lib().orc_dequant_nvfp4(_p(np.ascontiguousarray(packed)), _p(np.ascontiguousarray(scales)), float(gs), N, K,
                            _p(out))
    return out


def quant_act_nvfp4(x_bf16: np.ndarray, static_gs=None):
    """x [T, H] bf16 bits -> (codes u8 [T, H/2], scales u8 [T, H/16], gs f32 [T]).

    static_gs None: each row's own dynamic global scale; else that one fp32 scale for every row.
    """
    T, H = x_bf16.shape
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    q = np.empty((T, H // 2), np.uint8)
    s = np.empty((T, H // 16), np.uint8)
    if static_gs is None:
        g = np.empty(T, np.float32)
        lib().orc_quant_act_nvfp4(_p(x), T, H, _p(q), _p(s), _p(g))
    else:
        g = np.full(T, np.float32(static_gs), np.float32)
        lib().orc_quant_act_nvfp4_static(_p(x), T, H, C.c_float(float(np.float32(static_gs))), _p(q), _p(s))
    return q, s, g


def quant_act_fp8(x_bf16: np.ndarray):
    """x [T, H] bf16 bits -> (codes E4M3 u8 [T, H], scale_inv f32 [T, H/128]): one scale per
    1x128 group of a row."""
    T, H = x_bf16.shape
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    q = np.empty((T, H), np.uint8)
    s = np.empty((T, H // 128), np.float32)
    lib().orc_quant_act_fp8(_p(x), T, H, _p(q), _p(s))
    return q, s


def dequant_act_fp8(codes, scale_inv):
    T, H = codes.shape
    out = np.empty((T, H), np.float32)
    lib().orc_dequant_act_fp8(_p(np.ascontiguousarray(codes)), _p(np.ascontiguousarray(scale_inv, np.float32)), T, H,
                              _p(out))
    return out


# ---- routing ----------------------------------------------------------------------------
def route(logits: np.ndarray, k: int):
    """logits [T, E] f32 -> (idx int32 [T, k], w float64 [T, k])."""
    T, E = logits.shape
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().orc_route(_p(lg), T, E, k, _p(idx), _p(w))
    return idx, w


def permute(idx: np.ndarray, E: int):
    """idx [T, k] -> (offsets int32 [E+1], perm int32 [T*k], inv int32 [T*k])."""
    T, k = idx.shape
    ii = np.ascontiguousarray(idx, dtype=np.int32)
    off = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    lib().orc_permute(_p(ii), T, E, k, _p(off), _p(perm), _p(inv))
    return off, perm, inv


# ---- packing whole expert sets ----------------------------------------------------------
def pack_experts(fmt: int, wgu: np.ndarray, wd: np.ndarray, experts=None) -> dict:
    """Pack [E, 2I, H] / [E, H, I] bf16 weights per format into canonical per-expert tensors.

    Experts not in ``experts`` (when given) are left zero-filled: cheaper for full-size
    checks that only touch routed experts.
    """
    from concurrent.futures import ThreadPoolExecutor

    E, N2, H = wgu.shape
    I = N2 // 2
    sel = range(E) if experts is None else sorted(set(int(e) for e in experts))
    pool = ThreadPoolExecutor(max_workers=os.cpu_count() or 1)  # ctypes calls release the GIL
    out = {}
    for name, W, N, K in (("gu", wgu, 2 * I, H), ("d", wd, H, I)):
        if fmt == FMT_BF16:  # unquantized: the weights as given
            a = np.zeros((E, N, K), np.uint16)
            a[list(sel)] = np.asarray(W, dtype=np.uint16)[list(sel)]
            b = g = None
        elif fmt in (FMT_FP8, FMT_FP8_W8A8):  # W8A8 stores the same FP8 block weights
            a = np.zeros((E, N, K), np.uint8)
            b = np.zeros((E, N // 128, K // 128), np.float32)
            g = None
            for e, r in zip(sel, pool.map(lambda e: pack_fp8(W[e]), sel)):
                a[e], b[e] = r
        elif fmt == FMT_INT4:
            a = np.zeros((E, K // 8, N), np.int32)
            b = np.zeros((E, K // 128, N), np.uint16)
            g = None
            for e, r in zip(sel, pool.map(lambda e: pack_int4(W[e]), sel)):
                a[e], b[e] = r
        else:
            a = np.zeros((E, N, K // 2), np.uint8)
            b = np.zeros((E, N, K // 16), np.uint8)
            g = np.ones(E, np.float32)
            for e, r in zip(sel, pool.map(lambda e: pack_nvfp4(W[e]), sel)):
                a[e], b[e], g[e] = r
        out[name] = (a, b, g)
    pool.shutdown()
    return out


def moe_layer(fmt: int, x: np.ndarray, logits: np.ndarray, packed: dict, k: int, tokens=None,
              dense: bool = False, nthreads: int = 0, act_gs=None) -> np.ndarray:
    """Forward pass in fp64 for the given tokens (all when None). Returns [n_tok, H] float64.

    act_gs (W4A4): None for dynamic per-row activation scales, else the static (x, h) pair."""
    T, H = x.shape
    E = logits.shape[1]
    gu_a, gu_b, gu_g = packed["gu"]
    d_a, d_b, d_g = packed["d"]
    I = (gu_a.shape[1] // 2) if fmt != FMT_INT4 else gu_a.shape[2] // 2
    xx = np.ascontiguousarray(x, dtype=np.uint16)
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    if tokens is None:
        tok_p, n_tok = None, T
    else:
        tk = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        tok_p, n_tok = _p(tk), len(tk)
    out = np.empty((n_tok, H), np.float64)
    none = C.c_void_p(0)
    ags = None if act_gs is None else np.ascontiguousarray(np.asarray(act_gs, dtype=np.float32))
    rc = lib().orc_moe_layer(fmt, T, H, I, E, k, _p(xx), _p(lg), _p(gu_a), _p(gu_b) if gu_b is not None else none,
                             _p(gu_g) if gu_g is not None else none, _p(d_a), _p(d_b) if d_b is not None else none,
                             _p(d_g) if d_g is not None else none, tok_p, n_tok, int(dense), int(nthreads),
                             _p(ags) if ags is not None else none, _p(out))
    if rc != 0:
        raise ValueError(f"orc_moe_layer rejected its arguments (rc={rc})")
    return out


def max_threads() -> int:
    return lib().orc_max_threads()
