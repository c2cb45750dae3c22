"""Host-side checks of the C ABI (no GPU): the library loads, exports every function that
include/*.h declares, and the host-only calls (layouts, sizes, argument checks) behave."""
import ctypes as C
import glob
import os
import re

import numpy as np
import pytest

import nvfp4_expert_gemms_gb300 as M

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_function():
    lib = M.lib()
    names = declared_functions()
    assert {"moe_layer_forward", "moe_pack_experts", "moe_packed_size"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(M.EXPORTS) <= names


def test_packed_sizes_match_canonical_shapes(orc):
    H, I, E = 2048, 768, 128
    per_expert = {"fp8": 4_719_744, "int4": 2_433_024, "nvfp4_w4a16": 2_654_216}
    for fmt, want in per_expert.items():
        d = M.moe_packed_size(fmt, E, H, I)
        got = sum(int(d.size[i]) for i in range(6))  # the canonical tensors (no images)
        assert got == E * want, (fmt, got)
        assert all(int(d.offset[i]) % 256 == 0 for i in range(8))
        assert d.bytes >= got
    # the NVFP4 layer is the 0.32 GiB the page quotes (canonical tensors; the W4A4 buffer adds
    # the two matrices' tensor-core operand images, the same codes and scales rearranged)
    d = M.moe_packed_size("nvfp4_w4a4", E, H, I)
    assert round(sum(int(d.size[i]) for i in range(6)) / 2 ** 30, 2) == 0.32
    assert int(d.size[M.MOE_T_GU_IMG]) == int(d.size[M.MOE_T_GU_A]) + int(d.size[M.MOE_T_GU_B])
    assert int(d.size[M.MOE_T_D_IMG]) == int(d.size[M.MOE_T_D_A]) + int(d.size[M.MOE_T_D_B])
    # W4A16 repeats codes and scales as the bf16 converter's image: 9 KB per 128-row tile and chunk
    d = M.moe_packed_size("nvfp4_w4a16", E, H, I)
    assert int(d.size[M.MOE_T_GU_IMG]) == int(d.size[M.MOE_T_GU_A]) + int(d.size[M.MOE_T_GU_B])
    assert int(d.size[M.MOE_T_D_IMG]) == int(d.size[M.MOE_T_D_A]) + int(d.size[M.MOE_T_D_B])
    assert int(d.size[M.MOE_T_GU_IMG]) == E * (2 * I // 128) * (H // 128) * 9216
    # K not a multiple of 256 and H not of 256: whole 36 KB blocks per (tile pair, 256-column
    # chunk), the last chunk half used, the last down pair's second tile empty
    d = M.moe_packed_size("nvfp4_w4a4", 3, 384, 640)
    assert int(d.size[M.MOE_T_GU_IMG]) == 3 * (640 // 128) * 2 * 36864
    assert int(d.size[M.MOE_T_D_IMG]) == 3 * 2 * 3 * 36864


def test_packed_tensor_sizes_equal_oracle_outputs(orc):
    import synth

    wgu, wd = synth.gen_expert_weights(2, 256, 128, seed=0)
    for fmt_name, fid in (("fp8", 1), ("int4", 2), ("nvfp4_w4a16", 3), ("fp8_w8a8", 6)):
        p = orc.pack_experts(fid, wgu, wd)
        d = M.moe_packed_size(fmt_name, 2, 256, 128)
        assert int(d.size[M.MOE_T_GU_A]) == p["gu"][0].nbytes
        assert int(d.size[M.MOE_T_GU_B]) == p["gu"][1].nbytes
        assert int(d.size[M.MOE_T_D_A]) == p["d"][0].nbytes
        assert int(d.size[M.MOE_T_D_B]) == p["d"][1].nbytes


def test_argument_errors_are_synchronous():
    lib = M.lib()
    d = M.PackedDesc()
    assert lib.moe_packed_size(9, 8, 256, 128, C.byref(d)) == 1
    assert lib.moe_packed_size(1, 8, 200, 128, C.byref(d)) == 1
    assert lib.moe_packed_size(1, 300, 256, 128, C.byref(d)) == 1
    assert lib.moe_packed_size(1, 8, 256, 128, C.byref(d)) == 0
    n = C.c_size_t()
    assert lib.moe_workspace_size(C.byref(d), 16, 0, C.byref(n)) == 1
    assert lib.moe_workspace_size(C.byref(d), 16, 9, C.byref(n)) == 1
    assert lib.moe_workspace_size(C.byref(d), 16, 2, C.byref(n)) == 0 and n.value > 0
    # forward with a too-small workspace is refused before any CUDA call
    st = lib.moe_layer_forward(C.c_void_p(256), C.c_void_p(256), 16, C.byref(d), C.c_void_p(256), 2,
                               C.c_void_p(512), C.c_void_p(1024), 16, None)
    assert st == 3
    assert lib.moe_layer_forward(C.c_void_p(256), C.c_void_p(256), 16, C.byref(d), C.c_void_p(256), 2,
                                 C.c_void_p(256), C.c_void_p(1024), 1 << 30, None) == 1  # x aliases out
    assert M.moe_status_string(3) == "workspace too small"


def test_workspace_grows_with_tokens():
    d = M.moe_packed_size("nvfp4_w4a4", 128, 2048, 768)
    a = M.moe_workspace_size(d, 1, 8)
    b = M.moe_workspace_size(d, 16384, 8)
    assert b > a > 0
    assert M.moe_workspace_size_host_io(d, 16, 8) > M.moe_workspace_size(d, 16, 8)


def test_w8a8_layout_and_workspace():
    """W8A8 stores the W8A16 FP8 tensors unchanged; its workspace adds the E4M3 codes and the
    1x128-group scales of x and h for every permuted row; H not a multiple of 256 is refused
    by the forward pass before anything is launched."""
    E, H, I, T, k = 128, 2048, 768, 4096, 8
    a, b = M.moe_packed_size("fp8", E, H, I), M.moe_packed_size("fp8_w8a8", E, H, I)
    assert b.fmt == M.FMT_FP8_W8A8 and a.bytes == b.bytes
    assert [int(a.offset[i]) for i in range(8)] == [int(b.offset[i]) for i in range(8)]
    R = T * k
    sf_rows = R + 128
    act = R * H + 4 * sf_rows * (H // 128) + R * I + 4 * sf_rows * (I // 128)
    assert M.moe_workspace_size(b, T, k) >= act
    assert M.moe_workspace_size(b, T, k) > M.moe_workspace_size(b, T // 2, k)
    lib = M.lib()
    d = M.PackedDesc()
    assert lib.moe_packed_size(6, 8, 384, 128, C.byref(d)) == 0  # packing and layout: any multiple of 128
    n = C.c_size_t()
    assert lib.moe_workspace_size(C.byref(d), 16, 2, C.byref(n)) == 0
    st = lib.moe_layer_forward(C.c_void_p(256), C.c_void_p(256), 16, C.byref(d), C.c_void_p(256), 2,
                               C.c_void_p(512), C.c_void_p(1024), n.value, None)
    assert st == 2  # MOE_ERR_UNSUPPORTED: H = 384 is not a multiple of 256
    assert lib.moe_debug_quant_act_fp8(C.c_void_p(256), 4, 200, C.c_void_p(512), C.c_void_p(1024), None) == 1


def test_w4a16_converter_bit_order():
    """The header's W4A16 bit order uses every bit of a word once, and the converter's four
    shift-and-mask steps (pair 0: << 6, pair 1: << 2, pair 2: rotate right 4, pair 3: in place
    plus the mantissa bits >> 8, each masked to a bf16 pair's sign, low exponent bits and top
    mantissa bit) give, for every pair of codes, bf16 values equal to code * 2^-126 with the
    code's sign; and every normal E4M3 block scale, its 7 magnitude bits times 16 plus 0x7600,
    is bf16(scale * 2^116).  Their product is the weight * 2^-10, which the epilogue undoes."""
    import w4a16_bits

    assert sorted(b for d in w4a16_bits.DST for b in d) == list(range(32))
    e2m1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    c = np.arange(2 ** 16, dtype=np.uint64)
    canon = (c | (c << np.uint64(16))).astype("<u4")  # every (byte 0, byte 1) pair; bytes 2, 3 repeat them
    x = w4a16_bits.words(canon.view(np.uint8)).astype(np.uint64)
    m32, pair = np.uint64(0xFFFFFFFF), np.uint64(0x81C081C0)
    steps = [((x << np.uint64(6)) & m32) & pair, ((x << np.uint64(2)) & m32) & pair,
             (((x >> np.uint64(4)) | (x << np.uint64(28))) & m32) & pair,
             (x & np.uint64(0x81808180)) | ((x >> np.uint64(8)) & np.uint64(0x00400040))]
    for j, o in enumerate(steps):
        o = o.astype(np.uint32)
        for half in (0, 1):
            h = (o >> np.uint32(16 * half)) & np.uint32(0xFFFF)
            val = (h << np.uint32(16)).view(np.float32).astype(np.float64) * 2.0 ** 126
            code = ((canon.astype(np.uint64) >> np.uint64(8 * j + 4 * half)) & np.uint64(15)).astype(np.int64)
            assert np.array_equal(val, e2m1[code]), (j, half)
            assert np.array_equal(h >> np.uint32(15), (code >> 3).astype(np.uint32)), (j, half)  # signed zeros too
    for byte in range(1, 0x7F):
        e, m = byte >> 3, byte & 7
        if e == 0:
            continue  # zero and subnormal scales take the fp32 route
        want = 2.0 ** (e - 7) * (1 + m / 8) * 2.0 ** 116
        bits = np.array([(byte * 16 + 0x7600) << 16], np.uint32)
        assert float(bits.view(np.float32)[0]) == want, hex(byte)
