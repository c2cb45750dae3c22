"""GPU parity: the CUDA library against the CPU oracle on the same seeded inputs.

Integer work (packed codes, routing indices, permutation, activation codes) must be
bit-exact; dequantized weights bit-exact; routing weights within 1e-6 relative (expf is
not correctly rounded); layer outputs within relative Frobenius 1e-2 and per-element
2e-2 * max|ref| of the oracle's fp64 result.
"""
import numpy as np
import pytest
import torch

import nvfp4_expert_gemms_gb300 as M
import synth
import w4a16_bits

pytestmark = pytest.mark.gpu

FMTS = ["fp8", "int4", "nvfp4_w4a16", "nvfp4_w4a4", "bf16"]
FID = {"fp8": 1, "int4": 2, "nvfp4_w4a16": 3, "nvfp4_w4a4": 4, "bf16": 5, "fp8_w8a8": 6}
REL_FRO, REL_MAX = 1e-2, 2e-2


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_close(got, ref, what=""):
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64)
    assert np.all(np.isfinite(got)), what
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
    assert fro <= REL_FRO and mx <= REL_MAX, f"{what}: rel fro {fro:.3e}, rel max {mx:.3e}"
    return fro, mx


class Case:
    def __init__(self, fmt, T, H, I, E, k, seed=0, zipf=None, experts_for_oracle="routed"):
        self.fmt, self.T, self.H, self.I, self.E, self.k = fmt, T, H, I, E, k
        self.x = synth.gen_x(T, H, seed)
        self.lg = synth.gen_logits(T, E, seed, zipf_alpha=zipf)
        self.wgu, self.wd = synth.gen_expert_weights(E, H, I, seed)
        self.layer = M.MoELayer(fmt, dev_bf16(self.wgu), dev_bf16(self.wd))

    def run(self):
        x = dev_bf16(self.x)
        lg = torch.from_numpy(self.lg).cuda()
        out = self.layer.forward(x, lg, self.k)
        torch.cuda.synchronize()
        assert M.moe_get_device_error(self.layer.workspace) == 0
        return host_bits(out)

    def oracle(self, orc, tokens=None):
        idx, _ = orc.route(self.lg if tokens is None else self.lg[tokens], self.k)
        p = orc.pack_experts(FID[self.fmt], self.wgu, self.wd, experts=np.unique(idx))
        return orc.moe_layer(FID[self.fmt], self.x, self.lg, p, self.k, tokens=tokens)


# ------------------------------------------------------------------ packing and dequant
@pytest.mark.parametrize("fmt", ["fp8", "int4", "nvfp4_w4a16"])
def test_pack_bit_exact(orc, fmt):
    E, H, I = 3, 384, 256
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=5)
    wgu[1, 7, :] = 0  # a zero row: INT4 zero scale, NVFP4 zero blocks
    wd[2, :128, :128] = 0  # a zero FP8 tile
    layer = M.MoELayer(fmt, dev_bf16(wgu), dev_bf16(wd))
    torch.cuda.synchronize()
    ref = orc.pack_experts(FID[fmt], wgu, wd)
    d = layer.desc
    for which, name in ((M.MOE_T_GU_A, ("gu", 0)), (M.MOE_T_GU_B, ("gu", 1)), (M.MOE_T_D_A, ("d", 0)),
                        (M.MOE_T_D_B, ("d", 1))):
        got = M.packed_view(d, layer.packed, which).cpu().numpy()
        want = ref[name[0]][name[1]]
        assert got.tobytes() == np.ascontiguousarray(want).tobytes(), (fmt, which)
    if fmt.startswith("nvfp4"):
        for which, name in ((M.MOE_T_GU_GS, "gu"), (M.MOE_T_D_GS, "d")):
            got = M.packed_view(d, layer.packed, which).cpu().numpy()
            assert got.tobytes() == ref[name][2].tobytes()


def test_bf16_pack_and_dequant_are_the_weights():
    """BF16 'packing' stores the weights as given, and the dequant view widens them exactly."""
    E, H, I = 3, 256, 128
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=8)
    layer = M.MoELayer("bf16", dev_bf16(wgu), dev_bf16(wd))
    torch.cuda.synchronize()
    for which, w in ((M.MOE_T_GU_A, wgu), (M.MOE_T_D_A, wd)):
        got = M.packed_view(layer.desc, layer.packed, which).cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, w)
    for which, w in ((0, wgu), (1, wd)):
        for e in range(E):
            got = M.moe_debug_dequant(layer.desc, layer.packed, e, which).cpu().numpy()
            assert got.tobytes() == synth.bf16_bits_to_f32(w[e]).tobytes()


def _operand_image(codes, scales, N, K, gu):
    """The W4A4 weight operand image as the header defines it, built from canonical codes
    [E, N, K/2] and scales [E, N, K/16]: block [e, p, c] = codes of tile 0 and tile 1 (128 rows x
    128 bytes, 16-byte piece j of row l at piece j ^ (l % 8)), then their scales (byte
    512 s + 16 (l % 32) + 4 (l // 32) + i = scale of row l, block 16c + 4s + i); zero past N, K."""
    E = codes.shape[0]
    C, P = (K + 255) // 256, (N // 256 if gu else (N + 255) // 256)
    img = np.zeros((E, P, C, 36864), np.uint8)
    ln = np.arange(128)
    for p in range(P):
        for g in range(2):
            rows = (128 * p + ln if g == 0 else N // 2 + 128 * p + ln) if gu else 256 * p + 128 * g + ln
            ok = rows < N
            for c in range(C):
                kb = min(128, K // 2 - 128 * c)
                lines = np.zeros((E, 128, 128), np.uint8)
                lines[:, ok, :kb] = codes[:, rows[ok], 128 * c:128 * c + kb]
                sw = np.zeros((E, 128, 8, 16), np.uint8)
                pieces = lines.reshape(E, 128, 8, 16)
                for j in range(8):
                    sw[:, ln, j ^ (ln & 7)] = pieces[:, :, j]
                img[:, p, c, 16384 * g:16384 * (g + 1)] = sw.reshape(E, 16384)
                sb = np.zeros((E, 128, 16), np.uint8)
                sb[:, ok, :kb // 8] = scales[:, rows[ok], 16 * c:16 * c + kb // 8]
                atoms = sb.reshape(E, 4, 32, 4, 4).transpose(0, 3, 2, 1, 4)
                img[:, p, c, 32768 + 2048 * g:32768 + 2048 * (g + 1)] = atoms.reshape(E, 2048)
    return img


def test_w4a16_converter_image():
    """The W4A16 buffer's weight image holds the canonical codes (each 32-bit word's bits moved
    as the header's table says, pieces swizzled) and scales, per 128-row tile and 128-column
    chunk; gate/up tiles pair 64 gate rows with the same features' up rows."""
    E, H, I = 3, 384, 256
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=9)
    layer = M.MoELayer("nvfp4_w4a16", dev_bf16(wgu), dev_bf16(wd))
    torch.cuda.synchronize()
    d = layer.desc
    for ca, cb, im, (N, K), gu in ((M.MOE_T_GU_A, M.MOE_T_GU_B, M.MOE_T_GU_IMG, (2 * I, H), True),
                                   (M.MOE_T_D_A, M.MOE_T_D_B, M.MOE_T_D_IMG, (H, I), False)):
        codes = M.packed_view(d, layer.packed, ca).cpu().numpy().reshape(E, N, K // 2)
        sc = M.packed_view(d, layer.packed, cb).cpu().numpy().reshape(E, N, K // 16)
        got = M.packed_view(d, layer.packed, im).cpu().numpy()
        want = w4a16_bits.image(codes, sc, gu)
        assert got.shape == want.shape
        assert got.tobytes() == want.tobytes(), gu


@pytest.mark.parametrize("H,I", [(512, 256), (384, 640)])
def test_w4a4_weight_image(orc, H, I):
    """The W4A4 buffer's operand images hold exactly the canonical codes and scales (bit-exact
    with the oracle's packing), rearranged as the header's layout says -- including a last half
    chunk (K % 256 = 128) and a down tile pair whose second tile lies past H."""
    E = 3
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=6)
    layer = M.MoELayer("nvfp4_w4a4", dev_bf16(wgu), dev_bf16(wd))
    torch.cuda.synchronize()
    ref = orc.pack_experts(FID["nvfp4_w4a4"], wgu, wd)
    d = layer.desc
    for ca, cb, im, name, (N, K), gu in ((M.MOE_T_GU_A, M.MOE_T_GU_B, M.MOE_T_GU_IMG, "gu", (2 * I, H), True),
                                         (M.MOE_T_D_A, M.MOE_T_D_B, M.MOE_T_D_IMG, "d", (H, I), False)):
        codes = M.packed_view(d, layer.packed, ca).cpu().numpy()
        sc = M.packed_view(d, layer.packed, cb).cpu().numpy()
        assert codes.tobytes() == np.ascontiguousarray(ref[name][0]).tobytes()
        assert sc.tobytes() == np.ascontiguousarray(ref[name][1]).tobytes()
        got = M.packed_view(d, layer.packed, im).cpu().numpy()
        want = _operand_image(codes.reshape(E, N, K // 2), sc.reshape(E, N, K // 16), N, K, gu)
        assert got.shape == want.shape
        assert got.tobytes() == want.tobytes(), name


@pytest.mark.parametrize("fmt", ["fp8", "int4", "nvfp4_w4a16"])
def test_dequant_view_bit_exact(orc, fmt):
    E, H, I = 2, 256, 128
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=6)
    layer = M.MoELayer(fmt, dev_bf16(wgu), dev_bf16(wd))
    ref = orc.pack_experts(FID[fmt], wgu, wd)
    for e in range(E):
        for which, key in ((0, "gu"), (1, "d")):
            got = M.moe_debug_dequant(layer.desc, layer.packed, e, which).cpu().numpy()
            a, b, g = ref[key]
            if fmt == "fp8":
                want = orc.dequant_fp8(a[e], b[e])
            elif fmt == "int4":
                want = orc.dequant_int4(a[e], b[e])
            else:
                want = orc.dequant_nvfp4(a[e], b[e], g[e])
            assert got.tobytes() == want.tobytes()


def test_quant_act_bit_exact(orc):
    x = synth.gen_x(33, 2048, seed=7)
    x[5] = 0  # an all-zero row: amax clamp
    q, s, g = M.moe_debug_quant_act(dev_bf16(x))
    rq, rs, rg = orc.quant_act_nvfp4(x)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert g.cpu().numpy().tobytes() == rg.tobytes()


# ------------------------------------------------------------------ routing
def _tie_rows(T, K, seed):
    """Rows whose block quotients v/eff land exactly on the E2M1 rounding boundaries.

    Element 0 is 2688 * 2^m, so gs = 2^-m and eff = bs / gs keeps v/eff independent of m.
    Block 0 (eff = 448): the boundaries 0.25 .. 5 times 448, their negatives, and -1 (rounds
    to -0).  Block 1 (eff = 2, exact reciprocal): boundaries, one bf16 step either side, the
    saturating maximum 12.  Block 2: zeros and -0.0 (block scale 0).  Block 3 (eff = 3,
    inexact reciprocal): boundaries times 3.  The remaining blocks are ~N(0,1) * 2^m.
    """
    rng = np.random.default_rng(seed)
    bnd = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    b0 = [2688.0] + [t * 448 for t in bnd] + [-t * 448 for t in bnd] + [-1.0]
    def step(v, d):  # the bf16 value d units in the last place away from v (same sign)
        b = synth.f32_to_bf16_bits(np.array([v], np.float32)).astype(np.int32) + d
        return float(synth.bf16_bits_to_f32(b.astype(np.uint16))[0])

    b1 = [12.0] + [2 * t for t in bnd] + [step(2 * t, 1) for t in bnd[:4]] + [-step(2 * t, -1) for t in bnd[:4]]
    b2 = [0.0] * 15 + [-0.0]
    b3 = [18.0] + [3 * t for t in bnd] + [-3 * t for t in bnd] + [-(2.0 ** -7)]
    blocks = [b0, b1, b2, b3]
    nb = K // 16
    x = (rng.standard_normal((T, K))).astype(np.float32)
    for r in range(T):
        m = float(2.0 ** ((r % 9) - 4))
        row = x[r] * m
        for i, b in enumerate(blocks[:nb]):
            row[16 * i:16 * (i + 1)] = np.array(b, np.float32) * m
        x[r] = row
    bits = synth.f32_to_bf16_bits(x)
    n = 16 * min(nb, len(blocks))
    assert np.array_equal(synth.bf16_bits_to_f32(bits)[:, :n], x[:, :n])  # the planted values are exact in bf16
    return bits


@pytest.mark.parametrize("K", [48, 128, 256, 400, 768, 2048])
def test_quant_act_rounding_boundaries_bit_exact(orc, K):
    """Every register-resident row shape and the generic one, on exact E2M1 ties, signed
    zeros and values one step off a boundary: codes, block scales and gs equal the oracle's."""
    x = _tie_rows(37, K, seed=K)
    q, s, g = M.moe_debug_quant_act(dev_bf16(x))
    rq, rs, rg = orc.quant_act_nvfp4(x)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert g.cpu().numpy().tobytes() == rg.tobytes()
    assert np.array_equal(q.cpu().numpy(), rq)


def _gs_of(amax):
    """The quantize multiplier 2688 / amax in fp32, as the scale rule defines it."""
    return np.float32(2688.0) / np.float32(max(float(amax), 1e-12))


@pytest.mark.parametrize("K", [48, 256, 768, 2048])
def test_quant_act_static_bit_exact(orc, K):
    """Static activation scale: every row quantized with one given global scale (part of the
    rows exceed its range and saturate); codes and block scales equal the oracle's."""
    x = np.concatenate([_tie_rows(9, K, seed=K), synth.gen_x(23, K, seed=K + 1)])
    gs = _gs_of(3.0)
    q, s = M.moe_debug_quant_act_static(dev_bf16(x), torch.tensor([gs], device="cuda"))
    rq, rs, _ = orc.quant_act_nvfp4(x, static_gs=gs)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_quant_act_fp8_bit_exact(orc):
    """W8A8 activation quantizer (one E4M3 scale per 1x128 group of a row): codes and fp32
    scale_inv equal the oracle's, including an all-zero group and a tiny group whose codes are
    negative zeros."""
    x = synth.gen_x(37, 512, seed=31)
    x[3, 128:256] = 0
    x[5, :128] = synth.f32_to_bf16_bits(np.full(128, -1e-30, np.float32))
    q, s = M.moe_debug_quant_act_fp8(dev_bf16(x))
    torch.cuda.synchronize()
    rq, rs = orc.quant_act_fp8(x)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert s.cpu().numpy().tobytes() == rs.tobytes()


def test_quant_act_fp8_hand_worked_row():
    """The hand-worked two-group row of tests/golden/fp8_act_group_example.txt (an RNE tie, a
    subnormal tie, the same value coded differently under the two group scales)."""
    row = np.zeros((1, 256), np.float32)
    row[0, [0, 1, 4, 7, 128, 129]] = [3.5, -0.75, 0.07421875, 2.288818359375e-05, 0.21875, -0.109375]
    q, s = M.moe_debug_quant_act_fp8(dev_bf16(synth.f32_to_bf16_bits(row)))
    q = q.cpu().numpy()[0]
    assert [int(q[c]) for c in (0, 1, 4, 7, 128, 129)] == [0x7E, 0xEC, 0x52, 0x02, 0x7E, 0xF6]
    assert s.cpu().numpy().tolist() == [[0.0078125, 0.00048828125]]


def test_w8a8_pack_is_the_fp8_pack():
    """W8A8 stores the W8A16 FP8 tensors: the canonical tensors of the two packed buffers are
    identical (the alignment padding between them is never written)."""
    E, H, I = 2, 512, 256
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=9)
    a = M.MoELayer("fp8", dev_bf16(wgu), dev_bf16(wd))
    b = M.MoELayer("fp8_w8a8", dev_bf16(wgu), dev_bf16(wd))
    torch.cuda.synchronize()
    for which in (M.MOE_T_GU_A, M.MOE_T_GU_B, M.MOE_T_D_A, M.MOE_T_D_B):
        assert torch.equal(M.packed_view(a.desc, a.packed, which), M.packed_view(b.desc, b.packed, which))


@pytest.mark.parametrize("T,H,I,E,k", [(24, 256, 128, 8, 2), (700, 512, 256, 16, 4), (1, 256, 128, 8, 2),
                                       (300, 768, 384, 8, 8)])
def test_w8a8_layer_small(orc, T, H, I, E, k):
    """FP8 W8A8 layer (x and h quantized per 1x128 group, both GEMMs on E4M3 x E4M3 MMAs with
    per-K-block promotion) against the oracle: the tiny config, a ragged multi-tile shape with
    16 experts, one token, and H = 768 with top-8."""
    c = Case("fp8_w8a8", T, H, I, E, k, seed=T)
    got = synth.bf16_bits_to_f32(c.run())
    idx, _ = orc.route(c.lg, k)
    p = orc.pack_experts(FID["fp8_w8a8"], c.wgu, c.wd, experts=np.unique(idx))
    ref = orc.moe_layer(FID["fp8_w8a8"], c.x, c.lg, p, k)
    check_close(got, ref, f"w8a8 T={T}")


class StaticCase(Case):
    def __init__(self, T, H, I, E, k, seed, zipf=None, h_amax=1.0):
        super().__init__("nvfp4_w4a4", T, H, I, E, k, seed=seed, zipf=zipf)
        self.act_gs = np.array([_gs_of(np.abs(synth.bf16_bits_to_f32(self.x)).max()), _gs_of(h_amax)], np.float32)

    def run(self):
        out = torch.empty((self.T, self.H), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(M.moe_workspace_size(self.layer.desc, self.T, self.k), dtype=torch.uint8, device="cuda")
        M.moe_layer_forward_static_act(dev_bf16(self.x), torch.from_numpy(self.lg).cuda(), self.layer.desc,
                                       self.layer.packed, self.k, torch.from_numpy(self.act_gs).cuda(), out, ws)
        torch.cuda.synchronize()
        assert M.moe_get_device_error(ws) == 0
        return host_bits(out)

    def oracle(self, orc, tokens=None):
        idx, _ = orc.route(self.lg if tokens is None else self.lg[tokens], self.k)
        p = orc.pack_experts(FID[self.fmt], self.wgu, self.wd, experts=np.unique(idx))
        return orc.moe_layer(FID[self.fmt], self.x, self.lg, p, self.k, tokens=tokens, act_gs=self.act_gs)


@pytest.mark.parametrize("T,H,I,E,k", [(200, 512, 256, 16, 4), (64, 256, 128, 8, 2), (700, 512, 256, 4, 2)])
def test_layer_static_act_scales(orc, T, H, I, E, k):
    """W4A4 with static activation scales on the block-scaled FP4 path (h quantized inside the
    gate/up GEMM; several tiles per expert) and on the generic path (H, I not multiples of 256)."""
    c = StaticCase(T, H, I, E, k, seed=T + H, h_amax=0.5)
    check_close(synth.bf16_bits_to_f32(c.run()), c.oracle(orc), f"static T={T}")


def test_layer_static_act_scales_full_size_sampled(orc):
    c = StaticCase(16384, FULL["H"], FULL["I"], FULL["E"], FULL["k"], seed=0, zipf=1.1, h_amax=1.0)
    got = synth.bf16_bits_to_f32(c.run())
    toks = np.sort(np.random.default_rng(99).choice(16384, size=16, replace=False)).astype(np.int32)
    check_close(got[toks], c.oracle(orc, tokens=toks), "static full size")


def test_calibrate_act_scales(orc):
    """Calibration: x's scale is exactly 2688 / max|x|; h's is 2688 / max|h| over the routed rows,
    with h recomputed here from oracle primitives (x quantized with that scale, fp64 GEMVs,
    bf16 rounding), equal up to one bf16 step of the maximum."""
    T, H, I, E, k = 96, 512, 256, 8, 2
    c = Case("nvfp4_w4a4", T, H, I, E, k, seed=41)
    ws = torch.empty(M.moe_workspace_size(c.layer.desc, T, k), dtype=torch.uint8, device="cuda")
    gs = M.moe_calibrate_act_scales(dev_bf16(c.x), torch.from_numpy(c.lg).cuda(), c.layer.desc, c.layer.packed, k,
                                    ws).cpu().numpy()
    torch.cuda.synchronize()
    gx = _gs_of(np.abs(synth.bf16_bits_to_f32(c.x)).max())
    assert gs[0] == gx
    q, s, g = orc.quant_act_nvfp4(c.x, static_gs=gx)
    a = np.stack([orc.dequant_nvfp4(q[t:t + 1], s[t:t + 1], g[t])[0] for t in range(T)]).astype(np.float64)
    idx, _ = orc.route(c.lg, k)
    p = orc.pack_experts(FID["nvfp4_w4a4"], c.wgu, c.wd, experts=np.unique(idx))
    hmax = 0.0
    for e in np.unique(idx):
        w = orc.dequant_nvfp4(p["gu"][0][e], p["gu"][1][e], p["gu"][2][e]).astype(np.float64)
        toks = np.nonzero((idx == e).any(axis=1))[0]
        gu = a[toks] @ w.T
        h = gu[:, :I] / (1.0 + np.exp(-gu[:, :I])) * gu[:, I:]
        hmax = max(hmax, float(np.abs(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(h.astype(np.float32)))).max()))
    assert abs(gs[1] / _gs_of(hmax) - 1.0) <= 2.0 ** -7, (gs[1], _gs_of(hmax))


@pytest.mark.parametrize("T,E,k,zipf", [(64, 8, 2, None), (1, 128, 8, None), (300, 128, 8, 1.1), (257, 256, 8, None),
                                        (5, 6, 6, None), (1000, 37, 3, None), (100, 256, 8, 1.1), (50, 37, 3, None)])
def test_route_bit_exact(orc, T, E, k, zipf):
    lg = synth.gen_logits(T, E, seed=T + E, zipf_alpha=zipf)
    d = M.moe_packed_size("fp8", E, 128, 128)
    ws = torch.empty(M.moe_workspace_size(d, T, k), dtype=torch.uint8, device="cuda")
    idx, w, off, perm, inv = M.moe_debug_route(torch.from_numpy(lg).cuda(), k, ws)
    ridx, rw = orc.route(lg, k)
    roff, rperm, rinv = orc.permute(ridx, E)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.array_equal(off.cpu().numpy(), roff)
    assert np.array_equal(perm.cpu().numpy(), rperm)
    assert np.array_equal(inv.cpu().numpy(), rinv)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=1e-6, atol=0)


def test_route_ties_lower_index(orc):
    lg = np.array([[0.5, 2.0, 2.0, 1.0, 2.0, -1.0, 1.0, 1.0]], np.float32)
    d = M.moe_packed_size("fp8", 8, 128, 128)
    ws = torch.empty(M.moe_workspace_size(d, 1, 5), dtype=torch.uint8, device="cuda")
    idx, w, off, perm, inv = M.moe_debug_route(torch.from_numpy(lg).cuda(), 5, ws)
    assert idx.cpu().numpy().tolist() == [[1, 2, 4, 3, 6]] == orc.route(lg, 5)[0].tolist()


# ------------------------------------------------------------------ the layer
@pytest.mark.parametrize("fmt", FMTS)
def test_layer_tiny_config(orc, fmt):
    """64 tokens, hidden 256, intermediate 128, 8 experts, top-2 (seed 0)."""
    c = Case(fmt, 64, 256, 128, 8, 2)
    check_close(synth.bf16_bits_to_f32(c.run()), c.oracle(orc), fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_layer_ragged_multi_tile(orc, fmt):
    """Several row blocks per expert with ragged tails, several column and K tiles."""
    c = Case(fmt, 45, 384, 256, 16, 4, seed=3)
    check_close(synth.bf16_bits_to_f32(c.run()), c.oracle(orc), fmt)


@pytest.mark.parametrize("fmt,T,E,k", [("fp8", 1, 8, 1), ("nvfp4_w4a4", 3, 4, 4), ("int4", 9, 1, 1),
                                       ("nvfp4_w4a16", 17, 8, 8)])
def test_layer_edge_cases(orc, fmt, T, E, k):
    c = Case(fmt, T, 256, 128, E, k, seed=11)
    check_close(synth.bf16_bits_to_f32(c.run()), c.oracle(orc), fmt)


@pytest.mark.parametrize("T,H,I,E,k", [(1100, 256, 128, 8, 2), (1500, 384, 256, 16, 4), (530, 512, 384, 2, 1)])
def test_w4a16_wide_tiles(orc, T, H, I, E, k):
    """NVFP4 W4A16 at prefill sizes (more than 64 rows per active expert) takes 256-row routing
    tiles: full and ragged tiles, K of one to four chunks (fewer than the A ring's four stages)."""
    c = Case("nvfp4_w4a16", T, H, I, E, k, seed=T)
    check_close(synth.bf16_bits_to_f32(c.run()), c.oracle(orc), f"T={T}")


@pytest.mark.parametrize("fmt", ["fp8", "int4"])
@pytest.mark.parametrize("T,E,k,zipf", [(64, 64, 2, 1.1), (3, 16, 4, None), (40, 128, 8, None)])
def test_decode_gemv(orc, fmt, T, E, k, zipf):
    """FP8 and INT4 W4A16 decode steps with few active experts averaging at most two rows go
    through the CUDA-core GEMVs (the first two cases; the third takes the tensor-core kernels):
    Zipf-skewed routing gives tiles of up to 16 rows (several passes of four rows over the
    weights), K of 256 and 128 (FP8: a last partial 512-byte segment; INT4: 2 and 1 K groups)."""
    c = Case(fmt, T, 256, 128, E, k, seed=T + E, zipf=zipf)
    check_close(synth.bf16_bits_to_f32(c.run()), c.oracle(orc), f"T={T}")


def test_layer_zero_tokens_is_a_no_op():
    c = Case("fp8", 4, 256, 128, 8, 2)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    lg = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    out = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    ws = c.layer.ensure_workspace(0, 2)
    M.moe_layer_forward(x, lg, c.layer.desc, c.layer.packed, 2, out, ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_error(ws) == 0


def test_layer_forward_host_matches_device_path(orc):
    c = Case("nvfp4_w4a16", 20, 256, 128, 8, 2, seed=4)
    dev_out = c.run()
    ws = c.layer.ensure_workspace(c.T, c.k, host_io=True)
    xh = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    lh = torch.from_numpy(c.lg).pin_memory()
    oh = torch.empty((c.T, c.H), dtype=torch.bfloat16).pin_memory()
    M.moe_layer_forward_host(xh, lh, c.layer.desc, c.layer.packed, c.k, oh, ws)
    torch.cuda.synchronize()
    check_close(synth.bf16_bits_to_f32(host_bits(oh)), c.oracle(orc), "host io")
    check_close(synth.bf16_bits_to_f32(host_bits(oh)), synth.bf16_bits_to_f32(dev_out), "host vs device")


# ------------------------------------------------------------------ full-size workloads
FULL = dict(H=2048, I=768, E=128, k=8)


@pytest.mark.parametrize("fmt,T,zipf,sample", [("fp8", 16, None, None), ("int4", 256, None, 24),
                                               ("nvfp4_w4a16", 4096, 1.1, 24), ("nvfp4_w4a4", 16384, 1.1, 16),
                                               ("bf16", 16, None, None), ("bf16", 4096, 1.1, 24)])
def test_layer_full_size_sampled(orc, fmt, T, zipf, sample):
    c = Case(fmt, T, FULL["H"], FULL["I"], FULL["E"], FULL["k"], seed=0, zipf=zipf)
    got = synth.bf16_bits_to_f32(c.run())
    toks = None
    if sample:
        g = np.random.default_rng(T)
        toks = np.sort(g.choice(T, size=sample, replace=False)).astype(np.int32)
        got = got[toks]
    check_close(got, c.oracle(orc, tokens=toks), f"{fmt} T={T}")


@pytest.mark.parametrize("fmt,T", [("fp8", 1), ("fp8", 4), ("int4", 1), ("int4", 16), ("int4", 64)])
def test_layer_full_size_decode_all_tokens(orc, fmt, T):
    """The decode points of the FP8 and INT4 sweeps at the full 2048 / 768 / 128-expert / top-8
    shape, every token checked: the small row blocks whose CTAs walk several weight tiles each."""
    c = Case(fmt, T, FULL["H"], FULL["I"], FULL["E"], FULL["k"], seed=T + 1)
    check_close(synth.bf16_bits_to_f32(c.run()), c.oracle(orc), f"{fmt} T={T}")


def test_w8a8_layer_full_size_sampled(orc):
    """FP8 W8A8 at 16,384 tokens with Zipf-skewed routing: every CTA of both GEMMs takes many work
    items (the persistent item loop, the shared work counter, the promotion buffers reused across
    items); 48 sampled tokens against the oracle."""
    T = 16384
    c = Case("fp8_w8a8", T, FULL["H"], FULL["I"], FULL["E"], FULL["k"], seed=77, zipf=1.1)
    got = synth.bf16_bits_to_f32(c.run())
    toks = np.sort(np.random.default_rng(5).choice(T, 48, replace=False)).astype(np.int32)
    check_close(got[toks], c.oracle(orc, tokens=toks), "w8a8 full size")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (45, 16, 4), (300, 32, 8), (700, 4, 2)])
def test_layer_k256_shapes(orc, fmt, T, E, k):
    """Hidden and intermediate sizes that are multiples of 256 (the block-scaled FP4 path's
    K chunk): several tiles per expert, ragged tails, and row blocks from 16 to 128."""
    c = Case(fmt, T, 512, 256, E, k, seed=T + E)
    check_close(synth.bf16_bits_to_f32(c.run()), c.oracle(orc), f"{fmt} T={T}")


def test_mixed_format_stack_shared_workspace(orc):
    """A stack whose layers use different formats (FP8, then NVFP4 W4A4, as in the hybrid page's
    split) runs back to back on one workspace sized for the largest format; every layer matches
    its oracle."""
    T, H, I, E, k = 200, 512, 256, 16, 4
    cases = [Case("fp8", T, H, I, E, k, seed=31), Case("nvfp4_w4a4", T, H, I, E, k, seed=32, zipf=1.1)]
    ws = torch.empty(max(M.moe_workspace_size(c.layer.desc, T, k) for c in cases), dtype=torch.uint8, device="cuda")
    outs = []
    for c in cases:
        out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        M.moe_layer_forward(dev_bf16(c.x), torch.from_numpy(c.lg).cuda(), c.layer.desc, c.layer.packed, k, out, ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert M.moe_get_device_error(ws) == 0
    for c, out in zip(cases, outs):
        check_close(synth.bf16_bits_to_f32(host_bits(out)), c.oracle(orc), c.fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_layer_deterministic(fmt):
    """Two forward passes on the same inputs give bit-identical outputs (the combine sums each
    token's k rows in slot order; nothing reaches the output through atomics)."""
    c = Case(fmt, 300, 512, 256, 32, 8, seed=21)
    first = c.run()
    second = c.run()
    assert np.array_equal(first, second), fmt
