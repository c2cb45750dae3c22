"""Pins for the oracle's number formats and weight quantizers (CPU only).

Each check ties the oracle to something other than itself: torch's / numpy's own
conversions, hand-worked examples from the format definitions (tests/golden/), figures
printed on the model-card pages, closed-form error bounds and exhaustive enumeration.
"""
import math
import os

import numpy as np
import pytest
import torch

import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLD, name)) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                yield ln.split()


def bf16(vals):
    return synth.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


# ---------------------------------------------------------------- scalar formats
def test_e4m3_decode_all_codes_match_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.e4m3_decode(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok]))


def test_e4m3_golden_points(orc):
    for code, val in _lines("e4m3_points.txt"):
        got = orc.e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_encode_roundtrip_all_finite_codes(orc):
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert orc.e4m3_encode(orc.e4m3_decode(c)) == c


def test_e4m3_encode_matches_torch_rne_in_range(orc):
    g = np.random.default_rng(5)
    mags = np.concatenate([
        g.uniform(0, 448, 3000), np.exp(g.uniform(np.log(1e-6), np.log(448), 3000)),
        # every midpoint between neighbouring codes (ties)
        [(orc.e4m3_decode(c) + orc.e4m3_decode(c + 1)) / 2 for c in range(0, 0x7E)],
    ]).astype(np.float32)
    vals = np.concatenate([mags, -mags]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(v) for v in vals], dtype=np.uint8)
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates(orc):
    assert orc.e4m3_encode(470.0) == 0x7E
    assert orc.e4m3_encode(1e30) == 0x7E
    assert orc.e4m3_encode(-1e30) == 0xFE
    assert orc.e4m3_encode(-0.0) == 0x80  # reading: the sign of zero is kept


def test_e2m1_table_and_ties_golden(orc):
    for row in _lines("e2m1_grid.txt"):
        kind = row[0]
        if kind == "code":
            c, v = int(row[1]), float(row[2])
            got = orc.e2m1_decode(c)
            assert got == v and math.copysign(1, got) == math.copysign(1, v)
        elif kind in ("tie", "sat"):
            v, c = float(row[1]), int(row[2])
            assert orc.e2m1_encode(v) == c
            assert orc.e2m1_encode(-v) == c | 8


def test_e2m1_encode_is_nearest_grid_point_brute_force(orc):
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    g = np.random.default_rng(1)
    for v in np.concatenate([g.uniform(-8, 8, 4000), g.uniform(-1, 1, 1000)]).astype(np.float32):
        d = np.abs(grid - abs(float(v)))
        best = np.flatnonzero(d == d.min())
        mag = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        want = int(mag) | (8 if np.signbit(v) else 0)
        assert orc.e2m1_encode(float(v)) == want, v


def test_f16_matches_numpy(orc):
    g = np.random.default_rng(2)
    vals = np.concatenate([g.standard_normal(3000) * 0.01, np.exp(g.uniform(-20, 10, 3000)),
                           [6.103515625e-05, 5.960464477539063e-08, 2.98e-08, 65504.0, 1.0 + 2**-11]])
    for v in vals:
        want = int(np.float16(np.float32(v)).view(np.uint16)) if abs(v) < 65520 else None
        if want is None:
            continue
        # numpy rounds fp32 -> fp16 with round-half-even; the oracle takes the fp32 value too
        assert orc.f16_encode(float(np.float32(v))) == want, v
        assert orc.f16_decode(want) == float(np.float16(np.float32(v)))


def test_bf16_matches_torch(orc):
    g = np.random.default_rng(3)
    vals = np.concatenate([g.standard_normal(2000), g.standard_normal(2000) * 1e-3]).astype(np.float32)
    want = synth.f32_to_bf16_bits(vals)
    got = np.array([orc.bf16_encode(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(want, got)


# ---------------------------------------------------------------- FP8 block 128x128
def test_fp8_hand_worked_tile(orc):
    w = np.zeros((128, 128), np.float32)
    expect = {}
    sinv = None
    for row in _lines("fp8_tile_example.txt"):
        if row[0] == "scale_inv":
            sinv = float(row[1])
            continue
        r, c, v, code = int(row[0]), int(row[1]), float(row[2]), int(row[3], 16)
        w[r, c] = v
        expect[(r, c)] = code
    wb = bf16(w)
    assert np.array_equal(synth.bf16_bits_to_f32(wb), w), "example values must be bf16-exact"
    codes, s = orc.pack_fp8(wb)
    assert s.shape == (1, 1) and s[0, 0] == np.float32(sinv)
    for (r, c), code in expect.items():
        assert codes[r, c] == code, (r, c, hex(codes[r, c]), hex(code))
    mask = np.ones_like(codes, bool)
    for rc in expect:
        mask[rc] = False
    assert np.all(codes[mask] == 0)


def test_fp8_tiles_are_independent_and_bounded(orc):
    # 256 x 384 matrix whose 2 x 3 tiles have very different amax: a transposed or shifted
    # tile index would put elements under the wrong scale and break the bounds below.
    g = np.random.default_rng(4)
    mult = np.array([[1e-3, 1.0, 3e-2], [0.5, 7e-4, 2.0]], np.float32)
    w = g.standard_normal((256, 384)).astype(np.float32)
    w *= np.kron(mult, np.ones((128, 128), np.float32))
    wb = bf16(w)
    wf = synth.bf16_bits_to_f32(wb)
    codes, sinv = orc.pack_fp8(wb)
    deq = orc.dequant_fp8(codes, sinv)
    for tn in range(2):
        for tk in range(3):
            blk = wf[tn * 128:(tn + 1) * 128, tk * 128:(tk + 1) * 128]
            amax = np.abs(blk).max()
            # scale_inv = 1/(448/amax) ~= amax/448 (within an ulp or two)
            assert abs(sinv[tn, tk] - amax / 448) <= 4e-7 * amax / 448
            cb = codes[tn * 128:(tn + 1) * 128, tk * 128:(tk + 1) * 128]
            r, c = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert cb[r, c] & 0x7F == 0x7E
            db = deq[tn * 128:(tn + 1) * 128, tk * 128:(tk + 1) * 128]
            # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 for normals; absolute
            # error <= 2^-10 * scale_inv in the subnormal range
            err = np.abs(db - blk)
            assert np.all(err <= np.maximum(np.abs(blk) * 2.0 ** -4, sinv[tn, tk] * 2.0 ** -10) * (1 + 1e-6))


def test_fp8_requantize_grid_exact_is_identity(orc):
    g = np.random.default_rng(6)
    w = (g.standard_normal((128, 256)) * 0.02).astype(np.float32)
    codes, sinv = orc.pack_fp8(bf16(w))
    deq = orc.dequant_fp8(codes, sinv)
    # the dequantized tile is representable; re-packing it must give the same codes
    wb2 = bf16(deq)
    if np.array_equal(synth.bf16_bits_to_f32(wb2), deq):
        c2, s2 = orc.pack_fp8(wb2)
        assert np.array_equal(c2, codes) and np.array_equal(s2, sinv)


# ---------------------------------------------------------------- INT4 g128 auto_gptq
def test_int4_hand_worked_group(orc):
    w = np.zeros((2, 128), np.float32)
    scales, words = {}, {}
    for row in _lines("int4_group_example.txt"):
        if row[0] == "scale":
            scales[int(row[1])] = int(row[2], 16)
        elif row[0] == "word":
            words[(int(row[1]), int(row[2]))] = int(row[3], 16)
        else:
            w[int(row[0]), int(row[1])] = float(row[2])
    wb = bf16(w)
    assert np.array_equal(synth.bf16_bits_to_f32(wb), w)
    qw, sc = orc.pack_int4(wb)
    assert qw.shape == (16, 2) and sc.shape == (1, 2)
    for n, s in scales.items():
        assert sc[0, n] == s
    for (kr, n), word in words.items():
        assert int(qw[kr, n]) & 0xFFFFFFFF == word, (kr, n, hex(int(qw[kr, n]) & 0xFFFFFFFF))
    # every code of row 0 beyond k=7 and all of row 1 is the zero code 8
    u = qw.view(np.uint32)
    assert np.all(u[1:, 0] == 0x88888888) and np.all(u[:, 1] == 0x88888888)


def test_int4_unpack_independent_bit_ops(orc):
    g = np.random.default_rng(7)
    w = (g.standard_normal((256, 384)) * 0.02).astype(np.float32)
    wb = bf16(w)
    wf = synth.bf16_bits_to_f32(wb)
    qw, sc = orc.pack_int4(wb)
    u = qw.view(np.uint32)                          # [K/8, N]
    shifts = (4 * np.arange(8, dtype=np.uint32))[None, :, None]
    codes = ((u[:, None, :] >> shifts) & 0xF).reshape(384, 256).T  # [N, K]
    s = np.float16(0) + sc.view(np.float16).astype(np.float32)      # [K/128, N]
    deq = (codes.astype(np.float32) - 8) * np.repeat(s, 128, axis=0).T
    assert np.array_equal(deq, orc.dequant_int4(qw, sc))
    # symmetric scale: fp16(amax/7) per (row, group)
    amax = np.abs(wf.reshape(256, 3, 128)).max(-1).T            # [3, 256]
    assert np.array_equal(sc.view(np.float16), (amax / np.float32(7)).astype(np.float16))
    # round-to-nearest: |w - deq| <= scale/2
    assert np.all(np.abs(deq - wf) <= np.repeat(s, 128, axis=0).T / 2 * (1 + 1e-6))
    assert codes.min() >= 0 and codes.max() <= 15


# ---------------------------------------------------------------- NVFP4
def test_nvfp4_hand_worked_blocks(orc):
    d = {row[0]: row[1:] for row in _lines("nvfp4_block_example.txt")}
    vals = np.array([float(v) for v in d["values"]], np.float32)[None, :]
    wb = bf16(vals)
    assert np.array_equal(synth.bf16_bits_to_f32(wb), vals)
    pk, sc, gs = orc.pack_nvfp4(wb)
    assert gs == np.float32(float(d["gs"][0]))
    assert [int(b) for b in pk[0]] == [int(x, 16) for x in d["bytes"]]
    assert [int(b) for b in sc[0]] == [int(x, 16) for x in d["scales"]]
    codes = [(pk[0, i // 2] >> (4 * (i % 2))) & 0xF for i in range(32)]
    assert codes == [int(c) for c in d["codes"]]


def test_nvfp4_structure_and_error_bound(orc):
    g = np.random.default_rng(8)
    w = (g.standard_normal((128, 512)) * 0.02).astype(np.float32)
    w[3, 17] = 0.25  # the matrix amax, in block (3, 1)
    wb = bf16(w)
    wf = synth.bf16_bits_to_f32(wb)
    pk, sc, gs = orc.pack_nvfp4(wb)
    amax = np.abs(wf).max()
    assert abs(gs - 2688 / amax) <= 1e-6 * gs                     # 448*6/amax
    assert sc[3, 1] == 0x7E                                       # block holding amax: scale 448
    assert (pk[3, 8] >> 4) & 0x7 == 7                             # element 17: high nibble, 6.0
    deq = orc.dequant_nvfp4(pk, sc, gs)
    # per element: |w - deq| <= half the E2M1 grid spacing at |w|/eff, times eff
    bs = np.array([[orc.e4m3_decode(c) for c in r] for r in sc])
    eff = np.repeat(bs / gs, 16, axis=1)
    y = np.abs(wf) / eff
    half = np.where(y <= 2, 0.25, np.where(y <= 4, 0.5, 1.0))
    assert np.all(np.abs(deq - wf) <= half * eff * (1 + 1e-5))


def test_page_figure_nvfp4_layer_size(orc):
    figs = {row[0]: float(row[1]) for row in _lines("page_figures.txt")}
    E, H, I = int(figs["experts"]), 2048, 768
    wgu = np.zeros((2 * I, H), np.uint16)
    wd = np.zeros((H, I), np.uint16)
    nbytes = 0
    for W in (wgu, wd):
        pk, sc, gs = orc.pack_nvfp4(W)
        nbytes += pk.nbytes + sc.nbytes + 4
    gib = nbytes * E / 2 ** 30
    assert round(gib, 2) == figs["nvfp4_layer_gib"]
    assert figs["layers"] * E * 3 == figs["thinker_expert_matrices"]


@pytest.mark.parametrize("fmt,lo,hi", [("nvfp4", 0.085, 0.105), ("fp8", 0.016, 0.036), ("int4", 0.107, 0.127)])
def test_weight_error_statistics(orc, fmt, lo, hi):
    """NVFP4: 9.5% mean relative L2 on the page (clef-omni-NVFP4, "How close is it to the
    original"), +-1 point for Gaussian instead of trained weights.  FP8 / INT4: sanity bands."""
    figs = {row[0]: float(row[1]) for row in _lines("page_figures.txt")}
    wgu, wd = synth.gen_expert_weights(2, 1024, 384, seed=11)
    errs = []
    for W in (wgu[0], wgu[1], wd[0], wd[1]):
        wf = synth.bf16_bits_to_f32(W)
        if fmt == "nvfp4":
            d = orc.dequant_nvfp4(*orc.pack_nvfp4(W))
        elif fmt == "fp8":
            d = orc.dequant_fp8(*orc.pack_fp8(W))
        else:
            d = orc.dequant_int4(*orc.pack_int4(W))
        errs.append(np.linalg.norm(d - wf) / np.linalg.norm(wf))
    m = float(np.mean(errs))
    if fmt == "nvfp4":
        assert abs(m - figs["nvfp4_weight_rel_l2"]) <= 0.01
    assert lo <= m <= hi, m


# ---------------------------------------------------------------- dynamic activation quant
def test_act_quant_rows_are_independent_and_match_weight_rule(orc):
    x = synth.gen_x(5, 256, seed=3)
    q, s, gs = orc.quant_act_nvfp4(x)
    xf = synth.bf16_bits_to_f32(x)
    for t in range(5):
        assert abs(gs[t] - 2688 / np.abs(xf[t]).max()) <= 1e-6 * gs[t]
        # a row is quantized exactly like a one-row weight matrix
        pk, sc, g1 = orc.pack_nvfp4(x[t:t + 1])
        assert g1 == gs[t] and np.array_equal(pk[0], q[t]) and np.array_equal(sc[0], s[t])
    q1, s1, g1 = orc.quant_act_nvfp4(x[2:3])
    assert np.array_equal(q1[0], q[2]) and np.array_equal(s1[0], s[2]) and g1[0] == gs[2]


def test_act_quant_hand_worked_row(orc):
    d = {row[0]: row[1:] for row in _lines("nvfp4_block_example.txt")}
    vals = np.array([float(v) for v in d["values"]], np.float32)[None, :]
    q, s, gs = orc.quant_act_nvfp4(bf16(vals))
    assert gs[0] == np.float32(448.0)
    assert [int(b) for b in q[0]] == [int(x, 16) for x in d["bytes"]]
    assert [int(b) for b in s[0]] == [int(x, 16) for x in d["scales"]]


def test_static_activation_scale_reduces_to_dynamic_rows(orc):
    """With each row's own dynamic scale passed as the static one, the static quantizer returns
    the dynamic codes and block scales (the static path differs only in where gs comes from)."""
    import synth
    x = synth.gen_x(9, 512, seed=12)
    q, s, g = orc.quant_act_nvfp4(x)
    for t in range(len(x)):
        qs, ss, gs = orc.quant_act_nvfp4(x[t:t + 1], static_gs=g[t])
        assert np.array_equal(qs[0], q[t]) and np.array_equal(ss[0], s[t]) and gs[0] == g[t]


def test_static_activation_scale_saturates_outside_calibration(orc):
    """Calibrated amax 1 (gs = 2688): a block whose amax is 4 needs a block scale of 4 * 448,
    which saturates at 448 (E4M3 0x7E); its largest elements then need 24 on the E2M1 grid and
    saturate at 6 (code 7, sign kept); a block inside the range is unaffected."""
    import synth
    row = np.zeros((1, 32), np.float32)
    row[0, :16] = np.linspace(-4.0, 4.0, 16, dtype=np.float32)  # |max| 4: over range
    row[0, 16] = 1.0                                             # second block: amax 1
    q, s, g = orc.quant_act_nvfp4(synth.f32_to_bf16_bits(row), static_gs=2688.0)
    assert s[0, 0] == 0x7E and g[0] == np.float32(2688.0)
    assert q[0, 0] & 0x0F == 0xF and (q[0, 7] >> 4) == 0x7  # -4 -> -6 (0xF), +4 -> +6 (0x7)
    assert s[0, 1] == orc.e4m3_encode(np.float32(448.0)) and (q[0, 8] & 0x0F) == 0x7  # 1 -> 6 in its own block


# ---------------------------------------------------------------- dynamic FP8 1x128 activation quant
def test_fp8_act_quant_hand_worked_row(orc):
    row = np.zeros((1, 256), np.float32)
    expect, sinv = {}, {}
    for r in _lines("fp8_act_group_example.txt"):
        if r[0] == "scale_inv":
            sinv[int(r[1])] = float(r[2])
            continue
        row[0, int(r[0])] = float(r[1])
        expect[int(r[0])] = int(r[2], 16)
    xb = bf16(row)
    assert np.array_equal(synth.bf16_bits_to_f32(xb), row), "example values must be bf16-exact"
    q, s = orc.quant_act_fp8(xb)
    assert s.shape == (1, 2) and s[0, 0] == np.float32(sinv[0]) and s[0, 1] == np.float32(sinv[1])
    for c in range(256):
        assert q[0, c] == expect.get(c, 0), (c, hex(q[0, c]))


def _e4m3_nearest_brute_force(v):
    """Nearest finite E4M3 code to each fp32 value by exhaustive search over torch's decode of
    the 127 finite magnitudes (ties to the even code), sign kept, saturating at 448."""
    mags = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    a = np.abs(v.astype(np.float64))[..., None]
    d = np.abs(a - mags)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    even = cand & (np.arange(0x7F) % 2 == 0)
    code = np.where(even.any(-1), np.argmax(even, -1), np.argmax(cand, -1))
    return (code | (np.signbit(v) * 0x80)).astype(np.uint8)


def test_fp8_act_quant_is_nearest_grid_point_brute_force(orc):
    # groups of very different magnitude in one row: each must be scaled by its own amax
    g = np.random.default_rng(21)
    T, H = 6, 512
    x = g.standard_normal((T, H)).astype(np.float32)
    x *= np.repeat(np.array([1e-3, 1.0, 40.0, 3e-5], np.float32), 128)[None, :]
    xb = bf16(x)
    xf = synth.bf16_bits_to_f32(xb)
    q, s = orc.quant_act_fp8(xb)
    for t in range(T):
        for gi in range(H // 128):
            v = xf[t, gi * 128:(gi + 1) * 128]
            sc = np.float32(448.0) / np.float32(np.abs(v).max())  # IEEE fp32 division
            assert s[t, gi] == np.float32(1.0) / sc
            assert np.array_equal(q[t, gi * 128:(gi + 1) * 128], _e4m3_nearest_brute_force(v * sc))


def test_fp8_act_quant_groups_are_independent_and_bounded(orc):
    g = np.random.default_rng(22)
    x = g.standard_normal((4, 384)).astype(np.float32)
    x *= np.repeat(np.array([2e-3, 5.0, 1e-1], np.float32), 128)[None, :]
    xb = bf16(x)
    xf = synth.bf16_bits_to_f32(xb)
    q, s = orc.quant_act_fp8(xb)
    d = orc.dequant_act_fp8(q, s)
    for t in range(4):
        for gi in range(3):
            v = xf[t, gi * 128:(gi + 1) * 128]
            amax = np.abs(v).max()
            assert abs(s[t, gi] - amax / 448) <= 4e-7 * amax / 448
            assert q[t, gi * 128 + np.argmax(np.abs(v))] & 0x7F == 0x7E  # the group max maps to 448
            err = np.abs(d[t, gi * 128:(gi + 1) * 128] - v)
            # 3 mantissa bits: relative error <= 2^-4 for normals, absolute <= 2^-10 / s below
            assert np.all(err <= np.maximum(np.abs(v) * 2.0 ** -4, s[t, gi] * 2.0 ** -10) * (1 + 1e-6))
    # rows are independent: quantizing a subset gives the same rows
    q2, s2 = orc.quant_act_fp8(xb[2:3])
    assert np.array_equal(q2[0], q[2]) and np.array_equal(s2[0], s[2])


def test_fp8_act_quant_grid_exact_row_is_identity(orc):
    """A group made of E4M3 grid values scaled by 2^j, with its largest magnitude exactly
    448 * 2^j, has s = 2^-j: the codes are the ones the values were built from and the
    dequantized row is the row itself."""
    g = np.random.default_rng(23)
    mags = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    T, H = 3, 384
    codes = g.integers(0, 0x7E, size=(T, H)).astype(np.uint8) | (g.integers(0, 2, size=(T, H)) * 0x80).astype(np.uint8)
    codes[:, ::128] = 0x7E  # one element per group at the top of the range
    j = g.integers(-12, 4, size=(T, H // 128))
    vals = np.where(codes & 0x80, -1.0, 1.0) * mags[codes & 0x7F] * np.repeat(2.0 ** j, 128, axis=1)
    vals = vals.astype(np.float32)
    xb = bf16(vals)
    assert np.array_equal(synth.bf16_bits_to_f32(xb), vals)
    q, s = orc.quant_act_fp8(xb)
    assert np.array_equal(q, codes)
    assert np.array_equal(s, (2.0 ** j).astype(np.float32))
    assert np.array_equal(orc.dequant_act_fp8(q, s), vals)


def test_fp8_act_quant_zero_group(orc):
    """An all-zero group (amax clamped to 1e-12) gives zero codes, the sign of -0 kept."""
    row = np.zeros((1, 256), np.float32)
    row[0, 5] = -0.0
    row[0, 200] = 1.0
    q, s = orc.quant_act_fp8(bf16(row))
    assert q[0, 5] == 0x80 and np.all(np.delete(q[0, :128], 5) == 0)
    assert s[0, 0] == np.float32(1.0) / (np.float32(448.0) / np.float32(1e-12))
    assert q[0, 200] == 0x7E and s[0, 1] == np.float32(1.0) / np.float32(448.0)


def test_page_figures_whole_checkpoints(orc):
    """The assumed expert shapes (hidden 2048, intermediate 768: the pages never print them) and
    the oracle's FP8 and INT4 packings against three more page figures: the INT4 checkpoint's
    ~19.4 GiB of weights and the FP8 checkpoint's 34.5 GB (each = 48 x 128 packed experts plus
    the NVFP4 page's 3.1 + 2.4 GiB of non-expert bf16 weights), and experts = 97% of 30B
    parameters.  A wrong code width, scale type or shape misses these by far more than 2%."""
    figs = {row[0]: float(row[1]) for row in _lines("page_figures.txt")}
    L, E, H, I = int(figs["layers"]), int(figs["experts"]), 2048, 768
    nonexpert = (figs["nonexpert_text_gib"] + figs["nonexpert_towers_gib"]) * 2 ** 30
    shapes = ((2 * I, H), (H, I))
    fp8 = int4 = 0
    for N, K in shapes:
        w = np.zeros((N, K), np.uint16)
        c, s = orc.pack_fp8(w)
        fp8 += c.nbytes + s.nbytes
        q, s16 = orc.pack_int4(w)
        int4 += q.nbytes + s16.nbytes + (K // 128) * (N // 8) * 4  # + the checkpoint's qzeros [K/128, N/8] int32
    fp8_gb = (L * E * fp8 + nonexpert) / 1e9
    int4_gib = (L * E * int4 + nonexpert) / 2 ** 30
    assert abs(fp8_gb / figs["fp8_checkpoint_gb"] - 1) < 0.02, fp8_gb
    assert abs(int4_gib / figs["int4_weights_gib"] - 1) < 0.02, int4_gib
    expert_params = L * E * 3 * H * I
    assert abs(expert_params / (figs["total_params_b"] * 1e9) - figs["expert_param_fraction"]) < 0.01
