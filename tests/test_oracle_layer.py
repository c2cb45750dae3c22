"""Pins for the oracle's routing, permutation and layer (CPU only).

Top-k is checked against brute force over all k-subsets, the weights against the closed
form of a renormalised softmax, the permutation against Python's stable sort, and the
layer against an independent torch fp64 composition (dense all-experts einsum with the
routing mask, and the textbook SwiGLU MLP when one expert takes every token).
"""
import itertools

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth

FP8, INT4, W4A16, W4A4, BF16, W8A8 = 1, 2, 3, 4, 5, 6


def test_topk_brute_force_small(orc):
    g = np.random.default_rng(0)
    for E, k in [(8, 2), (8, 3), (6, 6), (5, 1)]:
        lg = g.standard_normal((40, E)).astype(np.float32)
        idx, w = orc.route(lg, k)
        for t in range(40):
            best = None
            for S in itertools.combinations(range(E), k):
                rest = [e for e in range(E) if e not in S]
                if not rest or min(lg[t, list(S)]) > max(lg[t, rest]):
                    best = S
            want = sorted(best, key=lambda e: -lg[t, e])
            assert list(idx[t]) == want


def test_topk_ties_go_to_lower_index(orc):
    lg = np.array([[1.0, 3.0, 3.0, 0.5, 3.0, 2.0]], np.float32)
    idx, _ = orc.route(lg, 4)
    assert list(idx[0]) == [1, 2, 4, 5]


def test_renormalised_softmax_closed_form(orc):
    g = np.random.default_rng(1)
    lg = (g.standard_normal((50, 16)) * 3).astype(np.float32)
    idx, w = orc.route(lg, 4)
    full = torch.softmax(torch.from_numpy(lg).double(), dim=-1).numpy()
    for t in range(50):
        sel = full[t, idx[t]]
        np.testing.assert_allclose(w[t], sel / sel.sum(), rtol=1e-13)
        assert abs(w[t].sum() - 1) < 1e-14
        np.testing.assert_allclose(w[t, 0] / w[t, 1], np.exp(np.float64(lg[t, idx[t, 0]]) - lg[t, idx[t, 1]]),
                                   rtol=1e-12)


def test_permutation_is_stable_sort_by_expert(orc):
    g = np.random.default_rng(2)
    T, E, k = 37, 9, 3
    idx, _ = orc.route(g.standard_normal((T, E)).astype(np.float32), k)
    off, perm, inv = orc.permute(idx, E)
    keys = sorted(((idx[t, j], t, j) for t in range(T) for j in range(k)))
    assert list(perm) == [t * k + j for (_, t, j) in keys]
    counts = np.bincount(idx.ravel(), minlength=E)
    assert list(off) == [0] + list(np.cumsum(counts))
    assert np.array_equal(inv[perm], np.arange(T * k))


def _torch_reference(fmt, x_bits, logits, packed, k, orc, act_gs=None):
    """Independent composition in torch fp64: dense einsum over all experts with the mask."""
    E = logits.shape[1]
    gu_a, gu_b, gu_g = packed["gu"]
    d_a, d_b, d_g = packed["d"]
    wgu, wd = [], []
    for e in range(E):
        if fmt in (FP8, W8A8):
            wgu.append(orc.dequant_fp8(gu_a[e], gu_b[e]))
            wd.append(orc.dequant_fp8(d_a[e], d_b[e]))
        elif fmt == INT4:
            wgu.append(orc.dequant_int4(gu_a[e], gu_b[e]))
            wd.append(orc.dequant_int4(d_a[e], d_b[e]))
        elif fmt == BF16:  # the stored bf16 bits, widened by numpy
            wgu.append(synth.bf16_bits_to_f32(gu_a[e]))
            wd.append(synth.bf16_bits_to_f32(d_a[e]))
        else:
            wgu.append(orc.dequant_nvfp4(gu_a[e], gu_b[e], gu_g[e]))
            wd.append(orc.dequant_nvfp4(d_a[e], d_b[e], d_g[e]))
    Wgu = torch.from_numpy(np.stack(wgu)).double()
    Wd = torch.from_numpy(np.stack(wd)).double()
    I = Wgu.shape[1] // 2
    if fmt == W4A4:
        q, s, gsa = orc.quant_act_nvfp4(x_bits, static_gs=None if act_gs is None else act_gs[0])
        a = torch.from_numpy(np.stack([orc.dequant_nvfp4(q[t:t + 1], s[t:t + 1], gsa[t])[0]
                                       for t in range(len(q))])).double()
    elif fmt == W8A8:
        a = torch.from_numpy(orc.dequant_act_fp8(*orc.quant_act_fp8(x_bits))).double()
    else:
        a = torch.from_numpy(synth.bf16_bits_to_f32(x_bits)).double()
    lg = torch.from_numpy(logits).double()
    topv, topi = torch.topk(lg, k, dim=-1)
    mask = torch.zeros_like(lg).scatter(1, topi, torch.softmax(topv, dim=-1))
    G = torch.einsum("eoh,th->teo", Wgu[:, :I], a)
    U = torch.einsum("eoh,th->teo", Wgu[:, I:], a)
    Hh = F.silu(G) * U
    if fmt == W4A4:
        T_ = Hh.shape[0]
        hb = synth.f32_to_bf16_bits(Hh.reshape(-1, I).float().numpy())  # fp32 then bf16: see below
        hq, hs, hg = orc.quant_act_nvfp4(hb, static_gs=None if act_gs is None else act_gs[1])
        hd = np.stack([orc.dequant_nvfp4(hq[r:r + 1], hs[r:r + 1], hg[r])[0] for r in range(len(hq))])
        Hh = torch.from_numpy(hd).double().reshape(T_, E, I)
    elif fmt == W8A8:
        T_ = Hh.shape[0]
        hb = synth.f32_to_bf16_bits(Hh.reshape(-1, I).float().numpy())
        hd = orc.dequant_act_fp8(*orc.quant_act_fp8(hb))
        Hh = torch.from_numpy(hd).double().reshape(T_, E, I)
    Y = torch.einsum("ehi,tei->teh", Wd, Hh)
    return torch.einsum("te,teh->th", mask, Y).numpy()


@pytest.mark.parametrize("fmt", [FP8, INT4, W4A16, W4A4, BF16, W8A8])
def test_layer_matches_torch_dense_composition(orc, fmt):
    E, H, I, T, k = 8, 256, 128, 24, 2
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=0)
    x = synth.gen_x(T, H, seed=0)
    lg = synth.gen_logits(T, E, seed=0)
    packed = orc.pack_experts(fmt, wgu, wd)
    got = orc.moe_layer(fmt, x, lg, packed, k)
    ref = _torch_reference(fmt, x, lg, packed, k, orc)
    if fmt in (W4A4, W8A8):
        # the torch side rounds h through fp32 before bf16, the oracle rounds fp64 -> bf16
        # once; a few h elements may land one bf16 ulp apart and change their code
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel < 2e-3, rel
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("fmt", [FP8, W4A4, BF16, W8A8])
def test_sparse_equals_dense_masked_definition(orc, fmt):
    E, H, I, T, k = 8, 256, 128, 16, 3
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=1)
    x = synth.gen_x(T, H, seed=1)
    lg = synth.gen_logits(T, E, seed=1)
    packed = orc.pack_experts(fmt, wgu, wd)
    a = orc.moe_layer(fmt, x, lg, packed, k)
    b = orc.moe_layer(fmt, x, lg, packed, k, dense=True)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)


def test_single_expert_reduces_to_swiglu_mlp(orc):
    H, I, T = 256, 128, 8
    wgu, wd = synth.gen_expert_weights(1, H, I, seed=2)
    x = synth.gen_x(T, H, seed=2)
    lg = synth.gen_logits(T, 1, seed=2)
    packed = orc.pack_experts(FP8, wgu, wd)
    got = orc.moe_layer(FP8, x, lg, packed, 1)
    Wg = torch.from_numpy(orc.dequant_fp8(packed["gu"][0][0][:I], packed["gu"][1][0][:1])).double()
    Wu = torch.from_numpy(orc.dequant_fp8(packed["gu"][0][0][I:], packed["gu"][1][0][1:])).double()
    Wd = torch.from_numpy(orc.dequant_fp8(packed["d"][0][0], packed["d"][1][0])).double()
    a = torch.from_numpy(synth.bf16_bits_to_f32(x)).double()
    ref = (F.silu(a @ Wg.T) * (a @ Wu.T)) @ Wd.T
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-11, atol=1e-14)


def test_token_subset_equals_full_rows(orc):
    E, H, I, T, k = 8, 256, 128, 20, 2
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=3)
    x = synth.gen_x(T, H, seed=3)
    lg = synth.gen_logits(T, E, seed=3)
    packed = orc.pack_experts(W4A4, wgu, wd)
    full = orc.moe_layer(W4A4, x, lg, packed, k)
    sub = orc.moe_layer(W4A4, x, lg, packed, k, tokens=[17, 3, 3, 0])
    assert np.array_equal(sub, full[[17, 3, 3, 0]])


def test_static_activation_scales_layer_matches_torch_composition(orc):
    """W4A4 with static (calibrated) activation scales, one too small for part of x so that
    some blocks saturate: the oracle layer equals the torch fp64 composition."""
    E, H, I, T, k = 8, 256, 128, 24, 2
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=4)
    x = synth.gen_x(T, H, seed=4)
    lg = synth.gen_logits(T, E, seed=4)
    packed = orc.pack_experts(W4A4, wgu, wd)
    act_gs = np.array([2688.0 / 2.5, 2688.0 / 0.05], np.float32)  # x beyond 2.5 saturates
    got = orc.moe_layer(W4A4, x, lg, packed, k, act_gs=act_gs)
    ref = _torch_reference(W4A4, x, lg, packed, k, orc, act_gs=act_gs)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 2e-3, rel  # h rounding to bf16 may differ by an ulp between the two (see above)
    dyn = orc.moe_layer(W4A4, x, lg, packed, k)
    assert not np.allclose(got, dyn)  # the static scales change the result


def test_w8a8_differs_from_w8a16_by_the_activation_quantization_only(orc):
    """W8A8 and W8A16 share the packed weights; W8A8 also quantizes x and h to E4M3 (3 mantissa
    bits, ~2.6% relative RMS each), so the two layers differ by a few percent, not by a scale
    factor, a sign or a permutation (each of which would give an O(1) difference)."""
    E, H, I, T, k = 8, 256, 128, 24, 2
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=5)
    x = synth.gen_x(T, H, seed=5)
    lg = synth.gen_logits(T, E, seed=5)
    packed = orc.pack_experts(W8A8, wgu, wd)
    a8 = orc.moe_layer(W8A8, x, lg, packed, k)
    a16 = orc.moe_layer(FP8, x, lg, packed, k)
    rel = np.linalg.norm(a8 - a16) / np.linalg.norm(a16)
    assert 0.01 < rel < 0.08, rel
