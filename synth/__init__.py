"""Seeded synthetic inputs for the quantized-expert MoE layer.

This module is shared by the oracle side (tests, the CPU baseline) and the
CUDA side (tests, bench).  It holds no arithmetic of the method: it only
draws random numbers and rounds them to the storage types the layer consumes
(bf16 activations and weights, fp32 router logits).

Workload shape (clef-omni-NVFP4 model card, "What you get" and "How it was
made"): a 30B-A3B MoE with 48 layers of 128 experts; gate and up projections
are one fused [2I, H] matrix per expert, down is [H, I].  The pages never
print H and I; the configurations use H = 2048, I = 768, top-8.

Recipe (all draws from numpy's PCG64 via SeedSequence, one independent stream
per (seed, layer, stream id, expert)):
  * x       ~ N(0, 1), rounded to bf16 (round-to-nearest-even)
  * logits  ~ N(0, 1) fp32; rows with a repeated value are redrawn so every
              row is tie-free; optional Zipf(alpha) skew adds the bias
              b_e = -alpha * ln(rank_e), rank a seeded permutation of 1..E
  * weights ~ N(0, 0.02), rounded to bf16, drawn per expert so that any
              subset of experts can be regenerated alone.
"""
from __future__ import annotations

import numpy as np

STREAM_X, STREAM_LOGITS, STREAM_WGU, STREAM_WD, STREAM_ZIPF = 0, 1, 2, 3, 4
WEIGHT_STD = 0.02


def _rng(seed: int, layer: int, stream: int, expert: int = -1) -> np.random.Generator:
    ent = [int(seed) & 0xFFFFFFFF, int(layer), int(stream), int(expert) + 1]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(ent)))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even) through torch's own conversion; returns uint16 bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def gen_x(T: int, H: int, seed: int, layer: int = 0) -> np.ndarray:
    """Activations [T, H] as bf16 bits (uint16)."""
    g = _rng(seed, layer, STREAM_X)
    return f32_to_bf16_bits(g.standard_normal((T, H), dtype=np.float32))


def zipf_bias(E: int, seed: int, layer: int = 0, alpha: float = 1.1) -> np.ndarray:
    """Per-expert logit bias -alpha*ln(rank): the log of a Zipf(alpha) pmf over a seeded ranking."""
    g = _rng(seed, layer, STREAM_ZIPF)
    rank = g.permutation(E) + 1
    return (-alpha * np.log(rank.astype(np.float64))).astype(np.float32)


def gen_logits(T: int, E: int, seed: int, layer: int = 0, zipf_alpha: float | None = None) -> np.ndarray:
    """Router logits [T, E] fp32, every row free of repeated values."""
    g = _rng(seed, layer, STREAM_LOGITS)
    lg = g.standard_normal((T, E), dtype=np.float32)
    if zipf_alpha is not None:
        lg = (lg + zipf_bias(E, seed, layer, zipf_alpha)[None, :]).astype(np.float32)
    srt = np.sort(lg, axis=1)
    tied = np.flatnonzero((np.diff(srt, axis=1) == 0).any(axis=1))
    for t in tied:
        while len(np.unique(lg[t])) != E:
            lg[t] = g.standard_normal(E, dtype=np.float32)
            if zipf_alpha is not None:
                lg[t] += zipf_bias(E, seed, layer, zipf_alpha)
    return lg


def gen_expert_weights(E: int, H: int, I: int, seed: int, layer: int = 0, experts=None):
    """Expert weights as bf16 bits: w_gate_up [E, 2I, H] (gate rows, then up rows), w_down [E, H, I].

    When ``experts`` is given only those experts are drawn; the rest stay zero.
    """
    import os
    from concurrent.futures import ThreadPoolExecutor

    wgu = np.zeros((E, 2 * I, H), dtype=np.uint16)
    wd = np.zeros((E, H, I), dtype=np.uint16)

    def one(e):  # each expert has its own streams, so drawing order across threads is irrelevant
        g1 = _rng(seed, layer, STREAM_WGU, e)
        g2 = _rng(seed, layer, STREAM_WD, e)
        wgu[e] = f32_to_bf16_bits(g1.standard_normal((2 * I, H), dtype=np.float32) * np.float32(WEIGHT_STD))
        wd[e] = f32_to_bf16_bits(g2.standard_normal((H, I), dtype=np.float32) * np.float32(WEIGHT_STD))

    sel = list(range(E) if experts is None else experts)
    with ThreadPoolExecutor(max_workers=min(len(sel), os.cpu_count() or 1) or 1) as pool:
        list(pool.map(one, sel))
    return wgu, wd


def gen_expert_weights_device(E: int, H: int, I: int, seed: int, layer: int, device):
    """Same distribution drawn with torch on ``device`` (for the 48-layer benchmark, where
    drawing 29 G values on the host would dominate set-up).  Not value-identical to
    gen_expert_weights; use that one wherever the oracle must see the same weights."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(layer) * 7919 + 17) & 0x7FFFFFFFFFFFFFFF)
    wgu = (torch.randn((E, 2 * I, H), generator=g, device=device) * WEIGHT_STD).to(torch.bfloat16)
    wd = (torch.randn((E, H, I), generator=g, device=device) * WEIGHT_STD).to(torch.bfloat16)
    return wgu, wd


# Named workloads (sizes only; the tests and the bench pick from these).
CONFIGS = {
    0: dict(name="tiny-fp8", fmt="fp8", T=[64], H=256, I=128, E=8, k=2, zipf=None, layers=1),
    1: dict(name="fp8-decode", fmt="fp8", T=[1, 4, 16], H=2048, I=768, E=128, k=8, zipf=None, layers=48),
    2: dict(name="int4-w4a16", fmt="int4", T=[1, 2, 4, 8, 16, 32, 64, 128, 256], H=2048, I=768, E=128, k=8,
            zipf=None, layers=48),
    3: dict(name="nvfp4-w4a16", fmt="nvfp4_w4a16", T=[4096], H=2048, I=768, E=128, k=8, zipf=1.1, layers=48),
    4: dict(name="nvfp4-w4a4", fmt="nvfp4_w4a4", T=[16384], H=2048, I=768, E=128, k=8, zipf=1.1, layers=48),
    # mixed per-layer formats: the first 17/32 of the stack FP8, the rest NVFP4 W4A4 (the hybrid
    # page's split of a 32-layer model, layers 0-16 FP8 and 17-31 NVFP4, scaled to the stack)
    # W4A4 with static activation global scales, calibrated on the batch before timing (the hybrid
    # page's calibrated activation scales; here from synthetic data)
    7: dict(name="nvfp4-w4a4-static", fmt="nvfp4_w4a4", T=[16384], H=2048, I=768, E=128, k=8, zipf=1.1, layers=48,
            static_act=True),
    # unquantized bf16 experts through the same kernels: the comparison point of the quantized formats
    6: dict(name="bf16", fmt="bf16", T=[16, 4096], H=2048, I=768, E=128, k=8, zipf=1.1, layers=48),
    5: dict(name="mixed-fp8-nvfp4-w4a4", fmt="nvfp4_w4a4", T=[16, 16384], H=2048, I=768, E=128, k=8, zipf=1.1,
            layers=48, fp8_fraction=17 / 32),
    # FP8 block weights with FP8 activations (one scale per 1x128 group), the large-batch workload
    8: dict(name="fp8-w8a8", fmt="fp8_w8a8", T=[16384], H=2048, I=768, E=128, k=8, zipf=1.1, layers=48),
}


def layer_formats(c: dict, L: int) -> list:
    """Format of each of L layers: c["fmt"] throughout, or with c["fp8_fraction"] the first
    round(L * fraction) layers FP8 and the rest c["fmt"]."""
    n = int(L * c["fp8_fraction"] + 0.5) if c.get("fp8_fraction") else 0
    return ["fp8"] * n + [c["fmt"]] * (L - n)
