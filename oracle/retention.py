"""Merged versus unmerged recovery LoRA on an int4 group-64 base -- TEST
INFRASTRUCTURE AND ANALYSIS ONLY (CPU, numpy fp64; nothing of the CUDA path
imports it).

"The Other Half of the Memory Wall", S3.3 "Recovery LoRA: Unmerged by Design".
The served path keeps the adapter unmerged: y = W_int4(x) + (alpha/r) B A x.
The alternative merges delta = (alpha/r) B A into the dequantized weight and
quantizes the sum again to int4 with per-group-of-64 scale and offset. The page
states that LoRA deltas (RMS about 1e-3) lie below the 4-bit group step, so the
requantization removes most of the delta. Its two measures:
  * weight level, per target matrix: sum(actual * delta) / sum(delta^2), where
    actual = dequant(requant(W + delta)) - W is what the merge really changed;
  * output level: 1 - |U - M| / |U - B|, for the outputs of the unmerged (U),
    merged (M) and base (B) models on the same input.
The page measures the output level on first-token logits. The synthetic stack
has no logits, so here the output is the shared expert's, with LoRA on its
gate, up and down projections.

Requantization follows the plain reading of the page's int4 format: affine,
in groups of 64 inputs along a row, with an fp16 scale and offset. Per group,
s = fp16((max - min) / 15), b = fp16(min), q = clip(round((w - b) / s), 0, 15),
w' = s q + b. The page does not say whether the merge recomputes the group
scales. keep_grid=True is the other reading: it rounds onto the base's own
grid, with the same s and b.
"""
from __future__ import annotations

import numpy as np

GROUP = 64


def fp16(x):
    """Round to the nearest fp16 value, returned as fp64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def quantize_g64(W):
    """Affine int4 quantization of W [out, in] per row and group of 64 inputs:
    returns nibbles q [out, in] and fp16 scales s, offsets b [out, in / 64]."""
    out, inp = W.shape
    assert inp % GROUP == 0
    G = W.reshape(out, inp // GROUP, GROUP)
    lo, hi = G.min(axis=2), G.max(axis=2)
    s = fp16((hi - lo) / 15.0)
    s = np.where(s > 0, s, fp16(np.float64(2.0 ** -24)))   # a constant group: any step
    b = fp16(lo)
    q = np.clip(np.rint((G - b[..., None]) / s[..., None]), 0, 15)
    return q.reshape(out, inp), s, b


def dequant_g64(q, s, b):
    """w = s q + b per group of 64 inputs."""
    out, inp = q.shape
    G = q.reshape(out, inp // GROUP, GROUP)
    return (s[..., None] * G + b[..., None]).reshape(out, inp)


def requant_on_grid(W, s, b):
    """W rounded onto a given grid: q = clip(round((w - b) / s), 0, 15)."""
    out, inp = W.shape
    G = W.reshape(out, inp // GROUP, GROUP)
    q = np.clip(np.rint((G - b[..., None]) / s[..., None]), 0, 15).reshape(out, inp)
    return dequant_g64(q, s, b)


def merge_requant(W, delta, keep_grid=False):
    """The merged weight: W + delta quantized again (fresh group scales, or the
    grid of W's own quantization) and dequantized."""
    if keep_grid:
        _, s, b = quantize_g64(W)
        return requant_on_grid(W + delta, s, b)
    return dequant_g64(*quantize_g64(W + delta))


def weight_retention(W, delta, keep_grid=False):
    """sum(actual * delta) / sum(delta^2), actual = merged - W."""
    actual = merge_requant(W, delta, keep_grid) - W
    return float(np.sum(actual * delta) / np.sum(delta * delta))


def output_retention(U, M, B):
    """1 - |U - M| / |U - B| (Frobenius norms over all outputs)."""
    return float(1.0 - np.linalg.norm(U - M) / np.linalg.norm(U - B))


def silu(z):
    return z / (1.0 + np.exp(-z))


def swiglu(Wg, Wu, Wd, X):
    """Rows of X are tokens: down(silu(gate x) * up x)."""
    return (silu(X @ Wg.T) * (X @ Wu.T)) @ Wd.T


def lora_study(Wg, Wu, Wd, loras, scale, X, keep_grid=False):
    """Unmerged, merged and base outputs of a SwiGLU expert whose three
    projections carry LoRA deltas; loras = ((Ag, Bg), (Au, Bu), (Ad, Bd)).
    Returns (weight retention per projection, output retention)."""
    (Ag, Bg), (Au, Bu), (Ad, Bd) = loras
    dg, du, dd = scale * Bg @ Ag, scale * Bu @ Au, scale * Bd @ Ad
    # unmerged: the base weights plus the parallel delta on each projection
    # (silu(g + dg x) * (u + du x), then down plus its delta applied to the act)
    g = X @ Wg.T + (X @ Ag.T) @ (scale * Bg).T
    u = X @ Wu.T + (X @ Au.T) @ (scale * Bu).T
    a = silu(g) * u
    U = a @ Wd.T + (a @ Ad.T) @ (scale * Bd).T
    M = swiglu(merge_requant(Wg, dg, keep_grid), merge_requant(Wu, du, keep_grid),
               merge_requant(Wd, dd, keep_grid), X)
    B = swiglu(Wg, Wu, Wd, X)
    w = {"gate": weight_retention(Wg, dg, keep_grid), "up": weight_retention(Wu, du, keep_grid),
         "down": weight_retention(Wd, dd, keep_grid)}
    return w, output_retention(U, M, B)


def synthetic_base(rng, out, inp):
    """An int4 group-64 matrix drawn like the synthetic stack's weights: nibbles
    and zero-points uniform over 0..15, s = fp16(U[0.5, 1.5) / (8 sqrt(in))),
    b = fp16(-s z); returns its dequantized value."""
    ng = inp // GROUP
    q = rng.integers(0, 16, size=(out, inp)).astype(np.float64)
    s = fp16(rng.uniform(0.5, 1.5, size=(out, ng)) / (8.0 * np.sqrt(inp)))
    z = rng.integers(0, 16, size=(out, ng)).astype(np.float64)
    b = fp16(-s * z)
    return dequant_g64(q, s, b)


def synthetic_lora(rng, out, inp, r, scale, rms):
    """LoRA factors A [r, in], B [out, r] with Gaussian entries, rescaled so that
    delta = scale B A has the given RMS."""
    A = rng.standard_normal((r, inp))
    B = rng.standard_normal((out, r))
    d = scale * B @ A
    f = np.sqrt(rms / np.sqrt(np.mean(d * d)))
    return A * f, B * f


def study_table(rms_values=(3e-4, 1e-3, 3e-3, 1e-2), seed=0):
    """Retention over LoRA delta RMS for the 35B-tier shared expert's shapes
    (d = 2048, I_s = 512, r = 16, alpha = 32) under both readings of the
    requantization; rows (rms, reading, weight retention per projection, output
    retention).  A fresh draw of the LoRA factors per RMS value."""
    rng = np.random.default_rng(seed)
    d, Is, r, alpha = 2048, 512, 16, 32.0
    sc = alpha / r
    Wg, Wu, Wd = synthetic_base(rng, Is, d), synthetic_base(rng, Is, d), synthetic_base(rng, d, Is)
    X = rng.standard_normal((64, d))
    rows = []
    for rms in rms_values:
        loras = (synthetic_lora(rng, Is, d, r, sc, rms), synthetic_lora(rng, Is, d, r, sc, rms),
                 synthetic_lora(rng, d, Is, r, sc, rms))
        for keep in (False, True):
            w, o = lora_study(Wg, Wu, Wd, loras, sc, X, keep_grid=keep)
            rows.append((rms, "base grid" if keep else "fresh scales", w, o))
    return rows


if __name__ == "__main__":
    print("| delta RMS | requantization | gate | up | down | output |")
    print("|---|---|---|---|---|---|")
    for rms, reading, w, o in study_table():
        print(f"| {rms:g} | {reading} | {w['gate']:.3f} | {w['up']:.3f} | {w['down']:.3f} | {o:.3f} |")
