"""Merged versus unmerged recovery LoRA ("The Other Half of the Memory Wall",
S3.3 "Recovery LoRA: Unmerged by Design"): the retention study in
oracle/retention.py, pinned against closed forms and special cases, then run in
the page's regime (LoRA delta RMS about 1e-3) on the 35B-tier shared expert's
synthetic shapes."""
import math

import numpy as np
import pytest

from oracle import retention as R


def on_grid(rng, out, inp, lo_q=0, hi_q=15):
    """Exactly representable int4 weights; each group holds nibbles 0 and 15 so
    that its range fixes the fresh scale to the drawn one."""
    ng = inp // R.GROUP
    q = rng.integers(lo_q, hi_q + 1, size=(out, ng, R.GROUP)).astype(np.float64)
    q[:, :, 0], q[:, :, 1] = 0, 15
    s = R.fp16(rng.uniform(0.5, 1.5, size=(out, ng)) / 64.0)
    b = R.fp16(-s * rng.integers(0, 16, size=(out, ng)))
    return R.dequant_g64(q.reshape(out, inp), s, b), q, s


def test_quantize_reproduces_an_exactly_representable_matrix():
    rng = np.random.default_rng(1)
    W, q, s = on_grid(rng, 8, 256)
    q2, s2, _ = R.quantize_g64(W)
    assert np.array_equal(s2, s)
    assert np.array_equal(q2, q.reshape(8, 256))
    assert np.array_equal(R.dequant_g64(*R.quantize_g64(W)), W)


@pytest.mark.parametrize("keep_grid", [False, True])
def test_deltas_on_the_grid_survive_whole(keep_grid):
    # whole steps on interior entries (the group's extremes untouched): the merge
    # lands exactly on W + delta
    rng = np.random.default_rng(2)
    W, q, s = on_grid(rng, 8, 256, 1, 14)
    k = rng.integers(-1, 2, size=q.shape).astype(np.float64)
    k[:, :, :2] = 0
    delta = (k * s[..., None]).reshape(W.shape)
    assert R.weight_retention(W, delta, keep_grid) == pytest.approx(1.0, abs=1e-12)


@pytest.mark.parametrize("keep_grid", [False, True])
def test_deltas_below_half_a_step_vanish(keep_grid):
    rng = np.random.default_rng(3)
    W, q, s = on_grid(rng, 8, 256, 1, 14)
    delta = rng.uniform(-0.45, 0.45, size=q.shape) * s[..., None]
    delta[:, :, :2] = 0
    delta = delta.reshape(W.shape)
    assert R.weight_retention(W, delta, keep_grid) == 0.0


def test_keep_grid_retention_matches_its_closed_form():
    # on the base grid, actual = s round(delta / s): for Gaussian delta of
    # deviation sigma (no clipping), E[actual delta] / E[delta^2] =
    # sum_k k s sigma (phi((k - 1/2) s / sigma) - phi((k + 1/2) s / sigma)) / sigma^2
    rng = np.random.default_rng(4)
    W, q, s = on_grid(rng, 256, 1024, 5, 10)
    s0 = s[..., None]
    sigma_steps = 0.4
    delta = rng.standard_normal(q.shape) * sigma_steps * s0
    delta[:, :, :2] = 0
    got = R.weight_retention(W, delta.reshape(W.shape), keep_grid=True)

    def phi(x):
        return math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)

    # in units of the step (the same ratio in every group)
    num = sum(k * sigma_steps * (phi((k - 0.5) / sigma_steps) - phi((k + 0.5) / sigma_steps))
              for k in range(-6, 7))
    want = num / sigma_steps ** 2
    assert got == pytest.approx(want, abs=0.02)


def test_large_deltas_survive_fresh_scales():
    # with fresh group scales the grid follows the merged range; (on the base's
    # own grid a delta of tens of steps clips at nibbles 0 and 15 instead)
    rng = np.random.default_rng(5)
    W = R.synthetic_base(rng, 64, 512)
    delta = rng.standard_normal(W.shape) * 0.1   # tens of steps
    assert R.weight_retention(W, delta) > 0.98


def test_output_retention_ends():
    rng = np.random.default_rng(6)
    U, B = rng.standard_normal((4, 8)), rng.standard_normal((4, 8))
    assert R.output_retention(U, U, B) == 1.0
    assert R.output_retention(U, B, B) == 0.0


def test_page_regime_on_the_35b_shared_expert():
    # The page's regime: LoRA delta RMS ~1e-3 on every projection of the shared
    # expert.  The synthetic steps are ~2.8e-3 for gate/up (d = 2048 inputs) and
    # ~5.5e-3 for down (512 inputs).  The output keeps a minority of the
    # unmerged effect under either reading of the requantization; deltas ten
    # times larger keep most of it.
    rng = np.random.default_rng(0)
    d, Is, r, alpha = 2048, 512, 16, 32.0
    sc = alpha / r
    Wg, Wu, Wd = R.synthetic_base(rng, Is, d), R.synthetic_base(rng, Is, d), R.synthetic_base(rng, d, Is)
    X = rng.standard_normal((64, d))
    out = {}
    for rms in (1e-3, 1e-2):
        loras = (R.synthetic_lora(rng, Is, d, r, sc, rms), R.synthetic_lora(rng, Is, d, r, sc, rms),
                 R.synthetic_lora(rng, d, Is, r, sc, rms))
        for keep in (False, True):
            out[rms, keep] = R.lora_study(Wg, Wu, Wd, loras, sc, X, keep_grid=keep)
    for keep in (False, True):
        assert out[1e-3, keep][1] < 0.5
        assert out[1e-2, keep][1] > 0.5
        # the down projection (the larger step) keeps less than gate/up
        w = out[1e-3, keep][0]
        assert w["down"] < w["gate"] and w["down"] < w["up"]
