"""Comparison helpers for the CUDA-vs-oracle parity tests.

Tolerances (fixed by the task's parity contract):
* fp16 outputs: max |gpu - ref| <= 2e-3 * max |ref|;
* routing ids: identical, except where the K-th and (K+1)-th selection scores of
  the oracle differ by less than 1e-3 (for sigmoid-group also the G-th and
  (G+1)-th group scores), where either choice is accepted;
* routing weights: compared only where the ids agree, within 2e-3 * max |w|.
"""
import numpy as np
import torch

REL_TOL = 2e-3
TIE = 1e-3


def assert_close(got, ref, what, rel=REL_TOL):
    got = got.detach().float().cpu()
    ref = ref.detach().double().cpu()
    err = (got.double() - ref).abs().max().item()
    scale = ref.abs().max().item()
    assert err <= rel * scale + 1e-12, f"{what}: max|diff| {err:.3e} > {rel:.0e} * {scale:.3e}"
    return err / max(scale, 1e-30)


def selection_scores(logits, kind, bias=None):
    """The scores the routing rule ranks (App. A): logits (+ bias) for softmax-topk,
    sigmoid(logits) (+ bias) for sigmoid-group, in fp32."""
    lg = np.asarray(logits, dtype=np.float32)
    b = None if bias is None else np.asarray(bias, dtype=np.float32)
    if kind == 1:
        s = (1.0 / (1.0 + np.exp(-lg.astype(np.float64)))).astype(np.float32)
        return s + b if b is not None else s
    return lg + b if b is not None else lg


def near_tie(scores, K, n_groups=None, G=None):
    """True when the K/(K+1) boundary (or the G/(G+1) group boundary) is closer than TIE."""
    s = np.sort(np.asarray(scores, dtype=np.float64))[::-1]
    if len(s) > K and s[K - 1] - s[K] < TIE:
        return True
    if n_groups and G and G < n_groups:
        per = len(scores) // n_groups
        gs = np.sort(np.sort(np.asarray(scores, np.float64).reshape(n_groups, per), axis=1)[:, -2:].sum(1))[::-1]
        if gs[G - 1] - gs[G] < TIE:
            return True
    return False


def routing_matches(got_ids, ref_ids, scores, K, n_groups=None, G=None, ordered=True):
    """Returns True when ids agree (as ordered lists when `ordered`, order swaps
    allowed between scores closer than TIE; as sets otherwise); returns 'tie' when
    they differ only at an allowed near-tie; raises otherwise."""
    got = [int(v) for v in got_ids]
    ref = [int(v) for v in ref_ids]
    if got == ref:
        return True
    sc = np.asarray(scores, dtype=np.float64)
    if not ordered and sorted(got) == sorted(ref):
        return True
    if sorted(got) == sorted(ref):
        # same set, different order: only allowed among near-equal scores
        for a, b in zip(got, ref):
            if a != b and abs(sc[a] - sc[b]) >= TIE:
                raise AssertionError(f"routing order differs beyond a tie: {got} vs {ref}")
        return True
    if near_tie(sc, K, n_groups, G):
        return "tie"
    srt = np.sort(sc)[::-1]
    raise AssertionError(f"routing differs with no near-tie: gpu {got} vs oracle {ref}; "
                         f"oracle K/K+1 gap {srt[K - 1] - srt[K]:.3e}")


def weights_by_id(got_ids, got_w, ref_ids, ref_w):
    """Weights reordered so that both follow the oracle's id order."""
    pos = {int(e): i for i, e in enumerate(got_ids)}
    return torch.tensor([float(got_w[pos[int(e)]]) for e in ref_ids]), torch.as_tensor(ref_w)
