"""Pins for the CPU oracle: each test ties one oracle routine to something other
than the oracle itself -- numbers the pages print (tests/golden), closed forms,
library routines (numpy / scipy) on special cases, invariants, or hand-checkable
tiny cases.  Chosen so that a dropped term, a wrong sign, a wrong index or a
transposed operand in the oracle fails at least one of them."""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy import special

import oracle
from int4_routed_expert_prerouter_gb300 import configs, inputs

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))


# ------------------------------------------------------------------ fp16 ----
def test_half_to_double_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_double_to_half_rounding_matches_numpy():
    rng = np.random.default_rng(0)
    vals = [0.0, -0.0, 1.0, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11, 65504.0, 65519.99, 65520.0, 1e6,
            2.0**-24, 2.0**-25, 3 * 2.0**-26, 2.0**-14, 2.0**-14 - 2.0**-25, 6.0e-8, 1e-12]
    vals += list(rng.standard_normal(4000) * np.exp(rng.uniform(-20, 12, 4000)))
    # exact midpoints between neighbouring halves (ties go to even)
    vals += list(rng.integers(0, 0x7bff, 2000).astype(np.uint16).view(np.float16).astype(np.float64))
    hv = np.arange(0, 0x7bff, 37, dtype=np.uint16)
    lo, hi = hv.view(np.float16).astype(np.float64), (hv + 1).view(np.float16).astype(np.float64)
    vals += list((lo + hi) / 2)
    vals += [-v for v in vals]
    vals = np.array(vals, dtype=np.float64)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_half(v) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ int4 ----
def test_int4_nibble_order_and_roundtrip():
    # word 0x76543210: nibble i (bits 4i..4i+3) holds input element 8j+i
    w = torch.tensor([0x76543210, -0x01234568 & 0xFFFFFFFF], dtype=torch.int64).to(torch.int32)
    nib = oracle.int4_unpack(w)
    assert nib[:8].tolist() == list(range(8))
    rng = torch.Generator().manual_seed(1)
    q = torch.randint(-2**31, 2**31 - 1, (999,), generator=rng, dtype=torch.int64).to(torch.int32)
    assert torch.equal(oracle.int4_pack(oracle.int4_unpack(q)), q)
    n = torch.randint(0, 16, (800,), generator=rng, dtype=torch.uint8)
    assert torch.equal(oracle.int4_unpack(oracle.int4_pack(n)), n)


def test_int4_dequant_hand_case_and_group_boundary():
    out, inp = 2, 128
    nib = torch.zeros(out, inp, dtype=torch.uint8)
    nib[0, :] = 3
    nib[1, :] = torch.arange(inp) % 16
    q = oracle.int4_pack(nib.reshape(-1)).view(out, inp // 8)
    # group 0 of row 0: s=2, b=-1 -> w = 5; group 1 of row 0: s=0.5, b=+4 -> 5.5
    s = torch.tensor([[2.0, 0.5], [1.0, -1.0]], dtype=torch.float16)
    b = torch.tensor([[-1.0, 4.0], [0.0, 16.0]], dtype=torch.float16)
    w = oracle.int4_dequant(q, s, b, out, inp)
    assert torch.all(w[0, :64] == 5.0) and torch.all(w[0, 64:] == 5.5)
    assert w[0, 63] == 5.0 and w[0, 64] == 5.5
    assert torch.equal(w[1, :64], (torch.arange(64) % 16).double())
    assert torch.equal(w[1, 64:], 16.0 - (torch.arange(64, 128) % 16).double())


def test_int4_matvec_equals_dequantised_dense_gemv():
    q, s, b = inputs.int4_stack(3, 0, 1, 1, 48, 256)
    v = torch.randn(256, dtype=torch.float64, generator=torch.Generator().manual_seed(2))
    W = oracle.int4_dequant(q[0], s[0], b[0], 48, 256)
    y = oracle.int4_matvec(q[0], s[0], b[0], 48, 256, v)
    ref = W.numpy() @ v.numpy()
    assert np.allclose(y.numpy(), ref, rtol=1e-13, atol=1e-13)


def test_f16_matvec_is_a_plain_gemv():
    W = (torch.randn(37, 70, generator=torch.Generator().manual_seed(4)) * 0.3).half()
    v = torch.randn(70, dtype=torch.float64, generator=torch.Generator().manual_seed(5))
    assert np.allclose(oracle.f16_matvec(W, v).numpy(), W.double().numpy() @ v.numpy(), rtol=1e-13)


# -------------------------------------------------------- activations ------
def test_gelu_erf_closed_form():
    assert oracle.gelu_erf(0.0) == 0.0
    assert abs(oracle.gelu_erf(1.0) - 0.8413447460685429) < 1e-15
    assert abs(oracle.gelu_erf(-1.0) + 0.15865525393145707) < 1e-15
    xs = np.linspace(-9, 9, 721)
    got = np.array([oracle.gelu_erf(x) for x in xs])
    ref = xs * special.ndtr(xs)                        # GELU(x) = x * Phi(x)
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-15)
    # erf form, not the tanh approximation (0.84119199 at 1)
    tanh_form = 0.5 * (1 + math.tanh(math.sqrt(2 / math.pi) * (1 + 0.044715)))
    assert abs(oracle.gelu_erf(1.0) - tanh_form) > 1e-4


def test_silu_is_x_sigmoid_x():
    xs = np.linspace(-30, 30, 601)
    got = np.array([oracle.silu(x) for x in xs])
    assert np.allclose(got, xs * special.expit(xs), rtol=1e-14, atol=1e-300)


# ------------------------------------------------------------- routing -----
def _brute_topk(score, k):
    score = np.asarray(score, dtype=np.float32)
    order = np.lexsort((np.arange(score.size), -score.astype(np.float64)))
    return order[:k]


@pytest.mark.parametrize("n,k", [(16, 2), (256, 4), (128, 8), (7, 7), (5, 1)])
def test_topk_against_full_sort(n, k):
    rng = np.random.default_rng(n * 31 + k)
    for trial in range(20):
        sc = rng.standard_normal(n).astype(np.float32)
        if trial % 3 == 0:                               # exact ties
            sc = np.round(sc * 2) / 2
        got = oracle.topk(torch.from_numpy(sc), k).numpy()
        assert np.array_equal(got, _brute_topk(sc, k))


def test_softmax_topk_closed_forms():
    rng = np.random.default_rng(7)
    for E, K in [(256, 4), (16, 2), (8, 8)]:
        lg = rng.standard_normal(E).astype(np.float32) * 2
        ids, w = oracle.route_softmax_topk(torch.from_numpy(lg), K)
        assert np.array_equal(ids.numpy(), _brute_topk(lg, K))
        assert abs(float(w.double().sum()) - 1.0) < 1e-6
        # renormalised softmax: w_i / w_j = exp(l_i - l_j)
        li = lg[ids.numpy()].astype(np.float64)
        assert np.allclose(w.numpy() / w.numpy()[0], np.exp(li - li[0]), rtol=1e-6)
        if K == E:                                       # K = E is the plain softmax
            assert np.allclose(w.numpy(), special.softmax(lg.astype(np.float64))[ids.numpy()], rtol=1e-6)
    # a selection bias is added to the logits in fp32 before softmax and selection
    lg = rng.standard_normal(64).astype(np.float32)
    bias = (-1.1 * np.log(rng.permutation(64) + 1.0)).astype(np.float32)
    a = oracle.route_softmax_topk(torch.from_numpy(lg), 4, torch.from_numpy(bias))
    b = oracle.route_softmax_topk(torch.from_numpy((lg + bias).astype(np.float32)), 4)
    assert torch.equal(a[0], b[0]) and torch.allclose(a[1], b[1], rtol=0, atol=0)


def test_sigmoid_group_all_groups_is_sigmoid_topk():
    rng = np.random.default_rng(9)
    g = GOLD["sigmoid_group_8b"]
    for _ in range(10):
        lg = rng.standard_normal(128).astype(np.float32)
        ids, w = oracle.route_sigmoid_group(torch.from_numpy(lg), g["K"], g["n"], g["n"], g["s"])
        assert np.array_equal(ids.numpy(), _brute_topk(lg, g["K"]))   # sigmoid is monotone
        sig = special.expit(lg.astype(np.float64))[ids.numpy()]
        assert np.allclose(w.numpy(), g["s"] * sig / sig.sum(), rtol=1e-6)
        assert abs(float(w.double().sum()) - g["s"]) < 1e-5


def test_sigmoid_group_drops_weak_groups_hand_case():
    # 4 groups of 2 experts, keep G=2, pick K=2.  Expert 0 has the largest score,
    # but its partner is very weak, so group 0's top-2 sum loses to groups 2 and 3.
    inv = lambda p: math.log(p / (1 - p))              # logit whose sigmoid is p
    p = [0.99, 0.01, 0.30, 0.30, 0.60, 0.55, 0.52, 0.51]
    lg = torch.tensor([inv(v) for v in p], dtype=torch.float32)
    ids, w = oracle.route_sigmoid_group(lg, K=2, n_groups=4, G=2, scale=2.5)
    assert ids.tolist() == [4, 5]
    assert np.allclose(w.numpy(), 2.5 * np.array([0.60, 0.55]) / 1.15, rtol=1e-6)
    # the bias decides selection only; weights keep the raw sigmoid
    bias = torch.tensor([0, 0, 0, 0, 0, 0, 0.2, 0.2], dtype=torch.float32)
    ids, w = oracle.route_sigmoid_group(lg, 2, 4, 2, 2.5, bias)
    assert ids.tolist() == [6, 7]
    assert np.allclose(w.numpy(), 2.5 * np.array([0.52, 0.51]) / 1.03, rtol=1e-6)


# ---------------------------------------------------------------- head -----
def _head_case(d=128, E=16, H=32, K=2, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(d, generator=g).half()
    ex = torch.randperm(E, generator=g)[:K].to(torch.int32)
    pv = torch.randperm(E, generator=g)[:K].to(torch.int32)
    return x, ex, pv


def test_f_in_and_head_parameter_count_match_the_pages():
    for key, cfg in (("f_in_35b", configs.STACK35), ("f_in_8b", configs.STACK8)):
        assert cfg.f_in == GOLD[key]["value"] == GOLD[key]["d_model"] + 2 * GOLD[key]["E"]
    c = configs.STACK35
    assert c.H == GOLD["head_hidden_35b"]["value"]
    params = c.H * c.f_in + c.E * c.H + c.E * c.f_in      # fc1 + fc2 + linear_init, no bias
    assert params == GOLD["head_params"]["value"]
    heads = c.head_owner_last - c.head_owner_first + 1
    assert heads == GOLD["heads_bytes_35b"]["heads"]
    assert heads * params * 2 == GOLD["heads_bytes_35b"]["value"]
    assert (c.head_owner_first, c.head_owner_last) == (GOLD["heads_35b_owners"]["first"],
                                                      GOLD["heads_35b_owners"]["last"])
    assert (min(c.prerouted), max(c.prerouted)) == (GOLD["heads_35b_owners"]["consumers_first"],
                                                    GOLD["heads_35b_owners"]["consumers_last"])


def test_head_with_zero_mlp_is_linear_init_and_warm_starts_to_the_router():
    d, E, H, K = 128, 16, 32, 2
    x, ex, pv = _head_case(d, E, H, K)
    Wr = (torch.randn(E, d, generator=torch.Generator().manual_seed(3)) / math.sqrt(d)).half()
    fc1 = torch.zeros(H, d + 2 * E, dtype=torch.float16)
    fc2 = torch.zeros(E, H, dtype=torch.float16)
    linit = torch.cat([Wr, torch.zeros(E, 2 * E, dtype=torch.float16)], 1)
    lg = oracle.prerouter_logits(fc1, fc2, linit, x, ex, pv, d, E, H, K)
    ref = oracle.f16_matvec(Wr, x.double()).float()
    assert torch.equal(lg, ref)
    assert torch.equal(oracle.route_softmax_topk(lg, K)[0], oracle.route_softmax_topk(ref, K)[0])


def test_head_one_hot_feature_layout():
    d, E, H, K = 64, 8, 16, 3
    x, ex, pv = _head_case(d, E, H, K, seed=5)
    eye = torch.eye(E, dtype=torch.float16)
    linit = torch.cat([torch.zeros(E, d, dtype=torch.float16), eye, 2 * eye], 1)
    fc1 = torch.zeros(H, d + 2 * E, dtype=torch.float16)
    fc2 = torch.zeros(E, H, dtype=torch.float16)
    lg = oracle.prerouter_logits(fc1, fc2, linit, x, ex, pv, d, E, H, K)
    ref = torch.zeros(E)
    ref[ex.long()] += 1.0                                # executed mask comes first
    ref[pv.long()] += 2.0                                # then the previous token's mask
    assert torch.equal(lg, ref)
    lg0 = oracle.prerouter_logits(fc1, fc2, linit, x, ex, None, d, E, H, K)
    ref0 = torch.zeros(E)
    ref0[ex.long()] = 1.0
    assert torch.equal(lg0, ref0)                        # no previous token: zero mask


def test_head_gelu_sits_between_fc1_and_fc2():
    d, E, H, K = 64, 16, 16, 2
    x, ex, pv = _head_case(d, E, H, K, seed=6)
    x = (x.float() * 2).half()
    fc1 = torch.zeros(H, d + 2 * E, dtype=torch.float16)
    fc1[:, :H] = torch.eye(H, dtype=torch.float16)
    fc2 = torch.diag(torch.arange(1, E + 1, dtype=torch.float32)).half()   # not symmetric in use
    linit = torch.zeros(E, d + 2 * E, dtype=torch.float16)
    lg = oracle.prerouter_logits(fc1, fc2, linit, x, ex, pv, d, E, H, K)
    xv = x.double().numpy()[:H]
    ref = np.arange(1, E + 1) * xv * special.ndtr(xv)
    assert np.allclose(lg.numpy(), ref.astype(np.float32), rtol=2e-7, atol=1e-7)


# ---------------------------------------------------------------- LoRA -----
def test_lora_zero_B_and_rank_one_closed_form():
    g = torch.Generator().manual_seed(11)
    r, inp, out, alpha = 16, 128, 48, 32.0
    A = (torch.randn(r, inp, generator=g) * 0.02).half()
    v = torch.randn(inp, dtype=torch.float64, generator=g)
    assert torch.all(oracle.lora_delta(A, torch.zeros(out, r, dtype=torch.float16), alpha, v) == 0)
    # A = e_i in row 0 only, B = column c in column 0 only: dy = (alpha/r) * c * v_i
    A1 = torch.zeros(r, inp, dtype=torch.float16)
    A1[0, 5] = 1.0
    c = torch.randn(out, generator=g).half()
    B1 = torch.zeros(out, r, dtype=torch.float16)
    B1[:, 0] = c
    dy = oracle.lora_delta(A1, B1, alpha, v)
    assert torch.allclose(dy, (alpha / r) * c.double() * v[5], rtol=1e-15, atol=0)
    assert GOLD["lora_35b"]["alpha"] / GOLD["lora_35b"]["r"] == 2.0


# ------------------------------------------------------------- RMSNorm -----
def test_rmsnorm_closed_form_and_scale_invariance():
    h = torch.tensor([3.0, 4.0], dtype=torch.float16)
    x = oracle.rmsnorm(h, eps=0.0)
    rms = math.sqrt((9 + 16) / 2)
    assert x.tolist() == torch.tensor([3 / rms, 4 / rms]).half().tolist()
    hr = torch.randn(2048, generator=torch.Generator().manual_seed(1)).half()
    assert torch.equal(oracle.rmsnorm(hr, eps=0.0), oracle.rmsnorm((hr.float() * 4).half(), eps=0.0))
    gam = torch.full((2,), 2.0, dtype=torch.float16)
    assert torch.equal(oracle.rmsnorm(h, gam, eps=0.0).float(), (x.float() * 2))


# ------------------------------------------------------- SwiGLU expert -----
def _const_q4(out, inp, value):
    """int4 matrix whose every dequantised weight equals `value` (s = 0, b = value)."""
    q = torch.zeros(out, inp // 8, dtype=torch.int32)
    s = torch.zeros(out, inp // 64, dtype=torch.float16)
    b = torch.full((out, inp // 64), value, dtype=torch.float16)
    return q, s, b


def test_swiglu_hand_checkable_case():
    d = I = 64
    gate, up, down = _const_q4(I, d, 1 / 64), _const_q4(I, d, 1 / 32), _const_q4(d, I, 1 / 64)
    y = oracle.expert_swiglu(gate, up, down, torch.ones(d, dtype=torch.float64))
    # g = 1, u = 2, act = silu(1) * 2 for every intermediate row; y_j = 64 * act / 64
    expect = special.expit(1.0) * 1.0 * 2.0
    assert np.allclose(y.numpy(), expect, rtol=1e-15)
    # gate feeds silu, up does not: with gate 2/64 and up 1/64 the value differs
    y2 = oracle.expert_swiglu(_const_q4(I, d, 1 / 32), _const_q4(I, d, 1 / 64), down,
                              torch.ones(d, dtype=torch.float64))
    assert np.allclose(y2.numpy(), 2.0 * special.expit(2.0) * 1.0, rtol=1e-15)


def test_swiglu_zero_cases_linearity_and_gate_up_swap():
    cfg = configs.TOY
    lw = inputs.make_layer(cfg, 0, seed=4)
    e = 3
    gate = tuple(t[e] for t in lw.gate)
    up = tuple(t[e] for t in lw.up)
    down = tuple(t[e] for t in lw.down)
    x = oracle.rmsnorm(inputs.hidden(cfg, 0)[0]).double()
    y = oracle.expert_swiglu(gate, up, down, x)
    zero_up = _const_q4(cfg.I, cfg.d, 0.0)
    assert torch.all(oracle.expert_swiglu(gate, zero_up, down, x) == 0)
    assert torch.all(oracle.expert_swiglu(zero_up, up, down, x) == 0)
    down2 = (down[0], (down[1].float() * 2).half(), (down[2].float() * 2).half())
    assert torch.equal(oracle.expert_swiglu(gate, up, down2, x), 2 * y)
    ysw = oracle.expert_swiglu(up, gate, down, x)
    rel = float((ysw - y).norm() / y.norm())
    assert rel > 0.5, rel          # the pages report ~100% error for a gate/up swap


# ------------------------------------------------------------ byte counts ---
def test_expert_byte_counts_match_the_pages():
    assert configs.expert_bytes(1536, 512) == GOLD["expert_bytes_8b"]["value"]
    b35 = configs.expert_bytes(2048, 512)
    g = GOLD["expert_mb_35b"]
    assert round(b35 / 1e6, 2) == g["value_mb"]
    assert round(b35 * g["experts"] / 1e6) == g["layer_mb"]
    assert round(b35 * g["experts"] * g["layers"] / 2**30, 1) == g["total_gib"]
    assert round(4 * b35 / 1e6) == GOLD["layer_set_k4_mb"]["value_mb"]


# ------------------------------------------------------------ MoE block -----
def test_moe_forward_is_weighted_sum_plus_shared():
    cfg = configs.TOY.with_(B=2)
    lw = inputs.make_layer(cfg, 0, seed=8)
    x = torch.stack([oracle.rmsnorm(h) for h in inputs.hidden(cfg, 3)])
    ids, w = inputs.routing(cfg, 8, 0)
    _, y = oracle.moe_forward(cfg, lw, x, ids, w)
    sh = oracle.expert_swiglu(lw.sh_gate, lw.sh_up, lw.sh_down, x[1].double())
    ref = sh.clone()
    for k in range(cfg.K):
        e = int(ids[1, k])
        ref += float(w[1, k]) * oracle.expert_swiglu(tuple(t[e] for t in lw.gate),
                                                     tuple(t[e] for t in lw.up),
                                                     tuple(t[e] for t in lw.down), x[1].double())
    assert torch.allclose(y[1], ref, rtol=1e-12, atol=1e-14)
    y0 = oracle.moe_forward(cfg, lw, x, ids, torch.zeros_like(w))[1]
    assert torch.allclose(y0[1], sh, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------ decode semantics ----
def test_decode_routing_state_machine_toy():
    cfg = configs.TOY
    m = inputs.make_model(cfg, seed=0)
    st = oracle.Stack(m)
    recs = []
    for t in range(4):
        h = inputs.hidden(cfg, t)
        recs.append(st.step(h, t))
    for t, r in enumerate(recs):
        for l in range(cfg.L):
            lw = m.layers[l]
            x = r["x"][l, 0]
            own = oracle.route_softmax_topk(oracle.f16_matvec(lw.router, x.double()).float(), cfg.K)
            if l in cfg.prerouted and t > 0:
                # prediction made at t-1 by the head owned by layer l-1, routed with layer l's rule
                pred = oracle.route_softmax_topk(recs[t - 1]["head_logits"][l - 1, 0], cfg.K)
                assert torch.equal(r["ids"][l, 0], pred[0]) and torch.equal(r["w"][l, 0], pred[1])
            else:
                assert torch.equal(r["ids"][l, 0], own[0]) and torch.equal(r["w"][l, 0], own[1])
        # head of layer 0 sees this step's executed ids and last step's (none at t = 0)
        hd = m.layers[0].head
        prev = recs[t - 1]["ids"][0, 0] if t > 0 else None
        lg = oracle.prerouter_logits(hd["fc1"], hd["fc2"], hd["linit"], r["x"][0, 0], r["ids"][0, 0],
                                     prev, cfg.d, cfg.E, cfg.H, cfg.K)
        assert torch.equal(lg, r["head_logits"][0, 0])


def test_decode_layer_without_lora_equals_h_plus_moe():
    cfg = configs.TOY
    m = inputs.make_model(cfg, seed=2)
    for lw in m.layers:                                  # B = 0 switches the adapter off
        for k in ("Bg", "Bu", "Bd"):
            lw.lora[k] = torch.zeros_like(lw.lora[k])
    st = oracle.Stack(m)
    h = inputs.hidden(cfg, 0)
    h_in = h.clone()
    r = st.step(h, 0)
    _, y = oracle.moe_forward(cfg, m.layers[0], r["x"][0], r["ids"][0], r["w"][0])
    ref = (h_in.double() + y).numpy().astype(np.float16)
    assert np.array_equal(r["hout"][0].numpy(), ref)
    assert torch.equal(r["x"][0], torch.stack([oracle.rmsnorm(v) for v in h_in]))


def test_decode_lora_changes_only_through_shared_expert():
    cfg = configs.TOY
    m = inputs.make_model(cfg, seed=2)
    st = oracle.Stack(m)
    h = inputs.hidden(cfg, 0)
    h_in = h.clone()
    r = st.step(h, 0, layers=[0])
    lw, x = m.layers[0], r["x"][0, 0].double()
    a = 2.0  # alpha / r
    g = oracle.int4_matvec(*[t[0] for t in lw.sh_gate], cfg.Is, cfg.d, x)
    g += oracle.lora_delta(lw.lora["Ag"], lw.lora["Bg"], cfg.alpha, x)
    u = oracle.int4_matvec(*[t[0] for t in lw.sh_up], cfg.Is, cfg.d, x)
    u += oracle.lora_delta(lw.lora["Au"], lw.lora["Bu"], cfg.alpha, x)
    act = g * torch.sigmoid(g) * u
    ys = oracle.int4_matvec(*[t[0] for t in lw.sh_down], cfg.d, cfg.Is, act)
    ys += oracle.lora_delta(lw.lora["Ad"], lw.lora["Bd"], cfg.alpha, act)
    _, yr = oracle.moe_forward(cfg, lw, r["x"][0], r["ids"][0], r["w"][0])
    ysh_base = oracle.expert_swiglu(lw.sh_gate, lw.sh_up, lw.sh_down, x)
    ref = (h_in[0].double() + (yr[0] - ysh_base) + ys).numpy().astype(np.float16)
    assert np.array_equal(r["hout"][0, 0].numpy(), ref)
    assert a == cfg.alpha / cfg.r


def test_head_warm_start_predicts_what_the_next_router_would_pick():
    cfg = configs.TOY
    m = inputs.make_model(cfg, seed=6)
    hd = m.layers[0].head
    hd["fc1"] = torch.zeros_like(hd["fc1"])
    hd["fc2"] = torch.zeros_like(hd["fc2"])
    hd["linit"] = torch.cat([m.layers[1].router, torch.zeros(cfg.E, 2 * cfg.E, dtype=torch.float16)], 1)
    st = oracle.Stack(m)
    recs = [st.step(inputs.hidden(cfg, t), t) for t in range(3)]
    for t in range(1, 3):
        x0 = recs[t - 1]["x"][0, 0]
        want = oracle.route_softmax_topk(oracle.f16_matvec(m.layers[1].router, x0.double()).float(), cfg.K)
        assert torch.equal(recs[t]["ids"][1, 0], want[0])
