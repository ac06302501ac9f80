"""CUDA path vs the CPU oracle on the same seeded inputs, through the C ABI.

Sizes: small cases the oracle finishes in seconds that still span several row
tiles and groups plus ragged batches; the 35B single layer and the 40-layer
35B stack at full size in the launch configuration the bench times (checked on
the first steps).  Tolerances are in tests/parity_util.py.
"""
import numpy as np
import pytest
import torch

import oracle
from int4_routed_expert_prerouter_gb300 import binding, configs, inputs
from parity_util import assert_close, routing_matches, selection_scores, weights_by_id

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _cpu_model(model):
    """Host copy of a model drawn on the device (for the oracle)."""
    m = inputs.Model(model.cfg, model.seed)
    for lw in model.layers:
        c = lambda trip: tuple(t.cpu() for t in trip)
        m.layers.append(inputs.LayerWeights(c(lw.gate), c(lw.up), c(lw.down), c(lw.sh_gate),
                                            c(lw.sh_up), c(lw.sh_down), lw.router.cpu(),
                                            lw.gamma.cpu(), {k: v.cpu() for k, v in lw.lora.items()},
                                            None if lw.bias is None else lw.bias.cpu(),
                                            None if lw.head is None else
                                            {k: (v.cpu() if torch.is_tensor(v) else v)
                                             for k, v in lw.head.items()},
                                            lw.prerouted))
    return m


# ------------------------------------------------------------- packing ----
# Reference packers written from the layout description in include/edge0.h:
# lane L = 4g + t of a row tile's 16-input step holds rows g and g + 8 at
# step-local inputs {2t, 2t+1, 2t+8, 2t+9}; matrices that multiply x are stored
# by halves of their input groups, down by halves of its output row tiles
# (half 0: the first n // 2).
_NIB = [(0, 0), (1, 0), (0, 8), (1, 8), (0, 1), (1, 1), (0, 9), (1, 9)]   # (row + 8?, k offset) of nibble p


def _nibbles(q):
    """q [..., in/8] int32 -> [..., in] int64 nibble values (input 8j+i = nibble i of word j)."""
    w = q.to(torch.int64) & 0xFFFFFFFF
    return torch.stack([(w >> (4 * i)) & 0xF for i in range(8)], dim=-1).flatten(-2)


def _q4_units(N, S, Bq):
    """N [..., 16, in] nibbles of one row tile, S/Bq [..., 16, in/64] fp16 ->
    words [..., in/64, 4, 32] (step, lane) int64 and scales [..., in/64, 8, 4] int16."""
    inp = N.shape[-1]
    ng = inp // 64
    Nv = N.reshape(*N.shape[:-1], ng, 4, 16)            # [..., 16 rows, group, step, k]
    words = torch.zeros(*N.shape[:-2], ng, 4, 32, dtype=torch.int64)
    for g in range(8):
        for t in range(4):
            w = torch.zeros(*N.shape[:-2], ng, 4, dtype=torch.int64)
            for pos, (hi, ko) in enumerate(_NIB):
                w |= Nv[..., g + 8 * hi, :, :, 2 * t + ko] << (4 * pos)
            words[..., 4 * g + t] = w
    sv = S.view(torch.int16).transpose(-1, -2)          # [..., group, 16 rows]
    bv = Bq.view(torch.int16).transpose(-1, -2)
    sc = torch.stack([sv[..., :8], bv[..., :8], sv[..., 8:], bv[..., 8:]], dim=-1)   # [..., group, 8, 4]
    return words, sc


def _to_u8(words, sc):
    """unit bytes: 4 step words per lane (lane-major, 16 B each) then 64 B of scales."""
    w32 = words.to(torch.int32)                          # wraps to the same bits
    lane_major = w32.transpose(-1, -2).contiguous()      # [..., group, 32 lanes, 4 steps]
    a = lane_major.view(torch.uint8).flatten(-3)         # [..., group * 512]
    return a, sc.contiguous().view(torch.uint8)


def _ref_pack_gate_up(gate, up):
    qg, sg, bg = gate
    qu, su, bu = up
    E, I, w8 = qg.shape
    Ng, Nu = _nibbles(qg), _nibbles(qu)                  # [E, I, d]
    rows = torch.cat([Ng.view(E, I // 8, 8, -1), Nu.view(E, I // 8, 8, -1)], dim=2)   # [E, tiles, 16, d]
    S = torch.cat([sg.view(E, I // 8, 8, -1), su.view(E, I // 8, 8, -1)], dim=2)
    Bq = torch.cat([bg.view(E, I // 8, 8, -1), bu.view(E, I // 8, 8, -1)], dim=2)
    words, sc = _q4_units(rows, S, Bq)                   # [E, tiles, ng, 4, 32], [E, tiles, ng, 8, 4]
    w32 = words.to(torch.int32).transpose(-1, -2).contiguous()              # [E, tiles, ng, 32, 4]
    units = torch.cat([w32.view(torch.uint8).flatten(-2), sc.contiguous().view(torch.uint8).flatten(-2)], -1)
    n0 = units.shape[2] // 2                             # [E, tiles, ng, 576] -> [E, half, tiles, groups, 576]
    halves = [units[:, :, :n0].reshape(E, -1), units[:, :, n0:].reshape(E, -1)]
    return torch.cat(halves, dim=1).reshape(-1)


def _ref_pack_down(trip):
    q, s, b = trip
    E, out, w8 = q.shape
    n_rt = (out + 15) // 16
    N = torch.zeros(E, n_rt * 16, w8 * 8, dtype=torch.int64)
    N[:, :out] = _nibbles(q)
    S = torch.zeros(E, n_rt * 16, s.shape[-1], dtype=torch.float16)
    Bq = torch.zeros_like(S)
    S[:, :out] = s
    Bq[:, :out] = b
    words, sc = _q4_units(N.view(E, n_rt, 16, -1), S.view(E, n_rt, 16, -1), Bq.view(E, n_rt, 16, -1))
    # words [E, rt, g, 4 steps, 32 lanes] -> per group and half of the row tiles:
    # [4 steps][rt of the half][32 lanes] words, then [rt of the half] scales
    w = words.to(torch.int32).permute(0, 2, 3, 1, 4).contiguous()           # [E, g, 4, rt, 32]
    scv = sc.permute(0, 2, 1, 3, 4).contiguous()                            # [E, g, rt, 8, 4]
    ng = w.shape[1]
    n0 = n_rt // 2
    parts = []
    for lo, hi in ((0, n0), (n0, n_rt)):
        parts.append(w[:, :, :, lo:hi].contiguous().view(torch.uint8).view(E, ng, -1))
        parts.append(scv[:, :, lo:hi].contiguous().view(torch.uint8).view(E, ng, -1))
    return torch.cat(parts, -1).reshape(-1)


def _ref_pack_f16(W, cols=None, kmajor=False):
    out, ld = W.shape
    inp = cols or ld
    n_rt, ns = (out + 15) // 16, inp // 16
    Wp = torch.zeros(n_rt * 16, inp, dtype=torch.int16)
    Wp[:out] = W[:, :inp].view(torch.int16)
    Wv = Wp.view(n_rt, 16, ns, 16)                       # [rt, row, step, k]
    blk = torch.zeros(n_rt, ns, 32, 8, dtype=torch.int16)
    for g in range(8):
        for t in range(4):
            L = 4 * g + t
            order = [(g, 2 * t), (g, 2 * t + 1), (g + 8, 2 * t), (g + 8, 2 * t + 1),
                     (g, 2 * t + 8), (g, 2 * t + 9), (g + 8, 2 * t + 8), (g + 8, 2 * t + 9)]
            for j, (row, k) in enumerate(order):
                blk[:, :, L, j] = Wv[:, row, :, k]
    if kmajor:
        return blk.transpose(0, 1).contiguous().view(torch.uint8).reshape(-1)
    ng = ns // 4
    n0 = ng // 2                                         # [rt, step, ...] -> [half, rt, groups, 4 steps, ...]
    blk = blk.view(n_rt, ng, 4, 32, 8)
    return torch.cat([blk[:, :n0].reshape(-1), blk[:, n0:].reshape(-1)]).view(torch.uint8).reshape(-1)


@pytest.mark.parametrize("E,I,d", [(3, 64, 256), (2, 128, 128), (1, 512, 2048), (2, 64, 192)])
def test_pack_q4_gate_up_layout(E, I, d):
    gate = inputs.int4_stack(5, 1, 1, E, I, d)
    up = inputs.int4_stack(5, 1, 2, E, I, d)
    got = binding.pack_q4_gate_up(tuple(t.to(DEV) for t in gate), tuple(t.to(DEV) for t in up)).cpu()
    assert torch.equal(got, _ref_pack_gate_up(gate, up))


@pytest.mark.parametrize("E,out,inp", [(3, 48, 256), (2, 20, 128), (1, 2048, 512), (2, 80, 192)])
def test_pack_q4_down_layout(E, out, inp):
    trip = inputs.int4_stack(6, 1, 3, E, out, inp)
    got = binding.pack_q4_down(tuple(t.to(DEV) for t in trip)).cpu()
    assert torch.equal(got, _ref_pack_down(trip))


@pytest.mark.parametrize("out,inp,cols", [(48, 256, None), (4, 128, None), (64, 288, 256), (32, 192, None)])
@pytest.mark.parametrize("kmajor", [False, True])
def test_pack_f16_layout(out, inp, cols, kmajor):
    W = (torch.randn(out, inp, generator=torch.Generator().manual_seed(3))).half()
    got = binding.pack_f16(W.to(DEV), cols=cols, kmajor=kmajor).cpu()
    assert torch.equal(got, _ref_pack_f16(W, cols, kmajor))
    T = binding.pack_cols_T(W.to(DEV), 8, 16).cpu()
    assert torch.equal(T, W[:, 8:24].t().contiguous())


# ------------------------------------------------------ standalone ops ----
def _moe_ws(cfg, B):
    n = binding.workspace_bytes(1, B, cfg.d, cfg.E)
    return torch.zeros(n, dtype=torch.uint8, device=DEV)


MOE_CASES = [
    configs.TOY.with_(B=1),
    configs.TOY.with_(B=3),
    configs.STACK35.with_(L=1, E=32, B=1),
    configs.STACK35.with_(L=1, E=32, B=2),
    configs.STACK8.with_(L=1, E=32, B=2, zipf=None),
]


@pytest.mark.parametrize("cfg", MOE_CASES, ids=lambda c: f"{c.name}-d{c.d}-E{c.E}-B{c.B}")
def test_moe_int4_forward(cfg):
    model = inputs.make_model(cfg.with_(L=1, head_owner_last=-1, prerouted=()), seed=11)
    lw = model.layers[0]
    dm = binding.DeviceModel(model, DEV)
    ws = _moe_ws(cfg, cfg.B)
    for trial in range(2):
        x = torch.stack([oracle.rmsnorm(h) for h in inputs.hidden(cfg, trial, seed=11)])
        ids, w = inputs.routing(cfg, 11, trial)
        if cfg.B > 1 and trial == 1:
            ids[1] = ids[0]          # two tokens on the same experts
        y = binding.moe_int4_forward(dm, 0, x.to(DEV), ids.to(DEV), w.to(DEV), ws)
        torch.cuda.synchronize()
        _, y_ref = oracle.moe_forward(cfg, lw, x, ids, w)
        assert_close(y, y_ref, f"moe y (trial {trial})")


@pytest.mark.parametrize("cfg", [configs.TOY.with_(B=2), configs.STACK35.with_(L=2, B=1),
                                 configs.STACK8.with_(L=2, B=2, head_owner_first=0,
                                                      head_owner_last=0)],
                         ids=lambda c: f"{c.name}-B{c.B}")
@pytest.mark.parametrize("with_prev", [False, True])
def test_prerouter_topk(cfg, with_prev):
    cfg = cfg.with_(head_owner_first=0, head_owner_last=0)
    model = inputs.make_model(cfg, seed=21)
    dm = binding.DeviceModel(model, DEV)
    hd = model.layers[0].head
    tgt_bias = model.layers[hd["target"]].bias
    n = binding.workspace_bytes(1, cfg.B, cfg.d, cfg.E)
    ws = torch.zeros(n, dtype=torch.uint8, device=DEV)
    x = torch.stack([oracle.rmsnorm(h) for h in inputs.hidden(cfg, 4, seed=21)])
    ex, _ = inputs.routing(cfg, 21, 1)
    pv, _ = inputs.routing(cfg, 21, 2)
    ids, w, lg = binding.prerouter_topk(dm, 0, x.to(DEV), ex.to(DEV), pv.to(DEV) if with_prev else None, ws)
    torch.cuda.synchronize()
    for b in range(cfg.B):
        ref_lg = oracle.prerouter_logits(hd["fc1"], hd["fc2"], hd["linit"], x[b], ex[b],
                                         pv[b] if with_prev else None, cfg.d, cfg.E, cfg.H, cfg.K)
        assert_close(lg[b], ref_lg, f"head logits b={b}")
        if cfg.route_kind == configs.SIGMOID_GROUP:
            rid, rw = oracle.route_sigmoid_group(ref_lg, cfg.K, cfg.n_groups, cfg.topk_groups,
                                                 cfg.route_scale, tgt_bias)
        else:
            rid, rw = oracle.route_softmax_topk(ref_lg, cfg.K, tgt_bias)
        sc = selection_scores(ref_lg.numpy(), cfg.route_kind,
                              None if tgt_bias is None else tgt_bias.numpy())
        ok = routing_matches(ids[b].cpu(), rid, sc, cfg.K, cfg.n_groups if cfg.route_kind else None,
                             cfg.topk_groups if cfg.route_kind else None)
        if ok is True:
            assert_close(w[b], rw, f"head weights b={b}")


@pytest.mark.parametrize("cfg", [configs.TOY.with_(B=3), configs.STACK35.with_(L=1, E=16, B=2)],
                         ids=lambda c: c.name)
def test_lora_delta(cfg):
    model = inputs.make_model(cfg.with_(L=1, head_owner_last=-1, prerouted=()), seed=31)
    dm = binding.DeviceModel(model, DEV)
    lo = model.layers[0].lora
    g = torch.Generator().manual_seed(31)
    for name, desc, A, Bm, inp, out in (("gate", dm.layers[0].lora_gate, lo["Ag"], lo["Bg"], cfg.d, cfg.Is),
                                        ("down", dm.layers[0].lora_down, lo["Ad"], lo["Bd"], cfg.Is, cfg.d)):
        v = torch.randn(cfg.B, inp, generator=g).half()
        y0 = (torch.randn(cfg.B, out, generator=g) * 0.1).half()
        y = y0.to(DEV).contiguous()
        binding.lora_delta(desc, v.to(DEV).contiguous(), y)
        torch.cuda.synchronize()
        for b in range(cfg.B):
            delta = oracle.lora_delta(A, Bm, cfg.alpha, v[b].double())
            ref = y0[b].double() + delta
            # fp16 output: one rounding of y0 + delta on top of the 2e-3 contract
            err = (y[b].cpu().double() - ref).abs().max().item()
            tol = 2e-3 * delta.abs().max().item() + 2.0**-11 * ref.abs().max().item()
            assert err <= tol, f"lora {name} b={b}: {err:.3e} > {tol:.3e}"


# ------------------------------------------------------------ decode ----
# Protocol.  The oracle runs each decode step from the routing state the GPU
# had before the step (predictions and executed ids), so steps are compared
# independently of each other.  Within a step, a batch-1 call records every
# layer's output h and every head's logits (edge0_route_state.record_*): the
# oracle then runs each layer on the GPU's own input to it (teacher-forced
# inside the single launch).  A near-tie (K-th and (K+1)-th selection scores
# closer than 1e-3) may let the GPU execute other experts: the oracle layer is
# then rerun with the GPU's ids (weights from the oracle's own logits under the
# layer's routing rule) and its output compared.  The batched path records no
# layers: there a near-tie excludes the affected sequence's row from that
# step's h comparison only, and is reported.

def _routing_kw(cfg):
    return dict(n_groups=cfg.n_groups if cfg.route_kind else None,
                G=cfg.topk_groups if cfg.route_kind else None)


def _state_of(st):
    return tuple(x.cpu().clone() for x in (st.pred_ids, st.pred_w, st.exec_ids))


def _oracle_layer(ref, l, h_in, t, state):
    """Oracle decode layer l at step t on h_in [B, d] fp16 from routing state
    `state` (pred_ids, pred_w, exec_ids); returns (h_out, record)."""
    ref.pred_ids.copy_(state[0])
    ref.pred_w.copy_(state[1])
    ref.exec_ids.copy_(state[2])
    h = h_in.clone().contiguous()
    rec = ref.step(h, t, layers=[l])
    return h, rec


def _oracle_layer_forced(ref, cfg, l, h_in, t, state, ids, logits, bias):
    """Layer l of one sequence with its routing forced to the GPU's `ids`: the
    layer's routing rule on the oracle's logits restricted to those ids gives
    the weights (softmax over them; sigmoid weights s sigma / sum sigma), and
    the layer runs on that routing as a prediction (step t + 2: same slots)."""
    lg = torch.full_like(logits, float("-inf"))
    idx = torch.as_tensor(ids).long()
    lg[idx] = logits[idx]
    if cfg.route_kind == configs.SIGMOID_GROUP:
        fi, fw = oracle.route_sigmoid_group(lg, cfg.K, 1, 1, cfg.route_scale, None)
    else:
        fi, fw = oracle.route_softmax_topk(lg, cfg.K, bias)
    assert sorted(fi.tolist()) == sorted(idx.tolist())
    pred_ids, pred_w, exec_ids = (x.clone() for x in state)
    t2 = t + 2
    pred_ids[(t2 - 1) & 1, l, 0] = fi
    pred_w[(t2 - 1) & 1, l, 0] = fw
    was = ref.layers[l].prerouted
    ref.layers[l].prerouted = 1
    try:
        return _oracle_layer(ref, l, h_in, t2, (pred_ids, pred_w, exec_ids))
    finally:
        ref.layers[l].prerouted = was


def _check_head(cfg, model, ref, l, t, rec, pred_after, predw_after, ties, what, gpu_logits=None):
    """A head's logits (when recorded) and its prediction for the next token."""
    lw = model.layers[l]
    tg = lw.head["target"]
    ref_lg = rec["head_logits"][l, 0]
    if gpu_logits is not None:
        assert_close(gpu_logits, ref_lg, f"{what}: head logits")
    tb = model.layers[tg].bias
    sc = selection_scores(ref_lg.numpy(), cfg.route_kind, None if tb is None else tb.cpu().numpy())
    r = routing_matches(pred_after[t & 1, tg, 0], ref.pred_ids[t & 1, tg, 0], sc, cfg.K, **_routing_kw(cfg),
                        ordered=False)
    if r is True:
        gw, rw = weights_by_id(pred_after[t & 1, tg, 0], predw_after[t & 1, tg, 0],
                               ref.pred_ids[t & 1, tg, 0], ref.pred_w[t & 1, tg, 0])
        assert_close(gw, rw, f"{what}: head weights")
    else:
        ties.append((t, l, "head"))


def _check_recorded_step(cfg, model, ref, st, before, h0, t, ties):
    """Every layer of one recorded batch-1 decode call, teacher-forced on the
    GPU's own per-layer inputs.  Returns the number of heads checked."""
    rec_h, rec_lg = st.rec_h.cpu(), st.rec_logits.cpu()
    exec_after, pred_after, predw_after = (x.cpu() for x in (st.exec_ids, st.pred_ids, st.pred_w))
    n_heads = 0
    for l in range(cfg.L):
        lw = model.layers[l]
        h_in = (h0 if l == 0 else rec_h[l - 1]).view(1, cfg.d)
        h_ref, rec = _oracle_layer(ref, l, h_in, t, before)
        gpu_ids = exec_after[t & 1, l, 0]
        what = f"step {t} layer {l}"
        if lw.prerouted and t > 0:
            # the prediction made one token earlier is the routing, as is
            assert gpu_ids.tolist() == before[0][(t - 1) & 1, l, 0].tolist(), what
        else:
            bias = None if lw.bias is None else lw.bias.cpu()
            lg = rec["router_logits"][l, 0]
            sc = selection_scores(lg.numpy(), cfg.route_kind, None if bias is None else bias.numpy())
            r = routing_matches(gpu_ids, rec["ids"][l, 0], sc, cfg.K, **_routing_kw(cfg), ordered=False)
            if r == "tie":
                ties.append((t, l, "layer"))
                h_ref, rec = _oracle_layer_forced(ref, cfg, l, h_in, t, before, gpu_ids, lg, bias)
        assert_close(rec_h[l], h_ref[0], f"{what}: h")
        if lw.head is not None:
            n_heads += 1
            _check_head(cfg, model, ref, l, t, rec, pred_after, predw_after, ties, what, rec_lg[l])
    return n_heads


def _run_stack(cfg, model, steps, use_layers=False, pool_slots=None, on_pool=None, inject=None,
               double_prefetch=False):
    """Decode `steps` steps on the GPU and check each against the oracle (see the
    protocol above).  Returns (steps compared, near-ties seen).  pool_slots: run
    the routed experts from a host tier with that many device slots per layer,
    prefetched after each step from the predictions (on_pool(pool) at the end);
    inject: (fail_every, delay_ns) for the pool's copy passes; double_prefetch:
    request each step's prefetch twice in a row (the second finds the layers'
    copies in flight).  Only the compute stream is synchronised between steps:
    the pool's copies run on."""
    dm = binding.DeviceModel(model, DEV)
    st = binding.DecodeState(cfg, device=DEV)
    recorded = cfg.B == 1 and not use_layers
    if recorded:
        st.record(True)
    pool = binding.ExpertPool(dm, pool_slots) if pool_slots else None
    if inject is not None:
        pool.inject(*inject)
    prerouted = [l for l in range(cfg.L) if model.layers[l].prerouted]
    ref = oracle.Stack(_cpu_model(model) if model.layers[0].gate[0].is_cuda else model)
    ties = []
    for t in range(steps):
        before = _state_of(st)
        h0 = inputs.hidden(cfg, t, seed=model.seed)
        h = h0.to(DEV).contiguous()
        if use_layers:
            for l in range(cfg.L):
                binding.decode_layer(dm, l, st, h, t)
        else:
            binding.decode_step(dm, st, h, t)
        if pool is not None:
            own = [l for l in range(cfg.L) if l not in prerouted]
            pool.prefetch(st, t, predicted=prerouted, cached=own)
            if double_prefetch:
                pool.prefetch(st, t, predicted=prerouted, cached=own)
        torch.cuda.current_stream().synchronize()
        assert st.error() == 0
        if recorded:
            assert torch.equal(h.cpu()[0], st.rec_h[cfg.L - 1].cpu())
            _check_recorded_step(cfg, model, ref, st, before, h0, t, ties)
            continue
        # whole step in the oracle from the GPU's state; rows without a near-tie
        ref.pred_ids.copy_(before[0])
        ref.pred_w.copy_(before[1])
        ref.exec_ids.copy_(before[2])
        h_ref = h0.clone()
        rec = ref.step(h_ref, t)
        exec_gpu, pred_gpu, predw_gpu = (x.cpu() for x in (st.exec_ids, st.pred_ids, st.pred_w))
        tied_rows = set()
        for l in range(cfg.L):
            lw = model.layers[l]
            bias = None if lw.bias is None else lw.bias.cpu().numpy()
            for b in range(cfg.B):
                if b in tied_rows:
                    continue
                if lw.prerouted and t > 0:
                    assert sorted(exec_gpu[t & 1, l, b].tolist()) == sorted(before[0][(t - 1) & 1, l, b].tolist())
                    continue
                sc = selection_scores(rec["router_logits"][l, b].numpy(), cfg.route_kind, bias)
                try:
                    r = routing_matches(exec_gpu[t & 1, l, b], rec["ids"][l, b], sc, cfg.K, **_routing_kw(cfg),
                                        ordered=False)
                except AssertionError as e:
                    raise AssertionError(f"step {t} layer {l} b {b} executed ids: {e}") from None
                if r == "tie":
                    tied_rows.add(b)
                    ties.append((t, l, f"row {b}"))
            if lw.head is not None:
                tg = lw.head["target"]
                tb = model.layers[tg].bias
                for b in range(cfg.B):
                    if b in tied_rows:
                        continue
                    sc = selection_scores(rec["head_logits"][l, b].numpy(), cfg.route_kind,
                                          None if tb is None else tb.cpu().numpy())
                    r = routing_matches(pred_gpu[t & 1, tg, b], ref.pred_ids[t & 1, tg, b], sc, cfg.K,
                                        **_routing_kw(cfg), ordered=False)
                    if r is True:
                        gw, rw = weights_by_id(pred_gpu[t & 1, tg, b], predw_gpu[t & 1, tg, b],
                                               ref.pred_ids[t & 1, tg, b], ref.pred_w[t & 1, tg, b])
                        assert_close(gw, rw, f"pred w t={t} l={l} b={b}")
                    else:
                        ties.append((t, l, f"head row {b}"))
        rows = [b for b in range(cfg.B) if b not in tied_rows]
        assert rows, f"step {t}: every row met a near-tie"
        assert_close(h.cpu()[rows], h_ref[rows], f"h after step {t}")
    if on_pool is not None:
        on_pool(pool)
    if ties:
        print(f"{cfg.name}: near-ties re-checked or excluded: {ties}")
    return steps, ties


def test_decode_toy_stack_8_steps():
    cfg = configs.TOY
    model = inputs.make_model(cfg, seed=0)
    assert _run_stack(cfg, model, cfg.steps)[0] == cfg.steps


def test_decode_toy_layer_by_layer_matches():
    cfg = configs.TOY
    model = inputs.make_model(cfg, seed=1, gamma="random")
    assert _run_stack(cfg, model, 4, use_layers=True)[0] == 4


def test_decode_toy_ragged_batch():
    cfg = configs.TOY.with_(B=3)
    model = inputs.make_model(cfg, seed=2)
    assert _run_stack(cfg, model, 5)[0] == 5


def test_decode_8b_shapes_small():
    cfg = configs.STACK8.with_(L=3, E=32, B=1, head_owner_first=0, head_owner_last=1,
                               prerouted=(1, 2))
    model = inputs.make_model(cfg, seed=3)
    assert _run_stack(cfg, model, 4)[0] == 4


def test_decode_35b_layer_ring_full_size():
    cfg = configs.LAYER35
    model = inputs.make_model(cfg, seed=0, device=DEV)
    assert _run_stack(cfg, model, 6)[0] == 6


def test_decode_35b_stack_first_8_layers_full_size():
    # one persistent launch over consecutive layers (own-routed 0-6, head owners
    # from 6, prerouted from 7) at full size
    cfg = configs.STACK35.with_(L=8, head_owner_last=6, prerouted=(7,))
    model = inputs.make_model(cfg, seed=0, device=DEV)
    assert _run_stack(cfg, model, 3)[0] == 3


def test_decode_35b_stack_benched_call_layer_by_layer():
    # The call bench.py times: one batch-1 launch of all 40 layers of the
    # 35B-tier stack followed by the 33-head flush, at full size.  Every layer's
    # output and every head's logits and prediction of each of 3 steps are
    # checked element by element (the protocol above).
    cfg = configs.STACK35
    model = inputs.make_model(cfg, seed=0, device=DEV)
    dm = binding.DeviceModel(model, DEV)
    st = binding.DecodeState(cfg, device=DEV)
    st.record(True)
    ref = oracle.Stack(_cpu_model(model))
    ties = []
    for t in range(3):
        before = _state_of(st)
        h0 = inputs.hidden(cfg, t)
        h = h0.to(DEV).contiguous()
        binding.decode_step(dm, st, h, t)
        torch.cuda.synchronize()
        assert st.error() == 0
        assert torch.equal(h.cpu()[0], st.rec_h[cfg.L - 1].cpu())
        assert _check_recorded_step(cfg, model, ref, st, before, h0, t, ties) == len(cfg.head_owners()) == 33
    print(f"near-ties re-checked with the GPU's ids: {ties}")


def test_decode_35b_stack_40_layers_full_size_properties():
    # what holds at any depth and for any step, free-running: distinct ids in
    # range, renormalised weights, predictions consumed as the next routing
    cfg = configs.STACK35
    model = inputs.make_model(cfg, seed=0, device=DEV)
    dm = binding.DeviceModel(model, DEV)
    st = binding.DecodeState(cfg, device=DEV)
    st_prev = None
    for t in range(3):
        h = inputs.hidden(cfg, t).to(DEV).contiguous()
        binding.decode_step(dm, st, h, t)
        torch.cuda.synchronize()
        assert st.error() == 0
        ex = st.exec_ids[t & 1].cpu()
        for l in range(cfg.L):
            ids = ex[l, 0].tolist()
            assert len(set(ids)) == cfg.K and all(0 <= e < cfg.E for e in ids)
        pr = st.pred_ids[t & 1].cpu()
        pw = st.pred_w[t & 1].cpu()
        for l in cfg.head_owners():
            tg = l + 1
            assert len(set(pr[tg, 0].tolist())) == cfg.K
            assert abs(float(pw[tg, 0].sum()) - 1.0) < 1e-5        # renormalised softmax
        if t > 0:
            for l in cfg.prerouted:
                assert sorted(ex[l, 0].tolist()) == sorted(st_prev[l, 0].tolist())
        st_prev = pr.clone()
        assert torch.isfinite(h.float()).all()


# ------------------------------------------------ batched decode path ----
# B > 4 sequences run on the batched path (experts grouped by token lists).
def test_batched_toy_ragged_batch():
    cfg = configs.TOY.with_(B=7)
    model = inputs.make_model(cfg, seed=6, gamma="random")
    assert _run_stack(cfg, model, 5)[0] == 5


def test_batched_toy_layer_by_layer():
    cfg = configs.TOY.with_(B=5)
    model = inputs.make_model(cfg, seed=8)
    assert _run_stack(cfg, model, 4, use_layers=True)[0] == 4


def test_batched_8b_shapes_small():
    # sigmoid-group routing with the Zipf selection bias, K = 8
    cfg = configs.STACK8.with_(L=3, E=32, B=16, head_owner_first=0, head_owner_last=1,
                               prerouted=(1, 2))
    model = inputs.make_model(cfg, seed=7)
    assert _run_stack(cfg, model, 4)[0] == 4


def test_batched_35b_shapes_small_zipf():
    # softmax-topK with the Zipf logit bias: a few experts take most tokens
    cfg = configs.HOST35.with_(L=3, E=64, B=37, head_owner_first=0, head_owner_last=1,
                               prerouted=(1, 2), pool_frac=None)
    model = inputs.make_model(cfg, seed=9)
    assert _run_stack(cfg, model, 3)[0] == 3


def _check_pool(pool, seen):
    """After the run: counters, residency counters, and every published slot
    holding its expert's bytes (device compare, bit-exact)."""
    st = pool.stats()
    tiers = pool.tiers()
    seen.update(stats=st, tiers=tiers)
    for l, ((sg, sd, tb), (hg, hd)) in enumerate(zip(pool.slots, pool.host)):
        table = tb.cpu().tolist()
        pub = [s for s in table if s >= 0]
        assert len(pub) == len(set(pub)), f"layer {l}: a slot published twice"
        for e, s in enumerate(table):
            if s < 0:
                continue
            g, d = pool.gu_bytes, pool.dn_bytes
            assert torch.equal(sg[s * g:(s + 1) * g].cpu(), hg[e * g:(e + 1) * g]), (l, e, s)
            assert torch.equal(sd[s * d:(s + 1) * d].cpu(), hd[e * d:(e + 1) * d]), (l, e, s)
    print(f"pool: {st}; active / host-tier experts per layer: {tiers.tolist()}")


def test_host_tier_batched_decode_matches_oracle():
    # 16 device slots for 64 experts: predicted experts are copied in ahead of
    # their layer, the rest (and own-routed layers) are read from host memory
    cfg = configs.HOST35.with_(L=3, E=64, B=24, head_owner_first=0, head_owner_last=1,
                               prerouted=(1, 2), pool_frac=0.25)
    model = inputs.make_model(cfg, seed=11)
    seen = {}
    n, _ = _run_stack(cfg, model, 4, pool_slots=16, on_pool=lambda p: _check_pool(p, seen))
    assert n == 4
    st, tiers = seen["stats"], seen["tiers"]
    assert st["published"] > 0 and st["hits"] > 0 and st["failed"] == 0 and st["bad_ids"] == 0
    assert 0 < tiers[:, 1].sum() < tiers[:, 0].sum()


def test_host_tier_full_cfg5_shapes_256_sequences():
    # E = 256 experts, 64 slots per layer, 256 sequences, 35B-tier expert
    # shapes: the predictions name more experts than there are slots, so each
    # prerouted layer runs partly from its slots and partly from host memory
    cfg = configs.HOST35.with_(L=3, head_owner_first=0, head_owner_last=1, prerouted=(1, 2))
    assert (cfg.E, cfg.B, int(cfg.E * cfg.pool_frac)) == (256, 256, 64)
    model = inputs.make_model(cfg, seed=13, device=DEV)
    seen = {}
    n, _ = _run_stack(cfg, model, 3, pool_slots=64, on_pool=lambda p: _check_pool(p, seen))
    assert n == 3
    st, tiers = seen["stats"], seen["tiers"]
    assert st["published"] > 0 and st["hits"] > 0
    assert tiers[1:, 1].sum() > 0 and tiers[1:, 1].sum() < tiers[1:, 0].sum()


def test_host_tier_delayed_and_failed_copies_keep_results_exact():
    # Host-side injection: every copy pass starts 0.4 s late and every third
    # copy fails; each step's prefetch is requested twice.  The steps do not
    # wait for copies: experts whose copies are late or failed are read from
    # host memory, plans of layers with copies in flight are skipped, and every
    # step still matches the oracle.
    cfg = configs.HOST35.with_(L=3, E=64, B=24, head_owner_first=0, head_owner_last=1,
                               prerouted=(1, 2), pool_frac=0.25)
    model = inputs.make_model(cfg, seed=12)
    seen = {}
    n, _ = _run_stack(cfg, model, 5, pool_slots=16, inject=(3, 400_000_000), double_prefetch=True,
                      on_pool=lambda p: _check_pool(p, seen))
    assert n == 5
    st, tiers = seen["stats"], seen["tiers"]
    assert st["skipped"] > 0 and st["failed"] > 0 and st["published"] > 0
    assert tiers[1:, 1].sum() > 0


def test_host_tier_bounded_wait_for_copies():
    # edge0_pool_wait polls from the host up to its limit: with the copy pass
    # held back 0.5 s it returns EDGE0_ETIMEOUT after 2 ms, then EDGE0_OK.
    import time
    cfg = configs.HOST35.with_(L=3, E=64, B=24, head_owner_first=0, head_owner_last=1,
                               prerouted=(1, 2), pool_frac=0.25)
    model = inputs.make_model(cfg, seed=14)
    dm = binding.DeviceModel(model, DEV)
    st = binding.DecodeState(cfg, device=DEV)
    pool = binding.ExpertPool(dm, 16)
    pool.inject(0, 500_000_000)
    binding.decode_step(dm, st, inputs.hidden(cfg, 0, seed=14).to(DEV), 0)
    pool.prefetch(st, 0, cached=[1, 2])
    t0 = time.time()
    assert pool.wait(2_000_000) == binding.EDGE0_ETIMEOUT
    assert time.time() - t0 < 0.4
    assert pool.wait(5_000_000_000) == binding.EDGE0_OK
    assert pool.stats()["published"] > 0


def test_batched_8b_full_shapes_64_sequences_teacher_forced():
    cfg = configs.STACK8.with_(L=3, head_owner_first=0, head_owner_last=1, prerouted=(1, 2))
    model = inputs.make_model(cfg, seed=0, device=DEV)
    calls, _ = _teacher_forced(cfg, model, steps=2)
    assert calls == 6


def test_batched_35b_full_shapes_256_sequences_teacher_forced():
    cfg = configs.HOST35.with_(L=2, head_owner_first=0, head_owner_last=0, prerouted=(1,),
                               pool_frac=None)
    model = inputs.make_model(cfg, seed=0, device=DEV)
    calls, _ = _teacher_forced(cfg, model, steps=2)
    assert calls == 4


# ------------------------------------------------- teacher-forced layers ----
def _teacher_forced(cfg, model, steps, layers=None, verbose=True):
    """Every layer call on the GPU gets the oracle's h and routing state as input
    (oracle -> GPU only); each layer's outputs are compared with the oracle's.
    A row whose routing meets a near-tie is compared with the oracle rerun on
    the GPU's ids (B == 1), or left out of that call's h check (B > 1).
    Returns (compared layer calls, fp16 elements that differ per call)."""
    dm = binding.DeviceModel(model, DEV)
    st = binding.DecodeState(cfg, device=DEV)
    ref = oracle.Stack(_cpu_model(model) if model.layers[0].gate[0].is_cuda else model)
    layers = list(range(cfg.L)) if layers is None else layers
    calls, flips, worst = 0, 0, 0.0
    head_logits_prev = None
    ties = []
    for t in range(steps):
        h_ref = inputs.hidden(cfg, t, seed=model.seed)
        rec_t = {}
        for l in range(cfg.L):
            before = (ref.pred_ids.clone(), ref.pred_w.clone(), ref.exec_ids.clone())
            st.pred_ids.copy_(ref.pred_ids)
            st.pred_w.copy_(ref.pred_w)
            st.exec_ids.copy_(ref.exec_ids)
            h_in = h_ref.clone()
            h = h_in.to(DEV).contiguous()
            if l in layers:
                binding.decode_layer(dm, l, st, h, t)
            rec = ref.step(h_ref, t, layers=[l])
            rec_t[l] = rec
            if l not in layers:
                continue
            torch.cuda.synchronize()
            assert st.error() == 0
            lw = model.layers[l]
            bias = None if lw.bias is None else lw.bias.cpu()
            rows = list(range(cfg.B))
            h_cmp = h_ref
            for b in range(cfg.B):
                if lw.prerouted and t > 0:
                    lg = head_logits_prev[l - 1 if not cfg.ring else l][b]
                else:
                    lg = rec["router_logits"][l, b]
                gpu_ids = st.exec_ids[t & 1, l, b].cpu()
                r = routing_matches(gpu_ids, rec["ids"][l, b],
                                    selection_scores(lg.numpy(), cfg.route_kind,
                                                     None if bias is None else bias.numpy()),
                                    cfg.K, **_routing_kw(cfg), ordered=False)
                if r == "tie":
                    ties.append((t, l, b))
                    if cfg.B == 1 and not (lw.prerouted and t > 0):
                        state = tuple(x.clone() for x in before)
                        h_cmp, rec_f = _oracle_layer_forced(ref, cfg, l, h_in, t, state, gpu_ids, lg, bias)
                        ref.pred_ids.copy_(before[0])   # the reference run continues on its own routing
                        ref.pred_w.copy_(before[1])
                        ref.exec_ids.copy_(before[2])
                        ref.step(h_in.clone(), t, layers=[l])
                    else:
                        rows.remove(b)
            if not rows:
                continue
            rel = assert_close(h.cpu()[rows], h_cmp[rows], f"h after step {t} layer {l}")
            worst = max(worst, rel)
            flips += int((h.cpu()[rows] != h_cmp[rows]).sum())
            calls += 1
            if lw.head is not None:
                tg = lw.head["target"]
                tb = model.layers[tg].bias
                for b in range(cfg.B):
                    sc = selection_scores(rec["head_logits"][l, b].numpy(), cfg.route_kind,
                                          None if tb is None else tb.cpu().numpy())
                    gi, gw = st.pred_ids[t & 1, tg, b].cpu(), st.pred_w[t & 1, tg, b].cpu()
                    ri, rw = ref.pred_ids[t & 1, tg, b], ref.pred_w[t & 1, tg, b]
                    r = routing_matches(gi, ri, sc, cfg.K, **_routing_kw(cfg), ordered=False)
                    if r is True:
                        gw2, rw2 = weights_by_id(gi, gw, ri, rw)
                        assert_close(gw2, rw2, f"pred w t={t} l={l}")
        head_logits_prev = {l: rec_t[l]["head_logits"][l] for l in rec_t}
    if verbose:
        print(f"{cfg.name}: {calls} layer calls, worst rel err {worst:.2e}, "
              f"{flips / max(calls, 1):.2f} fp16 elements differ per call (of {cfg.B * cfg.d}); "
              f"near-ties {ties}")
    return calls, flips / max(calls, 1)


def test_teacher_forced_35b_stack_full_size():
    cfg = configs.STACK35
    model = inputs.make_model(cfg, seed=0, device=DEV)
    calls, _ = _teacher_forced(cfg, model, steps=3)
    assert calls == 3 * cfg.L


def test_teacher_forced_toy_8_steps():
    cfg = configs.TOY
    model = inputs.make_model(cfg, seed=5, gamma="random")
    calls, _ = _teacher_forced(cfg, model, steps=cfg.steps)
    assert calls == cfg.steps * cfg.L


# ------------------------------------------------------- bounded waits ----
def test_bounded_wait_runs_out_then_the_state_recovers():
    # A short wait limit and the workspace's hold hook (the launch's first grid
    # barrier waits for one arrival more than the grid makes): every wait gives
    # up within the limit, the launch records EDGE0_ETIMEOUT and leaves; after
    # edge0_state_error reports it the state is clean and the next step matches
    # the oracle.  Nothing faults or traps: the kernel returns.
    import time
    cfg = configs.TOY
    model = inputs.make_model(cfg, seed=0)
    dm = binding.DeviceModel(model, DEV)
    st = binding.DecodeState(cfg, device=DEV)
    h = inputs.hidden(cfg, 0).to(DEV).contiguous()
    st.set_wait_limit(300_000)           # 0.3 ms
    st.hold_first_barrier(1)
    t0 = time.time()
    binding.decode_step(dm, st, h, 0)
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert st.error() == binding.EDGE0_ETIMEOUT
    assert st.error() == 0               # reported once; the state was re-initialised
    ref = oracle.Stack(model)
    for t in range(2):
        h0 = inputs.hidden(cfg, t)
        h = h0.to(DEV).contiguous()
        binding.decode_step(dm, st, h, t)
        torch.cuda.synchronize()
        assert st.error() == 0
        h_ref = h0.clone()
        ref.step(h_ref, t, record=False)
        assert_close(h.cpu(), h_ref, f"h after step {t} following a timeout")
