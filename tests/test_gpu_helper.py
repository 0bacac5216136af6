"""One MoE layer split between the active card and the idle-stage helper ("prefill: a layer
split's idle card streams a share of a one-chunk prompt's experts", What), both played by
this GPU one after the other: the helper groups, runs and hands back the rows of its
share of the routed experts through mapped host memory with a ready word; the active card
runs the rest, waits (bounded) for the word, copies the helper's rows in and combines.
The layer's output has the bits of the unsplit layer and matches the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import BOUND, bf16_dev, rel_err, to_f64
from host_offloaded_weight_gb300 import lstream as L
from oracle import forward as F
from oracle import helper as Hp

pytestmark = pytest.mark.gpu


def _layer(cfg, W, x, lg, rows_mask=None):
    """Route, group (optionally over a subset of experts), gather and run both grouped GEMMs.
    Returns (Y fp32 [T*k, H] with the kept rows written, table, bounds, kept row count)."""
    T, H, Fd, E, k = cfg.tokens, cfg.hidden, cfg.ffn, cfg.n_experts, cfg.top_k
    rows = T * k
    dev = x.device
    sel = torch.empty(rows, dtype=torch.int32, device=dev)
    w = torch.empty(rows, dtype=torch.float32, device=dev)
    table = torch.empty(rows, dtype=torch.int32, device=dev)
    bounds = torch.empty(E + 1, dtype=torch.int32, device=dev)
    used = torch.zeros(E, dtype=torch.uint8, device=dev)
    L.lsk_moe_route(lg, 1, T, E, k, sel, w)
    if rows_mask is None:
        L.lsk_moe_group(sel, 1, T, E, k, table, bounds, used)
    else:
        L.lsk_moe_group_masked(sel, 1, T, E, k, rows_mask, table, bounds, used)
    n = int(bounds[E].item())
    xs = torch.empty(max(n, 1), H, dtype=torch.bfloat16, device=dev)
    hsd = torch.empty(max(n, 1), Fd, dtype=torch.bfloat16, device=dev)
    Y = torch.full((rows, H), float("nan"), dtype=torch.float32, device=dev)
    seg = synth.segment_slot_bytes(cfg)
    eb = seg // E
    if n:
        L.lsk_moe_gather(x, table, n, k, H, xs)
        L.lsk_gemm_grouped_bf16(L.LSK_EPI_SWIGLU, xs, W, seg // (2 * H), 0, eb // (2 * H), Fd, bounds, E, hsd,
                                n, Fd, H)
        L.lsk_gemm_grouped_bf16(L.LSK_EPI_SCALE_F32, hsd, W, seg // (2 * Fd), 2 * H, eb // (2 * Fd), 0, bounds, E,
                                Y, n, H, Fd, row_table=table, row_weight=w)
    return Y, table, bounds, n, used, sel


CASES = {
    "small": synth.MOE.with_(n_segments=1, tokens=200, hidden=128, ffn=64, n_experts=16, top_k=4),
    "full_layer": synth.MOE.with_(n_segments=1),   # one layer at the stack's shapes: 2048 tokens, 128 experts
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_helper_split_keeps_the_bits_of_the_layer(name):
    cfg = CASES[name]
    T, H, E, k = cfg.tokens, cfg.hidden, cfg.n_experts, cfg.top_k
    hs = synth.HostStack(cfg)
    W = torch.from_numpy(hs.buffer[:synth.segment_slot_bytes(cfg)]).cuda()
    xb = synth.draw_x(cfg)
    x = bf16_dev(xb)
    lg_np = synth.draw_logits(cfg, 0)
    lg = torch.from_numpy(lg_np).cuda()

    # unsplit layer
    Y, table, bounds, n, used, sel = _layer(cfg, W, x, lg)
    out_full = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    L.lsk_moe_combine(x, Y, T, k, H, out_full)

    # the split: which experts the helper takes
    share = L.ls_helper_share(T)
    assert share > 0
    routed = used.cpu().numpy()
    helper = L.ls_helper_split(routed, share)
    mine = (routed.astype(bool) & ~helper.astype(bool)).astype(np.uint8)
    assert helper.sum() == int(np.floor(share * routed.sum())) > 0
    helper_dev, mine_dev = torch.from_numpy(helper).cuda(), torch.from_numpy(mine).cuda()

    # the idle card: its experts only, rows handed back through mapped host memory
    Yh, table_h, bounds_h, n_h, _, _ = _layer(cfg, W, x, lg, helper_dev)
    assert n_h > 0
    handoff = torch.empty(n_h, H, dtype=torch.float32).pin_memory()
    ready = torch.zeros(1, dtype=torch.int32, device="cuda")
    ticket = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.lsk_moe_rows_copy(Yh, handoff, n_h, H, src_table=table_h, ready=ready, ticket=ticket, epoch=7)

    # the active card: the other experts, then the bounded wait, the helper's rows, the combine
    Yp, table_p, bounds_p, n_p, _, _ = _layer(cfg, W, x, lg, mine_dev)
    assert n_p + n_h == T * k
    err = torch.zeros(1, dtype=torch.int32).pin_memory()
    L.lsk_wait_ready(ready, 7, 2000, err, 0)
    _, table_h2, _, _, _, _ = _layer(cfg, W, x, lg, helper_dev)       # the same table, built here
    L.lsk_moe_rows_copy(handoff, Yp, n_h, H, dst_table=table_h2)
    out_split = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    L.lsk_moe_combine(x, Yp, T, k, H, out_split)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "the hand-off wait ran out"
    assert torch.equal(table_h2[:n_h], table_h[:n_h])
    assert not torch.isnan(Yp).any(), "a row was written by neither card"
    assert torch.equal(out_split.view(torch.int16), out_full.view(torch.int16)), "the split changed the bits"

    # and the split matches the fp64 oracle's split (itself equal to the plain layer)
    specs = synth.segment_tensors(cfg)
    rows_t = np.arange(0, T, max(1, T // 64))

    def experts(e):
        return [F.as_f64(np.asarray(a), s.dtype) for a, s in zip(hs.seg_views[0][3 * e:3 * e + 3], specs[3 * e:3 * e + 3])]
    ref = Hp.moe_layer_split(F.as_f64(xb, "bf16")[rows_t], lg_np[rows_t], experts, k, share)
    assert rel_err(to_f64(out_split)[rows_t], ref) <= BOUND
