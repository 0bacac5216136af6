"""The idle-stage helper across two processes (gloo, CPU): rank 0 is the active card, rank 1
the idle card. For every MoE layer the active card hands the layer's input to the helper,
the helper computes the rows of its share of the routed experts and hands them back, and
the active card combines them with its own rows. The stack's output equals the oracle's
forward on one process ("prefill: a layer split's idle card streams a share of a one-chunk
prompt's experts", What). The gloo messages stand in for the mapped host memory the page
uses between the cards."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import synth

CFG = synth.MOE.with_(n_segments=3, tokens=16, hidden=16, ffn=8, n_experts=6, top_k=2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, out):
    import torch
    import torch.distributed as dist
    from oracle import forward as F
    from oracle import helper as Hp
    from oracle import stack as S
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    cfg = CFG
    share = Hp.helper_share(cfg.tokens)
    x = F.as_f64(synth.draw_x(cfg), cfg.dtype) if rank == 0 else np.zeros((cfg.tokens, cfg.hidden))
    sent = 0
    for layer in range(cfg.n_segments):
        xt = torch.from_numpy(np.ascontiguousarray(x))
        dist.broadcast(xt, src=0)                        # active card -> helper: the layer input
        x = xt.numpy()
        logits = synth.draw_logits(cfg, layer)
        sel, _ = F.route_topk(logits, cfg.top_k)
        mine, theirs = Hp.split_experts(np.unique(sel), share)

        def experts(e):
            specs = synth.segment_tensors(cfg)[3 * e:3 * e + 3]
            return [F.as_f64(a, s.dtype) for a, s in zip(synth.draw_expert(cfg, layer, e), specs)]
        keys = sorted((t, j) for t in range(cfg.tokens) for j in range(cfg.top_k) if sel[t, j] in set(theirs))
        if rank == 1:                                    # helper: only its share of the experts
            rows = Hp.expert_rows(x, logits, experts, cfg.top_k, theirs)
            buf = torch.from_numpy(np.stack([rows[key] for key in keys]) if keys else np.zeros((0, cfg.hidden)))
            dist.send(buf.contiguous(), dst=0)
            sent += len(keys)
        else:                                            # active card: its experts, then the combine
            rows = Hp.expert_rows(x, logits, experts, cfg.top_k, mine)
            buf = torch.zeros((len(keys), cfg.hidden), dtype=torch.float64)
            dist.recv(buf, src=1)
            rows.update({key: buf[i].numpy() for i, key in enumerate(keys)})
            x = Hp.combine(x, rows, cfg.top_k)
    if rank == 0:
        ref = S.stack_forward(cfg)
        out.put(("err", float(np.max(np.abs(x - ref)))))
    else:
        out.put(("rows", sent))
    dist.barrier()
    dist.destroy_process_group()


def test_helper_over_two_gloo_ranks_matches_the_oracle():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res["err"] < 1e-12
    assert res["rows"] > 0, "the helper computed no rows"
