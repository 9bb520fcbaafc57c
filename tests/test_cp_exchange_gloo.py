"""The context-parallel exchange across ranks, on CPU ranks with gloo.

What a multi-GPU version of this library would do per rank ("Add context
parallelism", Description: keys and values are all-gathered and queries are
sharded on the sequence; the key/value gradient goes back by the transpose of
the all-gather, a reduce-scatter):

  rank r holds the slots [r*S/cp, (r+1)*S/cp) of q, k, v, dout in
  load-balanced order (chunks r and 2cp-1-r);
  all-gather K and V (slot order = rank order);
  forward of its own query rows against the gathered K/V (what
  cp_attn_fwd_shard computes on one GPU);
  backward of its own rows: dq of those rows and fp32 dk/dv contributions
  over every key (what cp_attn_bwd_shard computes);
  reduce-scatter the dk/dv contributions, so rank r keeps the summed
  gradient of its own key slots.

The per-shard kernels are stood in for by the float64 oracle on the same
rows, so this checks the decomposition and the collectives, not the kernels
(unmeasured on hardware: no run here has more than one GPU).  The result
must equal unsharded causal attention and its gradients."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from context_causal_attention_load_gb300 import synth
from oracle import cp_attention as O

B, S, HQ, HKV, D = 1, 256, 4, 2, 64


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _reduce_scatter(full, world):
    """Sum over ranks of a [B, S, ...] tensor, each rank keeping its slots."""
    out = torch.empty((full.shape[0], full.shape[1] // world) + tuple(full.shape[2:]), dtype=full.dtype)
    chunks = [c.contiguous() for c in full.chunk(world, dim=1)]
    dist.reduce_scatter(out, chunks)
    return out


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cp = world
        pos = O.lb_positions(S, cp, True)
        rows = np.arange(rank * S // cp, (rank + 1) * S // cp)
        qn, kn, vn, dn = (synth.to_f64(t) for t in synth.attention_inputs(B, S, HQ, HKV, D, D, seed=3))
        # this rank's slots of the load-balanced tensors
        ql, kl, vl, dl = (torch.from_numpy(O.permute(x, pos)[:, rows].copy()) for x in (qn, kn, vn, dn))
        # all-gather of keys and values (slot order is rank order)
        kg = [torch.empty_like(kl) for _ in range(world)]
        vg = [torch.empty_like(vl) for _ in range(world)]
        dist.all_gather(kg, kl)
        dist.all_gather(vg, vl)
        kf = torch.cat(kg, dim=1).numpy()
        vf = torch.cat(vg, dim=1).numpy()
        # the per-shard forward and backward (oracle stand-ins for the shard kernels)
        out, lse = O.masked_attention_fwd(ql.numpy(), kf, vf, pos[rows], pos)
        dq, dk_part, dv_part = O.masked_attention_bwd(ql.numpy(), kf, vf, out, lse, dl.numpy(), pos[rows], pos)
        # reduce-scatter of the key/value gradient contributions
        dk = _reduce_scatter(torch.from_numpy(dk_part), world)
        dv = _reduce_scatter(torch.from_numpy(dv_part), world)
        q.put((rank, out, lse, dq, dk.numpy(), dv.numpy()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_exchange_reproduces_unsharded_attention(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    parts = sorted((q.get(timeout=300) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    cp = world
    pos = O.lb_positions(S, cp, True)
    got = [np.concatenate([t[i] for t in parts], axis=2 if i == 2 else 1) for i in range(1, 6)]
    out, lse, dq, dk, dv = (O.unpermute(x, pos) if x.ndim == 4 else x[:, :, np.argsort(pos)] for x in got)
    qn, kn, vn, dn = (synth.to_f64(t) for t in synth.attention_inputs(B, S, HQ, HKV, D, D, seed=3))
    o_ref, l_ref = O.causal_attention_fwd(qn, kn, vn)
    g_ref = O.causal_attention_bwd(qn, kn, vn, o_ref, l_ref, dn)
    np.testing.assert_allclose(out, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, l_ref, rtol=0, atol=1e-12)
    for a, b in zip((dq, dk, dv), g_ref):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)
