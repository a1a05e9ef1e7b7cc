"""Expert-parallel layer (experts partitioned over ranks, rows sent to the owning rank and back)
on CPU: the exchange logic of weight_only_int4_route_gb300.ep with the float64 oracle's steps
for the arithmetic, as gloo ranks (world size 2 and 3) and as ranks in one process, against the
single-rank oracle layer over all tokens."""
import dataclasses
import os
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import moe_oracle as O                      # noqa: E402
from weight_only_int4_route_gb300 import ep, synth     # noqa: E402


class OracleOps:
    """The phases' steps in float64 (oracle functions); rows travel as float64."""

    row_dtype = torch.float64

    def route(self, shard, x):
        w = shard.weights
        _, ids, gate = O.route(x, w.wr, w.bias, shard.cfg.k)
        return ids.to(torch.int32), gate

    def permute(self, shard, ids, x, E, k):
        _, offsets, perm, inv_perm = O.sort_by_expert(ids, E)
        return offsets, perm, inv_perm, O.permute_rows(x.to(torch.float64), perm, k)

    def experts(self, shard, xl, offsets_l):
        cfg, w = shard.cfg, shard.weights
        y = torch.zeros(xl.shape[0], cfg.d, dtype=torch.float64)
        for el in range(shard.E_local):
            lo, hi = int(offsets_l[el]), int(offsets_l[el + 1])
            if lo == hi:
                continue
            e = shard.e0 + el
            w1 = O.dequant(w.q1[e:e + 1], w.s1[e:e + 1], cfg.group)[0]
            w2 = O.dequant(w.q2[e:e + 1], w.s2[e:e + 1], cfg.group)[0]
            y[lo:hi] = O.expert_ffn(xl[lo:hi], w1, w2, cfg.act)
        return y

    def unpermute(self, shard, y, inv_l):
        return y[inv_l.long()]

    def shared(self, shard, x):
        w = shard.weights
        return None if w.ws_gu is None else O.shared_expert(x, w.ws_gu, w.ws_d)

    def combine(self, shard, yp, inv_perm, gate, shared):
        T, k = gate.shape
        out = torch.zeros(T, shard.cfg.d, dtype=torch.float64)
        for j in range(k):
            out += gate[:, j].to(torch.float64).unsqueeze(1) * yp[inv_perm[torch.arange(T) * k + j].long()]
        return out if shared is None else out + shared


def _case(name):
    if name == "tiny":
        return synth.CONFIGS["tiny"], 16, None
    if name == "shared_g128":      # group-128 scales, SwiGLU, a shared expert, E not divisible by world
        return synth.custom("qwen", d=256, F=128, E=7, k=2, Fs=128), 12, None
    if name == "skewed":           # every token picks experts 0 and 1: only rank 0 receives rows
        cfg = synth.CONFIGS["tiny"]
        bias = torch.zeros(cfg.E)
        bias[0], bias[1] = 60.0, 50.0
        return cfg, 10, bias
    raise KeyError(name)


def _inputs(name):
    cfg, T, bias = _case(name)
    w = synth.layer_weights(cfg, 0)
    if bias is not None:
        w = dataclasses.replace(w, bias=bias)
    return cfg, w, synth.activations(cfg, T)


def _token_split(T, world):
    base, extra = divmod(T, world)
    cuts = [0]
    for r in range(world):
        cuts.append(cuts[-1] + base + (1 if r < extra else 0))
    return cuts


def _shard(cfg, w, rank, world):
    e0, e1 = ep.expert_ranges(cfg.E, world)[rank]
    return ep.Shard(cfg, rank, world, e0, e1, w)


def test_expert_ranges_cover_every_expert():
    for E in (1, 5, 8, 60, 64):
        for W in (1, 2, 3, 8):
            rs = ep.expert_ranges(E, W)
            assert len(rs) == W and rs[0][0] == 0 and rs[-1][1] == E
            assert all(a <= b for a, b in rs) and all(rs[i][1] == rs[i + 1][0] for i in range(W - 1))
            sizes = [b - a for a, b in rs]
            assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("name", ["tiny", "shared_g128", "skewed"])
@pytest.mark.parametrize("world", [2, 3])
def test_ranks_in_one_process_match_the_oracle(name, world):
    cfg, w, x = _inputs(name)
    ref = O.moe_layer(x, w, cfg)["out"]
    cuts = _token_split(x.shape[0], world)
    shards = [_shard(cfg, w, r, world) for r in range(world)]
    outs = ep.ep_forward_local(shards, [x[cuts[r]:cuts[r + 1]] for r in range(world)], OracleOps())
    got = torch.cat(outs, 0)
    assert got.shape == ref.shape
    assert torch.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_skewed_routing_sends_every_row_to_rank_0():
    cfg, w, x = _inputs("skewed")
    shards = [_shard(cfg, w, r, 2) for r in range(2)]
    st, xp, counts = ep.phase_dispatch(shards[1], x[5:], OracleOps())
    assert st.send_rows == [xp.shape[0], 0] and counts[1].sum() == 0


class _NoReturnOrder(OracleOps):
    """Planted mistake: the expert rows are sent back in local-expert order, not received order."""

    def unpermute(self, shard, y, inv_l):
        return y


def test_planted_return_order_mistake_is_caught():
    cfg, w, x = _inputs("tiny")
    ref = O.moe_layer(x, w, cfg)["out"]
    shards = [_shard(cfg, w, r, 2) for r in range(2)]
    outs = ep.ep_forward_local(shards, [x[:8], x[8:]], _NoReturnOrder())
    assert not torch.allclose(torch.cat(outs, 0), ref, rtol=1e-6, atol=1e-6)


def _gloo_worker(rank, world, port, name, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg, w, x = _inputs(name)
        cuts = _token_split(x.shape[0], world)
        y = ep.ep_forward(_shard(cfg, w, rank, world), x[cuts[rank]:cuts[rank + 1]], OracleOps())
        out[rank] = y.numpy()
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,world,port", [("tiny", 2, 29541), ("shared_g128", 2, 29542), ("skewed", 2, 29543),
                                             ("tiny", 3, 29544)])
def test_gloo_ranks_match_the_oracle(name, world, port):
    out = mp.Manager().dict()
    mp.spawn(_gloo_worker, args=(world, port, name, out), nprocs=world, join=True)
    cfg, w, x = _inputs(name)
    ref = O.moe_layer(x, w, cfg)["out"]
    got = torch.cat([torch.from_numpy(out[r]) for r in range(world)], 0)
    assert torch.allclose(got, ref, rtol=1e-12, atol=1e-12)
