"""Expert-parallel form of the MoE layer: the experts are partitioned over ranks, every rank
routes its own tokens, sends each routed row to the rank that owns the row's expert, and gets
the expert outputs back before its combine.

"Who Says Elephants Can't Run", section 3 (model and training notes): the MoE models are
trained with expert parallelism -- whole experts live on different GPUs -- rather than with
experts sliced across GPUs.  The pages give no exchange protocol; this module uses the plainest
one that keeps every step of the single-GPU layer:

  1. dispatch  route (A1) and permute (A2/A3) the rank's tokens; the expert-sorted rows Xp are
               already contiguous per destination rank (experts [e0_q, e1_q) of rank q are
               the segment offsets[e0_q] .. offsets[e1_q]); send each segment to its rank,
               with the per-expert row counts so that the receiver knows which rows are whose.
  2. experts   regroup the received rows by local expert (a stable counting sort with k = 1:
               rows from source 0 first, then source 1, ...), FC1 + activation, FC2 (fp32),
               put the fp32 rows back in received order (an un-permute with gate 1.0, exact),
               and send each source its rows back.
  3. combine   the rank's own combine (A7) of the returned rows, with its gates, its inverse
               permutation and the shared expert (replicated on every rank).

Each phase is a function of one rank's state, so a caller can run the ranks as processes with
torch.distributed all-to-all exchanges (`ep_forward`), or as a loop in one process with the
exchange done by list transposition (`ep_forward_local`, what the single-GPU tests use).  The
arithmetic of each phase goes through an `ops` object (route, permute, experts, unpermute,
shared, combine, and `row_dtype`, the dtype of the expert rows sent back): `CudaOps` calls
libmoe's kernels (the product path, no fallback); tests pass the float64 oracle's steps instead
to check the exchange logic on CPU.

Numerics: for the same tokens, rank r's rows for expert e arrive in the order of the
single-GPU layer (tokens of rank 0 first, the layer's stable sort keeps token order), FC2
leaves fp32 rows and the way back is exact, so the combine sees what the single-GPU combine
sees.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np
import torch


def expert_ranges(E: int, world: int) -> List[tuple]:
    """[e0, e1) of every rank: contiguous blocks, the first E % world ranks one expert larger."""
    base, extra = divmod(E, world)
    out, e0 = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((e0, e0 + n))
        e0 += n
    return out


@dataclasses.dataclass
class Shard:
    """One rank's part of a layer: the full router, its experts' weights, the shared expert."""
    cfg: object
    rank: int
    world: int
    e0: int
    e1: int
    weights: object          # ops-specific handle to [e0, e1) experts' FC1 / FC2 weights + router + shared

    @property
    def E_local(self) -> int:
        return self.e1 - self.e0


@dataclasses.dataclass
class DispatchState:
    """What a rank keeps from dispatch to combine."""
    x: torch.Tensor
    gate: torch.Tensor
    inv_perm: torch.Tensor
    send_rows: List[int]            # rows sent to each rank (its segment of Xp)
    send_counts: np.ndarray         # (world, E_max) rows per (destination, local expert)


@dataclasses.dataclass
class ExpertState:
    recv_rows: List[int]            # rows received from each source


def _counts_matrix(offsets: np.ndarray, ranges: Sequence[tuple], E_max: int) -> np.ndarray:
    per_e = np.diff(offsets.astype(np.int64))
    m = np.zeros((len(ranges), E_max), dtype=np.int64)
    for q, (a, b) in enumerate(ranges):
        m[q, :b - a] = per_e[a:b]
    return m


def phase_dispatch(shard: Shard, x: torch.Tensor, ops):
    """Route and permute this rank's tokens.  Returns (state, xp, send_counts (world, E_max))."""
    cfg = shard.cfg
    assert x.shape[0] > 0, "a rank routes at least one token"
    ids, gate = ops.route(shard, x)
    offsets, perm, inv_perm, xp = ops.permute(shard, ids, x, cfg.E, cfg.k)
    ranges = expert_ranges(cfg.E, shard.world)
    E_max = max(b - a for a, b in ranges)
    off = offsets.cpu().numpy()                  # split sizes must be known on the host
    counts = _counts_matrix(off, ranges, E_max)
    send_rows = [int(c.sum()) for c in counts]
    return DispatchState(x, gate, inv_perm, send_rows, counts), xp, counts


def phase_experts(shard: Shard, recv_xp: torch.Tensor, recv_counts: np.ndarray, ops):
    """recv_xp: rows from every source, source-major, each source's rows sorted by local expert;
    recv_counts (world, E_max): rows per (source, local expert).  Returns (state, fp32 rows in
    received order)."""
    El = shard.E_local
    cnt = recv_counts[:, :El]
    recv_rows = [int(c.sum()) for c in cnt]
    R = int(cnt.sum())
    d = shard.cfg.d
    if R == 0:
        return ExpertState(recv_rows), torch.empty((0, d), dtype=ops.row_dtype, device=recv_xp.device)
    # local expert id of every received row (counts are on the host already)
    ids_l = np.concatenate([np.repeat(np.arange(El, dtype=np.int32), c) for c in cnt])
    ids_l = torch.from_numpy(ids_l).to(recv_xp.device).view(R, 1)
    offsets_l, _, inv_l, xl = ops.permute(shard, ids_l, recv_xp, El, 1)
    y = ops.experts(shard, xl, offsets_l)                     # (R, d) fp32, local-expert order
    back = ops.unpermute(shard, y, inv_l)                     # (R, d) fp32, received order
    return ExpertState(recv_rows), back


def phase_combine(shard: Shard, st: DispatchState, yp: torch.Tensor, ops) -> torch.Tensor:
    """yp: this rank's rows back in its own expert-sorted order (fp32)."""
    shared = ops.shared(shard, st.x)
    return ops.combine(shard, yp, st.inv_perm, st.gate, shared)


# ---------------------------------------------------------------- drivers


def _split(t: torch.Tensor, sizes: Sequence[int]) -> List[torch.Tensor]:
    return list(torch.split(t, list(sizes), dim=0))


def ep_forward_local(shards: Sequence[Shard], xs: Sequence[torch.Tensor], ops) -> List[torch.Tensor]:
    """Every rank in one process (the exchanges are list transpositions).  xs[r] = rank r's
    tokens; returns every rank's output."""
    W = len(shards)
    disp = [phase_dispatch(shards[r], xs[r], ops) for r in range(W)]
    # exchange 1: segment q of rank r's Xp goes to rank q
    seg = [_split(xp, st.send_rows) for st, xp, _ in disp]
    recv = [torch.cat([seg[s][q] for s in range(W)], 0) for q in range(W)]
    recv_counts = [np.stack([disp[s][2][q] for s in range(W)]) for q in range(W)]
    exp = [phase_experts(shards[q], recv[q], recv_counts[q], ops) for q in range(W)]
    # exchange 2: rank q's rows from source s go back to s
    back = [_split(y, est.recv_rows) for est, y in exp]
    outs = []
    for r in range(W):
        yp = torch.cat([back[q][r] for q in range(W)], 0)
        outs.append(phase_combine(shards[r], disp[r][0], yp, ops))
    return outs


def ep_forward(shard: Shard, x: torch.Tensor, ops, group=None) -> torch.Tensor:
    """One rank of a torch.distributed job (any backend with all_to_all_single: NCCL on GPUs,
    gloo on CPU).  Collective calls: one all-to-all of the per-expert counts, one of the rows
    out, one of the rows back."""
    import torch.distributed as dist
    W = shard.world
    st, xp, counts = phase_dispatch(shard, x, ops)
    E_max = counts.shape[1]
    dev = xp.device
    # counts: rank r sends row q of its matrix to rank q
    c_send = torch.from_numpy(counts.reshape(-1).astype(np.int64)).to(dev)
    c_recv = torch.empty_like(c_send)
    dist.all_to_all_single(c_recv, c_send, group=group)
    recv_counts = c_recv.cpu().numpy().reshape(W, E_max)
    recv_rows = [int(c.sum()) for c in recv_counts]
    recv_xp = torch.empty((sum(recv_rows), x.shape[1]), dtype=xp.dtype, device=dev)
    dist.all_to_all_single(recv_xp, xp.contiguous(), recv_rows, st.send_rows, group=group)
    est, y = phase_experts(shard, recv_xp, recv_counts, ops)
    yp = torch.empty((xp.shape[0], x.shape[1]), dtype=ops.row_dtype, device=dev)
    dist.all_to_all_single(yp, y.contiguous(), st.send_rows, est.recv_rows, group=group)
    return phase_combine(shard, st, yp, ops)


# ---------------------------------------------------------------- libmoe steps


@dataclasses.dataclass
class CudaShardWeights:
    wr: torch.Tensor
    bias: Optional[torch.Tensor]
    w1: Optional[torch.Tensor]       # packed FC1 of experts [e0, e1) (None when the rank owns none)
    w2: Optional[torch.Tensor]
    ws_gu: Optional[torch.Tensor]
    ws_d: Optional[torch.Tensor]


def cuda_shard(cfg, w, rank: int, world: int, device) -> Shard:
    """Pack rank `rank`'s experts of synthetic/host weights `w` (q1, s1, q2, s2 over all E)
    onto `device`; router and shared expert are replicated."""
    from . import moe as M
    dev = torch.device(device)
    e0, e1 = expert_ranges(cfg.E, world)[rank]
    w1 = w2 = None
    if e1 > e0:
        w1 = M.pack_weights(w.q1[e0:e1].to(dev), w.s1[e0:e1].to(dev), cfg.bits, cfg.group)
        w2 = M.pack_weights(w.q2[e0:e1].to(dev), w.s2[e0:e1].to(dev), cfg.bits, cfg.group)
    gu = dn = None
    if cfg.Fs:
        gu = M.pack_weights(w.ws_gu.to(dev)[None], None, 16, 0)
        dn = M.pack_weights(w.ws_d.to(dev)[None], None, 16, 0)
    bias = None if w.bias is None else w.bias.to(dev)
    sw = CudaShardWeights(w.wr.to(dev).contiguous(), bias, w1, w2, gu, dn)
    return Shard(cfg, rank, world, e0, e1, sw)


class CudaOps:
    """The phases' steps on libmoe's kernels (moe_route_topk, moe_permute, the grouped GEMMs,
    moe_unpermute_combine, moe_shared_expert)."""

    row_dtype = torch.float32   # expert output rows (FC2 accumulates and stores fp32)

    def route(self, shard, x):
        from . import moe as M
        return M.route_topk(x, shard.weights.wr, shard.weights.bias, shard.cfg.k)

    def permute(self, shard, ids, x, E, k):
        from . import moe as M
        return M.permute(ids, x, E)

    def experts(self, shard, xl, offsets_l):
        from . import moe as M
        cfg, sw = shard.cfg, shard.weights
        El = shard.E_local
        h = M.grouped_gemm(xl, sw.w1, cfg.bits, El, cfg.d, cfg.F1, cfg.group, offsets_l, cfg.act, cfg.torch_dtype)
        return M.grouped_gemm(h, sw.w2, cfg.bits, El, cfg.F, cfg.d, cfg.group, offsets_l, "none", torch.float32)

    def unpermute(self, shard, y, inv_l):
        from . import moe as M
        R = y.shape[0]
        ones = torch.ones((R, 1), dtype=torch.float32, device=y.device)
        return M.unpermute_combine(y, inv_l, ones, None, torch.float32)

    def shared(self, shard, x):
        from . import moe as M
        sw = shard.weights
        if sw.ws_gu is None:
            return None
        return M.shared_expert(x, sw.ws_gu, sw.ws_d, shard.cfg.Fs, torch.float32)

    def combine(self, shard, yp, inv_perm, gate, shared):
        from . import moe as M
        return M.unpermute_combine(yp, inv_perm, gate, shared, shard.cfg.torch_dtype)
