"""Zigzag context-parallel prefill.

("Day0 Inference Adaptation and Performance Optimization for New-Architecture LLMs",
§6.2, Zigzag layout; "Day0 Inference Optimization for New Architecture LLMs Based on
CANN", §4.2.)  The indexer's cost for a query grows with its position, so a prefill cut
into contiguous pieces overloads the devices that hold the tail.  The queries of a
sequence are cut into 2P chunks and device d takes chunks d and 2P-1-d: one
short-history and one long-history chunk each (8 chunks on 4 devices: 0+7, 1+6, 2+5,
3+4).  Every device sees the whole key side; after the computation the results are put
back in the original query order.

A chunk becomes a sequence of its own.  If a sequence's T queries are the last T of its
L keys, the chunk holding queries [a, e) sees keys [0, L - T + e): it is a sequence with
T_c = e - a queries and L_c = L - T + e keys, whose position formula
pos = L_c - T_c + i gives back the query's original position.  Its key rows are copied
from the key side, so positions (and with them Top-K indices) need no translation.

The local computation is a callable (``fused_forward_compute`` runs the DSA layer of this
package); the collectives are torch.distributed all-gathers of the key side and of the
outputs, so the same code runs on NCCL (GPU tensors) and gloo (CPU tensors).
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import torch

Compute = Callable[[List[int], List[int], Dict[str, torch.Tensor]], Dict[str, torch.Tensor]]

QUERY_SIDE = ("q_idx", "w", "q", "q_scale")   # one row per query
KEY_SIDE = ("k_idx", "kv", "k_scale")         # one row per key
OUTPUTS = ("out", "lse", "idx")               # one row per query


def chunk_bounds(T: int, n: int) -> List[Tuple[int, int]]:
    """[0, T) cut into n contiguous chunks whose sizes differ by at most one (larger first)."""
    base, extra = divmod(T, n)
    out, a = [], 0
    for c in range(n):
        e = a + base + (1 if c < extra else 0)
        out.append((a, e))
        a = e
    return out


def pair_of(rank: int, world: int) -> Tuple[int, int]:
    """The two chunk indices (of 2 * world) that rank `rank` takes: head d, tail 2P-1-d."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world of {world}")
    return rank, 2 * world - 1 - rank


@dataclasses.dataclass
class RankPlan:
    """One rank's share: its chunk-sequences and where their rows come from."""

    q_lens: List[int]                 # queries of each local chunk-sequence
    k_lens: List[int]                 # keys it sees
    chunks: List[Tuple[int, int, int]]  # (sequence, chunk index, first query in the sequence)
    q_rows: torch.Tensor              # int64 [ΣT_c]: global packed query row of each local row
    k_rows: torch.Tensor              # int64 [ΣL_c]: global packed key row of each local key row

    @property
    def total_q(self) -> int:
        return int(sum(self.q_lens))

    def causal_cost(self) -> int:
        """Indexer work of the share: Σ over its queries of (pos + 1) scored keys."""
        cost = 0
        for T_c, L_c in zip(self.q_lens, self.k_lens):
            first = L_c - T_c + 1                      # pos + 1 of the first query
            cost += T_c * first + T_c * (T_c - 1) // 2
        return cost


def plan(q_lens: Sequence[int], k_lens: Sequence[int], world: int) -> List[RankPlan]:
    """Zigzag shares of a packed varlen problem over `world` ranks (one plan per rank).

    Every sequence is cut on its own into 2 * world chunks; empty chunks (T < 2P) are
    left out.
    """
    if world < 1:
        raise ValueError("world must be >= 1")
    if len(q_lens) != len(k_lens):
        raise ValueError("q_lens and k_lens differ in length")
    cu_q = [0]
    cu_k = [0]
    for T, L in zip(q_lens, k_lens):
        if not 0 <= T <= L:
            raise ValueError(f"a sequence needs 0 <= T <= L (got T={T}, L={L})")
        cu_q.append(cu_q[-1] + int(T))
        cu_k.append(cu_k[-1] + int(L))
    plans = []
    for rank in range(world):
        ql, kl, chunks, qr, kr = [], [], [], [], []
        for b, (T, L) in enumerate(zip(q_lens, k_lens)):
            bounds = chunk_bounds(int(T), 2 * world)
            for c in pair_of(rank, world):
                a, e = bounds[c]
                if e == a:
                    continue
                L_c = int(L) - int(T) + e
                ql.append(e - a)
                kl.append(L_c)
                chunks.append((b, c, a))
                qr.append(torch.arange(cu_q[b] + a, cu_q[b] + e, dtype=torch.int64))
                kr.append(torch.arange(cu_k[b], cu_k[b] + L_c, dtype=torch.int64))
        cat = lambda xs: torch.cat(xs) if xs else torch.zeros(0, dtype=torch.int64)
        plans.append(RankPlan(ql, kl, chunks, cat(qr), cat(kr)))
    return plans


def local_inputs(p: RankPlan, query_side: Dict[str, torch.Tensor],
                 key_side: Dict[str, torch.Tensor]) -> Dict[str, torch.Tensor]:
    """A rank's tensors: its query rows (already local, in plan order) and its chunk-sequences'
    key rows copied out of the full key side, with their cu_q / cu_k."""
    out = {k: v for k, v in query_side.items() if v is not None}
    for k in KEY_SIDE:
        v = key_side.get(k)
        if v is not None:
            out[k] = v.index_select(0, p.k_rows.to(v.device))
    dev = next(iter(out.values())).device
    out["cu_q"] = torch.tensor([0] + list(_cumsum(p.q_lens)), dtype=torch.int32, device=dev)
    out["cu_k"] = torch.tensor([0] + list(_cumsum(p.k_lens)), dtype=torch.int32, device=dev)
    return out


def _cumsum(xs: Sequence[int]):
    s = 0
    for x in xs:
        s += int(x)
        yield s


def select_query_rows(p: RankPlan, query_side: Dict[str, torch.Tensor]) -> Dict[str, torch.Tensor]:
    """The rank's query rows out of global query-side tensors (how a caller that holds the
    whole batch hands a rank its share)."""
    return {k: v.index_select(0, p.q_rows.to(v.device)) for k, v in query_side.items()
            if v is not None and k in QUERY_SIDE}


def restore(plans: List[RankPlan], local_outs: List[Dict[str, torch.Tensor]], total_q: int
            ) -> Dict[str, torch.Tensor]:
    """Global outputs in the original query order from every rank's local outputs."""
    res = {}
    for k in OUTPUTS:
        parts = [o.get(k) for o in local_outs]
        ref = next((t for t in parts if t is not None and t.shape[0] > 0), None)
        if ref is None:
            continue
        g = torch.empty((total_q,) + tuple(ref.shape[1:]), dtype=ref.dtype, device=ref.device)
        for p, t in zip(plans, parts):
            if p.total_q:
                g.index_copy_(0, p.q_rows.to(g.device), t)
        res[k] = g
    return res


def forward_sequential(q_lens: Sequence[int], k_lens: Sequence[int], world: int,
                       query_side: Dict[str, torch.Tensor], key_side: Dict[str, torch.Tensor],
                       compute: Compute) -> Dict[str, torch.Tensor]:
    """All ranks' shares computed one after the other in this process (one device): the
    zigzag result without collectives, for checking the partition against the whole."""
    plans = plan(q_lens, k_lens, world)
    outs = []
    for p in plans:
        if p.total_q == 0:
            outs.append({})
            continue
        t = local_inputs(p, select_query_rows(p, query_side), key_side)
        outs.append(compute(p.q_lens, p.k_lens, t))
    return restore(plans, outs, int(sum(q_lens)))


def _all_gather_rows(x: torch.Tensor, group) -> List[torch.Tensor]:
    """Row-wise all-gather of tensors whose row counts differ between ranks."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    n = torch.tensor([x.shape[0]], dtype=torch.int64, device=x.device)
    ns = [torch.zeros_like(n) for _ in range(world)]
    dist.all_gather(ns, n, group=group)
    ns = [int(v.item()) for v in ns]
    m = max(ns)
    pad = torch.zeros((m,) + tuple(x.shape[1:]), dtype=x.dtype, device=x.device)
    pad[: x.shape[0]] = x
    bufs = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(bufs, pad, group=group)
    return [b[:k] for b, k in zip(bufs, ns)]


def forward_distributed(q_lens: Sequence[int], k_lens: Sequence[int],
                        query_rows: Dict[str, torch.Tensor], key_shard: Dict[str, torch.Tensor],
                        compute: Compute, group=None) -> Dict[str, torch.Tensor]:
    """This rank's zigzag share, with collectives.

    query_rows: this rank's query-side rows, in its plan order (``select_query_rows``).
    key_shard:  this rank's contiguous slice of the packed key side (any split; the slices
                are concatenated in rank order).
    Steps: all-gather the key side; compute the local chunk-sequences; all-gather the
    outputs and put them in the original query order (every rank returns the whole).
    """
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    plans = plan(q_lens, k_lens, world)
    key_side = {k: torch.cat(_all_gather_rows(v, group)) for k, v in key_shard.items()
                if v is not None}
    total_k = int(sum(k_lens))
    for k, v in key_side.items():
        if v.shape[0] != total_k:
            raise ValueError(f"key side {k} has {v.shape[0]} rows after the gather, not {total_k}")
    p = plans[rank]
    local = compute(p.q_lens, p.k_lens, local_inputs(p, query_rows, key_side)) if p.total_q else {}
    # row shape and dtype of every output, from whichever ranks computed one (a rank whose
    # share is empty contributes zero rows)
    meta = {k: (tuple(v.shape[1:]), v.dtype) for k, v in local.items() if k in OUTPUTS}
    metas: List[Optional[dict]] = [None] * world
    dist.all_gather_object(metas, meta, group=group)
    dev = next(iter(key_side.values())).device
    gathered: Dict[str, List[torch.Tensor]] = {}
    for k in OUTPUTS:
        m = next((mm[k] for mm in metas if k in mm), None)
        if m is None:
            continue
        ref = local.get(k)
        if ref is None:
            ref = torch.zeros((0,) + m[0], dtype=m[1], device=dev)
        gathered[k] = _all_gather_rows(ref, group)
    per_rank = [{k: gathered[k][r] for k in gathered} for r in range(world)]
    return restore(plans, per_rank, int(sum(q_lens)))


def fused_forward_compute(*, h_idx: int, d_idx: int, h: int, d_c: int, d_rope: int,
                          top_k: int, idx_dtype, kv_dtype, out_dtype=None,
                          sm_scale: float = 0.0) -> Compute:
    """A `compute` that runs this package's fused DSA layer on the local chunk-sequences."""
    from . import Problem, fused_forward

    def run(q_lens, k_lens, t):
        P = Problem(t["cu_q"], t["cu_k"], q_lens=q_lens, k_lens=k_lens, h_idx=h_idx,
                    d_idx=d_idx, h=h, d_c=d_c, d_rope=d_rope, top_k=top_k, idx_dtype=idx_dtype,
                    kv_dtype=kv_dtype, out_dtype=out_dtype, sm_scale=sm_scale)
        out, lse, idx, _ = fused_forward(P, t["q_idx"], t["k_idx"], t["w"], t["q"], t["kv"],
                                         t.get("q_scale"), t.get("k_scale"))
        return {"out": out, "lse": lse, "idx": idx}

    return run
