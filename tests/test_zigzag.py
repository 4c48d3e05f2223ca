"""Zigzag context-parallel prefill: the partition, its collectives, and its result.

The pairing is pinned to the pages' worked example (tests/golden/zigzag_pairs_8x4.txt).
The partitioned computation must give exactly what the whole problem gives: each query
row's result depends only on its own inputs and its sequence's history, so the fp64
oracle run per chunk-sequence reproduces the whole-problem oracle bit for bit, both
with the ranks run one after the other and as two gloo processes; on a GPU, the fused
CUDA layer run per share, with the results put back in query order, matches the fp64
oracle of the whole problem on every row.
"""
import os
import pathlib

import numpy as np
import pytest
import torch

from sparse_attention_lightning_gb300 import workloads as W
from sparse_attention_lightning_gb300 import zigzag as Z

GOLDEN = pathlib.Path(__file__).parent / "golden" / "zigzag_pairs_8x4.txt"


def _pages_pairs():
    rows = []
    for line in GOLDEN.read_text().splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(tuple(int(x) for x in line.split()))
    return rows


def test_pairing_matches_pages_example():
    rows = _pages_pairs()
    assert len(rows) == 4
    for dev, a, b in rows:
        assert Z.pair_of(dev, 4) == (a, b)
    # and the plan of a sequence of 8 queries puts exactly those chunks on each rank
    plans = Z.plan([8], [8], 4)
    for (dev, a, b), p in zip(rows, plans):
        assert [c for (_, c, _) in p.chunks] == [a, b]
        assert p.q_rows.tolist() == [a, b]


@pytest.mark.parametrize("T,n", [(256, 8), (1000, 6), (7, 8), (0, 4), (13, 1)])
def test_chunk_bounds_cover_exactly(T, n):
    b = Z.chunk_bounds(T, n)
    assert len(b) == n and b[0][0] == 0 and b[-1][1] == T
    sizes = [e - a for a, e in b]
    assert all(b[i][1] == b[i + 1][0] for i in range(n - 1))
    assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)


@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_plan_covers_every_query_once_at_its_position(world):
    q_lens, k_lens = [1000, 37, 5, 64], [1500, 37, 9, 64]
    plans = Z.plan(q_lens, k_lens, world)
    rows = torch.cat([p.q_rows for p in plans]).sort().values
    assert torch.equal(rows, torch.arange(sum(q_lens)))
    # a local row's position (from the local lengths) is its global position
    gpos = []
    for T, L in zip(q_lens, k_lens):
        gpos += [L - T + i for i in range(T)]
    cu_q = np.cumsum([0] + q_lens)
    cu_k = np.cumsum([0] + k_lens)
    for p in plans:
        r = 0
        for (b, c, a), T_c, L_c in zip(p.chunks, p.q_lens, p.k_lens):
            for i in range(T_c):
                assert L_c - T_c + i == gpos[int(p.q_rows[r + i])]
            # its keys are the first L_c keys of its sequence
            kr = p.k_rows[sum(p.k_lens[:p.chunks.index((b, c, a))]):][:L_c]
            assert kr.tolist() == list(range(int(cu_k[b]), int(cu_k[b]) + L_c))
            assert int(p.q_rows[r]) == int(cu_q[b]) + a
            r += T_c


def test_zigzag_balances_causal_work():
    # T divisible by 2P: every rank scores exactly the same number of (query, key) pairs
    for world in (2, 4, 8):
        costs = [p.causal_cost() for p in Z.plan([4096], [4096], world)]
        assert len(set(costs)) == 1, costs
        total = 4096 * 4097 // 2
        assert sum(costs) == total
        # a contiguous split of the same queries is far from balanced
        contiguous = [sum(range(a + 1, e + 1)) for a, e in Z.chunk_bounds(4096, world)]
        assert max(contiguous) / min(contiguous) > 2.0 and max(costs) == min(costs)


# ---- the result of the partitioned computation ---------------------------------------

CFG = W.custom([96, 40], [96, 72], top_k=16)   # prefill and a chunked-prefill sequence


def _oracle_compute(cfg):
    """Local compute for the tests: the fp64 oracle over a chunk-sequence problem."""
    from oracle import dsa_oracle as O

    def run(q_lens, k_lens, t):
        arrays = {k: v.contiguous().numpy() for k, v in t.items()}
        prob = O.Problem(arrays, idx_dtype=cfg.idx_dtype, kv_dtype=cfg.kv_dtype, d_c=cfg.d_c,
                         top_k=cfg.top_k)
        res = prob.forward()
        T = sum(q_lens)
        out = np.zeros((T, cfg.h, cfg.d_c))
        lse = np.zeros((T, cfg.h))
        idx = np.full((T, cfg.top_k), -1, dtype=np.int64)
        for r, v in res.items():
            out[r], lse[r] = v["out"], v["lse"]
            idx[r, : v["idx"].size] = v["idx"]
        return {"out": torch.from_numpy(out), "lse": torch.from_numpy(lse),
                "idx": torch.from_numpy(idx)}

    return run


def _whole(cfg, case):
    t = {k: v for k, v in case.tensors().items()}
    return _oracle_compute(cfg)(cfg.q_lens, cfg.k_lens, t)


def _split(case):
    t = case.tensors()
    query = {k: t[k] for k in Z.QUERY_SIDE if k in t}
    key = {k: t[k] for k in Z.KEY_SIDE if k in t}
    return query, key


@pytest.mark.parametrize("world", [2, 3])
def test_sequential_partition_reproduces_whole_problem(world):
    case = W.make_case(CFG, seed=5)
    whole = _whole(CFG, case)
    query, key = _split(case)
    part = Z.forward_sequential(CFG.q_lens, CFG.k_lens, world, query, key, _oracle_compute(CFG))
    for k in ("out", "lse", "idx"):
        assert torch.equal(part[k], whole[k]), k


def _gloo_worker(rank, world, port, q):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        import torch.distributed as dist
        dist.init_process_group("gloo", rank=rank, world_size=world)
        case = W.make_case(CFG, seed=5)
        query, key = _split(case)
        plans = Z.plan(CFG.q_lens, CFG.k_lens, world)
        mine = Z.select_query_rows(plans[rank], query)
        # this rank's contiguous slice of the key side
        total_k = CFG.total_k
        lo, hi = total_k * rank // world, total_k * (rank + 1) // world
        shard = {k: v[lo:hi] for k, v in key.items()}
        res = Z.forward_distributed(CFG.q_lens, CFG.k_lens, mine, shard, _oracle_compute(CFG))
        whole = _whole(CFG, case)
        ok = all(torch.equal(res[k], whole[k]) for k in ("out", "lse", "idx"))
        dist.destroy_process_group()
        q.put((rank, ok, ""))
    except Exception as e:  # reported to the parent
        q.put((rank, False, repr(e)))


def test_gloo_two_ranks_reproduce_whole_problem():
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_gloo_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ok, err in sorted(results):
        assert ok, f"rank {rank}: {err or 'result differs from the whole problem'}"


# ---- on a GPU: the fused layer per share against the oracle of the whole problem ---------

@pytest.mark.gpu
@pytest.mark.parametrize("cfg,world", [
    (W.custom([300, 120], [300, 500], top_k=32), 2),
    (W.custom([700], [700], h_idx=64, d_idx=128, h=128, d_c=512, d_rope=64, top_k=128,
              idx_dtype="bf16", kv_dtype="bf16"), 2),
    # T not divisible by 2P (chunks of unequal size), a chunked-prefill sequence (T < L)
    (W.custom([701, 97], [701, 2300], h_idx=64, d_idx=128, h=128, d_c=512, d_rope=64,
              top_k=256, idx_dtype="bf16", kv_dtype="bf16"), 3),
    (W.custom([301, 55], [301, 1200], h_idx=64, d_idx=128, h=128, d_c=512, d_rope=64,
              top_k=128, idx_dtype="e4m3", kv_dtype="bf16"), 3),
], ids=["f32-P2", "bf16-P2", "bf16-P3", "e4m3-P3"])
def test_gpu_zigzag_shares_match_oracle(cfg, world):
    """Every rank's share run through the fused CUDA layer, one after the other, the
    results put back in query order, and every row checked against the fp64 oracle of
    the WHOLE problem: the Top-K set (up to the tie band), the attention output and lse."""
    from sparse_attention_lightning_gb300 import build
    import sparse_attention_lightning_gb300 as dsa  # noqa: F401
    from oracle import dsa_oracle as O
    from parity import check_attn_row, check_topk_row, to_np, tol_for
    build.build()
    case = W.make_case(cfg, seed=9)
    d = {k: v.cuda() for k, v in case.tensors().items()}
    compute = Z.fused_forward_compute(h_idx=cfg.h_idx, d_idx=cfg.d_idx, h=cfg.h, d_c=cfg.d_c,
                                      d_rope=cfg.d_rope, top_k=cfg.top_k,
                                      idx_dtype=cfg.idx_dtype, kv_dtype=cfg.kv_dtype,
                                      out_dtype=cfg.out_dtype)
    query = {k: d[k] for k in Z.QUERY_SIDE if k in d}
    key = {k: d[k] for k in Z.KEY_SIDE if k in d}
    part = Z.forward_sequential(cfg.q_lens, cfg.k_lens, world, query, key, compute)
    torch.cuda.synchronize()
    p = O.problem_from_case(case)
    tol = tol_for(cfg)
    idx, out, lse = to_np(part["idx"]), to_np(part["out"]), to_np(part["lse"])
    assert idx.shape[0] == cfg.total_q
    for t in range(cfg.total_q):
        I = p.scores(t)
        ctx = f"{cfg.name} P={world} row {t}"
        check_topk_row(idx[t], I, cfg.top_k, ctx)
        n = min(cfg.top_k, I.shape[0])
        ref_out, ref_lse = p.sfa(t, idx[t, :n])
        check_attn_row(out[t], lse[t], ref_out, ref_lse, tol, ctx)
