"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on a GPU."""
import numpy as np
import pytest
import torch

import sparse_attention_lightning_gb300 as dsa
from sparse_attention_lightning_gb300 import workloads as W
from oracle import dsa_oracle as O
from parity import check_attn_row, check_scores_row, check_topk_row, to_np, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_lightning_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def to_dev(case):
    return {k: v.cuda() for k, v in case.tensors().items()}


def problem(case, d):
    return dsa.Problem.from_config(case.cfg, d["cu_q"], d["cu_k"])


def run_fused(case, d=None, ws=None):
    d = d or to_dev(case)
    P = problem(case, d)
    out, lse, idx, vals = dsa.fused_forward(P, d["q_idx"], d["k_idx"], d["w"], d["q"], d["kv"],
                                            d.get("q_scale"), d.get("k_scale"), want_vals=True,
                                            ws=ws)
    torch.cuda.synchronize()
    return P, out, lse, idx, vals


def check_rows(case, idx, vals, out, lse, rows):
    """Top-K, selected scores and attention of `rows` against the oracle."""
    p = O.problem_from_case(case)
    tol = tol_for(case.cfg)
    idx_n, vals_n, out_n, lse_n = to_np(idx), to_np(vals), to_np(out), to_np(lse)
    swaps = 0
    for t in rows:
        I = p.scores(t)
        ctx = f"{case.cfg.name} row {t}"
        swaps += check_topk_row(idx_n[t], I, case.cfg.top_k, ctx)["swaps"]
        n = min(case.cfg.top_k, I.shape[0])
        sel = idx_n[t, :n]
        m = np.abs(I).max()
        assert np.abs(vals_n[t, :n] - I[sel]).max() <= 1e-2 * m + 1e-30, ctx + ": vals"
        assert np.all(np.isneginf(vals_n[t, n:]))
        ref_out, ref_lse = p.sfa(t, sel)
        check_attn_row(out_n[t], lse_n[t], ref_out, ref_lse, tol, ctx)
        # end to end: against the oracle's attention over its own Top-K set (positions
        # swapped inside the tie band change the output by far less than the tolerance)
        own = np.argsort(-I, kind="stable")[:n]
        if not np.array_equal(np.sort(own), np.sort(sel)):
            e2e_out, e2e_lse = p.sfa(t, own)
            check_attn_row(out_n[t], lse_n[t], e2e_out, e2e_lse, tol, ctx + " (oracle's set)")
    return swaps


def test_tiny_prefill_fp32_all_rows():
    case = W.make_case(W.tiny_prefill(), W.WORKLOAD_SEEDS["tiny_prefill"])
    P, out, lse, idx, vals = run_fused(case)
    check_rows(case, idx, vals, out, lse, range(case.cfg.total_q))


SMALL = [
    # (q_lens, k_lens, dims, dtypes) — ragged tails, L < k, L = 1, T = L and T < L
    ([1, 7, 40, 1], [1, 300, 40, 2049], dict(top_k=32), ("f32", "f32")),
    ([3, 1, 130], [3, 77, 130], dict(top_k=64), ("bf16", "bf16")),
    ([1, 2, 1], [5000, 133, 2100], dict(h_idx=64, d_idx=128, h=128, d_c=512, d_rope=64,
                                        top_k=2048), ("bf16", "bf16")),
    ([1, 1, 4], [4100, 3000, 300], dict(h_idx=64, d_idx=128, h=128, d_c=512, d_rope=64,
                                        top_k=2048), ("e4m3", "bf16")),
    ([2, 1], [9, 65], dict(h_idx=3, d_idx=48, h=5, d_c=32, d_rope=16, top_k=5), ("e4m3", "f32")),
    # several query rows per sequence: the indexer scores blocks of four rows at once
    # (partial last blocks, chunked prefill T < L, a block straddling a 128-key tile edge)
    ([37, 1, 130, 6], [300, 2500, 1300, 6], dict(h_idx=64, d_idx=128, h=128, d_c=512,
                                                 d_rope=64, top_k=256), ("bf16", "bf16")),
    ([37, 1, 130, 6], [300, 2500, 1300, 6], dict(h_idx=64, d_idx=128, h=128, d_c=512,
                                                 d_rope=64, top_k=256), ("e4m3", "bf16")),
]


@pytest.mark.parametrize("qs,ks,dims,dts", SMALL)
def test_small_cases(qs, ks, dims, dts):
    cfg = W.custom(qs, ks, idx_dtype=dts[0], kv_dtype=dts[1], **dims)
    case = W.make_case(cfg, seed=123)
    P, out, lse, idx, vals = run_fused(case)
    check_rows(case, idx, vals, out, lse, range(cfg.total_q))


def test_materialised_scores_and_standalone_topk():
    cfg = W.custom([1, 5, 33], [700, 5, 100], h_idx=8, d_idx=64, idx_dtype="bf16",
                   kv_dtype="bf16", top_k=16)
    case = W.make_case(cfg, seed=7)
    d = to_dev(case)
    P = problem(case, d)
    s = dsa.indexer_scores(P, d["q_idx"], d["k_idx"], d["w"])
    idx, vals = dsa.topk(P, s, want_vals=True)
    torch.cuda.synchronize()
    p = O.problem_from_case(case)
    sn, idn = to_np(s), to_np(idx)
    for t in range(cfg.total_q):
        I = p.scores(t)
        check_scores_row(sn[t], I, f"row {t}")
        check_topk_row(idn[t], I, cfg.top_k, f"row {t}")


@pytest.mark.parametrize("idx_dtype", ["bf16", "e4m3"])
def test_tensor_core_indexer_scores(idx_dtype):
    # H_I = 64, d_I = 128 runs on tcgen05; rows cover decode (T=1), T<L and prefill,
    # tails that are not multiples of the 128-key tile, and a 1-key history.
    cfg = W.custom([1, 3, 130, 1], [1000, 300, 130, 1], h_idx=64, d_idx=128, h=8, d_c=64,
                   d_rope=16, top_k=64, idx_dtype=idx_dtype, kv_dtype="bf16")
    case = W.make_case(cfg, seed=17)
    d = to_dev(case)
    P = problem(case, d)
    s = dsa.indexer_scores(P, d["q_idx"], d["k_idx"], d["w"], d.get("q_scale"), d.get("k_scale"))
    idx, _ = dsa.topk(P, s)
    torch.cuda.synchronize()
    p = O.problem_from_case(case)
    sn, idn = to_np(s), to_np(idx)
    worst = 0.0
    for t in range(cfg.total_q):
        I = p.scores(t)
        worst = max(worst, check_scores_row(sn[t], I, f"row {t}"))
        check_topk_row(idn[t], I, cfg.top_k, f"row {t}")
    assert worst < 1e-4, worst  # fp32 accumulation of exact products: far inside 1e-2


@pytest.mark.parametrize("all_equal", [False, True], ids=["random", "all_scores_equal"])
def test_many_row_topk(all_equal):
    # more than 4096 query rows: the Top-K streams each row in its own CTA.  With q_I = 0
    # every score is 0, every key is a candidate (more than the kernel keeps in shared
    # memory) and the tie rule alone decides: positions 0 .. k-1.
    cfg = W.custom([4200], [4200], h_idx=64, d_idx=128, h=8, d_c=64, d_rope=16, top_k=256,
                   idx_dtype="bf16", kv_dtype="bf16")
    case = W.make_case(cfg, seed=41)
    if all_equal:
        case.q_idx.zero_()
    P, out, lse, idx, vals = run_fused(case)
    rng = np.random.default_rng(3)
    rows = sorted(set([0, 255, 256, 257, 4096, 4198, 4199] + rng.integers(0, 4200, 12).tolist()))
    check_rows(case, idx, vals, out, lse, rows)
    if all_equal:
        idn = to_np(idx)
        for t in rows:
            n = min(cfg.top_k, t + 1)
            assert np.array_equal(np.sort(idn[t, :n]), np.arange(n)), t


def test_topk_ties_match_oracle_exactly():
    # integer-valued scores with many ties: the tie rule (smaller position) fixes the set
    cfg = W.custom([3], [3000], top_k=100)
    case = W.make_case(cfg, seed=1)
    d = to_dev(case)
    P = problem(case, d)
    g = torch.Generator().manual_seed(3)
    scores = torch.randint(0, 6, (3, 3000), generator=g).to(torch.float32)
    idx, vals = dsa.topk(P, scores.cuda(), want_vals=True)
    torch.cuda.synchronize()
    for t in range(3):
        pos = 3000 - 3 + t
        ref = np.sort(O.topk_row(scores[t, :pos + 1].double().numpy(), 100))
        assert np.array_equal(to_np(idx)[t], ref)


def test_sfa_flags_bad_indices_and_skips_them():
    cfg = W.custom([2], [50], top_k=8, kv_dtype="bf16")
    case = W.make_case(cfg, seed=5)
    d = to_dev(case)
    P = problem(case, d)
    idx = torch.tensor([[3, -1, 49, 7, 60, 2, -1, 0],        # 49 > pos 48, 60 out of range
                        [-1, -1, -1, -1, -1, -1, -1, -1]], dtype=torch.int32).cuda()
    ws = dsa.Workspace()
    ws.clear_status()
    out, lse = dsa.sparse_mla_attn(P, d["q"], d["kv"], idx, ws=ws)
    flags = ws.status()
    assert flags & 0x1, "DSA_FLAG_BAD_INDEX not set"
    p = O.problem_from_case(case)
    ref_out, ref_lse = p.sfa(0, [3, 7, 2, 0])
    check_attn_row(to_np(out)[0], to_np(lse)[0], ref_out, ref_lse, tol_for(cfg))
    assert np.all(to_np(out)[1] == 0) and np.all(np.isneginf(to_np(lse)[1]))
    ws.clear_status()
    assert ws.status() == 0


@pytest.mark.parametrize("nq,out_dtype", [(3, "bf16"), (90, "bf16"), (5, "f32"), (310, "bf16")])
def test_tensor_core_sfa_standalone(nq, out_dtype):
    # H = 128, d_c = 512, d_rope = 64 runs on tcgen05 CTA pairs.  Few queries (fewer than
    # four per cluster) cut rows into pieces on equal shares of chunk slots, merged by the
    # row's last piece (3 rows: up to ~25 pieces a row, many of them empty); 310 rows run
    # whole rows.  Index rows mix valid positions, -1 padding anywhere, out-of-range
    # entries and a repeated entry.
    L = 3000
    cfg = W.custom([nq], [L], h_idx=4, d_idx=32, h=128, d_c=512, d_rope=64, top_k=2048,
                   idx_dtype="bf16", kv_dtype="bf16", out_dtype=out_dtype)
    case = W.make_case(cfg, seed=41)
    d = to_dev(case)
    P = problem(case, d)
    g = torch.Generator().manual_seed(nq)
    idx = torch.full((nq, 2048), -1, dtype=torch.int32)
    counts = []
    for t in range(nq):
        pos = L - nq + t
        n = [2048, 1, 65, 700, 2047][t % 5]
        sel = torch.randperm(pos + 1, generator=g)[:n].to(torch.int32)
        slots = torch.randperm(2048, generator=g)[:sel.numel()]
        idx[t, slots] = sel
        counts.append(sel.numel())
    idx[0, 5] = idx[0, 6]                # a repeated entry counts twice
    idx[1, 7] = L + 5                    # out of range: flagged and skipped
    ws = dsa.Workspace()
    ws.clear_status()
    out, lse = dsa.sparse_mla_attn(P, d["q"], d["kv"], idx.cuda(), ws=ws)
    flags = ws.status()
    assert flags == 0x1, hex(flags)
    p = O.problem_from_case(case)
    idn = idx.numpy()
    for t in range(nq):
        pos = L - nq + t
        row = idn[t]
        valid = row[(row >= 0) & (row <= pos)]
        ref_out, ref_lse = p.sfa(t, valid)
        check_attn_row(to_np(out)[t], to_np(lse)[t], ref_out, ref_lse, tol_for(cfg), f"row {t}")


@pytest.mark.parametrize("nq,top_k", [(3, 1984), (41, 1984)])
def test_tensor_core_sfa_rows_in_many_pieces(nq, top_k):
    # top_k = 1984 gives 31 chunk slots a row (odd): the rows' slots are cut into 76 equal
    # shares, so 3 rows spread over ~25 clusters each (pieces of 1-2 chunks, most of them
    # holding only -1 padding) and 41 rows into pieces of ~16 chunks; the merge kernel
    # combines every piece of a row.  Valid entries sit anywhere in the row.
    L = 2600
    cfg = W.custom([nq], [L], h_idx=4, d_idx=32, h=128, d_c=512, d_rope=64, top_k=top_k,
                   idx_dtype="bf16", kv_dtype="bf16", out_dtype="bf16")
    case = W.make_case(cfg, seed=43)
    d = to_dev(case)
    P = problem(case, d)
    g = torch.Generator().manual_seed(100 + nq)
    idx = torch.full((nq, top_k), -1, dtype=torch.int32)
    for t in range(nq):
        pos = L - nq + t
        n = [top_k, 1, 200, 1500][t % 4]
        sel = torch.randperm(pos + 1, generator=g)[:n].to(torch.int32)
        slots = torch.randperm(top_k, generator=g)[:sel.numel()]
        idx[t, slots] = sel
    ws = dsa.Workspace()
    ws.clear_status()
    out, lse = dsa.sparse_mla_attn(P, d["q"], d["kv"], idx.cuda(), ws=ws)
    assert ws.status() == 0
    out2, lse2 = dsa.sparse_mla_attn(P, d["q"], d["kv"], idx.cuda(), ws=ws)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), "merge not deterministic"
    p = O.problem_from_case(case)
    idn = idx.numpy()
    for t in range(nq):
        row = idn[t]
        valid = row[row >= 0]
        ref_out, ref_lse = p.sfa(t, valid)
        check_attn_row(to_np(out)[t], to_np(lse)[t], ref_out, ref_lse, tol_for(cfg), f"row {t}")


def test_repeat_runs_are_bitwise_identical():
    cfg = W.custom([1, 1], [3000, 2500], h_idx=64, d_idx=128, h=128, d_c=512, d_rope=64,
                   top_k=2048, idx_dtype="bf16", kv_dtype="bf16")
    case = W.make_case(cfg, seed=9)
    d = to_dev(case)
    r1 = run_fused(case, d)
    r2 = run_fused(case, d)
    assert torch.equal(r1[3], r2[3])
    assert torch.equal(r1[1].view(torch.int16), r2[1].view(torch.int16))


def test_decode_workload_full_size():
    """The bench's decode workload (B=32, L ~ U[8192, 32768], bf16), every row checked."""
    cfg = W.workload("decode")
    case = W.make_case(cfg, W.WORKLOAD_SEEDS["decode"])
    P, out, lse, idx, vals = run_fused(case)
    check_rows(case, idx, vals, out, lse, range(cfg.total_q))


def _sample_rows(T, k, n_random=24, seed=0):
    fixed = {0, 1, k - 2, k - 1, k, T // 2, T - 2, T - 1}
    rng = np.random.default_rng(seed)
    return sorted(fixed | set(rng.integers(0, T, n_random).tolist()))


@pytest.mark.parametrize("name", ["prefill_8k", pytest.param("prefill_64k", marks=pytest.mark.slow)])
def test_prefill_workloads_sampled_rows(name):
    cfg = W.workload(name)
    case = W.make_case(cfg, W.WORKLOAD_SEEDS[name])
    P, out, lse, idx, vals = run_fused(case)
    check_rows(case, idx, vals, out, lse, _sample_rows(cfg.total_q, cfg.top_k))


@pytest.mark.slow
def test_fp8_decode_workload_sampled_sequences():
    cfg = W.workload("fp8_decode")
    case = W.make_case(cfg, W.WORKLOAD_SEEDS["fp8_decode"])
    P, out, lse, idx, vals = run_fused(case)
    rows = sorted(set(np.random.default_rng(4).integers(0, cfg.total_q, 14).tolist()) | {0, 127})
    check_rows(case, idx, vals, out, lse, rows)


def test_fp8_decode_workload_first_sequences():
    """The FP8-indexer decode workload's shapes (L = 131072, H_I = 64, d_I = 128, E4M3 with
    per-token scales, bf16 latent), its first 16 sequences, every row checked."""
    import dataclasses
    cfg = W.workload("fp8_decode")
    cfg = dataclasses.replace(cfg, name=cfg.name + "_first16", q_lens=list(cfg.q_lens[:16]),
                              k_lens=list(cfg.k_lens[:16]))
    case = W.make_case(cfg, W.WORKLOAD_SEEDS["fp8_decode"])
    P, out, lse, idx, vals = run_fused(case)
    check_rows(case, idx, vals, out, lse, range(cfg.total_q))


BIG = dict(h_idx=64, d_idx=128, h=128, d_c=512, d_rope=64, top_k=2048)
PAGED = [
    # decode rows (the one-kernel fused indexer) with pages smaller than, equal to and
    # larger than the 128-key tile
    ([1, 1, 1], [3000, 700, 5000], BIG, ("bf16", "bf16"), 64),
    ([1, 1, 1], [3000, 700, 5000], BIG, ("bf16", "bf16"), 16),
    ([1, 1, 1], [3000, 700, 5000], BIG, ("e4m3", "bf16"), 256),
    # several queries per sequence: the persistent indexer on blocks of four rows, row
    # chunks selected by the streaming Top-K
    ([37, 1, 130, 6], [300, 2500, 1300, 6], dict(BIG, top_k=256), ("bf16", "bf16"), 128),
    ([37, 1, 130, 6], [300, 2500, 1300, 6], dict(BIG, top_k=256), ("e4m3", "bf16"), 32),
    # the CUDA-core paths (fp32, small heads)
    ([1, 7, 40, 1], [1, 300, 40, 2049], dict(top_k=32), ("f32", "f32"), 16),
]


@pytest.mark.parametrize("qs,ks,dims,dts,page_size", PAGED)
def test_paged_caches_match_oracle(qs, ks, dims, dts, page_size):
    """The key side scattered over pages in a random order (unused rows hold large values),
    read through the block table; every row checked against the oracle of the packed case."""
    cfg = W.custom(qs, ks, idx_dtype=dts[0], kv_dtype=dts[1], **dims)
    case = W.make_case(cfg, seed=11)
    pk = W.paged_keys(case, page_size, seed=12)
    d = to_dev(case)
    d.update({k: v.cuda() for k, v in pk.tensors().items()})
    P = dsa.Problem.from_config(cfg, d["cu_q"], d["cu_k"], block_table=d["block_table"],
                                page_size=page_size, num_pages=pk.num_pages)
    ws = dsa.Workspace()
    ws.clear_status()
    out, lse, idx, vals = dsa.fused_forward(P, d["q_idx"], d["k_idx"], d["w"], d["q"], d["kv"],
                                            d.get("q_scale"), d.get("k_scale"), want_vals=True,
                                            ws=ws)
    assert ws.status() == 0
    check_rows(case, idx, vals, out, lse, range(cfg.total_q))
    if cfg.idx_dtype != "f32":
        # the materialised scores read the pages the same way
        s = dsa.indexer_scores(P, d["q_idx"], d["k_idx"], d["w"], d.get("q_scale"),
                               d.get("k_scale"))
        torch.cuda.synchronize()
        p = O.problem_from_case(case)
        sn = to_np(s)
        for t in range(cfg.total_q):
            check_scores_row(sn[t], p.scores(t), f"paged scores row {t}")


@pytest.mark.parametrize("top_k,flag", [(256, 0x2), (2048, 0x1)],
                         ids=["indexer_reads_it", "every_key_kept"])
def test_paged_block_table_outside_cache_is_flagged(top_k, flag):
    # a block-table entry past the cache: the indexer reports it when it scores the row
    # (DSA_FLAG_BAD_SEQS); when the row keeps every key (k >= L) the indexer reads no key and
    # attention reports the entries it skips (DSA_FLAG_BAD_INDEX)
    cfg = W.custom([1, 1], [700, 300], idx_dtype="bf16", kv_dtype="bf16", **dict(BIG, top_k=top_k))
    case = W.make_case(cfg, seed=13)
    pk = W.paged_keys(case, 64, seed=14)
    bt = pk.block_table.clone()
    bt[1, 2] = pk.num_pages + 5          # a page that does not exist
    d = to_dev(case)
    d.update({k: v.cuda() for k, v in pk.tensors().items()})
    P = dsa.Problem.from_config(cfg, d["cu_q"], d["cu_k"], block_table=bt.cuda(),
                                page_size=64, num_pages=pk.num_pages)
    ws = dsa.Workspace()
    ws.clear_status()
    dsa.fused_forward(P, d["q_idx"], d["k_idx"], d["w"], d["q"], d["kv"], ws=ws)
    assert ws.status() & flag, f"flag {flag:#x} not set"
