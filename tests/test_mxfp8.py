"""The MXFP8 index path (E4M3 codes, one E8M0 scale per 32 elements of a query head or a
key): scores, Top-K and the attention behind them against the oracle, on the tensor-core
indexer (H_I = 64, d_I = 128) and the CUDA-core one, packed and paged, and the Top-K recall
against the bf16 indexer on the values the codes were quantised from."""
import dataclasses

import numpy as np
import pytest
import torch

import sparse_attention_lightning_gb300 as dsa
from sparse_attention_lightning_gb300 import _abi
from sparse_attention_lightning_gb300 import workloads as W
from oracle import dsa_oracle as O
from parity import check_attn_row, check_scores_row, check_topk_row, to_np, tol_for

BIG = dict(h_idx=64, d_idx=128, h=128, d_c=512, d_rope=64)


def test_mx_inputs_decode_within_half_a_spacing():
    # the generator's codes and E8M0 scales decode to the bf16 draws within half an E4M3
    # spacing of the group's scale grid (no element saturates: amax / 2^e <= 448)
    cfg = W.custom([1, 2], [300, 200], h_idx=4, d_idx=64, idx_dtype="mxfp8", kv_dtype="bf16")
    c = W.make_case(cfg, 3)
    cb = W.make_case(dataclasses.replace(cfg, idx_dtype="bf16"), 3)
    for codes, sc, ref in ((c.k_idx, c.k_scale, cb.k_idx),
                           (c.q_idx.reshape(-1, 64), c.q_scale.reshape(-1, 2),
                            cb.q_idx.reshape(-1, 64))):
        deq = O.mx_dequant(codes.numpy(), sc.numpy())
        x = O.bf16_to_f64(ref.contiguous().view(torch.int16).numpy())
        scale = O.e8m0_to_f64(np.repeat(sc.numpy(), 32, axis=-1))
        bound = np.maximum(np.abs(x) * 2.0 ** -4, scale * 2.0 ** -10) * (1 + 1e-9)
        assert np.all(np.abs(deq - x) <= bound)
        assert np.all(np.abs(deq) <= 448 * scale)


def _case(qs, ks, dims, top_k, seed):
    cfg = W.custom(qs, ks, idx_dtype="mxfp8", kv_dtype="bf16", top_k=top_k, **dims)
    return cfg, W.make_case(cfg, seed)


@pytest.mark.gpu
@pytest.mark.parametrize("qs,ks,dims", [
    ([1, 3, 130, 1], [1000, 300, 130, 1], BIG),        # tensor-core indexer
    ([1, 2, 33], [700, 5, 100], dict(h_idx=8, d_idx=64, h=8, d_c=64, d_rope=16)),  # CUDA cores
])
def test_mx_scores_and_topk(qs, ks, dims):
    cfg, case = _case(qs, ks, dims, 64, 17)
    d = {k: v.cuda() for k, v in case.tensors().items()}
    P = dsa.Problem.from_config(cfg, d["cu_q"], d["cu_k"])
    s = dsa.indexer_scores(P, d["q_idx"], d["k_idx"], d["w"], d["q_scale"], d["k_scale"])
    idx, _ = dsa.topk(P, s)
    torch.cuda.synchronize()
    p = O.problem_from_case(case)
    sn, idn = to_np(s), to_np(idx)
    worst = 0.0
    for t in range(cfg.total_q):
        I = p.scores(t)
        worst = max(worst, check_scores_row(sn[t], I, f"row {t}"))
        check_topk_row(idn[t], I, cfg.top_k, f"row {t}")
    assert worst < 1e-4, worst  # fp32 sums of exact products scaled by powers of two


@pytest.mark.gpu
@pytest.mark.parametrize("page_size", [0, 32])
def test_mx_fused_forward_matches_oracle(page_size):
    """The whole layer with the MXFP8 indexer: decode rows, a prefill-shaped sequence and a
    short one, packed and through a paged key cache."""
    cfg, case = _case([1, 1, 37, 6], [3000, 700, 1300, 6], BIG, 256, 11)
    d = {k: v.cuda() for k, v in case.tensors().items()}
    paging = {}
    if page_size:
        pk = W.paged_keys(case, page_size, seed=12)
        d.update({k: v.cuda() for k, v in pk.tensors().items()})
        paging = dict(block_table=d["block_table"], page_size=page_size, num_pages=pk.num_pages)
    P = dsa.Problem.from_config(cfg, d["cu_q"], d["cu_k"], **paging)
    ws = dsa.Workspace()
    ws.clear_status()
    out, lse, idx, vals = dsa.fused_forward(P, d["q_idx"], d["k_idx"], d["w"], d["q"], d["kv"],
                                            d["q_scale"], d["k_scale"], want_vals=True, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    p = O.problem_from_case(case)
    tol = tol_for(cfg)
    idx_n, vals_n, out_n, lse_n = to_np(idx), to_np(vals), to_np(out), to_np(lse)
    for t in range(cfg.total_q):
        I = p.scores(t)
        check_topk_row(idx_n[t], I, cfg.top_k, f"row {t}")
        n = min(cfg.top_k, I.shape[0])
        sel = idx_n[t, :n]
        assert np.abs(vals_n[t, :n] - I[sel]).max() <= 1e-2 * np.abs(I).max() + 1e-30
        ro, rl = p.sfa(t, sel)
        check_attn_row(out_n[t], lse_n[t], ro, rl, tol, f"row {t}")


@pytest.mark.gpu
def test_mx_recall_matches_oracle():
    import bench
    cfg = W.custom([1] * 4, [6000, 2100, 4096, 3000], top_k=512, idx_dtype="mxfp8",
                   kv_dtype="bf16", **BIG)
    rec = bench.fp8_recall(dsa, W, cfg, 11, "cuda:0", nseq=4)
    sets = {}
    for dt in ("mxfp8", "bf16"):
        c = dataclasses.replace(cfg, idx_dtype=dt)
        p = O.problem_from_case(W.make_case(c, 11))
        sets[dt] = [set(np.argsort(-p.scores(t), kind="stable")[:c.top_k].tolist())
                    for t in range(c.total_q)]
    ref = np.mean([len(a & b) / len(b) for a, b in zip(sets["mxfp8"], sets["bf16"])])
    assert abs(rec["mean"] - ref) <= 0.01, (rec, ref)
