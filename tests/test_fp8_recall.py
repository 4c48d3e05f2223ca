"""Top-K recall of the FP8 indexer against the bf16 indexer on the bf16 values the FP8 inputs
were quantised from (a measurement the pages ask for): the GPU's recall, computed from the two
GPU index sets, against the recall of the oracle's two exact sets."""
import dataclasses

import numpy as np
import pytest
import torch

import bench
import sparse_attention_lightning_gb300 as dsa
from sparse_attention_lightning_gb300 import workloads as W


def test_recall_counts_rows():
    a = torch.tensor([[3, 1, 2, -1], [5, 6, 7, 8]], dtype=torch.int32)
    b = torch.tensor([[1, 2, 9, -1], [8, 7, 6, 5]], dtype=torch.int32)
    r = bench.topk_recall(a, b)
    assert r.tolist() == [2 / 3, 1.0]


def test_indexer_only_case_is_a_prefix():
    cfg = W.custom([1, 1], [300, 200], h_idx=4, d_idx=32, h=8, d_c=64, d_rope=16, top_k=16,
                   idx_dtype="e4m3", kv_dtype="bf16")
    full = W.make_case(cfg, seed=3)
    sub = W.make_case(W.first_sequences(cfg, 1), seed=3, attention=False)
    assert torch.equal(sub.k_idx, full.k_idx[:300]) and torch.equal(sub.q_idx, full.q_idx[:1])
    assert torch.equal(sub.k_scale, full.k_scale[:300]) and sub.kv.numel() == 0


@pytest.mark.gpu
def test_fp8_recall_matches_oracle():
    from oracle import dsa_oracle as O
    cfg = W.custom([1] * 6, [6000, 2100, 4096, 3000, 700, 5000], h_idx=64, d_idx=128, h=128,
                   d_c=512, d_rope=64, top_k=512, idx_dtype="e4m3", kv_dtype="bf16")
    rec = bench.fp8_recall(dsa, W, cfg, 11, "cuda:0", nseq=6)
    ref = []
    sets = {}
    for dt in ("e4m3", "bf16"):
        c = dataclasses.replace(cfg, idx_dtype=dt)
        p = O.problem_from_case(W.make_case(c, 11))
        sets[dt] = []
        for t in range(c.total_q):
            I = p.scores(t)
            sets[dt].append(set(np.argsort(-I, kind="stable")[:min(c.top_k, I.shape[0])].tolist()))
    for a, b in zip(sets["e4m3"], sets["bf16"]):
        ref.append(len(a & b) / len(b))
    assert rec["rows"] == cfg.total_q
    assert abs(rec["mean"] - float(np.mean(ref))) <= 0.01, (rec, np.mean(ref))
    assert 0.5 < rec["mean"] <= 1.0
