"""Pins of the fp64 oracle against things other than itself (no GPU).

Each test checks the oracle against a closed form, a library routine, brute
force on tiny inputs, or an invariant, chosen so that a dropped term, a wrong
sign or index, or a transposed operand in the oracle fails one of them.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O


# ---------------------------------------------------------------------------
# Element decoding.

def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_closed_form_values():
    vals = O.e4m3_to_f64(np.array([0x7E, 0x08, 0x01, 0x38, 0xB8, 0x00, 0x07, 0x3C], dtype=np.uint8))
    assert list(vals) == [448.0, 2.0 ** -6, 2.0 ** -9, 1.0, -1.0, 0.0, 7 * 2.0 ** -9, 1.5]


def test_bf16_decode_matches_torch():
    x = torch.randn(4096, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_to_f64(bits), x.to(torch.float64).numpy())


# ---------------------------------------------------------------------------
# Positions.

def test_query_positions_closed_form():
    # seq0: decode (T=1, L=5) → pos 4; seq1: prefill T=L=3 → 0,1,2; seq2: T=2 of L=6 → 4,5.
    rows = O.query_rows([0, 1, 4, 6], [0, 5, 8, 14])
    assert rows == [(0, 0, 4), (1, 1, 0), (2, 1, 1), (3, 1, 2), (4, 2, 4), (5, 2, 5)]


# ---------------------------------------------------------------------------
# Indexer scoring.

def test_indexer_unit_queries_pick_key_columns():
    # q_I[j] = e_j makes z[j, s] = k_I[s, j]; shapes H_I=3 != d_I=5 expose a transposed operand.
    rng = np.random.default_rng(1)
    k = rng.standard_normal((7, 5))
    q = np.eye(3, 5)
    w = np.array([0.5, 2.0, 0.25])
    got = O.indexer_row(q, k, w, pos=6)
    want = [sum(w[j] * max(0.0, k[s, j]) for j in range(3)) for s in range(7)]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def test_indexer_relu_sign_and_weights_closed_form():
    # q_I[j] = a_j·u and k_I[s] = c_s·u with |u| = 1, so z[j, s] = a_j·c_s.
    u = np.array([0.6, 0.0, 0.8])
    a = np.array([1.0, -2.0, 3.0])
    w = np.array([0.5, 0.25, 2.0])
    c = np.arange(8) - 3.0                     # c_s = s - 3 takes both signs
    q = a[:, None] * u[None, :]
    k = c[:, None] * u[None, :]
    got = O.indexer_row(q, k, w, pos=7)
    # c > 0: heads 0 and 2 fire: (0.5·1 + 2·3)·c = 6.5c; c < 0: head 1 fires: 0.25·(-2)·c = -0.5c.
    want = np.where(c > 0, 6.5 * c, -0.5 * c)
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=1e-15)


def test_indexer_is_causal_inclusive():
    k = np.zeros((6, 2))
    k[3] = [1.0, 0.0]                          # the query's own position
    k[4] = [100.0, 0.0]                        # a future key, must not be seen
    got = O.indexer_row(np.array([[1.0, 0.0]]), k, np.array([1.0]), pos=3)
    assert got.shape == (4,)
    assert list(got) == [0.0, 0.0, 0.0, 1.0]


def test_indexer_fp8_scales_dequantise_per_key_and_per_query_head():
    # Powers-of-two scales keep code·scale exact in fp32, so the fp8 problem must equal
    # the fp32 problem holding the dequantised values.
    rng = np.random.default_rng(2)
    T, L, HI, DI = 1, 9, 3, 4
    qc = rng.integers(0, 256, (T, HI, DI)).astype(np.uint8)
    kc = rng.integers(0, 256, (L, DI)).astype(np.uint8)
    qc[(qc & 0x7F) == 0x7F] = 0x3C              # no NaN codes
    kc[(kc & 0x7F) == 0x7F] = 0x3C
    qs = np.array([[0.5, 4.0, 0.125]], dtype=np.float32)   # distinct per head
    ks = (2.0 ** rng.integers(-3, 3, L)).astype(np.float32)
    w = rng.uniform(0, 1, (T, HI)).astype(np.float32)
    base = dict(cu_q=np.array([0, 1]), cu_k=np.array([0, L]), w=w,
                q=np.zeros((T, 1, 8), np.float32), kv=np.zeros((L, 8), np.float32))
    p8 = O.Problem(dict(base, q_idx=qc, k_idx=kc, q_scale=qs, k_scale=ks),
                   idx_dtype="e4m3", kv_dtype="f32", d_c=4, top_k=4)
    qf = (O.e4m3_to_f64(qc) * qs[:, :, None]).astype(np.float32)
    kf = (O.e4m3_to_f64(kc) * ks[:, None]).astype(np.float32)
    p32 = O.Problem(dict(base, q_idx=qf, k_idx=kf), idx_dtype="f32", kv_dtype="f32", d_c=4,
                    top_k=4)
    assert np.array_equal(p8.scores(0), p32.scores(0))
    # and a scale on the wrong axis would change the scores
    assert not np.allclose(O.indexer_row(O.e4m3_to_f64(qc[0]) * ks[:HI, None],
                                         O.e4m3_to_f64(kc) * qs[0, :1], w[0], L - 1),
                           p8.scores(0))


def test_e8m0_decode_matches_torch_for_every_code():
    # OCP E8M0: 2^(code - 127), 255 = NaN (the library's own float8_e8m0fnu)
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).double().numpy()
    got = O.e8m0_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[:255], ref[:255])
    assert O.e8m0_to_f64(np.array([127, 128, 126], np.uint8)).tolist() == [1.0, 2.0, 0.5]


def test_mxfp8_group_scales_sit_on_their_32_elements():
    # codes all 1.0 (0x38); query groups scaled 1, 2, 4, 8 and key groups 8, 4, 2, 1: the dot
    # is 32·(8 + 8 + 8 + 8) = 1024, while a reversed or transposed group axis gives 2720
    HI, DI, L = 2, 128, 3
    qc = np.full((1, HI, DI), 0x38, np.uint8)
    kc = np.full((L, DI), 0x38, np.uint8)
    qs = np.array([[[127, 128, 129, 130], [130, 129, 128, 127]]], np.uint8)
    ks = np.tile(np.array([[130, 129, 128, 127]], np.uint8), (L, 1))
    w = np.array([[1.0, 0.25]], np.float32)
    p = O.Problem(dict(cu_q=np.array([0, 1]), cu_k=np.array([0, L]), w=w, q_idx=qc, k_idx=kc,
                       q_scale=qs, k_scale=ks, q=np.zeros((1, 1, 8), np.float32),
                       kv=np.zeros((L, 8), np.float32)),
                  idx_dtype="mxfp8", kv_dtype="f32", d_c=4, top_k=2)
    # head 0: 32·(1·8 + 2·4 + 4·2 + 8·1) = 1024; head 1: 32·(8·8 + 4·4 + 2·2 + 1·1) = 2720
    assert p.scores(0).tolist() == [1.0 * 1024 + 0.25 * 2720] * L


def test_indexer_mxfp8_equals_fp32_on_dequantised_values():
    rng = np.random.default_rng(3)
    T, L, HI, DI = 1, 7, 3, 64
    qc = rng.integers(0, 256, (T, HI, DI)).astype(np.uint8)
    kc = rng.integers(0, 256, (L, DI)).astype(np.uint8)
    qc[(qc & 0x7F) == 0x7F] = 0x3C
    kc[(kc & 0x7F) == 0x7F] = 0x3C
    qs = rng.integers(120, 134, (T, HI, DI // 32)).astype(np.uint8)
    ks = rng.integers(120, 134, (L, DI // 32)).astype(np.uint8)
    w = rng.uniform(0, 1, (T, HI)).astype(np.float32)
    base = dict(cu_q=np.array([0, 1]), cu_k=np.array([0, L]), w=w,
                q=np.zeros((T, 1, 8), np.float32), kv=np.zeros((L, 8), np.float32))
    pmx = O.Problem(dict(base, q_idx=qc, k_idx=kc, q_scale=qs, k_scale=ks),
                    idx_dtype="mxfp8", kv_dtype="f32", d_c=4, top_k=4)
    # code · 2^k is exact in fp32 for these exponents
    qf = (O.e4m3_to_f64(qc) * np.exp2(np.repeat(qs.astype(np.float64) - 127, 32, -1)))
    kf = (O.e4m3_to_f64(kc) * np.exp2(np.repeat(ks.astype(np.float64) - 127, 32, -1)))
    p32 = O.Problem(dict(base, q_idx=qf.astype(np.float32), k_idx=kf.astype(np.float32)),
                    idx_dtype="f32", kv_dtype="f32", d_c=4, top_k=4)
    assert np.array_equal(pmx.scores(0), p32.scores(0))


# ---------------------------------------------------------------------------
# Top-K.

@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_subset_brute_force(seed):
    # For distinct scores the top-n set is the unique n-subset with the largest sum.
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 10))
    k = int(rng.integers(1, 6))
    s = rng.permutation(L).astype(np.float64) + rng.uniform(0, 0.5)
    n = min(k, L)
    best = max(itertools.combinations(range(L), n), key=lambda c: sum(s[i] for i in c))
    assert sorted(O.topk_row(s, k).tolist()) == sorted(best)


def test_topk_ties_go_to_smaller_positions():
    assert O.topk_row(np.zeros(10), 4).tolist() == [0, 1, 2, 3]
    assert sorted(O.topk_row(np.array([1.0, 3.0, 3.0, 3.0, 0.0]), 2).tolist()) == [1, 2]
    assert O.topk_row(np.array([2.0, 1.0]), 5).tolist() == [0, 1]        # fewer than k


def test_topk_threshold_invariant_random():
    rng = np.random.default_rng(3)
    for _ in range(20):
        s = rng.integers(0, 5, int(rng.integers(1, 40))).astype(np.float64)  # many ties
        k = int(rng.integers(1, 20))
        sel = O.topk_row(s, k)
        rest = np.setdiff1d(np.arange(s.size), sel)
        assert sel.size == min(k, s.size) and np.unique(sel).size == sel.size
        if rest.size:
            assert s[sel].min() >= s[rest].max()
            # every tied-but-unselected position lies after every tied selected one
            tau = s[sel].min()
            assert rest[s[rest] == tau].min(initial=10 ** 9) > sel[s[sel] == tau].max()


# ---------------------------------------------------------------------------
# Sparse attention.

def _sdpa(q, k, v, mask=None):
    # torch's math backend in fp64, default scale 1/sqrt(q.size(-1))
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), attn_mask=mask).numpy()


def test_sfa_full_history_equals_dense_causal_attention():
    # k >= pos+1 selects the whole prefix: SFA must equal standard causal attention.
    rng = np.random.default_rng(4)
    T, H, dc, dr = 12, 3, 6, 2
    q = rng.standard_normal((T, H, dc + dr))
    kv = rng.standard_normal((T, dc + dr))
    outs = np.stack([O.sfa_row(q[t], kv, range(t + 1), dc, 1 / math.sqrt(dc + dr))[0]
                     for t in range(T)])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(0, 1), torch.from_numpy(kv)[None].expand(H, T, -1),
        torch.from_numpy(kv[:, :dc])[None].expand(H, T, -1), is_causal=True).transpose(0, 1).numpy()
    np.testing.assert_allclose(outs, ref, rtol=1e-12, atol=1e-13)


def test_sfa_equals_dense_attention_with_minus_inf_mask_outside_selection():
    rng = np.random.default_rng(5)
    L, H, dc, dr = 20, 4, 8, 3
    q = rng.standard_normal((H, dc + dr))
    kv = rng.standard_normal((L, dc + dr))
    sel = rng.choice(L, 7, replace=False)
    out, lse = O.sfa_row(q, kv, sel, dc, 1 / math.sqrt(dc + dr))
    mask = np.full((H, L), -np.inf)
    mask[:, sel] = 0.0
    ref = _sdpa(q[:, None, :], np.broadcast_to(kv, (H, L, dc + dr)).copy(),
                np.broadcast_to(kv[:, :dc], (H, L, dc)).copy(), torch.from_numpy(mask[:, None, :]))
    np.testing.assert_allclose(out, ref[:, 0], rtol=1e-12, atol=1e-13)
    # lse against torch.logsumexp of the masked dense logits
    dense = (q @ kv.T) / math.sqrt(dc + dr) + mask
    np.testing.assert_allclose(lse, torch.logsumexp(torch.from_numpy(dense), 1).numpy(), rtol=1e-13)


def test_sfa_zero_query_gives_mean_and_log_n():
    rng = np.random.default_rng(6)
    kv = rng.standard_normal((9, 5))
    sel = [1, 4, 7]
    out, lse = O.sfa_row(np.zeros((2, 5)), kv, sel, 3, 0.5)
    np.testing.assert_allclose(out, np.broadcast_to(kv[sel, :3].mean(0), (2, 3)), atol=1e-15)
    np.testing.assert_allclose(lse, [math.log(3)] * 2, rtol=1e-15)


def test_sfa_single_row_and_two_row_closed_forms():
    kv = np.array([[1.0, 2.0, 3.0], [4.0, -1.0, 0.5], [0.0, 0.0, 2.0]])
    q = np.array([[0.0, 0.0, 1.0]])            # logit = scale·kv[r, 2]
    out, lse = O.sfa_row(q, kv, [1], 2, 0.5)
    assert out.tolist() == [[4.0, -1.0]] and lse.tolist() == [0.25]
    out, lse = O.sfa_row(q, kv, [0, 2], 2, 0.5)
    # logits 1.5 and 1.0: weights σ(0.5) and σ(-0.5)
    p = 1 / (1 + math.exp(-0.5))
    np.testing.assert_allclose(out[0], p * kv[0, :2] + (1 - p) * kv[2, :2], rtol=1e-15)
    np.testing.assert_allclose(lse[0], math.log(math.exp(1.5) + math.exp(1.0)), rtol=1e-15)


def test_sfa_empty_selection():
    out, lse = O.sfa_row(np.ones((2, 3)), np.ones((4, 3)), [], 2, 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_default_scale_is_inverse_sqrt_of_full_row_width():
    arr = dict(cu_q=np.array([0, 1]), cu_k=np.array([0, 2]), q_idx=np.zeros((1, 1, 4), np.float32),
               k_idx=np.zeros((2, 4), np.float32), w=np.ones((1, 1), np.float32),
               q=np.zeros((1, 1, 80), np.float32), kv=np.zeros((2, 80), np.float32))
    p = O.Problem(arr, idx_dtype="f32", kv_dtype="f32", d_c=64, top_k=2)
    assert p.sm_scale == 1 / math.sqrt(80)


# ---------------------------------------------------------------------------
# The whole row: planted structure pins selection → output.

def test_planted_keys_are_selected_and_pull_the_output():
    rng = np.random.default_rng(7)
    L, HI, DI, H, dc, dr, k = 64, 4, 8, 2, 6, 2, 4
    qi = np.abs(rng.standard_normal((1, HI, DI))).astype(np.float32)
    ki = (rng.standard_normal((L, DI)) * 0.01).astype(np.float32)
    planted = [5, 17, 40, 63]
    ki[planted] = 1.0                           # aligned with every (positive) query head
    q = rng.standard_normal((1, H, dc + dr)).astype(np.float32)
    kv = rng.standard_normal((L, dc + dr)).astype(np.float32)
    kv[planted, :dc] = 50.0                     # marker in the value columns
    arr = dict(cu_q=np.array([0, 1]), cu_k=np.array([0, L]), q_idx=qi, k_idx=ki,
               w=np.ones((1, HI), np.float32), q=q, kv=kv)
    r = O.Problem(arr, idx_dtype="f32", kv_dtype="f32", d_c=dc, top_k=k).forward_row(0)
    assert sorted(r["idx"].tolist()) == planted
    np.testing.assert_allclose(r["out"], 50.0, rtol=1e-12)


def test_invariants_on_tiny_workload():
    from sparse_attention_lightning_gb300 import workloads as W
    case = W.make_case(W.custom([16, 1], [16, 40], top_k=8), seed=11)
    p = O.problem_from_case(case)
    res = p.forward()
    for t, r in res.items():
        _, b, pos = p.rows[t]
        idx = r["idx"]
        assert idx.size == min(8, pos + 1) and np.unique(idx).size == idx.size
        assert idx.min() >= 0 and idx.max() <= pos
        assert np.all(r["scores"] >= 0)          # ReLU with w >= 0
        kvb = p.kv_seq(b)[idx, :64]
        assert np.all(r["out"] <= kvb.max(0) + 1e-12) and np.all(r["out"] >= kvb.min(0) - 1e-12)
