"""Indexer prolog: Q quantisation and head-weight projection.

CPU tests pin the oracle (oracle/prolog.py) to what the E4M3 format, the
library's own fp8 conversion and closed forms fix; GPU tests compare the fused
prolog kernel with it (codes and scales bit-exact, weights within an fp32
summation bound) and run prolog -> FP8 fused indexer end to end.
"""
import numpy as np
import pytest
import torch

from oracle import prolog as P
from oracle.dsa_oracle import e4m3_to_f64


# ---------------------------------------------------------------------------
# The E4M3 encoder.

def test_e4m3_named_values():
    # values fixed by the format: 1 = 0.0111.000, 448 = 0.1111.110, smallest subnormal 2^-9
    y = np.array([0.0, -0.0, 1.0, -1.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -6, 1.875, 0.5],
                 np.float32)
    want = [0x00, 0x80, 0x38, 0xB8, 0x7E, 0xFE, 0x01, 0x08, 0x3F, 0x30]
    assert P.e4m3_encode(y).tolist() == want


def test_e4m3_ties_go_to_even():
    # midpoints between neighbours: the code with an even mantissa wins
    y = np.array([1.0625,          # between 1 (0x38) and 1.125 (0x39) -> 0x38
                  1.1875,          # between 1.125 (0x39) and 1.25 (0x3A) -> 0x3A
                  2.0 ** -10,      # between 0 and 2^-9 -> 0
                  3 * 2.0 ** -10,  # between 2^-9 (0x01) and 2^-8 (0x02) -> 0x02
                  15 * 2.0 ** -10,  # between 7·2^-9 (0x07) and 2^-6 (0x08) -> 0x08
                  432.0,           # between 416 (0x7D) and 448 (0x7E) -> 0x7E
                  240.0 + 8.0],    # between 240 (0x77) and 256 (0x78) -> 0x78
                 np.float32)
    assert P.e4m3_encode(y).tolist() == [0x38, 0x3A, 0x00, 0x02, 0x08, 0x7E, 0x78]


def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = e4m3_to_f64(codes).astype(np.float32)
    assert np.array_equal(P.e4m3_encode(vals), codes)


def test_e4m3_saturates():
    y = np.array([448.5, 463.9, 464.0, 480.0, 1e6, -1e30], np.float32)
    assert P.e4m3_encode(y).tolist() == [0x7E] * 5 + [0xFE]


def test_e4m3_matches_torch_cast():
    # the library's own float32 -> float8_e4m3fn cast (round to nearest even) over random
    # magnitudes spanning the subnormals to the top binade, and every midpoint
    rng = np.random.default_rng(0)
    y = (np.exp2(rng.uniform(-12, np.log2(448), 200_000)) *
         rng.choice([-1.0, 1.0], 200_000)).astype(np.float32)
    grid = np.sort(e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    y = np.concatenate([y, mids, -mids])
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(P.e4m3_encode(y), ref)


# ---------------------------------------------------------------------------
# Per-token quantisation.

def _tokens(seed, T=6, n=512):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1 / np.sqrt(128), (T, n)).astype(np.float32)
    # bf16-valued, like the indexer queries
    return (torch.from_numpy(x).to(torch.bfloat16).float()).numpy()


def test_quantise_amax_maps_to_448_and_error_bound():
    x = _tokens(1)
    codes, scale = P.quantise_tokens(x)
    deq = e4m3_to_f64(codes) * scale[:, None]
    for t in range(x.shape[0]):
        j = np.argmax(np.abs(x[t]))
        assert codes[t, j] & 0x7F == 0x7E
    # 3 mantissa bits: at most half a spacing, 2^-4 relative on normals, 2^-10·scale below
    bound = np.maximum(np.abs(x) * 2.0 ** -4, scale[:, None] * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound)


def test_quantise_sign_scale_and_zero():
    x = _tokens(2)
    c, s = P.quantise_tokens(x)
    cn, sn = P.quantise_tokens(-x)
    assert np.array_equal(cn, c ^ 0x80) and np.array_equal(sn, s)
    c4, s4 = P.quantise_tokens(4 * x)  # a power of two commutes with both fp32 divisions
    assert np.array_equal(c4, c) and np.array_equal(s4, 4 * s)
    z, sz = P.quantise_tokens(np.zeros((2, 64), np.float32))
    assert np.all(z == 0) and np.all(sz == 1.0)


def test_quantise_matches_torch_quantiser():
    # an independent statement of the same per-row rule through the library's fp8 cast:
    # scale = amax / 448 (fp32), codes = cast(x / scale)
    x = _tokens(3, T=9, n=1024)
    codes, scale = P.quantise_tokens(x)
    xt = torch.from_numpy(x)
    amax = xt.abs().amax(dim=1)
    st = amax / 448.0
    ct = (xt / st[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(scale, st.numpy()) and np.array_equal(codes, ct)


# ---------------------------------------------------------------------------
# Head-weight projection.

def test_head_weights_one_hot_picks_columns():
    rng = np.random.default_rng(4)
    w_h = rng.normal(size=(5, 12))
    x = np.eye(12)[[3, 0, 11]]          # token t is the unit vector e_c
    w = P.head_weights(x, w_h)
    assert w.shape == (3, 5)
    assert np.array_equal(w, w_h[:, [3, 0, 11]].T)


def test_head_weights_ones_give_row_sums():
    rng = np.random.default_rng(5)
    x = rng.integers(-4, 5, size=(4, 20)).astype(np.float64)
    w = P.head_weights(x, np.ones((3, 20)))
    assert np.array_equal(w, np.repeat(x.sum(axis=1)[:, None], 3, axis=1))


# ---------------------------------------------------------------------------
# The library: argument checks (no GPU work) and, on the GPU, parity.

def test_prolog_argument_checks():
    from sparse_attention_lightning_gb300 import _abi
    L = _abi.lib()
    a = 1 << 20  # an aligned address that is never dereferenced: every check fails first
    assert L.dsa_indexer_prolog(4, 4, 32, 64, None, None, None, None, None, None, None) == \
        _abi.DSA_ERR_INVALID_ARG
    assert L.dsa_indexer_prolog(4, 4, 12, 64, a, None, None, a, a, None, None) == \
        _abi.DSA_ERR_UNSUPPORTED
    assert L.dsa_indexer_prolog(4, 4, 32, 60, None, a, a, None, None, a, None) == \
        _abi.DSA_ERR_UNSUPPORTED
    assert L.dsa_indexer_prolog(4, 4, 32, 64, None, a, None, None, None, a, None) == \
        _abi.DSA_ERR_INVALID_ARG
    assert L.dsa_indexer_prolog(4, 4, 32, 64, a + 8, None, None, a, a, None, None) == \
        _abi.DSA_ERR_INVALID_ARG
    assert L.dsa_indexer_prolog(-1, 4, 32, 64, a, None, None, a, a, None, None) == \
        _abi.DSA_ERR_INVALID_ARG


def _w_bound(x: np.ndarray, w_h: np.ndarray) -> np.ndarray:
    # fp32 accumulation of exact bf16 products: each output is rounded at most
    # d_model/512 + 8 (a thread's chunks) + 5 (warp butterfly) + 16 (warps) times,
    # each time by at most 2^-24 of a partial sum bounded by Σ|terms|; 1e-5 covers
    # d_model <= 65536
    return 1e-5 * (np.abs(x) @ np.abs(w_h).T) + 1e-30


def _run_prolog(T, h, d, d_model, seed, parts=("q", "w")):
    import sparse_attention_lightning_gb300 as dsa
    from sparse_attention_lightning_gb300 import workloads as W
    cfg = W.custom([1] * T, [64] * T, h_idx=h, d_idx=d, idx_dtype="e4m3", kv_dtype="bf16")
    inp = W.prolog_inputs(cfg, seed, d_model)
    dev = "cuda:0"
    qp = inp["q_proj"].to(dev) if "q" in parts else None
    x = inp["x"].to(dev) if "w" in parts else None
    wh = inp["w_h"].to(dev) if "w" in parts else None
    codes, scale, w = dsa.indexer_prolog(qp, x, wh)
    torch.cuda.synchronize()
    return inp, codes, scale, w


@pytest.mark.gpu
@pytest.mark.parametrize("T,h,d,d_model", [
    (3, 4, 32, 64),        # one partial tile of each kind
    (37, 64, 128, 7168),   # decode shapes: five token tiles, the last ragged
    (32, 64, 128, 7168),   # the 32-sequence decode batch
    (129, 12, 16, 200),    # ragged head tile, d_model not a multiple of the thread stride
    (1, 1, 8, 8),          # smallest sizes
])
def test_prolog_matches_oracle(T, h, d, d_model):
    inp, codes, scale, w = _run_prolog(T, h, d, d_model, seed=T + h)
    qf = inp["q_proj"].float().reshape(T, h * d).numpy()
    rc, rs = P.quantise_tokens(qf)
    assert np.array_equal(codes.cpu().reshape(T, -1).numpy(), rc)      # bit-exact codes
    assert np.array_equal(scale.cpu().numpy(), np.repeat(rs[:, None], h, axis=1))
    x = inp["x"].float().numpy().astype(np.float64)
    wh = inp["w_h"].float().numpy().astype(np.float64)
    ref = P.head_weights(x, wh)
    err = np.abs(w.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= _w_bound(x, wh)), float((err / _w_bound(x, wh)).max())


@pytest.mark.gpu
def test_prolog_parts_and_edge_tokens():
    import sparse_attention_lightning_gb300 as dsa
    dev = "cuda:0"
    # quantisation only, with an all-zero token and a token holding one huge value
    q = torch.randn(5, 8, 64).to(torch.bfloat16)
    q[1] = 0
    q[3, 2, 7] = 3.0e38
    codes, scale, w = dsa.indexer_prolog(q.to(dev))
    assert w is None
    rc, rs = P.quantise_tokens(q.float().reshape(5, -1).numpy())
    assert np.array_equal(codes.cpu().reshape(5, -1).numpy(), rc)
    assert np.array_equal(scale.cpu().numpy()[:, 0], rs) and rs[1] == 1.0
    # projection only
    inp, codes, scale, w = _run_prolog(9, 16, 32, 520, seed=7, parts=("w",))
    assert codes is None and scale is None
    x = inp["x"].float().numpy().astype(np.float64)
    wh = inp["w_h"].float().numpy().astype(np.float64)
    assert np.all(np.abs(w.cpu().numpy() - P.head_weights(x, wh)) <= _w_bound(x, wh))
    # no tokens: nothing launched, empty results
    c0, s0, w0 = dsa.indexer_prolog(torch.empty(0, 4, 32, dtype=torch.bfloat16, device=dev))
    assert c0.numel() == 0 and s0.numel() == 0


@pytest.mark.gpu
def test_prolog_feeds_the_fp8_fused_indexer():
    """prolog -> FP8 fused indexer on the GPU against the oracle's prolog -> indexer -> Top-K:
    the GPU prolog's query codes and scales are those of the FP8 workload's inputs, and the
    selected positions match the oracle's under the Top-K tie rule."""
    import dataclasses

    import sparse_attention_lightning_gb300 as dsa
    from oracle import dsa_oracle as O
    from sparse_attention_lightning_gb300 import workloads as W
    from tests.parity import check_topk_row
    cfg = W.custom([1] * 5, [3000, 700, 4096, 1500, 2200], h_idx=64, d_idx=128, h=128, d_c=512,
                   d_rope=64, top_k=512, idx_dtype="e4m3", kv_dtype="bf16")
    case = W.make_case(cfg, seed=21)
    inp = W.prolog_inputs(cfg, 21, 1024)
    dev = "cuda:0"
    codes, scale, w = dsa.indexer_prolog(inp["q_proj"].to(dev), inp["x"].to(dev),
                                         inp["w_h"].to(dev))
    assert torch.equal(codes.cpu(), case.q_idx) and torch.equal(scale.cpu(), case.q_scale)
    Pb = dsa.Problem.from_config(cfg, case.cu_q.to(dev), case.cu_k.to(dev))
    idx, _ = dsa.fused_indexer(Pb, codes, case.k_idx.to(dev), w, scale, case.k_scale.to(dev))
    idx = idx.cpu().numpy()
    x = inp["x"].float().numpy().astype(np.float64)
    wh = inp["w_h"].float().numpy().astype(np.float64)
    ref_w = P.head_weights(x, wh).astype(np.float32)
    prob = O.problem_from_case(dataclasses.replace(case, w=torch.from_numpy(ref_w)))
    for t in range(cfg.total_q):
        check_topk_row(idx[t], prob.scores(t), cfg.top_k, ctx=f"row {t}")
