"""dsa_fused_indexer_static against dsa_fused_indexer, on a GPU.

dsa_fused_indexer_static is the fused indexer for callers that cannot allocate
device memory: code inside a host framework that owns every byte of device
memory and forbids raw cudaMalloc, or a latency-critical loop where cudaMalloc
would synchronise the device.  It keeps its scratch in a static device array
instead of a caller workspace.  Two calls in a row (different shapes, so the
shared array is reused) must give what the workspace entry point gives.

Kept in a file that pytest collects last, so a stop-at-first-failure run has
already run every other test when this one runs.
"""
import ctypes

import numpy as np
import pytest
import torch

import sparse_attention_lightning_gb300 as dsa
from sparse_attention_lightning_gb300 import _abi
from sparse_attention_lightning_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_lightning_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _static_call(P, d, idx, vals, flags):
    ptr = lambda t: None if t is None else t.data_ptr()
    return _abi.lib().dsa_fused_indexer_static(
        ctypes.byref(P.c), d["q_idx"].data_ptr(), d["k_idx"].data_ptr(), d["w"].data_ptr(),
        ptr(d.get("q_scale")), ptr(d.get("k_scale")), idx.data_ptr(), vals.data_ptr(),
        flags.data_ptr(), torch.cuda.current_stream().cuda_stream)


CASES = [
    W.custom([1, 1, 1], [5000, 1700, 2600], h_idx=64, d_idx=128, h=128, d_c=512, d_rope=64,
             top_k=2048, idx_dtype="bf16", kv_dtype="bf16"),
    W.custom([40, 3], [40, 900], top_k=32, idx_dtype="f32", kv_dtype="f32"),
]


def test_static_scratch_entry_point_matches_workspace_entry_point():
    for n, cfg in enumerate(CASES):          # two calls in a row share the static array
        case = W.make_case(cfg, seed=31 + n)
        d = {k: v.cuda() for k, v in case.tensors().items()}
        P = dsa.Problem.from_config(cfg, d["cu_q"], d["cu_k"])
        ref_idx, ref_vals = dsa.fused_indexer(P, d["q_idx"], d["k_idx"], d["w"], want_vals=True)
        idx = torch.full_like(ref_idx, 7)
        vals = torch.zeros_like(ref_vals)
        flags = torch.full((4,), 0xFF, dtype=torch.int32, device="cuda")
        _abi.check(_static_call(P, d, idx, vals, flags))
        torch.cuda.synchronize()
        assert int(flags[0]) == 0
        a, b = idx.cpu().numpy(), ref_idx.cpu().numpy()
        va, vb = vals.cpu().numpy(), ref_vals.cpu().numpy()
        for t in range(cfg.total_q):
            # same selected set, up to swaps of positions whose scores sit within 1e-3
            # (relative) of the k-th score; the order inside a row is free
            sa = dict(zip(a[t][a[t] >= 0].tolist(), va[t][a[t] >= 0].tolist()))
            sb = dict(zip(b[t][b[t] >= 0].tolist(), vb[t][b[t] >= 0].tolist()))
            assert len(sa) == len(sb) == (a[t] >= 0).sum() == (b[t] >= 0).sum()
            assert np.all(a[t][len(sa):] == -1) and np.all(b[t][len(sb):] == -1)
            kth = min(sb.values())
            for p_, v_ in list(set(sa.items()) - set(sb.items())):
                if p_ in sb:  # same position: scores agree to the score tolerance
                    assert abs(v_ - sb[p_]) <= 1e-2 * max(abs(x) for x in sb.values())
                else:
                    assert abs(v_ - kth) <= 1e-3 * abs(kth), (t, p_, v_, kth)
            for p_, v_ in sb.items():
                if p_ not in sa:
                    assert abs(v_ - kth) <= 1e-3 * abs(kth), (t, p_, v_, kth)


def test_static_scratch_rejects_oversized_problems():
    cu = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    P = dsa.Problem(cu, torch.tensor([0, 3_000_000], dtype=torch.int32, device="cuda"),
                    q_lens=[2], k_lens=[3_000_000], h_idx=4, d_idx=32, h=8, d_c=64, d_rope=16,
                    top_k=8, idx_dtype="f32", kv_dtype="f32")
    A = 1 << 20
    rc = _abi.lib().dsa_fused_indexer_static(ctypes.byref(P.c), A, A, A, None, None, A, None,
                                             None, None)
    assert rc == _abi.DSA_ERR_UNSUPPORTED
    assert b"static scratch" in _abi.lib().dsa_last_error()
