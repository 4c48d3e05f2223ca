"""The bounded-wait path, made to run out without faulting or hanging the GPU: a wait on an
mbarrier that nothing arrives at gives up after a short limit and reports DSA_FLAG_TIMEOUT in
the workspace status word; the status block is cleared and a normal call on the same context and
workspace then runs clean and matches the oracle."""
import numpy as np
import pytest
import torch

import sparse_attention_lightning_gb300 as dsa
from sparse_attention_lightning_gb300 import _abi
from sparse_attention_lightning_gb300 import workloads as W


def test_selftest_argument_checks():
    L = _abi.lib()
    assert L.dsa_selftest_wait_timeout(None, 1000, None) == _abi.DSA_ERR_WORKSPACE
    assert L.dsa_selftest_wait_timeout(1 << 20, 0, None) == _abi.DSA_ERR_INVALID_ARG
    assert L.dsa_selftest_wait_timeout(1 << 20, 10 ** 9, None) == _abi.DSA_ERR_INVALID_ARG
    assert L.dsa_selftest_wait_timeout((1 << 20) + 4, 1000, None) == _abi.DSA_ERR_WORKSPACE


@pytest.mark.gpu
def test_wait_gives_up_then_context_stays_usable():
    from oracle import dsa_oracle as O
    ws = dsa.Workspace("cuda:0")
    ws.clear_status()
    assert ws.status() == 0
    ws.selftest_wait_timeout(2_000_000)  # 2 ms
    flags = ws.status()
    assert flags & _abi.DSA_FLAG_TIMEOUT
    f = __import__("ctypes").c_uint32(0)
    assert _abi.lib().dsa_read_status(ws.ptr, None, __import__("ctypes").byref(f)) == \
        _abi.DSA_ERR_TIMEOUT
    ws.clear_status()
    assert ws.status() == 0
    # a normal call afterwards (the fused decode indexer, whose row counters live in the same
    # status block, and the attention)
    cfg = W.custom([1, 1, 1], [3000, 900, 2100], h_idx=64, d_idx=128, h=128, d_c=512,
                   d_rope=64, top_k=256, idx_dtype="bf16", kv_dtype="bf16")
    case = W.make_case(cfg, seed=5)
    d = {k: v.to("cuda:0") for k, v in case.tensors().items()}
    P = dsa.Problem.from_config(cfg, d["cu_q"], d["cu_k"])
    out, lse, idx, _ = dsa.fused_forward(P, d["q_idx"], d["k_idx"], d["w"], d["q"], d["kv"], ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    p = O.problem_from_case(case)
    idx_n = idx.cpu().numpy()
    for t in range(cfg.total_q):
        I = p.scores(t)
        n = min(cfg.top_k, I.shape[0])
        ref = np.argsort(-I, kind="stable")[:n]
        s_k = I[ref[-1]]
        diff = np.setxor1d(idx_n[t, :n], ref)
        assert np.all(np.abs(I[diff] - s_k) <= 1e-3 * abs(s_k))
