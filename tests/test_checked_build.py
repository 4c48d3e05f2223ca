"""The checked build (libdsa_checked.so, -DDSA_CHECKED): the kernels test their internal
invariants on the device (gather rows inside the cache, tile coordinates and query rows in
range, output slots below top_k) and report a failure as DSA_FLAG_CHECK, never by a trap.
Run through it, the main paths must raise no flag and give the same bytes as the ordinary
build."""
import pytest
import torch

import sparse_attention_lightning_gb300 as dsa
from sparse_attention_lightning_gb300 import _abi
from sparse_attention_lightning_gb300 import workloads as W

BIG = dict(h_idx=64, d_idx=128, h=128, d_c=512, d_rope=64)


def test_check_flag_is_declared():
    hdr = open(_abi.os.path.join(_abi._PKG, "..", "include", "dsa.h")).read()
    assert "#define DSA_FLAG_CHECK     0x8u" in hdr and _abi.DSA_FLAG_CHECK == 0x8


def test_checked_library_builds_and_exports_every_symbol():
    # compiles for sm_103a without a GPU (about 20 s); nothing runs on a device
    from sparse_attention_lightning_gb300 import build
    assert build.build(checked=True) == _abi.CHECKED_LIB_PATH
    with _abi.using(_abi.CHECKED_LIB_PATH) as L:
        assert L.dsa_abi_version() == _abi.ABI_VERSION
        for name in _abi.EXPORTS:
            assert hasattr(L, name), name
    assert _abi.lib()._name == _abi.LIB_PATH  # the ordinary library again outside the block


CASES = [
    # (q_lens, k_lens, dims, idx dtype, page size): decode rows on the fused indexer (bf16,
    # FP8), several queries per sequence on the chunked indexer and streaming Top-K, MXFP8,
    # a paged cache, and the CUDA-core paths
    ([1, 1, 1], [3000, 700, 5000], dict(BIG, top_k=2048), "bf16", 0),
    ([1, 1, 4], [4100, 3000, 300], dict(BIG, top_k=2048), "e4m3", 0),
    ([37, 1, 130, 6], [300, 2500, 1300, 6], dict(BIG, top_k=256), "bf16", 0),
    ([1, 3, 1], [2000, 900, 64], dict(BIG, top_k=512), "mxfp8", 0),
    ([1, 1, 1], [3000, 700, 5000], dict(BIG, top_k=2048), "bf16", 64),
    ([1, 7, 40, 1], [1, 300, 40, 2049], dict(top_k=32), "f32", 0),
]


def _run(case, cfg, page_size):
    d = {k: v.cuda() for k, v in case.tensors().items()}
    paging = {}
    if page_size:
        pk = W.paged_keys(case, page_size, seed=12)
        d.update({k: v.cuda() for k, v in pk.tensors().items()})
        paging = dict(block_table=d["block_table"], page_size=page_size, num_pages=pk.num_pages)
    P = dsa.Problem.from_config(cfg, d["cu_q"], d["cu_k"], **paging)
    ws = dsa.Workspace()
    ws.clear_status()
    out, lse, idx, _ = dsa.fused_forward(P, d["q_idx"], d["k_idx"], d["w"], d["q"], d["kv"],
                                         d.get("q_scale"), d.get("k_scale"), ws=ws)
    torch.cuda.synchronize()
    return ws.status(), out.cpu(), lse.cpu(), idx.cpu()


@pytest.mark.gpu
def test_checked_build_raises_no_flag_and_matches():
    from sparse_attention_lightning_gb300 import build
    build.build(checked=True)
    for qs, ks, dims, idt, page in CASES:
        kvd = "f32" if idt == "f32" else "bf16"
        cfg = W.custom(qs, ks, idx_dtype=idt, kv_dtype=kvd, **dims)
        case = W.make_case(cfg, seed=31)
        ref = _run(case, cfg, page)
        with _abi.using(_abi.CHECKED_LIB_PATH):
            got = _run(case, cfg, page)
        assert ref[0] == 0 and got[0] == 0, (qs, idt, page, ref[0], got[0])
        for a, b in zip(ref[1:], got[1:]):
            assert torch.equal(a, b), (qs, idt, page)
