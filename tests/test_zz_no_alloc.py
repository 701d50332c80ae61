"""msa_build_k2q_noalloc: the key-block -> query CSR built with the library's
fixed scratch array instead of a caller workspace, for callers that may not
allocate device memory (a framework allocator or memory pool owns it all, or
cudaMalloc's implicit synchronisation is not acceptable on their path).

Its tables must equal those of msa_build_k2q (the entry point that takes a
workspace) bit for bit, on two calls in a row and after another problem has
left its own contents in the shared array.  This file is collected last so a
run that stops at the first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest

from block_sparse_top_attn_gb300 import workloads as W
from tests._util import upload


@pytest.fixture(scope="module")
def B():
    from block_sparse_top_attn_gb300 import build_lib
    build_lib.build()
    from block_sparse_top_attn_gb300 import binding
    return binding


def _cases():
    return {
        "tiny": W.make_problem("tiny", values=False),
        "zipf64k": W.make_problem("zipf64k", values=False),
        "ragged_aligned": W.make_problem(lengths=[200, 77, 130, 1, 9, 513, 2048], num_index_heads=3, topk=5,
                                         policy="diag_uniform", kv_layout="aligned", seed=11, values=False),
        "long128k": W.make_problem("long128k", values=False),
    }


def _with_workspace(B, pb):
    import torch
    prob, t = upload(pb)
    bw = B.Backward(prob)
    B.msa_build_k2q(prob, t["sel"], bw.row_ptr, bw.q_indices, bw.edge_cap, bw.status, bw.ws)
    torch.cuda.synchronize()
    assert int(bw.status[0].item()) == 0
    return prob, t, bw.row_ptr.cpu().numpy(), bw.q_indices.cpu().numpy(), bw.edge_cap


def _no_alloc(B, prob, t, edge_cap):
    import torch
    Hi, NB = prob.num_index_heads, prob.num_blocks
    row_ptr = torch.full((Hi, NB + 1), -7, dtype=torch.int32, device="cuda")
    q_indices = torch.full((Hi, edge_cap), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    B.msa_build_k2q_noalloc(prob, t["sel"], row_ptr, q_indices, edge_cap, status)
    torch.cuda.synchronize()
    assert int(status[0].item()) == 0
    return row_ptr.cpu().numpy(), q_indices.cpu().numpy()


def _same(ref, got):
    rp, qi = ref
    g_rp, g_qi = got
    np.testing.assert_array_equal(g_rp, rp)
    for hi in range(rp.shape[0]):
        n = int(rp[hi, -1])
        np.testing.assert_array_equal(g_qi[hi, :n], qi[hi, :n])


@pytest.mark.gpu
def test_no_alloc_matches_workspace_build_twice(B):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    cases = _cases()
    refs = {}
    for name, pb in cases.items():
        prob, t, rp, qi, cap = _with_workspace(B, pb)
        refs[name] = (prob, t, (rp, qi), cap)
    # every case twice in a row, then the cases again in a different order so
    # each call finds another problem's leftovers in the shared array
    for name in list(cases) + list(reversed(list(cases))):
        prob, t, ref, cap = refs[name]
        for _ in range(2):
            _same(ref, _no_alloc(B, prob, t, cap))


@pytest.mark.gpu
def test_no_alloc_reports_device_errors_like_the_workspace_build(B):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    pb = W.make_problem(lengths=[700, 300], num_index_heads=1, topk=3, policy="diag_uniform", values=False)
    pb.sel = pb.sel.copy()
    pb.sel[0, 20, 1] = 3                      # non-causal: chunk 20 starts at 160 < 3 * 64
    prob, t = upload(pb)
    row_ptr = torch.empty((1, prob.num_blocks + 1), dtype=torch.int32, device="cuda")
    q_indices = torch.empty((1, prob.edge_capacity()), dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    B.msa_build_k2q_noalloc(prob, t["sel"], row_ptr, q_indices, prob.edge_capacity(), status)
    torch.cuda.synchronize()
    assert int(status[0].item()) == B.MSA_ERR_INVALID_SELECTION


def test_no_alloc_rejects_problems_beyond_the_scratch_array(B):
    """Host-side check: nothing is launched, so fake device pointers are safe."""
    p = B.msa_problem()
    T = 49152 * 64                            # the largest key-block count one call accepts
    p.num_docs, p.total_tokens, p.kv_rows = 1, T, T
    p.cu_seqlens, p.kv_doc_starts = 4096, 8192
    p.num_q_heads, p.num_index_heads, p.num_kv_heads = 16 * 64, 64, 64
    p.head_dim, p.block_size, p.query_chunk, p.topk = 128, 64, 8, 32
    p.num_blocks, p.num_chunks, p.softmax_scale = T // 64, T // 8, 0.1
    fake = ctypes.c_void_p(1 << 20)
    rc = B.lib.msa_build_k2q_noalloc(ctypes.byref(p), fake, fake, fake, 1 << 30, fake, None)
    assert rc == B.MSA_ERR_SCRATCH_TOO_SMALL
    assert "no-allocation" in B.status_string(rc)
