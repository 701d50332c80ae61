"""GPU: the CSR, task tables and walk from msa_build_k2q / msa_build_tasks are
bit-exact against the oracle on every named workload and on ragged custom
cases, and device-detected errors land in the status word."""
import numpy as np
import pytest

from oracle import msa_oracle as O
from block_sparse_top_attn_gb300 import workloads as W
from tests._util import upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from block_sparse_top_attn_gb300 import binding
    return binding


def _check_tables(B, pb, tile, sms=None):
    import torch
    prob, t = upload(pb)
    bw = B.Backward(prob, task_tile_chunks=tile, num_sms=sms or 0)
    bw.build_tables(t["sel"])
    torch.cuda.synchronize()
    bw.check_status()
    rp, qi = O.build_k2q(pb.sel, pb.cu_seqlens, pb.block, pb.chunk)
    g_rp = bw.row_ptr.cpu().numpy()
    np.testing.assert_array_equal(g_rp, rp)
    g_qi = bw.q_indices.cpu().numpy()
    for hi in range(rp.shape[0]):
        n = int(rp[hi, -1])
        np.testing.assert_array_equal(g_qi[hi, :n], qi[hi, :n])
    meta, qr, qp = O.build_tasks(rp, qi, pb.cu_seqlens, pb.block, pb.chunk, tile_chunks=tile)
    n = meta.shape[0]
    walk = bw.walk.cpu().numpy()
    S = sms or B.msa_device_sm_count(torch.cuda.current_device())
    R = O.rows_per_cta(n)
    full, tail, grid = O.chunk_map(n, R, S)
    assert walk[:6].tolist() == [n, R, full, tail, grid, S]
    np.testing.assert_array_equal(bw.task_meta[:n].cpu().numpy(), meta)
    np.testing.assert_array_equal(bw.task_q_rows[:n].cpu().numpy(), qr)
    np.testing.assert_array_equal(bw.task_q_pos[:n].cpu().numpy(), qp)
    return n


@pytest.mark.parametrize("name", ["tiny", "single8k", "varlen32k", "zipf64k", "long128k", "single8k_b128",
                                  "long128k_b128"])
def test_tables_bit_exact_named(B, name):
    pb = W.make_problem(name, values=False)
    tile = 1024 if name.startswith("long128k") else 0
    _check_tables(B, pb, tile)


@pytest.mark.parametrize("tile", [0, 3])
@pytest.mark.parametrize("seed", [0, 1])
def test_tables_bit_exact_ragged_block128(B, tile, seed):
    # 128-key blocks: documents that end inside a block's lower or upper
    # half, a single token, and chunks whose last query stops short of the
    # upper half of their own diagonal block
    rng = np.random.default_rng(200 + seed)
    lengths = [65, 127, 1, 129, 200, 64, 700] if seed == 0 else [int(x) for x in rng.integers(1, 1200, size=6)]
    pb = W.make_problem(lengths=lengths, num_index_heads=2, topk=5, policy="diag_uniform", seed=seed,
                        values=False, block=128, kv_layout="aligned" if seed else "compact")
    _check_tables(B, pb, tile, sms=int(rng.integers(1, 200)))


@pytest.mark.parametrize("tile", [0, 1, 5, 64])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tables_bit_exact_ragged(B, tile, seed):
    rng = np.random.default_rng(100 + seed)
    lengths = [int(x) for x in rng.integers(1, 900, size=int(rng.integers(1, 7)))]
    pb = W.make_problem(lengths=lengths, num_index_heads=int(rng.integers(1, 4)), topk=int(rng.integers(1, 9)),
                        policy="diag_uniform", seed=seed, values=False,
                        kv_layout="aligned" if seed % 2 else "compact")
    sel = pb.sel.copy()
    for hi in range(sel.shape[0]):        # -1 pads at random slots, some chunks left empty
        for g in range(sel.shape[1]):
            sel[hi, g] = sel[hi, g][rng.permutation(sel.shape[2])]
            if rng.random() < 0.05:
                sel[hi, g] = -1
    pb.sel = sel
    _check_tables(B, pb, tile, sms=int(rng.integers(1, 200)))


def test_tables_are_deterministic(B):
    import torch
    pb = W.make_problem("zipf64k", values=False)
    prob, t = upload(pb)
    outs = []
    for _ in range(3):
        bw = B.Backward(prob)
        bw.build_tables(t["sel"])
        torch.cuda.synchronize()
        assert int(bw.status[0].item()) == 0
        n = bw.num_tasks()
        e = int(bw.row_ptr[:, -1].max().item())
        outs.append((bw.row_ptr.cpu().numpy().copy(), bw.q_indices[:, :e].cpu().numpy().copy(),
                     bw.task_meta[:n].cpu().numpy().copy(), bw.task_q_rows[:n].cpu().numpy().copy(),
                     bw.task_q_pos[:n].cpu().numpy().copy(), bw.walk.cpu().numpy().copy()))
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("bad", ["range", "causal", "dup"])
def test_invalid_selection_sets_status(B, bad):
    import torch
    pb = W.make_problem(lengths=[700, 300], num_index_heads=1, topk=3, policy="diag_uniform", values=False)
    sel = pb.sel.copy()
    if bad == "range":
        sel[0, 10, 1] = 11                   # doc 0 has 11 blocks: 0..10
    elif bad == "causal":
        sel[0, 20, 1] = 3                    # chunk 20 starts at 160 < 3 * 64
    else:
        sel[0, 40, :2] = [2, 2]
    pb.sel = sel
    prob, t = upload(pb)
    bw = B.Backward(prob)
    bw.build_tables(t["sel"])
    torch.cuda.synchronize()
    assert int(bw.status[0].item()) == B.MSA_ERR_INVALID_SELECTION


def test_capacity_errors_set_status(B):
    import torch
    pb = W.make_problem("tiny", values=False)
    prob, t = upload(pb)
    bw = B.Backward(prob, edge_cap=100)
    bw.build_tables(t["sel"])
    torch.cuda.synchronize()
    assert int(bw.status[0].item()) == B.MSA_ERR_CAPACITY
    bw = B.Backward(prob, task_cap=100)
    bw.build_tables(t["sel"])
    torch.cuda.synchronize()
    assert int(bw.status[0].item()) == B.MSA_ERR_CAPACITY


def test_inconsistent_documents_set_status(B):
    import torch
    pb = W.make_problem(lengths=[300, 200], num_index_heads=1, topk=2, policy="diag_uniform", values=False)
    prob, t = upload(pb)
    prob.d_kvs[1] = 100                      # overlaps document 0's K/V rows
    bw = B.Backward(prob)
    bw.build_tables(t["sel"])
    torch.cuda.synchronize()
    assert int(bw.status[0].item()) == B.MSA_ERR_INVALID_DOCUMENTS


@pytest.mark.slow
def test_tables_bit_exact_row_windows(B):
    # more key-block rows than one shared-memory row window of the CSR build
    # (16384): a 1.1M-token document and a short one, with duplicates planted
    # past the first window checked separately below
    pb = W.make_problem(lengths=[1_100_000, 5000], num_index_heads=1, topk=3, policy="diag_uniform", seed=21,
                        values=False)
    assert O.DocLayout(pb.cu_seqlens, pb.block, pb.chunk).NB > 16384
    _check_tables(B, pb, 4096)


def test_duplicate_past_the_first_row_window_sets_status(B):
    import torch
    pb = W.make_problem(lengths=[1_100_000], num_index_heads=1, topk=3, policy="diag_uniform", seed=22,
                        values=False)
    sel = pb.sel.copy()
    g = sel.shape[1] - 5                       # a late chunk: its diagonal row is in the second window
    sel[0, g, 1] = sel[0, g, 0]
    pb.sel = sel
    prob, t = upload(pb)
    bw = B.Backward(prob)
    bw.build_tables(t["sel"])
    torch.cuda.synchronize()
    assert int(bw.status[0].item()) == B.MSA_ERR_INVALID_SELECTION
