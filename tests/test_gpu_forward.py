"""GPU: O and LSE from msa_fwd (the flat forward) against the fp64 oracle."""
import numpy as np
import pytest

from oracle import msa_oracle as O
from block_sparse_top_attn_gb300 import workloads as W
from tests._util import assert_grad_close, from_bf16_tensor, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from block_sparse_top_attn_gb300 import binding
    return binding


@pytest.mark.parametrize("case", ["tiny", "ragged", "single8k", "single8k_b128", "ragged_block128"])
def test_forward_matches_oracle(B, case):
    import torch
    if case == "ragged":
        pb = W.make_problem(lengths=[200, 77, 1, 130, 9], num_index_heads=2, topk=4, policy="diag_uniform",
                            kv_layout="aligned", seed=3)
    elif case == "ragged_block128":
        pb = W.make_problem(lengths=[65, 127, 1, 129, 300, 9], num_index_heads=2, topk=3, policy="diag_uniform",
                            kv_layout="aligned", seed=13, block=128)
    else:
        pb = W.make_problem(case)
    prob, t = upload(pb)
    o, lse, st = B.forward(prob, t["sel"], t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    assert int(st[0].item()) == 0
    ro, rl = O.forward_blocked(pb.q, pb.k, pb.v, pb.cu_seqlens, pb.kv_doc_starts, pb.sel, pb.block, pb.chunk,
                               pb.softmax_scale)
    assert_grad_close("o", from_bf16_tensor(o), ro)
    gl = lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(gl - rl)) < 2e-3


@pytest.mark.parametrize("case", ["empty_chunks", "single_tokens", "topk1", "tail_T", "zipf_shuffled"])
def test_forward_edge_cases(B, case):
    """Chunks with no selected block (O = 0, LSE = -inf), -1 pads and blocks in
    any slot order, one-token documents, top-k 1, a partial last chunk, and a
    zipf selection whose block order is shuffled so the running max moves."""
    import torch
    rng = np.random.default_rng(11)
    if case == "empty_chunks":
        pb = W.make_problem(lengths=[300, 260], num_index_heads=2, topk=3, policy="diag_uniform", seed=4)
        sel = pb.sel.copy()
        for hi in range(sel.shape[0]):
            for g in range(sel.shape[1]):
                sel[hi, g] = sel[hi, g][rng.permutation(sel.shape[2])]
                if rng.random() < 0.1:
                    sel[hi, g] = -1
        pb.sel = sel
    elif case == "single_tokens":
        pb = W.make_problem(lengths=[1, 1, 2, 1, 3], num_index_heads=1, topk=2, policy="diag_uniform", seed=2)
    elif case == "topk1":
        pb = W.make_problem(lengths=[64 * 5 + 3], num_index_heads=1, topk=1, policy="diag_uniform", seed=3)
    elif case == "tail_T":
        pb = W.make_problem(lengths=[555], num_index_heads=1, topk=5, policy="diag_recent3_uniform", seed=5)
    else:
        pb = W.make_problem(lengths=[4096, 1500], num_index_heads=2, topk=16, policy="zipf", seed=6)
        sel = pb.sel.copy()
        for hi in range(sel.shape[0]):
            for g in range(sel.shape[1]):
                sel[hi, g] = sel[hi, g][rng.permutation(sel.shape[2])]
        pb.sel = sel
    prob, t = upload(pb)
    o, lse, st = B.forward(prob, t["sel"], t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    assert int(st[0].item()) == 0
    ro, rl = O.forward_blocked(pb.q, pb.k, pb.v, pb.cu_seqlens, pb.kv_doc_starts, pb.sel, pb.block, pb.chunk,
                               pb.softmax_scale)
    assert_grad_close("o", from_bf16_tensor(o), ro)
    gl = lse.cpu().numpy().astype(np.float64)
    empty = ~np.isfinite(rl)
    assert np.array_equal(empty, ~np.isfinite(gl))          # exactly the rows with no key
    assert np.all(from_bf16_tensor(o)[empty] == 0)
    assert np.max(np.abs(gl[~empty] - rl[~empty])) < 2e-3


def _forward_parity(B, pb):
    import torch
    prob, t = upload(pb)
    o, lse, st = B.forward(prob, t["sel"], t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    assert int(st[0].item()) == 0
    ro, rl = O.forward_blocked(pb.q, pb.k, pb.v, pb.cu_seqlens, pb.kv_doc_starts, pb.sel, pb.block, pb.chunk,
                               pb.softmax_scale)
    assert_grad_close("o", from_bf16_tensor(o), ro)
    gl = lse.cpu().numpy().astype(np.float64)
    assert np.array_equal(~np.isfinite(rl), ~np.isfinite(gl))
    fin = np.isfinite(rl)
    assert np.max(np.abs(gl[fin] - rl[fin])) < 2e-3


def test_forward_many_documents(B):
    """Sixty documents of 1..599 tokens with K/V rows at aligned, gapped
    offsets: every item looks its document up among many and reads its keys
    at a document-local block offset."""
    rng = np.random.default_rng(21)
    lengths = [int(x) for x in rng.integers(1, 600, size=60)]
    pb = W.make_problem(lengths=lengths, num_index_heads=2, topk=6, policy="diag_uniform", kv_layout="aligned",
                        seed=21)
    _forward_parity(B, pb)


@pytest.mark.parametrize("name", ["varlen32k", "zipf64k"])
def test_forward_large_sampled(B, name):
    """The mid-size workloads at full size: 300 random (index head, document,
    chunk) items, each checked against the oracle's per-chunk forward."""
    import torch
    pb = W.make_problem(name)
    prob, t = upload(pb)
    o, lse, st = B.forward(prob, t["sel"], t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    assert int(st[0].item()) == 0
    go = from_bf16_tensor(o)
    gl = lse.cpu().numpy().astype(np.float64)
    lay = O.DocLayout(pb.cu_seqlens, pb.block, pb.chunk)
    G = pb.num_q_heads // pb.sel.shape[0]
    rng = np.random.default_rng(5)
    got_o, ref_o, got_l, ref_l = [], [], [], []
    for _ in range(300):
        hi = int(rng.integers(pb.sel.shape[0]))
        d = int(rng.integers(lay.num_docs))
        c = int(rng.integers(int(lay.nc[d])))
        qp, oc, lc = O.chunk_forward(pb.q, pb.k, pb.v, lay, pb.kv_doc_starts, pb.sel, hi, d, c, G,
                                     pb.softmax_scale)
        rows = int(lay.cu[d]) + qp
        got_o.append(go[rows, hi * G:(hi + 1) * G])
        ref_o.append(oc.transpose(1, 0, 2))
        got_l.append(gl[rows, hi * G:(hi + 1) * G])
        ref_l.append(lc.T)
    assert_grad_close("o", np.concatenate(got_o), np.concatenate(ref_o))
    gl_s, rl_s = np.concatenate(got_l), np.concatenate(ref_l)
    assert np.array_equal(np.isfinite(gl_s), np.isfinite(rl_s))
    fin = np.isfinite(rl_s)
    assert np.max(np.abs(gl_s[fin] - rl_s[fin])) < 2e-3


def _rows_with_rescale(pb, lay, chunks):
    """Rows of the given (hi, d, c) chunks whose running max, taken over the
    selected blocks in slot order, rises by more than 8 (log2 units) after
    the row's first key: the kernel rescales O in TMEM for those."""
    qf, kf = O.bf16_to_f64(pb.q), O.bf16_to_f64(pb.k)
    G = pb.num_q_heads // pb.sel.shape[0]
    n = 0
    for hi, d, c in chunks:
        t0, k0 = int(lay.cu[d]), int(pb.kv_doc_starts[d])
        qp = lay.chunk_positions(d, c)
        m = np.full((qp.size, G), -np.inf)
        hit = np.zeros((qp.size, G), dtype=bool)
        for b in (int(x) for x in pb.sel[hi, int(lay.chunk_off[d]) + c] if x >= 0):
            keys = np.arange(b * 64, min(b * 64 + 64, int(lay.lengths[d])))
            s = np.einsum("qhd,kd->qhk", qf[t0 + qp, hi * G:(hi + 1) * G], kf[k0 + keys, hi])
            s = np.where(keys[None, None, :] <= qp[:, None, None], s * pb.softmax_scale / np.log(2.0), -np.inf)
            bm = s.max(axis=2)
            up = bm > m + 8
            hit |= up & (m > -np.inf)
            m = np.where(up, bm, m)
        n += int(hit.sum())
    return n


def test_forward_rescales_o_when_the_max_jumps(B):
    """K of about a third of the key blocks scaled by 8 (exact in bf16) and
    block order shuffled: most rows meet a block that raises their running
    max by more than 2^8, so the kernel's O rescale in TMEM runs."""
    rng = np.random.default_rng(31)
    pb = W.make_problem(lengths=[2048, 700], num_index_heads=2, topk=8, policy="diag_uniform", seed=31)
    kf = O.bf16_to_f64(pb.k)
    lay = O.DocLayout(pb.cu_seqlens, pb.block, pb.chunk)
    for d in range(lay.num_docs):
        k0 = int(pb.kv_doc_starts[d])
        for b in range(int(lay.nb[d])):
            if rng.random() < 0.35:
                kf[k0 + b * 64:k0 + b * 64 + 64] *= 8.0
    pb.k = O.f64_to_bf16(kf)
    sel = pb.sel.copy()
    for hi in range(sel.shape[0]):
        for g in range(sel.shape[1]):
            sel[hi, g] = sel[hi, g][rng.permutation(sel.shape[2])]
    pb.sel = sel
    sample = [(int(rng.integers(2)), d, int(rng.integers(int(lay.nc[d])))) for d in (0, 1) for _ in range(20)]
    assert _rows_with_rescale(pb, lay, sample) > 0
    _forward_parity(B, pb)
