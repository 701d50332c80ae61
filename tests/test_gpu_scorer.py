"""GPU: the block scorer and top-k selection (msa_select_topk, through the C
ABI) against the oracle, bit for bit: the top-k decision is taken in the same
fp32 arithmetic on both sides (pooled means rounded to bf16, dot products
summed in index-dim order), so the selected blocks, their order and the -1
pads must be identical.  Covers ragged documents, partial chunks and blocks,
top-k 1 and 32, ties between blocks, every named workload but the 128k one in
full, and sampled rows of the 128k one."""
import numpy as np
import pytest

from oracle import msa_oracle as O
from block_sparse_top_attn_gb300 import workloads as W
from tests._util import to_bf16_tensor, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from block_sparse_top_attn_gb300 import binding
    return binding


def _gpu_sel(B, pb, qi, ki):
    import torch
    prob, _ = upload(pb)
    sel, st = B.select_topk(prob, to_bf16_tensor(qi, "cuda"), to_bf16_tensor(ki, "cuda"))
    torch.cuda.synchronize()
    assert int(st[0].item()) == 0
    return sel.cpu().numpy()


@pytest.mark.parametrize("case", ["tiny", "single8k", "varlen32k", "zipf64k", "ragged", "topk1", "topk32",
                                  "ties", "single8k_b128", "ragged_block128"])
def test_selection_bit_exact(B, case):
    if case in W.WORKLOADS:
        pb = W.make_problem(case, values=False)
    elif case == "ragged":
        pb = W.make_problem(lengths=[200, 77, 130, 1, 9, 513, 2049], num_index_heads=3, topk=6,
                            policy="diag_uniform", seed=3, values=False)
    elif case == "ragged_block128":
        pb = W.make_problem(lengths=[200, 77, 130, 1, 9, 513, 2049], num_index_heads=3, topk=6,
                            policy="diag_uniform", seed=3, values=False, block=128)
    elif case == "topk1":
        pb = W.make_problem(lengths=[700, 90], num_index_heads=2, topk=1, policy="diag_uniform", seed=4,
                            values=False)
    elif case == "topk32":
        pb = W.make_problem(lengths=[5000, 3000], num_index_heads=2, topk=32, policy="diag_uniform", seed=5,
                            values=False)
    else:
        pb = W.make_problem(lengths=[3000], num_index_heads=1, topk=8, policy="diag_uniform", seed=6,
                            values=False)
    qi, ki = W.index_values(pb)
    if case == "ties":
        # coarse index keys: many blocks pool to the same vector and tie
        rng = np.random.default_rng(9)
        vals = rng.integers(-1, 2, size=ki.shape).astype(np.float32)
        ki = W.f32_to_bf16_bits(vals)
    exp = O.select_topk(qi, ki, pb.cu_seqlens, pb.block, pb.chunk, pb.topk)
    got = _gpu_sel(B, pb, qi, ki)
    np.testing.assert_array_equal(got, exp)
    O.validate_selection(got, O.DocLayout(pb.cu_seqlens, pb.block, pb.chunk))


def test_selection_long128k_sampled_rows(B):
    """Full 131k-token workload on the device; the oracle recomputes sampled
    rows from the pooled vectors of their chunk and of every causal block."""
    import torch
    pb = W.make_problem("long128k", values=False)
    qi, ki = W.index_values(pb)
    got = _gpu_sel(B, pb, qi, ki)
    lay = O.DocLayout(pb.cu_seqlens, pb.block, pb.chunk)
    rng = np.random.default_rng(0)
    kpool = O.pool_index(ki, pb.cu_seqlens, pb.block)               # [Hi, NB, D]
    for hi, g in [(int(rng.integers(0, 8)), int(c)) for c in rng.integers(0, lay.NC, size=24)] + [(0, 0), (7, lay.NC - 1)]:
        rows = slice(g * pb.chunk, (g + 1) * pb.chunk)
        qpool = O.pool_index(qi[rows], np.array([0, pb.chunk]), pb.chunk)[hi]   # [1, D]
        diag = g * pb.chunk // pb.block
        sc = O.block_scores(qpool, kpool[hi, :diag])[0] if diag else np.zeros(0, np.float32)
        ranked = sorted(range(diag), key=lambda b: (-float(sc[b]), b))[:pb.topk - 1]
        exp = [diag] + ranked
        exp += [-1] * (pb.topk - len(exp))
        assert got[hi, g].tolist() == exp, (hi, g)
    O.validate_selection(got, lay)


def test_selection_feeds_the_backward(B):
    """The scorer's selection is a valid input of the table build and the
    backward: CSR and tasks bit-exact, gradients within tolerance."""
    import torch
    from tests._util import assert_grad_close, from_bf16_tensor, oracle_backward, oracle_forward_stored
    pb = W.make_problem(lengths=[900, 350], num_index_heads=2, topk=5, policy="diag_uniform", seed=8)
    qi, ki = W.index_values(pb)
    pb.sel = _gpu_sel(B, pb, qi, ki)
    np.testing.assert_array_equal(pb.sel, O.select_topk(qi, ki, pb.cu_seqlens, pb.block, pb.chunk, pb.topk))
    o_bits, lse32 = oracle_forward_stored(pb)
    ref = oracle_backward(pb, o_bits, lse32)
    prob, t = upload(pb)
    bw = B.Backward(prob)
    outs = bw.run(t["sel"], t["q"], t["k"], t["v"], to_bf16_tensor(o_bits, "cuda"), t["do"],
                  torch.from_numpy(np.ascontiguousarray(lse32)).cuda())
    torch.cuda.synchronize()
    bw.check_status()
    for name, g, r in zip(("dq", "dk", "dv"), outs, ref):
        assert_grad_close(name, from_bf16_tensor(g), r)
