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


@pytest.mark.parametrize("case", ["tiny", "ragged", "single8k"])
def test_forward_matches_oracle(B, case):
    import torch
    if case == "ragged":
        pb = W.make_problem(lengths=[200, 77, 1, 130, 9], num_index_heads=2, topk=4, policy="diag_uniform",
                            kv_layout="aligned", seed=3)
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
