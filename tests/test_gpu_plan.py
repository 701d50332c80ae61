"""GPU: the forward work plan (msa_plan_forward, through the C ABI) is bit-exact
against the oracle's plan (scheduler_metadata rows and work_count), and the
forward that walks it (msa_fwd_planned) writes the same O and LSE, bit for
bit, as the forward in index order."""
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


def _case(name):
    if name in W.WORKLOADS:
        return W.make_problem(name, values=False)
    rng = np.random.default_rng(4)
    pb = W.make_problem(lengths=[300, 260, 5, 1100], num_index_heads=2, topk=6, policy="diag_uniform", seed=4,
                        values=False)
    sel = pb.sel.copy()
    for hi in range(sel.shape[0]):
        for g in range(sel.shape[1]):
            sel[hi, g] = sel[hi, g][rng.permutation(sel.shape[2])]
            if rng.random() < 0.1:
                sel[hi, g] = -1
    pb.sel = sel
    return pb


@pytest.mark.parametrize("name", ["tiny", "single8k", "varlen32k", "zipf64k", "long128k", "ragged_empty",
                                  "single8k_b128"])
def test_plan_bit_exact(B, name):
    import torch
    pb = _case(name)
    prob, t = upload(pb)
    meta, wc, st = B.plan_forward(prob, t["sel"])
    torch.cuda.synchronize()
    assert int(st[0].item()) == 0
    exp_meta, exp_work = O.plan_forward(pb.sel, pb.cu_seqlens, pb.block, pb.chunk)
    np.testing.assert_array_equal(meta.cpu().numpy(), exp_meta)
    assert int(wc[0].item()) == exp_work


@pytest.mark.parametrize("name", ["varlen32k", "ragged_empty"])
def test_planned_forward_equals_forward(B, name):
    import torch
    pb = _case(name)
    prob, t = upload(pb)
    q, k, v, _ = W.device_values(pb, "cuda", seed=1)
    o0, l0, s0 = B.forward(prob, t["sel"], q, k, v)
    meta, _, sp = B.plan_forward(prob, t["sel"])
    o1, l1, s1 = B.forward(prob, t["sel"], q, k, v, plan=meta)
    torch.cuda.synchronize()
    assert int(s0[0].item()) == int(s1[0].item()) == int(sp[0].item()) == 0
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0.view(torch.int32), l1.view(torch.int32))
