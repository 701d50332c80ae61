"""GPU: a bounded device wait that runs out reports MSA_ERR_TIMEOUT and leaves
the context usable.  The wait is on an mbarrier phase that nothing completes
(no fault, no trap, no unbounded loop); afterwards a forward on the same device
still matches the oracle."""
import time

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


def test_bounded_wait_times_out_and_the_context_survives(B):
    import torch
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    B.msa_selftest_wait_timeout(st)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(st[0].item()) == B.MSA_ERR_TIMEOUT
    assert 1.0 < elapsed < 60.0
    pb = W.make_problem("tiny")
    prob, t = upload(pb)
    o, lse, fst = B.forward(prob, t["sel"], t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    assert int(fst[0].item()) == 0
    ro, rl = O.forward_blocked(pb.q, pb.k, pb.v, pb.cu_seqlens, pb.kv_doc_starts, pb.sel, pb.block, pb.chunk,
                               pb.softmax_scale)
    assert_grad_close("o", from_bf16_tensor(o), ro)
    assert np.max(np.abs(lse.cpu().numpy().astype(np.float64) - rl)) < 2e-3
