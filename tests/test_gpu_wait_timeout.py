"""GPU: a bounded device wait that runs out reports MSA_ERR_TIMEOUT and leaves
the context usable.  The waits are on mbarrier phases that nothing completes
(no fault, no trap, no unbounded loop): a one-wait kernel, and the main
backward kernel with one role held idle; afterwards a forward or a backward on
the same device still matches the oracle."""
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


def test_backward_aborts_cleanly_when_a_role_stalls(B):
    """The main backward kernel with its reduce warps held idle (a self-test
    instance): the task-info ring and the dQ buffers are never released, the
    waits on them run out their bound, every role aborts and waits for the
    copies it started, and the status reads MSA_ERR_TIMEOUT.  A normal backward
    on the same context and buffers then matches the oracle."""
    import torch
    from tests._util import oracle_backward, oracle_forward_stored, to_bf16_tensor
    pb = W.make_problem("tiny")
    prob, t = upload(pb)
    o_bits, lse32 = oracle_forward_stored(pb)
    o = to_bf16_tensor(o_bits, "cuda")
    lse = torch.from_numpy(np.ascontiguousarray(lse32)).cuda()
    bw = B.Backward(prob)
    bw.build_tables(t["sel"])
    bw.backward_stage(B.MSA_STAGE_PREPROCESS, t["q"], t["k"], t["v"], o, t["do"], lse)
    torch.cuda.synchronize()
    bw.check_status()
    t0 = time.monotonic()
    bw.backward_stage(B.MSA_STAGE_MAIN | B.MSA_BWD_SELFTEST_HOLD_REDUCE, t["q"], t["k"], t["v"], o, t["do"], lse)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(bw.status[0].item()) == B.MSA_ERR_TIMEOUT
    assert 1.0 < elapsed < 60.0
    bw.status.zero_()
    dq, dk, dv = bw.run(t["sel"], t["q"], t["k"], t["v"], o, t["do"], lse)
    torch.cuda.synchronize()
    bw.check_status()
    ref = oracle_backward(pb, o_bits, lse32)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_grad_close(name, from_bf16_tensor(g), r)
