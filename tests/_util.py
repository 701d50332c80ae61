"""Shared helpers of the test suite (inputs to device, oracle references, tolerances)."""
from __future__ import annotations

import numpy as np

from oracle import msa_oracle as O

# Tolerances of the backward against the fp64 oracle: relative Frobenius error
# <= 1e-2 and max-abs error <= 3e-2, the latter applied on top of the bf16
# rounding every output must undergo (half a bf16 ulp of the exact value).
REL_FRO = 1e-2
MAX_ABS = 3e-2


def to_bf16_tensor(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def from_bf16_tensor(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def upload(pb, device="cuda"):
    """Device tensors and the binding's Problem for a workloads.Problem."""
    import torch
    from block_sparse_top_attn_gb300 import binding as B
    prob = B.make_problem(pb.cu_seqlens, pb.kv_doc_starts, pb.kv_rows, pb.num_q_heads, pb.topk,
                          pb.softmax_scale, device=device)
    t = {"sel": torch.from_numpy(np.ascontiguousarray(pb.sel)).to(device)}
    if pb.q is not None:
        for name in ("q", "k", "v", "do"):
            t[name] = to_bf16_tensor(getattr(pb, name), device)
    return prob, t


def oracle_forward_stored(pb):
    """O rounded to bf16 bits and LSE rounded to fp32, from the blocked oracle."""
    o, lse = O.forward_blocked(pb.q, pb.k, pb.v, pb.cu_seqlens, pb.kv_doc_starts, pb.sel, pb.block, pb.chunk,
                               pb.softmax_scale)
    return O.f64_to_bf16(o), lse.astype(np.float32)


def oracle_backward(pb, o_bits, lse32):
    return O.backward_blocked(pb.q, pb.k, pb.v, o_bits, pb.do, lse32.astype(np.float64), pb.cu_seqlens,
                              pb.kv_doc_starts, pb.sel, pb.block, pb.chunk, pb.softmax_scale, kv_rows=pb.kv_rows)


def grad_errors(gpu_bits: np.ndarray, ref: np.ndarray) -> dict:
    g = O.bf16_to_f64(gpu_bits)
    err = g - ref
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(err)) / nref if nref > 0 else float(np.linalg.norm(err))
    bound = MAX_ABS + 0.5 * O.bf16_ulp(ref)
    over = np.abs(err) > bound
    return {
        "rel_fro": rel,
        "max_abs": float(np.max(np.abs(err))) if err.size else 0.0,
        "max_abs_vs_rounded_ref": float(np.max(np.abs(g - O.bf16_to_f64(O.f64_to_bf16(ref))))) if err.size else 0.0,
        "n_over_bound": int(over.sum()),
        "n_raw_over_3e-2": int((np.abs(err) > MAX_ABS).sum()),
        "finite": bool(np.all(np.isfinite(g))),
    }


def assert_grad_close(name: str, gpu_bits: np.ndarray, ref: np.ndarray):
    e = grad_errors(gpu_bits, ref)
    assert e["finite"], (name, e)
    assert e["rel_fro"] <= REL_FRO, (name, e)
    assert e["n_over_bound"] == 0, (name, e)
    return e
