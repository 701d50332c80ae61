"""Shared helpers of the test suite (inputs to device, oracle references, tolerances)."""
from __future__ import annotations

import json
import os

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
                          pb.softmax_scale, device=device, block_size=pb.block)
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


# Below this magnitude half a bf16 ulp is at most 2**-6 = 0.0156, so the
# mandatory output rounding cannot by itself exceed MAX_ABS.  Elements there
# that still exceed the flat 3e-2 are counted (not excused by the output
# rounding alone: P and dS enter the tensor-core GEMMs as bf16, as on the
# pages, and that input rounding adds up over a key's queries).
FLAT_BELOW = 8.0


def grad_errors(gpu_bits: np.ndarray, ref: np.ndarray) -> dict:
    g = O.bf16_to_f64(gpu_bits)
    err = g - ref
    aerr = np.abs(err)
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(err)) / nref if nref > 0 else float(np.linalg.norm(err))
    bound = MAX_ABS + 0.5 * O.bf16_ulp(ref)
    over = aerr > bound
    raw_over = aerr > MAX_ABS
    rounded = O.bf16_to_f64(O.f64_to_bf16(ref))
    # elements over the flat 3e-2 whose correctly rounded exact value is itself
    # more than 3e-2 away: those the bf16 output format alone forces over
    floor_over = np.abs(rounded - ref) > MAX_ABS
    return {
        "rel_fro": rel,
        "max_abs": float(np.max(aerr)) if err.size else 0.0,
        "max_abs_vs_rounded_ref": float(np.max(np.abs(g - rounded))) if err.size else 0.0,
        "max_abs_of_rounding_alone": float(np.max(np.abs(rounded - ref))) if err.size else 0.0,
        "max_abs_ref": float(np.max(np.abs(ref))) if err.size else 0.0,
        "n_over_bound": int(over.sum()),
        "n_raw_over_3e-2": int(raw_over.sum()),
        "n_raw_over_3e-2_rounding_forced": int((raw_over & floor_over).sum()),
        "n_raw_over_3e-2_below_8": int((raw_over & (np.abs(ref) < FLAT_BELOW)).sum()),
        "n": int(err.size),
        "finite": bool(np.all(np.isfinite(g))),
    }


def report(record: dict):
    """One JSON line per parity case: printed (visible with pytest -s) and, when
    MSA_PARITY_LOG names a file, appended to it."""
    line = json.dumps(record, sort_keys=True)
    print("PARITY " + line, flush=True)
    path = os.environ.get("MSA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")


def assert_grad_close(name: str, gpu_bits: np.ndarray, ref: np.ndarray, case: str | None = None):
    e = grad_errors(gpu_bits, ref)
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    report({"case": case or test, "grad": name, **e})
    assert e["finite"], (name, e)
    assert e["rel_fro"] <= REL_FRO, (name, e)
    assert e["n_over_bound"] == 0, (name, e)
    return e
