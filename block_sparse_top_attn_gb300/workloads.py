"""Seeded synthetic inputs for the MSA block-sparse attention backward.

This module draws inputs only: document lengths, the top-k key-block selection
and the bf16 tensors Q, K, V and dO.  It holds none of the method's arithmetic
(no attention, no softmax, no gradient), so that the fp64 oracle and the CUDA
library can both be fed from it without sharing any of the computation.

Every draw goes through one ``numpy.random.default_rng(seed)`` in a fixed
order: document lengths, selection, Q, K, V, dO.  Dense values are standard
normal fp32 draws rounded to bf16 (round to nearest even); tensors travel as
``uint16`` bf16 bit patterns.

The five named workloads follow the MiniMax-M3 MSA backward statement (packed
THD tensors, 16 query heads per index/KV head, head dim 128, key block 64,
query chunk 8, causal within each document):

* ``tiny``      1 doc x 512 tokens, 1 index head, 16 q heads, top-k 4
                (diagonal block + 3 uniform earlier blocks).
* ``single8k``  1 doc x 8192, 4 index heads, 64 q heads, top-k 16
                (diagonal + 15 uniform earlier blocks).
* ``varlen32k`` 32768 tokens packed from lengths drawn uniformly in
                [512, 8192] (last document truncated), 4/64 heads, top-k 16
                (diagonal + 15 uniform earlier blocks of the same document).
* ``long128k``  1 doc x 131072, 8 index heads, 128 q heads, top-k 32
                (diagonal + 3 most recent + 28 uniform earlier blocks).
* ``zipf64k``   8 docs x 8192, 4/64 heads, top-k 16 drawn by sequential
                weighted sampling without replacement with weight
                (b + 1) ** -1.2 over the causal blocks b of the chunk.

Chunks that have fewer causal blocks than top-k take all of them and pad the
remaining slots with -1.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

HEAD_DIM = 128
BLOCK = 64
CHUNK = 8
GROUP = 16

WORKLOADS = {
    "tiny": dict(lengths=[512], num_index_heads=1, topk=4, policy="diag_uniform"),
    "single8k": dict(lengths=[8192], num_index_heads=4, topk=16, policy="diag_uniform"),
    "varlen32k": dict(total=32768, len_range=(512, 8192), num_index_heads=4, topk=16,
                      policy="diag_uniform"),
    "long128k": dict(lengths=[131072], num_index_heads=8, topk=32, policy="diag_recent3_uniform"),
    "zipf64k": dict(lengths=[8192] * 8, num_index_heads=4, topk=16, policy="zipf", zipf_s=1.2),
    # one index head of long128k (an eighth of its tasks, same causal and
    # per-tile structure): the small case for hardware-counter captures
    "long128k_1head": dict(lengths=[131072], num_index_heads=1, topk=32, policy="diag_recent3_uniform"),
    # 128-key blocks: the same keys per chunk (16 x 128 = 32 x 64)
    "single8k_b128": dict(lengths=[8192], num_index_heads=4, topk=8, policy="diag_uniform", block=128),
    "long128k_b128": dict(lengths=[131072], num_index_heads=8, topk=16, policy="diag_recent3_uniform", block=128),
}


@dataclasses.dataclass
class Problem:
    """One seeded problem instance.  Arrays are host numpy arrays.

    q, do: uint16 bf16 bits [T, Hq, D]; k, v: uint16 bf16 bits [W, Hkv, D];
    cu_seqlens int32 [N + 1]; kv_doc_starts int32 [N]; sel int32 [Hi, NC, K]
    (document-local key-block ids, -1 = empty slot), indexed by the global
    query chunk (chunks of each document numbered after those of the previous
    documents).
    """

    name: str
    cu_seqlens: np.ndarray
    kv_doc_starts: np.ndarray
    kv_rows: int
    num_q_heads: int
    num_index_heads: int
    head_dim: int
    block: int
    chunk: int
    topk: int
    sel: np.ndarray
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray
    softmax_scale: float

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_docs(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_index_heads


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even) and return the 16-bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat.size, step):
        n = min(step, flat.size - s)
        flat[s:s + n] = f32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32))
    return out


def _draw_lengths(rng, spec) -> list[int]:
    if "lengths" in spec:
        return list(spec["lengths"])
    lo, hi = spec["len_range"]
    total = spec["total"]
    out, acc = [], 0
    while acc < total:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def _uniform_subset(rng, n_rows: int, pool: int, k: int) -> np.ndarray:
    """k distinct values from range(pool) per row (uniform, without replacement)."""
    if k <= 0 or pool <= 0:
        return np.zeros((n_rows, 0), dtype=np.int64)
    if k >= pool:
        return np.tile(np.arange(pool, dtype=np.int64), (n_rows, 1))
    keys = rng.random((n_rows, pool))
    return np.argpartition(keys, k - 1, axis=1)[:, :k].astype(np.int64)


def draw_selection(rng, lengths, num_index_heads: int, topk: int, policy: str,
                   block: int = BLOCK, chunk: int = CHUNK, zipf_s: float = 1.2) -> np.ndarray:
    """Selection sel[Hi, NC, K] of document-local key blocks per query chunk."""
    nc = [math.ceil(n / chunk) for n in lengths]
    sel = np.full((num_index_heads, sum(nc), topk), -1, dtype=np.int32)
    g0 = 0
    for n, ncd in zip(lengths, nc):
        for hi in range(num_index_heads):
            # chunks sharing one diagonal block draw together
            for bd in range(math.ceil(n / block)):
                c_lo = bd * block // chunk
                c_hi = min(ncd, (bd + 1) * block // chunk)
                if c_lo >= c_hi:
                    continue
                rows = c_hi - c_lo
                if policy == "diag_uniform":
                    fixed = [bd]
                    pool = bd
                elif policy == "diag_recent3_uniform":
                    fixed = [bd] + [b for b in (bd - 1, bd - 2, bd - 3) if b >= 0]
                    pool = max(bd - 3, 0)
                elif policy == "zipf":
                    fixed, pool = [], bd + 1
                else:
                    raise ValueError(policy)
                if policy == "zipf":
                    w = (np.arange(pool, dtype=np.float64) + 1.0) ** (-zipf_s)
                    w = w / w.sum()
                    kk = min(topk, pool)
                    for i in range(rows):
                        pick = rng.choice(pool, size=kk, replace=False, p=w)
                        sel[hi, g0 + c_lo + i, :kk] = pick
                else:
                    kk = min(topk - len(fixed), pool)
                    pick = _uniform_subset(rng, rows, pool, kk)
                    sel[hi, g0 + c_lo:g0 + c_hi, :len(fixed)] = fixed
                    sel[hi, g0 + c_lo:g0 + c_hi, len(fixed):len(fixed) + kk] = pick
        g0 += ncd
    return sel


def make_problem(name: str | None = None, *, seed: int = 0, lengths=None,
                 num_index_heads: int | None = None, topk: int | None = None,
                 policy: str | None = None, group: int = GROUP, head_dim: int = HEAD_DIM,
                 block: int = BLOCK, chunk: int = CHUNK, kv_layout: str = "compact",
                 kv_align: int = 128, values: bool = True, zipf_s: float = 1.2) -> Problem:
    """Draw a named workload (``name``) or a custom one (explicit keywords).

    ``kv_layout='aligned'`` places each document's keys at a multiple of
    ``kv_align`` rows in the K/V workspace, the padding rows holding finite
    random values.  ``values=False`` skips the dense tensors (tables only).
    """
    rng = np.random.default_rng(seed)
    if name is not None:
        spec = dict(WORKLOADS[name])
        lengths = _draw_lengths(rng, spec)
        num_index_heads = spec["num_index_heads"]
        topk = spec["topk"]
        policy = spec["policy"]
        zipf_s = spec.get("zipf_s", zipf_s)
        block = spec.get("block", block)
    lengths = [int(n) for n in lengths]
    sel = draw_selection(rng, lengths, num_index_heads, topk, policy, block, chunk, zipf_s)
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    if kv_layout == "compact":
        kv_starts = cu[:-1].copy()
        kv_rows = int(cu[-1])
    elif kv_layout == "aligned":
        padded = [-(-n // kv_align) * kv_align for n in lengths]
        kv_starts = np.zeros(len(lengths), dtype=np.int32)
        kv_starts[1:] = np.cumsum(padded)[:-1]
        kv_rows = int(sum(padded))
    else:
        raise ValueError(kv_layout)
    T = int(cu[-1])
    hq = num_index_heads * group
    hkv = num_index_heads
    if values:
        q = _normal_bf16(rng, (T, hq, head_dim))
        k = _normal_bf16(rng, (kv_rows, hkv, head_dim))
        v = _normal_bf16(rng, (kv_rows, hkv, head_dim))
        do = _normal_bf16(rng, (T, hq, head_dim))
    else:
        q = k = v = do = None
    return Problem(name or "custom", cu, kv_starts, kv_rows, hq, num_index_heads, head_dim,
                   block, chunk, topk, sel, q, k, v, do, float(head_dim) ** -0.5)


def device_values(pb: Problem, device="cuda", seed: int = 0):
    """bf16 N(0, 1) Q, K, V, dO drawn on the device with torch's seeded Philox
    generator (for workloads whose host draw would take tens of seconds).
    Returns torch bf16 tensors (q, k, v, do); the host draw order is kept."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    T, Hq, Hkv, D, W = pb.total_tokens, pb.num_q_heads, pb.num_index_heads, pb.head_dim, pb.kv_rows

    def draw(shape):
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = out.view(-1)
        step = 1 << 28
        for s in range(0, flat.numel(), step):
            n = min(step, flat.numel() - s)
            flat[s:s + n] = torch.randn(n, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
        return out

    return draw((T, Hq, D)), draw((W, Hkv, D)), draw((W, Hkv, D)), draw((T, Hq, D))


INDEX_DIM = 128


def index_values(pb: Problem, seed: int = 0, index_dim: int = INDEX_DIM):
    """Index projections for the block scorer: per token and index head, an
    index query and an index key, bf16 N(0, 1) as uint16 bit patterns of shape
    [T, Hi, index_dim] each.  They come from their own generator
    (``default_rng([seed, 1])``: index queries, then index keys), so drawing
    them leaves every other input of the workload unchanged."""
    rng = np.random.default_rng([seed, 1])
    shape = (pb.total_tokens, pb.num_index_heads, index_dim)
    return _normal_bf16(rng, shape), _normal_bf16(rng, shape)


def device_index_values(pb: Problem, device="cuda", seed: int = 0, index_dim: int = INDEX_DIM):
    """index_values drawn on the device with torch's seeded Philox generator
    (same distribution; for workloads whose host draw is slow).  Returns torch
    bf16 tensors (q_index, k_index)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed + 1_000_003)
    shape = (pb.total_tokens, pb.num_index_heads, index_dim)
    return tuple(torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
                 for _ in range(2))


def effective_flops(pb: Problem) -> int:
    """Effective FLOP of the backward over full selected blocks: every
    (query, q-head, selected block) costs 5 GEMMs x 2 x block x head_dim."""
    lengths = np.diff(pb.cu_seqlens.astype(np.int64))
    chunk_len = np.concatenate([np.minimum(pb.chunk, n - np.arange(0, n, pb.chunk)) for n in lengths])
    slots = (pb.sel >= 0).sum(axis=2)                      # [Hi, NC]
    rows = int((slots * chunk_len[None, :]).sum()) * pb.group
    return rows * 10 * pb.block * pb.head_dim
