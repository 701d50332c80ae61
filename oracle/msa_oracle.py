"""Plain fp64 CPU oracle for the MSA block-sparse top-k attention backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA library.

Sources (NVIDIA NeMo AutoModel API pages for MiniMax-M3-VL MSA):

* ``msa_backward_sm100`` page, module docstring: the backward is KV-parallel
  over task rows of 8 queries x 16 main heads, bucketed by (batch, index head,
  key block); it forms S, dP, dV, dK and dQ.  ``run_backward`` parameters: q,
  grad_out, out are bf16 [T, Hq, 128] THD tensors, lse fp32 [T, Hq], k and v
  bf16 [W, Hkv, 128] in a document workspace; it returns bf16 dq, dk, dv.
* ``msa_schedule`` page, ``MSABackwardSchedule``: ``row_ptr`` [Hi, rows+1] and
  ``q_indices`` [Hi, edge_capacity] form the key-block -> query CSR map whose
  entries are document-local query positions; ``scheduler_metadata`` columns
  are (index_head, row_linear, q_begin, q_count, document_ordinal,
  document_local_kblock); ``cu_seqlens`` gives compact document offsets;
  ``document_workspace_starts`` gives each document's K/V workspace row.
* ``msa_schedule`` page, ``rows_per_cta`` / ``chunk_map`` /
  ``grid_launch_bound`` and the constants ROWS_PER_CTA_SMALL = 4,
  ROWS_PER_CTA_LARGE = 64, ROWS_PER_CTA_SWITCH = 2400, SOFTMAX_SCALE =
  HEAD_DIM ** -0.5, QUERY_CHUNK = 8.

Attention being differentiated (the plain definition; the pages state the
topology, the text of the problem statement states the math):

  For query i at document-local position p_i of document d, q-head h, index
  head hi = h // G (G = Hq / Hi q-heads share one index/KV head), query chunk
  c = p_i // C, the attended keys are
      M(i, h) = { key j of document d : p_j <= p_i  and  p_j // B in sel[hi][g(d, c)] }
  s_ij = scale * q_i . k_j,  LSE_i = ln sum_{j in M} exp(s_ij),
  O_i = sum_{j in M} exp(s_ij - LSE_i) v_j.
  Backward with O, LSE and dO as supplied:
      D_i = dO_i . O_i,  P_ij = exp(s_ij - LSE_i) on M (0 elsewhere),
      dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i),
      dQ_i = scale * sum_j dS_ij k_j,
      dK_j = scale * sum_{i, h in group} dS_ij q_i,
      dV_j = sum_{i, h in group} P_ij dO_i.

The block scorer that produces ``sel`` (``pool_index``, ``block_scores``,
``select_topk``) follows a reading stated above its functions: the pages name
the scorer and its index dimension but not the score.

Readings where the pages are silent (each also listed in the design notes):
block size B and chunk C are parameters (the configs use B = 64, C = 8);
``sel`` is int32 [Hi, NC, K] of document-local block ids with -1 for an empty
slot, entries distinct and causal (b * B <= first position of the chunk);
LSE is the natural-log form; D uses the supplied bf16 O; K/V rows outside
every document get zero gradient.

Parity status: every function here is pinned by tests in ``tests/``
(finite differences, torch fp64 SDPA/autograd, hand-worked golden fixtures,
invariants and exhaustive sweeps); none is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

ROWS_PER_CTA_SMALL = 4
ROWS_PER_CTA_LARGE = 64
ROWS_PER_CTA_SWITCH = 2400


class InvalidSelection(ValueError):
    """A selection entry is out of range, non-causal or repeated in its chunk."""


# ---------------------------------------------------------------------------
# scalar formats
# ---------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, correctly rounded to nearest (ties to even).

    The two bf16 neighbours of x are formed from its float32 rounding (a bf16
    midpoint has 9 significant bits, so float32 keeps it exact) and the one
    nearer to x, measured in float64, is kept; ties go to the even mantissa.
    """
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    u = f.view(np.uint32)
    down = u & np.uint32(0xFFFF0000)                       # truncate toward zero
    up = down + np.uint32(0x10000)                         # next bf16 away from zero
    vd = down.view(np.float32).astype(np.float64)
    vu = up.view(np.float32).astype(np.float64)
    dd = np.abs(x - vd)
    du = np.abs(vu - x)
    even_down = ((down >> np.uint32(16)) & np.uint32(1)) == 0
    pick_up = (du < dd) | ((du == dd) & ~even_down)
    out = np.where(pick_up, up, down) >> np.uint32(16)
    return out.astype(np.uint16)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits): 2**(e - 7) for |x|
    in [2**e, 2**(e+1)); below the smallest normal, the subnormal spacing
    2**-133."""
    ax = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7.0)


# ---------------------------------------------------------------------------
# document layout
# ---------------------------------------------------------------------------

class DocLayout:
    """Per-document derived counts for packed (THD) sequences.

    cu_seqlens[d] .. cu_seqlens[d+1] are the compact token rows of document d;
    its key blocks are numbered r = blk_off[d] + b and its query chunks
    g = chunk_off[d] + c (global numbering, documents in order).
    """

    def __init__(self, cu_seqlens, block: int, chunk: int):
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        if cu.ndim != 1 or cu.size < 2 or cu[0] != 0 or np.any(np.diff(cu) <= 0):
            raise ValueError("cu_seqlens must start at 0 and increase strictly")
        self.cu = cu
        self.block = block
        self.chunk = chunk
        self.lengths = np.diff(cu)
        self.nb = -(-self.lengths // block)
        self.nc = -(-self.lengths // chunk)
        self.blk_off = np.concatenate([[0], np.cumsum(self.nb)[:-1]]).astype(np.int64)
        self.chunk_off = np.concatenate([[0], np.cumsum(self.nc)[:-1]]).astype(np.int64)
        self.NB = int(self.nb.sum())
        self.NC = int(self.nc.sum())
        self.num_docs = len(self.lengths)

    def chunk_positions(self, d: int, c: int) -> np.ndarray:
        lo = c * self.chunk
        return np.arange(lo, min(lo + self.chunk, int(self.lengths[d])), dtype=np.int64)

    def block_positions(self, d: int, b: int) -> np.ndarray:
        lo = b * self.block
        return np.arange(lo, min(lo + self.block, int(self.lengths[d])), dtype=np.int64)


def selected_blocks(sel: np.ndarray, lay: DocLayout, hi: int, d: int, c: int) -> list[int]:
    """The valid (non -1) document-local blocks chunk c of document d selected."""
    row = sel[hi, lay.chunk_off[d] + c]
    return sorted(int(b) for b in row if b >= 0)


def validate_selection(sel: np.ndarray, lay: DocLayout) -> None:
    """Raise InvalidSelection unless every entry is -1 or a distinct causal block."""
    sel = np.asarray(sel)
    if sel.ndim != 3 or sel.shape[1] != lay.NC:
        raise InvalidSelection(f"sel shape {sel.shape} does not match NC={lay.NC}")
    for d in range(lay.num_docs):
        for c in range(int(lay.nc[d])):
            first = c * lay.chunk
            for hi in range(sel.shape[0]):
                vals = [int(b) for b in sel[hi, lay.chunk_off[d] + c] if b != -1]
                if len(set(vals)) != len(vals):
                    raise InvalidSelection(f"repeated block in chunk {c} of doc {d}")
                for b in vals:
                    if b < 0 or b >= lay.nb[d] or b * lay.block > first:
                        raise InvalidSelection(f"block {b} invalid for chunk {c} of doc {d}")


# ---------------------------------------------------------------------------
# attention: dense-masked variant (one T x T mask per document and index head)
# ---------------------------------------------------------------------------

def attend_mask(sel, lay: DocLayout, hi: int, d: int) -> np.ndarray:
    """Boolean [len_d, len_d] mask: query position (row) attends key position (col)."""
    n = int(lay.lengths[d])
    m = np.zeros((n, n), dtype=bool)
    for p in range(n):
        blocks = set(selected_blocks(sel, lay, hi, d, p // lay.chunk))
        for j in range(p + 1):
            if j // lay.block in blocks:
                m[p, j] = True
    return m


def _heads(t_bits_or_f64):
    a = np.asarray(t_bits_or_f64)
    return bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def forward_dense(q, k, v, cu_seqlens, kv_doc_starts, sel, block, chunk, scale):
    """O [T, Hq, D] and LSE [T, Hq] in float64 (natural log), dense-masked."""
    q, k, v = _heads(q), _heads(k), _heads(v)
    lay = DocLayout(cu_seqlens, block, chunk)
    T, Hq, D = q.shape
    Hi = sel.shape[0]
    G = Hq // Hi
    o = np.zeros((T, Hq, D))
    lse = np.full((T, Hq), -np.inf)
    for d in range(lay.num_docs):
        t0, n, k0 = int(lay.cu[d]), int(lay.lengths[d]), int(kv_doc_starts[d])
        for hi in range(Hi):
            mask = attend_mask(sel, lay, hi, d)
            kd, vd = k[k0:k0 + n, hi], v[k0:k0 + n, hi]
            for h in range(hi * G, (hi + 1) * G):
                s = scale * (q[t0:t0 + n, h] @ kd.T)
                s = np.where(mask, s, -np.inf)
                mx = np.max(s, axis=1, keepdims=True)
                mx = np.where(np.isfinite(mx), mx, 0.0)
                e = np.where(mask, np.exp(s - mx), 0.0)
                ssum = e.sum(axis=1)
                with np.errstate(divide="ignore"):
                    lse[t0:t0 + n, h] = mx[:, 0] + np.log(ssum)
                p = np.where(mask, np.exp(s - lse[t0:t0 + n, h][:, None]), 0.0)
                o[t0:t0 + n, h] = p @ vd
    return o, lse


def backward_dense(q, k, v, o, do, lse, cu_seqlens, kv_doc_starts, sel, block, chunk, scale,
                   kv_rows=None):
    """dQ [T, Hq, D], dK/dV [W, Hkv, D] in float64 from supplied O, dO, LSE."""
    q, k, v, o, do = _heads(q), _heads(k), _heads(v), _heads(o), _heads(do)
    lse = np.asarray(lse, dtype=np.float64)
    lay = DocLayout(cu_seqlens, block, chunk)
    T, Hq, D = q.shape
    W = k.shape[0] if kv_rows is None else kv_rows
    Hi = sel.shape[0]
    G = Hq // Hi
    dq = np.zeros((T, Hq, D))
    dk = np.zeros((W, Hi, D))
    dv = np.zeros((W, Hi, D))
    delta = np.sum(do * o, axis=2)
    for d in range(lay.num_docs):
        t0, n, k0 = int(lay.cu[d]), int(lay.lengths[d]), int(kv_doc_starts[d])
        for hi in range(Hi):
            mask = attend_mask(sel, lay, hi, d)
            kd, vd = k[k0:k0 + n, hi], v[k0:k0 + n, hi]
            for h in range(hi * G, (hi + 1) * G):
                qh, doh = q[t0:t0 + n, h], do[t0:t0 + n, h]
                s = scale * (qh @ kd.T)
                p = np.where(mask, np.exp(s - lse[t0:t0 + n, h][:, None]), 0.0)
                dp = doh @ vd.T
                ds = p * (dp - delta[t0:t0 + n, h][:, None])
                dq[t0:t0 + n, h] = scale * (ds @ kd)
                dk[k0:k0 + n, hi] += scale * (ds.T @ qh)
                dv[k0:k0 + n, hi] += p.T @ doh
    return dq, dk, dv


# ---------------------------------------------------------------------------
# attention: blocked variant (gathers only the selected key blocks per chunk)
# ---------------------------------------------------------------------------

def _gather(a, rows, cols) -> np.ndarray:
    """a[rows][:, cols] as float64 (bf16 bit patterns are decoded exactly)."""
    return _heads(np.asarray(a)[rows][:, cols])


def _chunk_keys(sel, lay: DocLayout, hi: int, d: int, c: int) -> np.ndarray:
    blocks = selected_blocks(sel, lay, hi, d, c)
    if not blocks:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([lay.block_positions(d, b) for b in blocks])


def chunk_forward(q, k, v, lay, kv_doc_starts, sel, hi, d, c, G, scale):
    """Forward for one (document, index head, query chunk).

    Returns (query positions, O [G, nq, D], LSE [G, nq]) for the q-heads
    hi*G .. hi*G+G-1 of that chunk, in float64.
    """
    qp = lay.chunk_positions(d, c)
    kp = _chunk_keys(sel, lay, hi, d, c)
    t0, k0 = int(lay.cu[d]), int(kv_doc_starts[d])
    qc = _gather(q, t0 + qp, slice(hi * G, (hi + 1) * G)).transpose(1, 0, 2)   # [G, nq, D]
    D = qc.shape[2]
    if kp.size == 0:
        return qp, np.zeros((G, qp.size, D)), np.full((G, qp.size), -np.inf)
    kc = _gather(k, k0 + kp, hi)                                               # [nk, D]
    vc = _gather(v, k0 + kp, hi)
    mask = kp[None, :] <= qp[:, None]                                          # [nq, nk]
    s = scale * (qc @ kc.T)                                                   # [G, nq, nk]
    s = np.where(mask[None], s, -np.inf)
    mx = np.max(s, axis=2, keepdims=True)
    mx = np.where(np.isfinite(mx), mx, 0.0)
    e = np.where(mask[None], np.exp(s - mx), 0.0)
    with np.errstate(divide="ignore"):
        lse = mx[..., 0] + np.log(e.sum(axis=2))
    p = np.where(mask[None], np.exp(s - lse[..., None]), 0.0)
    return qp, p @ vc, lse


def chunk_backward(q, k, v, do, oc, lc, lay, kv_doc_starts, sel, hi, d, c, G, scale):
    """Backward contributions of one (document, index head, query chunk).

    ``oc`` [G, nq, D] and ``lc`` [G, nq] are that chunk's O and LSE.  Returns
    (query positions, dQ [G, nq, D], key positions, dK part [nk, D], dV part
    [nk, D]); the key parts are this chunk's share of the sums over queries.
    """
    qp = lay.chunk_positions(d, c)
    kp = _chunk_keys(sel, lay, hi, d, c)
    t0, k0 = int(lay.cu[d]), int(kv_doc_starts[d])
    hs = slice(hi * G, (hi + 1) * G)
    qc = _gather(q, t0 + qp, hs).transpose(1, 0, 2)
    D = qc.shape[2]
    if kp.size == 0:
        z = np.zeros((0, D))
        return qp, np.zeros((G, qp.size, D)), kp, z, z
    doc_ = _gather(do, t0 + qp, hs).transpose(1, 0, 2)
    oc = np.asarray(oc, dtype=np.float64)
    lc = np.asarray(lc, dtype=np.float64)
    kc = _gather(k, k0 + kp, hi)
    vc = _gather(v, k0 + kp, hi)
    mask = (kp[None, :] <= qp[:, None])[None]
    s = scale * (qc @ kc.T)                                                   # [G, nq, nk]
    p = np.where(mask, np.exp(s - lc[..., None]), 0.0)
    dp = doc_ @ vc.T
    delta = np.sum(doc_ * oc, axis=2)
    ds = p * (dp - delta[..., None])
    dq = scale * (ds @ kc)
    n = G * qp.size                                                           # sum over (head, query)
    dk = scale * (ds.reshape(n, -1).T @ qc.reshape(n, D))
    dv = p.reshape(n, -1).T @ doc_.reshape(n, D)
    return qp, dq, kp, dk, dv


def forward_blocked(q, k, v, cu_seqlens, kv_doc_starts, sel, block, chunk, scale):
    """Same result as forward_dense, computed per chunk over its selected blocks."""
    lay = DocLayout(cu_seqlens, block, chunk)
    T, Hq, D = np.asarray(q).shape
    Hi = sel.shape[0]
    G = Hq // Hi
    o = np.zeros((T, Hq, D))
    lse = np.full((T, Hq), -np.inf)
    for d in range(lay.num_docs):
        t0 = int(lay.cu[d])
        for hi in range(Hi):
            for c in range(int(lay.nc[d])):
                qp, oc, lc = chunk_forward(q, k, v, lay, kv_doc_starts, sel, hi, d, c, G, scale)
                o[t0 + qp, hi * G:(hi + 1) * G] = oc.transpose(1, 0, 2)
                lse[t0 + qp, hi * G:(hi + 1) * G] = lc.T
    return o, lse


def backward_blocked(q, k, v, o, do, lse, cu_seqlens, kv_doc_starts, sel, block, chunk, scale,
                     kv_rows=None):
    """Same result as backward_dense, accumulated chunk by chunk."""
    lay = DocLayout(cu_seqlens, block, chunk)
    T, Hq, D = np.asarray(q).shape
    W = np.asarray(k).shape[0] if kv_rows is None else kv_rows
    Hi = sel.shape[0]
    G = Hq // Hi
    lse = np.asarray(lse, dtype=np.float64)
    dq = np.zeros((T, Hq, D))
    dk = np.zeros((W, Hi, D))
    dv = np.zeros((W, Hi, D))
    for d in range(lay.num_docs):
        t0, k0 = int(lay.cu[d]), int(kv_doc_starts[d])
        for hi in range(Hi):
            hs = slice(hi * G, (hi + 1) * G)
            for c in range(int(lay.nc[d])):
                rows = t0 + lay.chunk_positions(d, c)
                oc = _gather(o, rows, hs).transpose(1, 0, 2)
                lc = lse[rows][:, hs].T
                qp, dqc, kp, dkc, dvc = chunk_backward(q, k, v, do, oc, lc, lay, kv_doc_starts,
                                                       sel, hi, d, c, G, scale)
                dq[t0 + qp, hs] = dqc.transpose(1, 0, 2)
                # key positions of one chunk are distinct, so fancy-index add is exact
                dk[k0 + kp, hi] += dkc
                dv[k0 + kp, hi] += dvc
    return dq, dk, dv


# ---------------------------------------------------------------------------
# sampled outputs for workloads too large for a full oracle pass
# ---------------------------------------------------------------------------

def _stored(oc, lc):
    """O and LSE as the forward stores them: O rounded to bf16, LSE to fp32."""
    return bf16_to_f64(f64_to_bf16(oc)), np.asarray(lc, np.float64).astype(np.float32).astype(np.float64)


def sampled_query_grads(q, k, v, do, cu_seqlens, kv_doc_starts, sel, block, chunk, scale,
                        picks):
    """dQ of sampled (document, index head, chunk) triples.

    O and LSE of those queries are recomputed here by ``chunk_forward`` and
    stored-rounded, so nothing is taken from the device.  Returns a list of
    (token rows, head slice, dQ [nq, G, D]).
    """
    lay = DocLayout(cu_seqlens, block, chunk)
    G = np.asarray(q).shape[1] // sel.shape[0]
    out = []
    for d, hi, c in picks:
        _, oc, lc = chunk_forward(q, k, v, lay, kv_doc_starts, sel, hi, d, c, G, scale)
        oc, lc = _stored(oc, lc)
        qp, dqc, _, _, _ = chunk_backward(q, k, v, do, oc, lc, lay, kv_doc_starts, sel,
                                          hi, d, c, G, scale)
        out.append((int(lay.cu[d]) + qp, slice(hi * G, (hi + 1) * G), dqc.transpose(1, 0, 2)))
    return out


def sampled_key_grads(q, k, v, do, cu_seqlens, kv_doc_starts, sel, block, chunk, scale, picks):
    """dK/dV of sampled (document, index head, key block) triples.

    Every chunk of the document that selected the block contributes; its O
    and LSE are recomputed by ``chunk_forward`` and stored-rounded first.
    Returns a list of (K/V rows, index head, dK [nk, D], dV [nk, D]).
    """
    lay = DocLayout(cu_seqlens, block, chunk)
    G = np.asarray(q).shape[1] // sel.shape[0]
    out = []
    for d, hi, b in picks:
        kp_blk = lay.block_positions(d, b)
        k0 = int(kv_doc_starts[d])
        D = np.asarray(q).shape[2]
        dk = np.zeros((kp_blk.size, D))
        dv = np.zeros_like(dk)
        for c in range(int(lay.nc[d])):
            if b not in selected_blocks(sel, lay, hi, d, c):
                continue
            _, oc, lc = chunk_forward(q, k, v, lay, kv_doc_starts, sel, hi, d, c, G, scale)
            oc, lc = _stored(oc, lc)
            _, _, kp, dkc, dvc = chunk_backward(q, k, v, do, oc, lc, lay, kv_doc_starts,
                                                sel, hi, d, c, G, scale)
            idx = np.searchsorted(kp, kp_blk)
            dk += dkc[idx]
            dv += dvc[idx]
        out.append((k0 + kp_blk, hi, dk, dv))
    return out


# ---------------------------------------------------------------------------
# block scorer and top-k selection (produces sel)
# ---------------------------------------------------------------------------
#
# The msa_bindings page names a scorer launcher (MSAKernels.fmha_sm100) among
# the entry points and the msa_schedule page fixes INDEX_DIM = 128 per index
# head, but neither says how a key block is scored.  The reading used here:
#   * pooled index query of query chunk c:  the mean of the chunk's tokens'
#     index queries; pooled index key of key block b: the mean of the block's
#     tokens' index keys (both within the document; a partial last chunk or
#     block averages the tokens it has);
#   * each mean is an fp32 sum over the tokens in order, divided by the token
#     count in fp32, and stored rounded to bf16, like every other tensor;
#   * score(c, b) = the fp32 dot product of the two pooled bf16 vectors,
#     accumulated over the index dims in ascending order (every product of two
#     bf16 values is exact in fp32, so this is a fixed sequence of rounded
#     fp32 additions);
#   * the diagonal block b = (first position of c) // B is always selected
#     first; the other K - 1 slots take the causal blocks b < diagonal with the
#     highest scores, a tie going to the lower block; the row of sel lists the
#     diagonal, then those blocks by descending score, then -1 pads.

def pool_index(x_bits, cu_seqlens, size: int) -> np.ndarray:
    """Mean over consecutive groups of ``size`` tokens of each document.

    x_bits: bf16 bits [T, Hi, D].  Returns bf16 bits [Hi, n_groups, D], groups
    numbered document by document (so chunks for size = C, blocks for size = B).
    """
    x = bf16_to_f64(np.asarray(x_bits)).astype(np.float32)        # exact
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, Hi, D = x.shape
    out = []
    for d in range(len(cu) - 1):
        t0, n = int(cu[d]), int(cu[d + 1] - cu[d])
        for g0 in range(0, n, size):
            rows = range(t0 + g0, t0 + min(g0 + size, n))
            acc = np.zeros((Hi, D), dtype=np.float32)
            for t in rows:                                        # fp32 adds in token order
                acc = acc + x[t]
            mean = acc / np.float32(len(rows))                    # fp32 division, correctly rounded
            out.append(f64_to_bf16(mean.astype(np.float64)))
    return np.stack(out, axis=1)


def block_scores(qpool_bits, kpool_bits) -> np.ndarray:
    """fp32 scores [..., nq, nk] of pooled queries [..., nq, D] against pooled
    keys [..., nk, D] (bf16 bits), accumulated over D in ascending order."""
    qp = bf16_to_f64(np.asarray(qpool_bits)).astype(np.float32)
    kp = bf16_to_f64(np.asarray(kpool_bits)).astype(np.float32)
    acc = np.zeros(qp.shape[:-1] + (kp.shape[-2],), dtype=np.float32)
    for i in range(qp.shape[-1]):
        acc = acc + qp[..., :, None, i] * kp[..., None, :, i]     # exact products, rounded sums
    return acc


def select_topk(q_index, k_index, cu_seqlens, block: int, chunk: int, topk: int) -> np.ndarray:
    """sel int32 [Hi, NC, K] from index projections q_index, k_index (bf16 bits
    [T, Hi, D]) by the scorer reading above."""
    lay = DocLayout(cu_seqlens, block, chunk)
    qpool = pool_index(q_index, cu_seqlens, chunk)                 # [Hi, NC, D]
    kpool = pool_index(k_index, cu_seqlens, block)                 # [Hi, NB, D]
    Hi = qpool.shape[0]
    sel = np.full((Hi, lay.NC, topk), -1, dtype=np.int32)
    for d in range(lay.num_docs):
        g0, r0 = int(lay.chunk_off[d]), int(lay.blk_off[d])
        nc, nb = int(lay.nc[d]), int(lay.nb[d])
        for hi in range(Hi):
            sc = block_scores(qpool[hi, g0:g0 + nc], kpool[hi, r0:r0 + nb])   # [nc, nb]
            for c in range(nc):
                diag = (c * chunk) // block
                ranked = sorted(range(diag), key=lambda b: (-float(sc[c, b]), b))[:topk - 1]
                row = [diag] + ranked
                sel[hi, g0 + c, :len(row)] = row
    return sel


# ---------------------------------------------------------------------------
# index tables: key-block -> query CSR, task rows, CTA walk
# ---------------------------------------------------------------------------

def build_k2q(sel, cu_seqlens, block, chunk, validate=True):
    """CSR of the key-block -> query map, one row set per index head.

    Row r = blk_off[d] + b lists, in ascending order, every document-local
    query position p of document d whose chunk p // C selected block b.
    Returns (row_ptr int32 [Hi, NB + 1], q_indices int32 [Hi, E_max]) where
    E_max is the largest per-head edge count (tail entries of shorter heads
    are -1).  Built as a sort of the (head, row, position) triples.
    """
    sel = np.asarray(sel)
    lay = DocLayout(cu_seqlens, block, chunk)
    if validate:
        validate_selection(sel, lay)
    Hi = sel.shape[0]
    heads, rows, pos = [], [], []
    for d in range(lay.num_docs):
        n = int(lay.lengths[d])
        p = np.arange(n, dtype=np.int64)
        g = lay.chunk_off[d] + p // chunk                                  # chunk of each query
        for hi in range(Hi):
            s = sel[hi, g]                                                 # [n, K]
            valid = s >= 0
            pp = np.broadcast_to(p[:, None], s.shape)[valid]
            rr = lay.blk_off[d] + s[valid].astype(np.int64)
            heads.append(np.full(pp.size, hi, dtype=np.int64))
            rows.append(rr)
            pos.append(pp)
    heads = np.concatenate(heads) if heads else np.zeros(0, np.int64)
    rows = np.concatenate(rows) if rows else np.zeros(0, np.int64)
    pos = np.concatenate(pos) if pos else np.zeros(0, np.int64)
    order = np.lexsort((pos, rows, heads))
    heads, rows, pos = heads[order], rows[order], pos[order]
    counts = np.zeros((Hi, lay.NB), dtype=np.int64)
    np.add.at(counts, (heads, rows), 1)
    row_ptr = np.zeros((Hi, lay.NB + 1), dtype=np.int64)
    row_ptr[:, 1:] = np.cumsum(counts, axis=1)
    e_max = int(row_ptr[:, -1].max()) if Hi else 0
    q_indices = np.full((Hi, e_max), -1, dtype=np.int64)
    for hi in range(Hi):
        m = heads == hi
        q_indices[hi, :m.sum()] = pos[m]
    return row_ptr.astype(np.int32), q_indices.astype(np.int32)


def build_tasks(row_ptr, q_indices, cu_seqlens, block, chunk, tile_chunks=0, key_tile=64):
    """Task rows of the KV-parallel backward.

    Each CSR row's entries are cut into consecutive groups of ``chunk``
    entries; a group is one task row (at most C queries x the q-heads of the
    index head, one 128-row tile at C = 8, G = 16).  Tasks are ordered by
    index head, then query tile (global chunk index of the group's first
    query // tile_chunks; a single tile when tile_chunks is 0), then key-block
    row, then CSR offset.

    Key tiles (not in the pages; the kernel's tile is 64 keys): a block wider
    than ``key_tile`` keys is cut into block // key_tile tiles, and a group
    becomes one task per tile whose first key is at or before the group's last
    query (the tiles after it would be fully masked).  Row r, tile h is task
    row r * (block // key_tile) + h and its document-local kblock is counted
    in key tiles (b * (block // key_tile) + h); the order is (index head,
    query tile, that task row, CSR offset).  Blocks of at most ``key_tile``
    keys are one tile, so the rows and kblocks are the CSR's.

    Returns task_meta int32 [n, 6] with columns (index_head, row_linear,
    q_begin, q_count, document_ordinal, document_local_kblock), q_begin being
    the CSR offset of the task's first entry; task_q_rows int32 [n, C]
    (compact token row, -1 pad) and task_q_pos int32 [n, C] (document-local
    position, -1 pad).
    """
    nh = 1
    if block > key_tile:
        assert block % key_tile == 0, "a block must be a whole number of key tiles"
        nh = block // key_tile
    lay = DocLayout(cu_seqlens, block, chunk)
    row_ptr = np.asarray(row_ptr, dtype=np.int64)
    q_indices = np.asarray(q_indices, dtype=np.int64)
    Hi = row_ptr.shape[0]
    doc_of_row = np.repeat(np.arange(lay.num_docs), lay.nb)
    cols = []
    for hi in range(Hi):
        rp = row_ptr[hi]
        counts = np.diff(rp)
        r_of_entry = np.repeat(np.arange(lay.NB), counts)
        j = np.arange(int(rp[-1]), dtype=np.int64)
        k_in_row = j - rp[r_of_entry]
        starts = j[k_in_row % chunk == 0]                     # first entry of each group
        r = r_of_entry[starts]
        cnt = np.minimum(starts + chunk, rp[r + 1]) - starts
        d = doc_of_row[r]
        b = r - lay.blk_off[d]
        g = lay.chunk_off[d] + q_indices[hi, starts] // chunk
        tile = g // tile_chunks if tile_chunks > 0 else np.zeros_like(g)
        last = q_indices[hi, starts + cnt - 1]                # the group's last query
        for h in range(nh):
            reach = b * block + h * key_tile <= last
            cols.append((np.full(int(reach.sum()), hi), tile[reach], r[reach] * nh + h, starts[reach],
                         cnt[reach], d[reach], b[reach] * nh + h))
    hi_, tile, r, starts, cnt, d, b = (np.concatenate(c) for c in zip(*cols))
    order = np.lexsort((starts, r, tile, hi_))
    hi_, r, starts, cnt, d, b = (a[order] for a in (hi_, r, starts, cnt, d, b))
    n = starts.size
    meta = np.stack([hi_, r, starts, cnt, d, b], axis=1).astype(np.int32)
    slot = np.arange(chunk)[None, :]
    valid = slot < cnt[:, None]
    src = np.where(valid, starts[:, None] + slot, 0)
    pos = q_indices[hi_[:, None], src]
    q_pos = np.where(valid, pos, -1).astype(np.int32)
    q_rows = np.where(valid, lay.cu[d][:, None] + pos, -1).astype(np.int32)
    return meta.reshape(n, 6), q_rows.reshape(n, chunk), q_pos.reshape(n, chunk)


def plan_forward(sel, cu_seqlens, block: int, chunk: int):
    """Forward work plan (the planner launcher of the msa_bindings page,
    MSAKernels.fmha_sm100_plan; scheduler_metadata and work_count of the
    msa_schedule page).

    One work item per (index head, query chunk), in the scheduler_metadata
    column order (index_head, row_linear, q_begin, q_count, document_ordinal,
    document_local_kblock) read for query-chunk items: row_linear is the global
    chunk, q_begin its first token row, q_count its token count, and
    document_local_kblock the document-local key block holding its first query
    (its diagonal block).  Items are ordered longest first: descending number
    of selected blocks, ties in (index head, chunk) order; items that select no
    block come last.  Returns (meta int32 [Hi * NC, 6], work_count = number of
    items that select at least one block).
    """
    sel = np.asarray(sel)
    lay = DocLayout(cu_seqlens, block, chunk)
    Hi = sel.shape[0]
    items = []
    for hi in range(Hi):
        for d in range(lay.num_docs):
            for c in range(int(lay.nc[d])):
                g = int(lay.chunk_off[d]) + c
                nsel = int((sel[hi, g] >= 0).sum())
                q0 = c * chunk
                row = (hi, g, int(lay.cu[d]) + q0, min(chunk, int(lay.lengths[d]) - q0), d, q0 // block)
                items.append((nsel, row))
    # stable: sorted() keeps the (index head, chunk) order among equal counts
    items = sorted(items, key=lambda it: -it[0])
    meta = np.array([row for _, row in items], dtype=np.int32).reshape(-1, 6)
    work = sum(1 for n, _ in items if n > 0)
    return meta, work


def rows_per_cta(num_rows: int) -> int:
    """Walk length: ROWS_PER_CTA_SMALL below ROWS_PER_CTA_SWITCH rows, else LARGE."""
    return ROWS_PER_CTA_SMALL if num_rows < ROWS_PER_CTA_SWITCH else ROWS_PER_CTA_LARGE


def chunk_map(num_rows: int, rows_per: int, num_sms: int):
    """(num_full_ctas, tail_rows, grid_ctas): full CTAs of rows_per rows each,
    then the remaining tail rows spread one per CTA over at most num_sms CTAs."""
    full = num_rows // rows_per
    tail = num_rows - full * rows_per
    return full, tail, full + min(tail, num_sms)


def walk_units(num_rows: int, num_sms: int):
    """Rows of each walk unit (CTA) in order: full units take consecutive
    rows_per rows; tail unit j takes rows full*R + j, full*R + j + S, ..."""
    R = rows_per_cta(num_rows)
    full, tail, grid = chunk_map(num_rows, R, num_sms)
    units = [list(range(i * R, (i + 1) * R)) for i in range(full)]
    ntail = grid - full
    for j in range(ntail):
        units.append(list(range(full * R + j, num_rows, ntail)))
    return units


def grid_launch_bound(capacity: int, num_sms: int) -> int:
    """max over n in [0, capacity] of chunk_map(n, rows_per_cta(n), S)[2]."""
    n = np.arange(capacity + 1, dtype=np.int64)
    R = np.where(n < ROWS_PER_CTA_SWITCH, ROWS_PER_CTA_SMALL, ROWS_PER_CTA_LARGE)
    full = n // R
    tail = n - full * R
    return int(np.max(full + np.minimum(tail, num_sms)))
