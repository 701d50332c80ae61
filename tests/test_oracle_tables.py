"""Pins of the oracle's index tables: hand-worked golden, invariants, brute force,
and an exhaustive sweep of the CTA-walk rule (msa_schedule page: rows_per_cta,
chunk_map, grid_launch_bound; "the CPU tests exhaust the walk rule")."""
import json
import os

import numpy as np
import pytest

from oracle import msa_oracle as O
from block_sparse_top_attn_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    return json.load(open(os.path.join(GOLD, "k2q_tasks_two_docs.json")))


def test_k2q_and_tasks_match_hand_worked_golden():
    g = _golden()
    sel = np.array(g["sel"], np.int32)
    rp, qi = O.build_k2q(sel, g["cu_seqlens"], g["block"], g["chunk"])
    assert rp.tolist() == g["row_ptr"]
    assert qi.tolist() == g["q_indices"]
    m, qr, qp = O.build_tasks(rp, qi, g["cu_seqlens"], g["block"], g["chunk"])
    assert m.tolist() == g["tasks_untiled"]["meta"]
    assert qp.tolist() == g["tasks_untiled"]["q_pos"]
    assert qr.tolist() == g["tasks_untiled"]["q_rows"]
    m2, _, _ = O.build_tasks(rp, qi, g["cu_seqlens"], g["block"], g["chunk"],
                             tile_chunks=g["tasks_tile2"]["tile_chunks"])
    assert m2.tolist() == g["tasks_tile2"]["meta"]


def _brute_rows(sel, lay):
    """Brute force: for every (head, row), scan every query of the document."""
    Hi = sel.shape[0]
    rows = {}
    for hi in range(Hi):
        for d in range(lay.num_docs):
            for b in range(int(lay.nb[d])):
                lst = []
                for p in range(int(lay.lengths[d])):
                    if b in sel[hi, lay.chunk_off[d] + p // lay.chunk]:
                        lst.append(p)
                rows[(hi, int(lay.blk_off[d]) + b)] = lst
    return rows


@pytest.mark.parametrize("seed", range(6))
def test_k2q_equals_brute_force_inversion(seed):
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(1, 300, size=int(rng.integers(1, 5)))]
    pb = W.make_problem(lengths=lengths, num_index_heads=2, topk=5, policy="diag_uniform", seed=seed,
                        values=False, block=16, chunk=8)
    # scatter -1 pads to random slots
    sel = pb.sel.copy()
    for hi in range(sel.shape[0]):
        for g in range(sel.shape[1]):
            sel[hi, g] = sel[hi, g][rng.permutation(sel.shape[2])]
    lay = O.DocLayout(pb.cu_seqlens, 16, 8)
    rp, qi = O.build_k2q(sel, pb.cu_seqlens, 16, 8)
    brute = _brute_rows(sel, lay)
    for (hi, r), lst in brute.items():
        assert qi[hi, rp[hi, r]:rp[hi, r + 1]].tolist() == lst
    # invariant: edges = sum over chunks of (#valid slots x chunk length)
    for hi in range(sel.shape[0]):
        tot = 0
        for d in range(lay.num_docs):
            for c in range(int(lay.nc[d])):
                tot += int((sel[hi, lay.chunk_off[d] + c] >= 0).sum()) * lay.chunk_positions(d, c).size
        assert rp[hi, -1] == tot


@pytest.mark.parametrize("tile", [0, 1, 3, 16])
def test_tasks_are_chunks_and_cover_every_edge_once(tile):
    pb = W.make_problem(lengths=[200, 77, 130], num_index_heads=3, topk=4, policy="diag_uniform", seed=9,
                        values=False, block=16, chunk=8)
    lay = O.DocLayout(pb.cu_seqlens, 16, 8)
    rp, qi = O.build_k2q(pb.sel, pb.cu_seqlens, 16, 8)
    m, qr, qp = O.build_tasks(rp, qi, pb.cu_seqlens, 16, 8, tile_chunks=tile)
    seen = set()
    keys = []
    for t in range(m.shape[0]):
        hi, r, s, cnt, d, b = (int(x) for x in m[t])
        pos = qp[t, :cnt]
        c = int(pos[0]) // 8
        # one whole chunk: consecutive positions, all of chunk c
        assert pos.tolist() == lay.chunk_positions(d, c).tolist()
        assert (qp[t, cnt:] == -1).all() and (qr[t, cnt:] == -1).all()
        assert (qr[t, :cnt] == pb.cu_seqlens[d] + pos).all()
        assert r == lay.blk_off[d] + b and b in pb.sel[hi, lay.chunk_off[d] + c]
        assert qi[hi, s:s + cnt].tolist() == pos.tolist()
        assert (hi, d, c, b) not in seen
        seen.add((hi, d, c, b))
        g = int(lay.chunk_off[d]) + c
        keys.append((hi, g // tile if tile else 0, r, s))
    assert keys == sorted(keys)
    assert len(seen) == int((pb.sel >= 0).sum())


def test_walk_rule_threshold_and_constants():
    assert O.rows_per_cta(0) == 4 and O.rows_per_cta(2399) == 4
    assert O.rows_per_cta(2400) == 64 and O.rows_per_cta(10 ** 7) == 64


@pytest.mark.parametrize("sms", [1, 7, 132, 148, 152])
def test_walk_rule_exhaustive(sms):
    cap = 20000
    bound = O.grid_launch_bound(cap, sms)
    worst = 0
    for n in range(cap + 1):
        R = O.rows_per_cta(n)
        full, tail, grid = O.chunk_map(n, R, sms)
        assert full * R + tail == n and 0 <= tail < R
        assert grid <= n // R + sms
        worst = max(worst, grid)
    assert bound == worst
    # cover-once on a sample of counts (the unit lists are explicit)
    for n in list(range(0, 300)) + [2399, 2400, 2401, 4095, 9999, 19999]:
        units = O.walk_units(n, sms)
        flat = sorted(x for u in units for x in u)
        assert flat == list(range(n))
        assert len(units) == O.chunk_map(n, O.rows_per_cta(n), sms)[2]


@pytest.mark.parametrize("bad", ["range", "causal", "dup"])
def test_invalid_selection_is_rejected(bad):
    pb = W.make_problem(lengths=[100], num_index_heads=1, topk=3, policy="diag_uniform", seed=1, values=False,
                        block=16, chunk=8)
    sel = pb.sel.copy()
    if bad == "range":
        sel[0, 12, 0] = 7                 # doc has 7 blocks: 0..6
    elif bad == "causal":
        sel[0, 3, 0] = 2                  # chunk 3 starts at 24 < 2 * 16... block 2 starts at 32
    else:
        sel[0, 10, :2] = [1, 1]
    with pytest.raises(O.InvalidSelection):
        O.build_k2q(sel, pb.cu_seqlens, 16, 8)


@pytest.mark.parametrize("name,tasks", [("tiny", 208), ("single8k", 61696), ("long128k", 4162560),
                                        ("zipf64k", 493568)])
def test_named_workload_task_counts(name, tasks):
    pb = W.make_problem(name, values=False)
    # one task per valid (index head, chunk, block) selection entry
    assert int((pb.sel >= 0).sum()) == tasks


def test_forward_plan_orders_longest_first_and_counts_nonempty_items():
    """The forward plan is a permutation of every (index head, chunk) item,
    ordered by descending selected-block count with ties in (head, chunk)
    order (checked against numpy's lexsort), empty items last, and work_count
    counts the non-empty ones; each row's columns follow from the layout."""
    from block_sparse_top_attn_gb300 import workloads as W
    pb = W.make_problem(lengths=[200, 77, 130, 1, 9, 513], num_index_heads=2, topk=5, policy="diag_uniform",
                        seed=3, values=False)
    sel = pb.sel.copy()
    sel[1, 10:14] = -1                                  # a few chunks that select nothing
    meta, work = O.plan_forward(sel, pb.cu_seqlens, pb.block, pb.chunk)
    lay = O.DocLayout(pb.cu_seqlens, pb.block, pb.chunk)
    Hi, NC = sel.shape[:2]
    nsel = (sel >= 0).sum(axis=2)                       # [Hi, NC]
    hh, gg = np.meshgrid(np.arange(Hi), np.arange(NC), indexing="ij")
    order = np.lexsort((gg.ravel(), hh.ravel(), -nsel.ravel()))
    np.testing.assert_array_equal(meta[:, 0], hh.ravel()[order])
    np.testing.assert_array_equal(meta[:, 1], gg.ravel()[order])
    assert work == int((nsel > 0).sum()) == Hi * NC - 4
    assert (nsel[meta[work:, 0], meta[work:, 1]] == 0).all()
    for hi, g, q_begin, q_count, d, kb in meta:
        c = g - lay.chunk_off[d]
        assert lay.chunk_off[d] <= g < lay.chunk_off[d] + lay.nc[d]
        assert q_begin == lay.cu[d] + c * pb.chunk
        assert q_count == min(pb.chunk, lay.lengths[d] - c * pb.chunk)
        assert kb == c * pb.chunk // pb.block


@pytest.mark.parametrize("block,key_tile", [(32, 16), (128, 64)])
def test_key_tiles_cover_every_attended_pair_once(block, key_tile):
    # Blocks wider than the kernel's key tile become one task per reached tile:
    # brute force over (head, document, query, key) pairs that the selection
    # and the causal mask admit, each in exactly one task, and no task whose
    # tile no query of the group reaches.
    lengths = [300, 129, 64] if block == 128 else [100, 33, 70]
    pb = W.make_problem(lengths=lengths, num_index_heads=2, topk=3, policy="diag_uniform", seed=4,
                        values=False, block=block, chunk=8)
    lay = O.DocLayout(pb.cu_seqlens, block, 8)
    rp, qi = O.build_k2q(pb.sel, pb.cu_seqlens, block, 8)
    tile_chunks = 2
    m, qr, qp = O.build_tasks(rp, qi, pb.cu_seqlens, block, 8, tile_chunks=tile_chunks, key_tile=key_tile)
    nh = block // key_tile
    want = set()
    for hi in range(2):
        for d in range(lay.num_docs):
            n = int(lay.lengths[d])
            for p in range(n):
                for b in pb.sel[hi, lay.chunk_off[d] + p // 8]:
                    if b >= 0:
                        want.update((hi, d, p, key) for key in range(b * block, min((b + 1) * block, p + 1)))
    got, order = [], []
    for t in range(m.shape[0]):
        hi, rt, s, cnt, d, kb = (int(x) for x in m[t])
        assert rt == (int(lay.blk_off[d]) + kb // nh) * nh + kb % nh
        n = int(lay.lengths[d])
        pairs = [(hi, d, int(p), key) for p in qp[t, :cnt]
                 for key in range(kb * key_tile, min((kb + 1) * key_tile, n)) if key <= p]
        assert pairs, "a task whose key tile no query of the group reaches"
        got.extend(pairs)
        order.append((hi, (int(lay.chunk_off[d]) + int(qp[t, 0]) // 8) // tile_chunks, rt, s))
    assert len(got) == len(set(got))
    assert set(got) == want
    assert order == sorted(order)
