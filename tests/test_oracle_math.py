"""Pins of the fp64 oracle's attention arithmetic against things other than itself.

* central finite differences of L = sum(dO * O(Q, K, V)) (backward vs forward);
* torch's scaled_dot_product_attention in fp64 on CPU (a library routine),
  with is_causal=True when top-k covers every causal block (textbook causal
  attention with grouped KV heads), and with an explicit boolean mask
  expanded from the selection for sparse cases, forward and autograd;
* the hand-worked attended key sets of tests/golden/k2q_tasks_two_docs.json;
* closed forms: a query that sees only one key has dS = 0, so dQ = 0 and
  dV of that key receives P = 1;
* the dense-masked and blocked oracles agree to rounding.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand_sel(rng, lengths, Hi, K, B, C, full=False):
    nc = [-(-n // C) for n in lengths]
    sel = np.full((Hi, sum(nc), K), -1, np.int32)
    g = 0
    for n, ncd in zip(lengths, nc):
        for c in range(ncd):
            allowed = np.arange(0, (c * C) // B + 1)
            for hi in range(Hi):
                if full:
                    pick = allowed
                else:
                    k = int(rng.integers(1, min(K, allowed.size) + 1))
                    pick = rng.choice(allowed, size=k, replace=False)
                slots = rng.permutation(K)[:pick.size]
                sel[hi, g + c, slots] = pick
        g += ncd
    return sel


def _problem(seed, lengths, Hi, G, D, K, B, C, full=False, aligned=False):
    rng = np.random.default_rng(seed)
    sel = _rand_sel(rng, lengths, Hi, K, B, C, full)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    if aligned:
        pad = [-(-n // 16) * 16 for n in lengths]
        kvs = np.concatenate([[0], np.cumsum(pad)[:-1]]).astype(np.int32)
        W = int(sum(pad))
    else:
        kvs = cu[:-1].copy()
        W = int(cu[-1])
    T = int(cu[-1])
    q = rng.standard_normal((T, Hi * G, D))
    k = rng.standard_normal((W, Hi, D))
    v = rng.standard_normal((W, Hi, D))
    do = rng.standard_normal((T, Hi * G, D))
    return dict(q=q, k=k, v=v, do=do, cu=cu, kvs=kvs, sel=sel, B=B, C=C, scale=D ** -0.5, W=W)


def _loss(p, q, k, v):
    o, _ = O.forward_dense(q, k, v, p["cu"], p["kvs"], p["sel"], p["B"], p["C"], p["scale"])
    return float(np.sum(p["do"] * o))


def test_finite_differences_match_backward():
    p = _problem(1, [21, 16], Hi=2, G=2, D=8, K=2, B=8, C=4)
    o, lse = O.forward_dense(p["q"], p["k"], p["v"], p["cu"], p["kvs"], p["sel"], p["B"], p["C"], p["scale"])
    dq, dk, dv = O.backward_dense(p["q"], p["k"], p["v"], o, p["do"], lse, p["cu"], p["kvs"], p["sel"],
                                  p["B"], p["C"], p["scale"])
    rng = np.random.default_rng(7)
    eps = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        arr = p[name]
        for _ in range(25):
            idx = tuple(int(rng.integers(0, s)) for s in arr.shape)
            args = {x: p[x].copy() for x in ("q", "k", "v")}
            args[name][idx] += eps
            lp = _loss(p, args["q"], args["k"], args["v"])
            args[name][idx] -= 2 * eps
            lm = _loss(p, args["q"], args["k"], args["v"])
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def _torch_ref(p, mask_fn):
    """Per document: torch fp64 SDPA forward + autograd backward."""
    T, Hq, D = p["q"].shape
    Hi = p["sel"].shape[0]
    G = Hq // Hi
    out = np.zeros_like(p["q"]); dq = np.zeros_like(p["q"])
    dk = np.zeros((p["W"], Hi, D)); dv = np.zeros_like(dk)
    cu = p["cu"]
    for d in range(len(cu) - 1):
        t0, n, k0 = int(cu[d]), int(cu[d + 1] - cu[d]), int(p["kvs"][d])
        q = torch.tensor(p["q"][t0:t0 + n].transpose(1, 0, 2), requires_grad=True)
        k = torch.tensor(p["k"][k0:k0 + n].transpose(1, 0, 2), requires_grad=True)
        v = torch.tensor(p["v"][k0:k0 + n].transpose(1, 0, 2), requires_grad=True)
        kk = k.repeat_interleave(G, dim=0)
        vv = v.repeat_interleave(G, dim=0)
        m = mask_fn(d, n)
        if m is None:
            o = torch.nn.functional.scaled_dot_product_attention(q[None], kk[None], vv[None],
                                                                 is_causal=True, scale=p["scale"])[0]
        else:
            mm = torch.tensor(np.repeat(m[None], Hi, 0)).repeat_interleave(G, dim=0)
            o = torch.nn.functional.scaled_dot_product_attention(q[None], kk[None], vv[None],
                                                                 attn_mask=mm[None], scale=p["scale"])[0]
        g = torch.tensor(p["do"][t0:t0 + n].transpose(1, 0, 2))
        (o * g).sum().backward()
        out[t0:t0 + n] = o.detach().numpy().transpose(1, 0, 2)
        dq[t0:t0 + n] = q.grad.numpy().transpose(1, 0, 2)
        dk[k0:k0 + n] = k.grad.numpy().transpose(1, 0, 2)
        dv[k0:k0 + n] = v.grad.numpy().transpose(1, 0, 2)
    return out, dq, dk, dv


def _oracle_all(p, blocked):
    fw = O.forward_blocked if blocked else O.forward_dense
    bw = O.backward_blocked if blocked else O.backward_dense
    o, lse = fw(p["q"], p["k"], p["v"], p["cu"], p["kvs"], p["sel"], p["B"], p["C"], p["scale"])
    g = bw(p["q"], p["k"], p["v"], o, p["do"], lse, p["cu"], p["kvs"], p["sel"], p["B"], p["C"], p["scale"],
           kv_rows=p["W"])
    return (o,) + g


@pytest.mark.parametrize("blocked", [False, True])
def test_full_selection_is_textbook_causal_attention(blocked):
    p = _problem(2, [37, 70, 9], Hi=2, G=3, D=16, K=16, B=8, C=4, full=True, aligned=True)
    ref = _torch_ref(p, lambda d, n: None)
    got = _oracle_all(p, blocked)
    for a, b, name in zip(got, ref, ("o", "dq", "dk", "dv")):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11, err_msg=name)


@pytest.mark.parametrize("blocked", [False, True])
def test_sparse_selection_matches_masked_sdpa(blocked):
    p = _problem(3, [45, 30], Hi=2, G=2, D=16, K=3, B=8, C=4)
    sel, B, C = p["sel"], p["B"], p["C"]
    nc = [-(-int(n) // C) for n in np.diff(p["cu"])]
    goff = np.concatenate([[0], np.cumsum(nc)])

    # torch reference per index head (masks differ per index head)
    T, Hq, D = p["q"].shape
    Hi = sel.shape[0]
    G = Hq // Hi
    ref = [np.zeros_like(p["q"]), np.zeros_like(p["q"]), np.zeros((p["W"], Hi, D)), np.zeros((p["W"], Hi, D))]
    for hi in range(Hi):
        ph = dict(p)
        ph["q"] = p["q"][:, hi * G:(hi + 1) * G]
        ph["do"] = p["do"][:, hi * G:(hi + 1) * G]
        ph["k"] = p["k"][:, hi:hi + 1]
        ph["v"] = p["v"][:, hi:hi + 1]
        ph["sel"] = sel[hi:hi + 1]

        def mf(d, n, hi=hi):
            nb = -(-n // B)
            member = np.zeros((nc[d], nb), bool)
            for c in range(nc[d]):
                for b in sel[hi, goff[d] + c]:
                    if b >= 0:
                        member[c, b] = True
            pos = np.arange(n)
            return member[pos // C][:, pos // B] & (pos[None, :] <= pos[:, None])

        o, dq, dk, dv = _torch_ref(ph, mf)
        ref[0][:, hi * G:(hi + 1) * G] = o
        ref[1][:, hi * G:(hi + 1) * G] = dq
        ref[2][:, hi:hi + 1] = dk
        ref[3][:, hi:hi + 1] = dv
    got = _oracle_all(p, blocked)
    for a, b, name in zip(got, ref, ("o", "dq", "dk", "dv")):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11, err_msg=name)


def test_attended_sets_match_hand_worked_golden():
    g = json.load(open(os.path.join(GOLD, "k2q_tasks_two_docs.json")))
    sel = np.array(g["sel"], np.int32)
    lay = O.DocLayout(g["cu_seqlens"], g["block"], g["chunk"])
    for d, per_query in enumerate(g["attended"]):
        got = O.attend_mask(sel, lay, 0, d)
        exp = np.zeros_like(got)
        for qpos, ranges in enumerate(per_query):
            for a, b in ranges:
                exp[qpos, a:b + 1] = True
        assert (got == exp).all()


def test_single_key_query_has_zero_dq_and_unit_probability():
    # every document's first chunk can only select block 0; its first query sees key 0 alone
    p = _problem(4, [19, 12], Hi=1, G=2, D=8, K=2, B=8, C=4)
    o, lse = O.forward_dense(p["q"], p["k"], p["v"], p["cu"], p["kvs"], p["sel"], p["B"], p["C"], p["scale"])
    for d in range(2):
        t0, k0 = int(p["cu"][d]), int(p["kvs"][d])
        np.testing.assert_array_equal(o[t0], p["v"][k0, 0][None].repeat(2, 0))
        np.testing.assert_allclose(lse[t0], p["scale"] * p["q"][t0] @ p["k"][k0, 0], rtol=1e-15)
    dq, dk, dv = O.backward_dense(p["q"], p["k"], p["v"], o, p["do"], lse, p["cu"], p["kvs"], p["sel"],
                                  p["B"], p["C"], p["scale"])
    for d in range(2):
        # dS = 1 * (dO.v0 - dO.O) with O = v0 exactly: zero up to summation-order rounding
        assert np.max(np.abs(dq[int(p["cu"][d])])) < 1e-14


def test_blocked_equals_dense_on_tiny_workload():
    from block_sparse_top_attn_gb300 import workloads as W
    pb = W.make_problem("tiny")
    args = (pb.q, pb.k, pb.v, pb.cu_seqlens, pb.kv_doc_starts, pb.sel, pb.block, pb.chunk, pb.softmax_scale)
    o1, l1 = O.forward_dense(*args)
    o2, l2 = O.forward_blocked(*args)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13)
    ob = O.bf16_to_f64(O.f64_to_bf16(o1))
    lf = l1.astype(np.float32).astype(np.float64)
    bargs = (pb.q, pb.k, pb.v, ob, pb.do, lf, pb.cu_seqlens, pb.kv_doc_starts, pb.sel, pb.block, pb.chunk,
             pb.softmax_scale)
    g1 = O.backward_dense(*bargs)
    g2 = O.backward_blocked(*bargs)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_sampled_grads_equal_full_blocked():
    p = _problem(5, [70, 41], Hi=2, G=2, D=16, K=3, B=16, C=8, aligned=True)
    o, lse = O.forward_blocked(p["q"], p["k"], p["v"], p["cu"], p["kvs"], p["sel"], p["B"], p["C"], p["scale"])
    ob = O.bf16_to_f64(O.f64_to_bf16(o))
    lf = lse.astype(np.float32).astype(np.float64)
    dq, dk, dv = O.backward_blocked(p["q"], p["k"], p["v"], ob, p["do"], lf, p["cu"], p["kvs"], p["sel"],
                                    p["B"], p["C"], p["scale"], kv_rows=p["W"])
    picks = [(0, 0, 0), (0, 1, 8), (1, 1, 5), (1, 0, 2)]
    for rows, hs, g in O.sampled_query_grads(p["q"], p["k"], p["v"], p["do"], p["cu"], p["kvs"], p["sel"],
                                              p["B"], p["C"], p["scale"], picks):
        np.testing.assert_allclose(g, dq[rows][:, hs], rtol=1e-12, atol=1e-13)
    kp = [(0, 0, 0), (0, 1, 3), (1, 1, 2), (1, 0, 0)]
    for rows, hi, gk, gv in O.sampled_key_grads(p["q"], p["k"], p["v"], p["do"], p["cu"], p["kvs"], p["sel"],
                                                 p["B"], p["C"], p["scale"], kp):
        np.testing.assert_allclose(gk, dk[rows, hi], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(gv, dv[rows, hi], rtol=1e-11, atol=1e-12)


def test_bf16_rounding_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-20, 20, 200000))).astype(np.float32)
    # exact ties: bf16 midpoints (9 significant bits) round to the even neighbour
    ties = (np.arange(1, 513, dtype=np.float32) * 2.0 + 1.0) * np.float32(2.0 ** -9)
    x = np.concatenate([x, ties, -ties])
    got = O.f64_to_bf16(x.astype(np.float64))
    ref = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(O.bf16_to_f64(got), torch.tensor(x).to(torch.bfloat16).double().numpy())


def test_bf16_rounding_of_float64_between_neighbours():
    # values just off a float32-representable midpoint must round by their float64 side
    mid = 1.0 + 2.0 ** -8                      # midpoint of 1.0 and 1.0078125
    assert O.f64_to_bf16(np.array([mid - 2.0 ** -40]))[0] == 0x3F80
    assert O.f64_to_bf16(np.array([mid + 2.0 ** -40]))[0] == 0x3F81
    assert O.f64_to_bf16(np.array([mid]))[0] == 0x3F80          # tie -> even


def _bf16_bits_to_f64_torch(bits):
    """Decode bf16 bit patterns with torch (independent of the oracle's decoder)."""
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_bf16_ulp_is_the_spacing_of_adjacent_bf16_values():
    """bf16_ulp(x) must equal the gap between x and the next larger-magnitude
    bf16 value, for every positive and negative exponent of the format,
    including the subnormal range (spacing 2**-133) and zero."""
    bits = np.arange(0, 0x7F7F, dtype=np.uint32)          # all finite non-negative bf16 but the largest
    rng = np.random.default_rng(5)
    pick = np.unique(np.concatenate([bits[::7], bits[:300], rng.choice(bits, 4000)])).astype(np.uint16)
    x = _bf16_bits_to_f64_torch(pick)
    nxt = _bf16_bits_to_f64_torch(pick + np.uint16(1))
    spacing = nxt - x
    np.testing.assert_array_equal(O.bf16_ulp(x), spacing)
    np.testing.assert_array_equal(O.bf16_ulp(-x), spacing)
    # values strictly inside a binade (not bf16 values themselves) have the binade's spacing
    inner = x * (1.0 + rng.uniform(0, 2.0 ** -9, x.size))
    normal = x >= 2.0 ** -126
    np.testing.assert_array_equal(O.bf16_ulp(inner[normal]), spacing[normal])
    # a few values written out: 1 -> 2**-7, 8 -> 2**-4 (so half an ulp is 0.03125 on [8, 16)), 0 -> 2**-133
    np.testing.assert_array_equal(O.bf16_ulp(np.array([1.0, 1.5, 8.0, 15.9, 0.0])),
                                  [2.0 ** -7, 2.0 ** -7, 2.0 ** -4, 2.0 ** -4, 2.0 ** -133])


def test_empty_chunk_attends_nothing():
    """A chunk whose selection holds only -1 attends no key: its rows get O = 0
    and LSE = -inf (dense and blocked forms alike), dQ = 0, and dK/dV do not
    depend on those rows' dO."""
    p = _problem(11, [70, 45], Hi=2, G=2, D=8, K=3, B=8, C=4)
    sel = p["sel"].copy()
    empty = [(0, 2), (1, 5), (0, 19), (1, 19)]            # (index head, global chunk)
    for hi, g in empty:
        sel[hi, g] = -1
    p["sel"] = sel
    lay = O.DocLayout(p["cu"], p["B"], p["C"])
    G = 2
    rows = {}
    for hi, g in empty:
        d = int(np.searchsorted(lay.chunk_off, g, side="right") - 1)
        c = g - int(lay.chunk_off[d])
        rows[(hi, g)] = int(lay.cu[d]) + lay.chunk_positions(d, c)
    for fwd in (O.forward_dense, O.forward_blocked):
        # the dense form evaluates exp(-inf - -inf) in a branch its mask discards
        with np.errstate(invalid="ignore"):
            o, lse = fwd(p["q"], p["k"], p["v"], p["cu"], p["kvs"], sel, p["B"], p["C"], p["scale"])
        for (hi, g), r in rows.items():
            assert np.all(o[r][:, hi * G:(hi + 1) * G] == 0.0)
            assert np.all(np.isneginf(lse[r][:, hi * G:(hi + 1) * G]))
        assert np.isfinite(o).all()
    o, lse = O.forward_blocked(p["q"], p["k"], p["v"], p["cu"], p["kvs"], sel, p["B"], p["C"], p["scale"])
    dq, dk, dv = O.backward_blocked(p["q"], p["k"], p["v"], o, p["do"], lse, p["cu"], p["kvs"], sel, p["B"],
                                    p["C"], p["scale"])
    do2 = p["do"].copy()
    for (hi, g), r in rows.items():
        assert np.all(dq[r][:, hi * G:(hi + 1) * G] == 0.0)
        do2[np.ix_(r, np.arange(hi * G, (hi + 1) * G))] += 100.0
    _, dk2, dv2 = O.backward_blocked(p["q"], p["k"], p["v"], o, do2, lse, p["cu"], p["kvs"], sel, p["B"],
                                     p["C"], p["scale"])
    assert np.array_equal(dk, dk2) and np.array_equal(dv, dv2)
