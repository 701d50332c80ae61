#!/usr/bin/env python
"""Benchmark of the MSA block-sparse attention backward on GB300.

One step = the whole hot path over one batch: msa_build_k2q (CSR),
msa_build_tasks (task rows + CTA walk), and msa_bwd (preprocess D, main
KV-parallel tcgen05 kernel, postprocess casts).  Inputs (Q, K, V, dO drawn
bf16 N(0,1); O and LSE produced by msa_fwd) are resident in HBM before the
timed region; they are larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long128k]
    python bench.py --impl reference     # the fp64 CPU oracle on a bounded sample

Prints one JSON line (rank 0).  Under torchrun each rank runs its own
independent batch (seed = rank): no data-path collective, weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MSA backward effective TFLOP/s (selected blocks) and % of GB300 bf16 peak"
UNIT = "TFLOP/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["bf16_tflops"]), float(m["bf16_tflops_sustained"]), float(m["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def _rank():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's);
    x itself when the job has one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, flop_per_rank: float, ms: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own batch of flop_per_rank (weak
    scaling, no data-path collective), the job takes ms."""
    return world * flop_per_rank / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu)], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(parts)
            except Exception:
                pass
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle leg (bounded sample)
# ---------------------------------------------------------------------------
def oracle_sample(pb, host, budget_s: float, seed: int = 1):
    """Time the fp64 oracle backward on random (index head, chunk) units of the
    workload until about budget_s of CPU time; returns (TFLOP/s, seconds,
    units, flop).  O/LSE of each unit come from the oracle forward (untimed)."""
    from oracle import msa_oracle as O
    lay = O.DocLayout(pb.cu_seqlens, pb.block, pb.chunk)
    rng = np.random.default_rng(seed)
    q, k, v, do = host
    G = pb.group
    t_spent, flop, units = 0.0, 0, 0
    while t_spent < budget_s and units < 100000:
        g = int(rng.integers(0, lay.NC))
        hi = int(rng.integers(0, pb.num_index_heads))
        d = int(np.searchsorted(lay.chunk_off, g, side="right") - 1)
        c = g - int(lay.chunk_off[d])
        _, oc, lc = O.chunk_forward(q, k, v, lay, pb.kv_doc_starts, pb.sel, hi, d, c, G, pb.softmax_scale)
        oc = O.bf16_to_f64(O.f64_to_bf16(oc))
        lc = lc.astype(np.float32).astype(np.float64)
        t0 = time.perf_counter()
        O.chunk_backward(q, k, v, do, oc, lc, lay, pb.kv_doc_starts, pb.sel, hi, d, c, G, pb.softmax_scale)
        t_spent += time.perf_counter() - t0
        nq = lay.chunk_positions(d, c).size
        flop += nq * G * int((pb.sel[hi, g] >= 0).sum()) * 10 * pb.block * pb.head_dim
        units += 1
    return flop / t_spent / 1e12, t_spent, units, flop


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    rank, world, _ = _rank()
    if rank != 0:
        return 0
    from block_sparse_top_attn_gb300 import workloads as W
    pb = W.make_problem(args.workload, values=False)
    host = _host_values(pb)
    for _ in range(args.warmup):
        oracle_sample(pb, host, 0.5, seed=99)
    times, flops = [], 0
    tot_t = 0.0
    for s in range(args.steps):
        v, t, units, f = oracle_sample(pb, host, args.ref_budget, seed=s)
        tot_t += t
        flops += f
    value = flops / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "tokens": pb.total_tokens, "q_heads": pb.num_q_heads,
                       "index_heads": pb.num_index_heads, "topk": pb.topk},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                             "sample": f"{args.steps} steps x ~{args.ref_budget:.0f} s of random (index head, "
                                       f"query chunk) units of the workload, fp64 NumPy backward"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _host_values(pb):
    """Host bf16 bit arrays for the oracle leg: drawn on the GPU when one is
    present (fast), else with numpy."""
    try:
        import torch
        if torch.cuda.is_available():
            from block_sparse_top_attn_gb300 import workloads as W
            vals = W.device_values(pb, "cuda", seed=0)
            return tuple(t.view(torch.int16).cpu().numpy().view(np.uint16) for t in vals)
    except Exception:
        pass
    rng = np.random.default_rng(12345)
    from block_sparse_top_attn_gb300 import workloads as W
    T, Hq, D, Hkv, Wr = pb.total_tokens, pb.num_q_heads, pb.head_dim, pb.num_index_heads, pb.kv_rows
    return (W._normal_bf16(rng, (T, Hq, D)), W._normal_bf16(rng, (Wr, Hkv, D)), W._normal_bf16(rng, (Wr, Hkv, D)),
            W._normal_bf16(rng, (T, Hq, D)))


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------
MAIN_KERNEL_SOURCES = ("msa_bwd.cu", "msa_bwd_ws.cuh", "msa_common.cuh")
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "bwd_main_traffic.json")


def kernel_source_sha1() -> str:
    """SHA-1 over the sources the main backward kernel is compiled from."""
    h = hashlib.sha1()
    for name in MAIN_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "block_sparse_top_attn_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_record(workload: str, tile: int):
    """(bytes per launch, note) of the main kernel's DRAM traffic from the
    committed ncu record, or (None, why not).  The record holds counters taken
    on a small case and scaled to the named workload by its task count; it is
    valid only for that workload and tiling and while the kernel sources it was
    taken on are unchanged."""
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, "no traffic record"
    if rec.get("source_sha1") != kernel_source_sha1():
        return None, "kernel changed since the ncu counters were taken"
    scaled = rec.get("scaled", {}).get(f"{workload}/tile{tile}")
    if scaled is None:
        return None, f"no record scaled to {workload} with query tiles of {tile}"
    return float(scaled["bytes_per_launch"]), scaled.get("how", "")


# fp32 FMA issue peak of the GPU: 152 SMs x 128 FMA lanes x 2 FLOP x 2.07 GHz.
FP32_FMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def scorer_flops(pb) -> int:
    """Score FLOPs of the block scorer: one 128-dim dot product (2 x 128 FLOP)
    per index head, query chunk and key block strictly before the chunk's
    diagonal block (the diagonal is selected without a score)."""
    cu = np.asarray(pb.cu_seqlens, dtype=np.int64)
    pairs = 0
    for d in range(len(cu) - 1):
        n = int(cu[d + 1] - cu[d])
        c = np.arange((n + pb.chunk - 1) // pb.chunk, dtype=np.int64)
        pairs += int(((c * pb.chunk) // pb.block).sum())
    return pairs * pb.num_index_heads * 2 * 128


def aux_bytes(pb, n_tasks: int) -> dict:
    """Algorithmic (compulsory) DRAM bytes of each auxiliary stage per step."""
    Hi, NC, K = pb.num_index_heads, pb.sel.shape[1], pb.topk
    NB = int(sum(-(-int(n) // pb.block) for n in np.diff(pb.cu_seqlens)))
    T, Hq, W, D = pb.total_tokens, pb.num_q_heads, pb.kv_rows, pb.head_dim
    sizes = _chunk_sizes(pb)
    edges = int(sum(int(np.count_nonzero(pb.sel[hi] >= 0, axis=1) @ sizes) for hi in range(Hi)))
    sel_b, qi_b, rp_b = Hi * NC * K * 4, edges * 4, Hi * (NB + 1) * 4
    return {
        # sel read, row_ptr and q_indices written
        "k2q": sel_b + qi_b + rp_b,
        # row_ptr and q_indices read; task_meta (6), task_q_rows and task_q_pos (8 + 8) ints written per task
        "tasks": rp_b + qi_b + n_tasks * (6 + 8 + 8) * 4,
        # O, dO read; D written; dK/dV fp32 accumulators and the bf16 dQ output zeroed
        "preprocess": 2 * T * Hq * D * 2 + T * Hq * 4 + 2 * W * Hi * D * 4 + T * Hq * D * 2,
        # dK/dV fp32 accumulators read, bf16 dK/dV written
        "postprocess": 2 * W * Hi * D * 4 + 2 * W * Hi * D * 2,
    }


def _chunk_sizes(pb) -> np.ndarray:
    """Tokens of every query chunk, documents in order."""
    out = []
    for n in np.diff(pb.cu_seqlens):
        n = int(n)
        c = -(-n // pb.chunk)
        sz = np.full(c, pb.chunk, np.int64)
        sz[-1] = n - (c - 1) * pb.chunk
        out.append(sz)
    return np.concatenate(out)


def run_gpu(args):
    import torch
    import torch.distributed as dist
    rank, world, local = _rank()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from block_sparse_top_attn_gb300 import binding as B
    from block_sparse_top_attn_gb300 import workloads as W

    dev = torch.device("cuda", local)
    pb = W.make_problem(args.workload, values=False, seed=rank)
    prob = B.make_problem(pb.cu_seqlens, pb.kv_doc_starts, pb.kv_rows, pb.num_q_heads, pb.topk, pb.softmax_scale,
                          device=dev, block_size=pb.block)
    sel = torch.from_numpy(pb.sel).to(dev)
    q, k, v, do = W.device_values(pb, dev, seed=rank)
    o, lse, st = B.forward(prob, sel, q, k, v)
    torch.cuda.synchronize()
    if int(st[0].item()) != 0:
        raise B.MSAError(int(st[0].item()), "msa_fwd")
    flop = W.effective_flops(pb)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)

    # The forward (the next row on the path: it produces O and LSE) timed on its
    # own, outside the backward step: CUDA events around msa_fwd after one
    # warm-up call.  Effective FLOP count: QK^T and PV per selected block, 2/5
    # of the backward's five GEMMs.
    fwd_out = (torch.empty_like(o), torch.empty_like(lse), torch.zeros(4, dtype=torch.int32, device=dev))
    fwd_ws = torch.empty(max(256, 8 * (pb.num_docs + 1) + 256), dtype=torch.uint8, device=dev)
    fwd_runs = 3
    B.msa_fwd(prob, q, k, v, sel, *fwd_out[:2], fwd_out[2], fwd_ws)
    f0, f1 = ev(), ev()
    f0.record(stream)
    for _ in range(fwd_runs):
        B.msa_fwd(prob, q, k, v, sel, *fwd_out[:2], fwd_out[2], fwd_ws)
    f1.record(stream)
    torch.cuda.synchronize()
    if int(fwd_out[2][0].item()) != 0:
        raise B.MSAError(int(fwd_out[2][0].item()), "msa_fwd")
    fwd_ms = f0.elapsed_time(f1) / fwd_runs
    fwd_flop = flop * 2 / 5

    # The planner and the forward walking its plan, timed the same way.
    plan_meta, plan_wc, plan_st = B.plan_forward(prob, sel)
    plan_ws = torch.empty(B.msa_workspace_bytes(prob, 1, 1, 0), dtype=torch.uint8, device=dev)
    B.msa_fwd_planned(prob, q, k, v, sel, plan_meta, *fwd_out[:2], fwd_out[2], fwd_ws)
    f0.record(stream)
    for _ in range(fwd_runs):
        B.msa_plan_forward(prob, sel, plan_meta, plan_wc, plan_st, plan_ws)
    f1.record(stream)
    f2 = ev()
    for _ in range(fwd_runs):
        B.msa_fwd_planned(prob, q, k, v, sel, plan_meta, *fwd_out[:2], fwd_out[2], fwd_ws)
    f2.record(stream)
    torch.cuda.synchronize()
    for t, what in ((plan_st, "msa_plan_forward"), (fwd_out[2], "msa_fwd_planned")):
        if int(t[0].item()) != 0:
            raise B.MSAError(int(t[0].item()), what)
    plan_ms = f0.elapsed_time(f1) / fwd_runs
    fwd_planned_ms = f1.elapsed_time(f2) / fwd_runs
    del fwd_out, fwd_ws, plan_meta, plan_wc, plan_st, plan_ws

    # The block scorer + top-k on seeded index projections of the same shape.
    qi_idx, ki_idx = W.device_index_values(pb, dev, seed=rank)
    sel_scored = torch.empty_like(sel)
    sc_st = torch.zeros(4, dtype=torch.int32, device=dev)
    sc_ws = torch.empty(B.msa_workspace_bytes(prob, 1, 1, 0), dtype=torch.uint8, device=dev)
    B.msa_select_topk(prob, qi_idx, ki_idx, sel_scored, sc_st, sc_ws)
    f0.record(stream)
    for _ in range(fwd_runs):
        B.msa_select_topk(prob, qi_idx, ki_idx, sel_scored, sc_st, sc_ws)
    f1.record(stream)
    torch.cuda.synchronize()
    if int(sc_st[0].item()) != 0:
        raise B.MSAError(int(sc_st[0].item()), "msa_select_topk")
    score_ms = f0.elapsed_time(f1) / fwd_runs
    score_flop = scorer_flops(pb)
    del qi_idx, ki_idx, sel_scored, sc_st, sc_ws

    bw = B.Backward(prob, task_tile_chunks=args.tile)
    STAGES = ("k2q", "tasks", "preprocess", "main", "postprocess")

    def step(evs=None):
        """One pass of the hot path; evs (6 events) bracket its five stages on
        the launching stream."""
        rec = (lambda i: evs[i].record(stream)) if evs is not None else (lambda i: None)
        rec(0)
        B.msa_build_k2q(bw.p, sel, bw.row_ptr, bw.q_indices, bw.edge_cap, bw.status, bw.ws)
        rec(1)
        B.msa_build_tasks(bw.p, bw.row_ptr, bw.q_indices, bw.edge_cap, bw.tile, bw.task_meta, bw.task_q_rows,
                          bw.task_q_pos, bw.walk, bw.task_cap, bw.num_sms, bw.status, bw.ws)
        rec(2)
        bw.backward_stage(B.MSA_STAGE_PREPROCESS, q, k, v, o, do, lse)
        rec(3)
        bw.backward_stage(B.MSA_STAGE_MAIN, q, k, v, o, do, lse)
        rec(4)
        bw.backward_stage(B.MSA_STAGE_POSTPROCESS, q, k, v, o, do, lse)
        rec(5)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    bw.check_status()
    n_tasks = bw.num_tasks()

    stage_ev = [[ev() for _ in range(6)] for _ in range(args.steps)]
    t_start, t_end = ev(), ev()
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    t_start.record(stream)
    for i in range(args.steps):
        step(stage_ev[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    bw.check_status()
    ms = max_over_ranks(t_start.elapsed_time(t_end) / args.steps, dev)
    stage_ms = {name: sum(e[i].elapsed_time(e[i + 1]) for e in stage_ev) / args.steps
                for i, name in enumerate(STAGES)}
    main_ms = stage_ms["main"]
    value = job_value(world, flop, ms)

    # End to end through the public API with host buffers (pinned), copies timed.
    # Each step copies its inputs host->device, runs the backward and reads dQ,
    # dK, dV back; the steps are pipelined over two device input/output sets
    # and three streams (H2D of step i+1 and D2H of step i-1 overlap step i's
    # compute), as a serving loop would run them.  Every copy batch is
    # bracketed by events on its own stream, so the link rates below come from
    # the same timed region as the end-to-end figure.  The timed region spans
    # the same K steps as the device-timed loop and includes the pipeline's
    # fill (the first host->device batch) and drain (the last backward and its
    # device->host batch).
    pin = lambda t: t.cpu().pin_memory()
    host_in = {"q": pin(q), "k": pin(k), "v": pin(v), "o": pin(o), "do": pin(do), "lse": pin(lse), "sel": pin(sel)}
    host_out = [{n: torch.empty_like(getattr(bw, n), device="cpu").pin_memory() for n in ("dq", "dk", "dv")}
                for _ in range(2)]
    dev_in = [{"q": q, "k": k, "v": v, "o": o, "do": do, "lse": lse, "sel": sel},
              {n: torch.empty_like(t) for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do),
                                                   ("lse", lse), ("sel", sel))}]
    bws = [bw, B.Backward(prob, task_tile_chunks=args.tile)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_run(n_steps):
        """Runs n_steps pipelined steps; returns (start, end, [(h2d start, end)], [(d2h start, end)])."""
        done = [None, None]      # compute of the last step that used set b finished
        out_free = [None, None]  # D2H of the last step that used set b finished
        start = ev()
        start.record(s_h2d)
        end_events, h2d_ev, d2h_ev = [], [], []
        for i in range(n_steps):
            b = i % 2
            din, bwb = dev_in[b], bws[b]
            with torch.cuda.stream(s_h2d):
                if done[b] is not None:
                    s_h2d.wait_event(done[b])
                c0 = ev()
                c0.record(s_h2d)
                for name, t in host_in.items():
                    din[name].copy_(t, non_blocking=True)
                ready = ev()
                ready.record(s_h2d)
                h2d_ev.append((c0, ready))
            stream.wait_event(ready)
            if out_free[b] is not None:
                stream.wait_event(out_free[b])
            bwb.run(din["sel"], din["q"], din["k"], din["v"], din["o"], din["do"], din["lse"], stream=stream)
            done[b] = ev()
            done[b].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(done[b])
                c1 = ev()
                c1.record(s_d2h)
                for name in ("dq", "dk", "dv"):
                    host_out[b][name].copy_(getattr(bwb, name), non_blocking=True)
                out_free[b] = ev()
                out_free[b].record(s_d2h)
                d2h_ev.append((c1, out_free[b]))
            end_events.append(out_free[b])
        return start, end_events[-1], h2d_ev, d2h_ev

    e2e_steps = max(2, args.steps)
    e2e_run(2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1, h2d_ev, d2h_ev = e2e_run(e2e_steps)
    torch.cuda.synchronize()
    for b_ in bws:
        b_.check_status()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    e2e_value = job_value(world, flop, e2e_ms)
    h2d_ms = sum(a_.elapsed_time(b_) for a_, b_ in h2d_ev)
    d2h_ms = sum(a_.elapsed_time(b_) for a_, b_ in d2h_ev)

    # The fp32 dQ accumulator option on the same tables: preprocess, main and
    # postprocess timed with events, after one untimed backward.
    del bws
    bw32 = B.Backward(prob, task_tile_chunks=args.tile, dq_fp32=True)
    bw32.build_tables(sel)
    bw32.backward(q, k, v, o, do, lse)
    reps32 = 2
    ev32 = [[ev() for _ in range(4)] for _ in range(reps32)]
    for e in ev32:
        e[0].record(stream)
        for i_, stage_ in enumerate((B.MSA_STAGE_PREPROCESS, B.MSA_STAGE_MAIN, B.MSA_STAGE_POSTPROCESS)):
            bw32.backward_stage(stage_, q, k, v, o, do, lse)
            e[i_ + 1].record(stream)
    torch.cuda.synchronize()
    bw32.check_status()
    dq32_ms = {name: sum(e[i].elapsed_time(e[i + 1]) for e in ev32) / reps32
               for i, name in enumerate(("preprocess", "main", "postprocess"))}
    del bw32

    burst, sustained, hbm, src = _peaks()
    achieved = flop / (main_ms * 1e-3) / 1e12
    traffic, traffic_note = traffic_record(args.workload, args.tile)
    abytes = aux_bytes(pb, n_tasks)
    aux = {name: {"ms": stage_ms[name], "algorithmic_bytes": abytes[name],
                  "gbs": abytes[name] / (stage_ms[name] * 1e-3) / 1e9,
                  "frac_of_hbm": abytes[name] / (stage_ms[name] * 1e-3) / 1e9 / hbm}
           for name in ("k2q", "tasks", "preprocess", "postprocess")}
    n_launches = 5 + 6 + 3 + 1 + 1  # CSR build, task build, preprocess, counter reset + main, postprocess
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "tokens": pb.total_tokens, "documents": pb.num_docs,
                   "q_heads": pb.num_q_heads, "index_heads": pb.num_index_heads, "head_dim": pb.head_dim,
                   "block": pb.block, "chunk": pb.chunk, "topk": pb.topk, "tasks": n_tasks,
                   "effective_tflop_per_step": flop / 1e12, "task_tile_chunks": args.tile,
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"},
        "fraction_of_peak": {"value": value / burst, "peak_tflops": burst, "peak_kind": f"bf16 burst ({src})",
                             "value_vs_sustained": value / sustained, "sustained_tflops": sustained},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
                     "frac": achieved / burst, "traffic": traffic, "kernel": "bwd_main_ws",
                     "kernel_ms": main_ms, "peak_kind": f"bf16 burst, of {src}",
                     "frac_vs_sustained": achieved / sustained, "sustained_peak": sustained,
                     "traffic_note": traffic_note},
        "stages_ms": stage_ms,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "pipeline": "H2D of step i+1 and D2H of step i-1 overlap step i (two device sets, three streams)",
                "h2d_gbs": h2d * e2e_steps / (h2d_ms * 1e-3) / 1e9,
                "d2h_gbs": d2h * e2e_steps / (d2h_ms * 1e-3) / 1e9,
                "h2d_ms_per_step": h2d_ms / e2e_steps, "d2h_ms_per_step": d2h_ms / e2e_steps,
                "copy_timing": "per-step events on the copy streams inside the timed region"},
        "gpu_launches": args.steps * n_launches,
        "next_rows": {"forward": {"kernel_ms": fwd_ms, "effective_tflops": fwd_flop / (fwd_ms * 1e-3) / 1e12,
                                  "frac": fwd_flop / (fwd_ms * 1e-3) / 1e12 / burst,
                                  "frac_vs_sustained": fwd_flop / (fwd_ms * 1e-3) / 1e12 / sustained,
                                  "flop_convention": "QK^T and PV per selected block (2 of the 5 backward GEMMs)",
                                  "timed": "3 msa_fwd calls after one warm-up, outside the backward step"},
                      "forward_planned": {"plan_ms": plan_ms, "kernel_ms": fwd_planned_ms,
                                          "effective_tflops": fwd_flop / (fwd_planned_ms * 1e-3) / 1e12,
                                          "timed": "3 msa_plan_forward then 3 msa_fwd_planned calls after "
                                                   "one warm-up"},
                      "scorer": {"ms": score_ms, "score_gflop": score_flop / 1e9,
                                 "score_tflops": score_flop / (score_ms * 1e-3) / 1e12,
                                 "bound": "alu", "fp32_fma_peak_tflops": FP32_FMA_PEAK_TFLOPS,
                                 "frac": score_flop / (score_ms * 1e-3) / 1e12 / FP32_FMA_PEAK_TFLOPS,
                                 "timed": "3 msa_select_topk calls on seeded index projections after one warm-up"},
                      "dq_fp32": {"stages_ms": dq32_ms, "step_ms": sum(dq32_ms.values()),
                                  "main_tflops": flop / (dq32_ms["main"] * 1e-3) / 1e12,
                                  "timed": "2 x (preprocess, main, postprocess) with the fp32 dQ accumulator "
                                           "option, after one untimed backward"},
                      "aux_kernels": aux},
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = tuple(t.view(torch.int16).numpy().view(np.uint16) for t in (host_in["q"], host_in["k"],
                                                                             host_in["v"], host_in["do"]))
        cv, ct, units, cf = oracle_sample(pb, host, args.cpu_budget)
        line["cpu_baseline"] = {"value": cv, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                                "sample": f"{units} random (index head, query chunk) units, {cf / 1e9:.1f} GFLOP, "
                                          f"{ct:.1f} s fp64 NumPy backward"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_tables(args):
    """The index-side kernels alone (no attention tensors on the device): the
    CSR and task builds on the workload's selection (per-stage CUDA-event
    times and GB/s of the algorithmic bytes), the scorer + top-k on seeded
    index projections and the forward planner.  For profiling those kernels
    on a small footprint."""
    import torch
    from block_sparse_top_attn_gb300 import binding as B
    from block_sparse_top_attn_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pb = W.make_problem(args.workload, values=False)
    prob = B.make_problem(pb.cu_seqlens, pb.kv_doc_starts, pb.kv_rows, pb.num_q_heads, pb.topk, pb.softmax_scale,
                          device=dev, block_size=pb.block)
    sel = torch.from_numpy(pb.sel).to(dev)
    bw = B.Backward(prob, task_tile_chunks=args.tile)
    stream = torch.cuda.current_stream()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for _ in range(args.warmup):
        bw.build_tables(sel)
    torch.cuda.synchronize()
    for e in evs:
        e[0].record(stream)
        B.msa_build_k2q(bw.p, sel, bw.row_ptr, bw.q_indices, bw.edge_cap, bw.status, bw.ws)
        e[1].record(stream)
        B.msa_build_tasks(bw.p, bw.row_ptr, bw.q_indices, bw.edge_cap, bw.tile, bw.task_meta, bw.task_q_rows,
                          bw.task_q_pos, bw.walk, bw.task_cap, bw.num_sms, bw.status, bw.ws)
        e[2].record(stream)
    torch.cuda.synchronize()
    bw.check_status()
    n_tasks = bw.num_tasks()
    ms = {name: sum(e[i].elapsed_time(e[i + 1]) for e in evs) / args.steps for i, name in enumerate(("k2q", "tasks"))}
    # the scorer + top-k and the forward planner on the same problem
    qi_idx, ki_idx = W.device_index_values(pb, dev, seed=0)
    sel2 = torch.empty_like(sel)
    meta = torch.empty((pb.num_index_heads * pb.sel.shape[1], B.MSA_TASK_META_COLS), dtype=torch.int32, device=dev)
    wc = torch.zeros(4, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        B.msa_select_topk(prob, qi_idx, ki_idx, sel2, bw.status, bw.ws)
        B.msa_plan_forward(prob, sel, meta, wc, bw.status, bw.ws)
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for e in ev2:
        e[0].record(stream)
        B.msa_select_topk(prob, qi_idx, ki_idx, sel2, bw.status, bw.ws)
        e[1].record(stream)
        B.msa_plan_forward(prob, sel, meta, wc, bw.status, bw.ws)
        e[2].record(stream)
    torch.cuda.synchronize()
    bw.check_status()
    ms2 = {name: sum(e[i].elapsed_time(e[i + 1]) for e in ev2) / args.steps for i, name in enumerate(("scorer", "plan"))}
    ab = aux_bytes(pb, n_tasks)
    _, _, hbm, _ = _peaks()
    sf = scorer_flops(pb)
    out = {"metric": "CSR and task build time", "unit": "ms", "workload": args.workload, "tasks": n_tasks,
           "steps": args.steps, "warmup": args.warmup,
           "stages": {k: {"ms": ms[k], "algorithmic_bytes": ab[k], "gbs": ab[k] / (ms[k] * 1e-3) / 1e9,
                          "frac_of_hbm": ab[k] / (ms[k] * 1e-3) / 1e9 / hbm} for k in ms},
           "scorer": {"ms": ms2["scorer"], "score_gflop": sf / 1e9,
                      "frac_of_fp32_fma_peak": sf / (ms2["scorer"] * 1e-3) / 1e12 / FP32_FMA_PEAK_TFLOPS},
           "plan": {"ms": ms2["plan"]}}
    print(json.dumps(out), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long128k")
    ap.add_argument("--tile", type=int, default=1024, help="query chunks per task tile (0 = untiled)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tables-only", action="store_true",
                    help="time only the index-side kernels: CSR, tasks, scorer, planner (a small footprint)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.tables_only:
        return run_tables(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
