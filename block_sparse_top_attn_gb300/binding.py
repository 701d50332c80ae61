"""Thin ctypes binding over libmsa.so (the C ABI in include/msa.h).

Only argument marshalling lives here: every step of the path runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  There
is no fallback: if libmsa.so cannot be loaded, importing this module raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmsa.so")

MSA_OK = 0
MSA_ERR_INVALID_ARGUMENT = 1
MSA_ERR_UNSUPPORTED_DEVICE = 2
MSA_ERR_UNSUPPORTED_SHAPE = 3
MSA_ERR_CAPACITY = 4
MSA_ERR_INVALID_SELECTION = 5
MSA_ERR_TIMEOUT = 6
MSA_ERR_CUDA = 7
MSA_ERR_INVALID_DOCUMENTS = 8
MSA_ERR_SCRATCH_TOO_SMALL = 9
MSA_NOALLOC_SCRATCH_BYTES = 16 << 20
MSA_TASK_META_COLS = 6
MSA_STAGE_PREPROCESS, MSA_STAGE_MAIN, MSA_STAGE_POSTPROCESS, MSA_STAGE_ALL = 1, 2, 4, 7
MSA_BWD_DQ_FP32 = 8
MSA_BWD_SELFTEST_HOLD_REDUCE = 16
MSA_WALK_LEN = 8

HEAD_DIM, BLOCK, CHUNK, GROUP = 128, 64, 8, 16


class MSAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


class msa_problem(ctypes.Structure):
    _fields_ = [
        ("num_docs", ctypes.c_int32),
        ("total_tokens", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p),
        ("kv_doc_starts", ctypes.c_void_p),
        ("kv_rows", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_index_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("query_chunk", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("num_chunks", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmsa.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                          "or python -m block_sparse_top_attn_gb300.build_lib")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(msa_problem)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "msa_workspace_bytes": (sz, [P, i64, i64, i32]),
        "msa_workspace_bytes_opts": (sz, [P, i64, i64, i32, ctypes.c_uint32]),
        "msa_build_k2q": (ctypes.c_int, [P, vp, vp, vp, i64, vp, vp, sz, vp]),
        "msa_build_k2q_noalloc": (ctypes.c_int, [P, vp, vp, vp, i64, vp, vp]),
        "msa_build_tasks": (ctypes.c_int, [P, vp, vp, i64, i32, vp, vp, vp, vp, i64, i32, vp, vp, sz, vp]),
        "msa_bwd": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, sz, vp]),
        "msa_bwd_staged": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, sz, vp,
                                          ctypes.c_uint32]),
        "msa_fwd": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "msa_rows_per_cta": (i32, [i64]),
        "msa_chunk_map": (None, [i64, i32, i32, ctypes.POINTER(i64)]),
        "msa_grid_launch_bound": (i64, [i64, i32]),
        "msa_device_capability": (ctypes.c_int, [i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]),
        "msa_device_sm_count": (ctypes.c_int, [i32, ctypes.POINTER(i32)]),
        "msa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "msa_selftest_wait_timeout": (ctypes.c_int, [vp, vp]),
        "msa_select_topk": (ctypes.c_int, [P, vp, vp, vp, vp, vp, sz, vp]),
        "msa_plan_forward": (ctypes.c_int, [P, vp, vp, vp, vp, vp, sz, vp]),
        "msa_fwd_planned": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def msa_selftest_wait_timeout(d_status, stream=None):
    """Run the bounded-wait self-test kernel: *d_status becomes MSA_ERR_TIMEOUT
    about two seconds later, with no fault and the context still usable."""
    _check(lib.msa_selftest_wait_timeout(_ptr(d_status), _stream(stream)), "msa_selftest_wait_timeout")


def status_string(code: int) -> str:
    return lib.msa_status_string(int(code)).decode()


def _check(rc: int, where: str):
    if rc != MSA_OK:
        raise MSAError(rc, where)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---------------------------------------------------------------------------
# host-side walk rule and device queries
# ---------------------------------------------------------------------------

def msa_rows_per_cta(num_rows: int) -> int:
    return int(lib.msa_rows_per_cta(int(num_rows)))


def msa_chunk_map(num_rows: int, rows_per_cta: int, num_sms: int):
    out = (ctypes.c_int64 * 3)()
    lib.msa_chunk_map(int(num_rows), int(rows_per_cta), int(num_sms), out)
    return int(out[0]), int(out[1]), int(out[2])


def msa_grid_launch_bound(capacity: int, num_sms: int) -> int:
    return int(lib.msa_grid_launch_bound(int(capacity), int(num_sms)))


def msa_device_sm_count(device: int = 0) -> int:
    v = ctypes.c_int32()
    _check(lib.msa_device_sm_count(int(device), ctypes.byref(v)), "msa_device_sm_count")
    return int(v.value)


def msa_device_capability(device: int = 0):
    a, b = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.msa_device_capability(int(device), ctypes.byref(a), ctypes.byref(b)), "msa_device_capability")
    return int(a.value), int(b.value)


# ---------------------------------------------------------------------------
# problem description
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Problem:
    """Host description plus the device copies the C struct points at."""
    cu_seqlens: np.ndarray
    kv_doc_starts: np.ndarray
    kv_rows: int
    num_q_heads: int
    topk: int
    softmax_scale: float
    d_cu: object = None
    d_kvs: object = None
    block_size: int = BLOCK   # keys per selectable block: 64, or 128 (two 64-key tiles)

    @property
    def num_docs(self):
        return len(self.cu_seqlens) - 1

    @property
    def total_tokens(self):
        return int(self.cu_seqlens[-1])

    @property
    def num_index_heads(self):
        return self.num_q_heads // GROUP

    @property
    def lengths(self):
        return np.diff(np.asarray(self.cu_seqlens, np.int64))

    @property
    def num_blocks(self):
        return int(sum(-(-n // self.block_size) for n in self.lengths))

    @property
    def num_chunks(self):
        return int(sum(-(-n // CHUNK) for n in self.lengths))

    def edge_capacity(self) -> int:
        """Upper bound on CSR entries per index head: every chunk selects topk blocks."""
        return max(1, int(sum(min(self.topk, -(-int(n) // self.block_size)) * int(n) for n in self.lengths)))

    def task_capacity(self) -> int:
        """Upper bound on task rows: one per valid selection slot and 64-key tile."""
        return max(1, self.num_index_heads * self.num_chunks * self.topk * max(1, self.block_size // BLOCK))

    def c_struct(self) -> msa_problem:
        s = msa_problem()
        s.num_docs = self.num_docs
        s.total_tokens = self.total_tokens
        s.cu_seqlens = self.d_cu.data_ptr()
        s.kv_doc_starts = self.d_kvs.data_ptr()
        s.kv_rows = int(self.kv_rows)
        s.num_q_heads = int(self.num_q_heads)
        s.num_index_heads = self.num_index_heads
        s.num_kv_heads = self.num_index_heads
        s.head_dim = HEAD_DIM
        s.block_size = int(self.block_size)
        s.query_chunk = CHUNK
        s.topk = int(self.topk)
        s.num_blocks = self.num_blocks
        s.num_chunks = self.num_chunks
        s.softmax_scale = float(self.softmax_scale)
        return s


def make_problem(cu_seqlens, kv_doc_starts, kv_rows, num_q_heads, topk, softmax_scale=HEAD_DIM ** -0.5,
                 device="cuda", block_size=BLOCK) -> Problem:
    import torch
    cu = np.asarray(cu_seqlens, np.int32)
    kvs = np.asarray(kv_doc_starts, np.int32)
    p = Problem(cu, kvs, int(kv_rows), int(num_q_heads), int(topk), float(softmax_scale), block_size=int(block_size))
    p.d_cu = torch.tensor(cu, dtype=torch.int32, device=device)
    p.d_kvs = torch.tensor(kvs, dtype=torch.int32, device=device)
    return p


# ---------------------------------------------------------------------------
# the C entry points, same names
# ---------------------------------------------------------------------------

def msa_workspace_bytes(p: Problem, edge_cap: int, task_cap: int, task_tile_chunks: int = 0) -> int:
    s = p.c_struct() if p.d_cu is not None else None
    return int(lib.msa_workspace_bytes(ctypes.byref(s), int(edge_cap), int(task_cap), int(task_tile_chunks)))


def msa_workspace_bytes_opts(p: Problem, edge_cap: int, task_cap: int, task_tile_chunks: int = 0,
                             options: int = 0) -> int:
    s = p.c_struct() if p.d_cu is not None else None
    return int(lib.msa_workspace_bytes_opts(ctypes.byref(s), int(edge_cap), int(task_cap), int(task_tile_chunks),
                                            int(options)))


def msa_build_k2q(p: Problem, sel, row_ptr, q_indices, edge_cap, d_status, ws, stream=None):
    s = p.c_struct()
    _check(lib.msa_build_k2q(ctypes.byref(s), _ptr(sel), _ptr(row_ptr), _ptr(q_indices), int(edge_cap),
                             _ptr(d_status), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "msa_build_k2q")


def msa_build_k2q_noalloc(p: Problem, sel, row_ptr, q_indices, edge_cap, d_status, stream=None):
    """msa_build_k2q without a caller workspace: the library's fixed scratch
    array stands in for it, for callers that may not allocate device memory."""
    s = p.c_struct()
    _check(lib.msa_build_k2q_noalloc(ctypes.byref(s), _ptr(sel), _ptr(row_ptr), _ptr(q_indices), int(edge_cap),
                                     _ptr(d_status), _stream(stream)),
           "msa_build_k2q_noalloc")


def msa_build_tasks(p: Problem, row_ptr, q_indices, edge_cap, task_tile_chunks, task_meta, task_q_rows,
                    task_q_pos, walk, task_cap, num_sms, d_status, ws, stream=None):
    s = p.c_struct()
    _check(lib.msa_build_tasks(ctypes.byref(s), _ptr(row_ptr), _ptr(q_indices), int(edge_cap),
                               int(task_tile_chunks), _ptr(task_meta), _ptr(task_q_rows), _ptr(task_q_pos),
                               _ptr(walk), int(task_cap), int(num_sms), _ptr(d_status), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)),
           "msa_build_tasks")


def msa_bwd(p: Problem, q, k, v, o, dout, lse, task_meta, task_q_rows, task_q_pos, walk, task_cap, dq, dk, dv,
            d_status, ws, stream=None):
    s = p.c_struct()
    _check(lib.msa_bwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                       _ptr(task_meta), _ptr(task_q_rows), _ptr(task_q_pos), _ptr(walk), int(task_cap),
                       _ptr(dq), _ptr(dk), _ptr(dv), _ptr(d_status), _ptr(ws), ws.numel() * ws.element_size(),
                       _stream(stream)),
           "msa_bwd")


def msa_bwd_staged(p: Problem, q, k, v, o, dout, lse, task_meta, task_q_rows, task_q_pos, walk, task_cap, dq, dk,
                   dv, d_status, ws, stages, stream=None):
    s = p.c_struct()
    _check(lib.msa_bwd_staged(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                              _ptr(task_meta), _ptr(task_q_rows), _ptr(task_q_pos), _ptr(walk), int(task_cap),
                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(d_status), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream), int(stages)),
           "msa_bwd_staged")


def msa_fwd(p: Problem, q, k, v, sel, o, lse, d_status, ws, stream=None):
    s = p.c_struct()
    _check(lib.msa_fwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(sel), _ptr(o), _ptr(lse),
                       _ptr(d_status), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "msa_fwd")


def msa_select_topk(p: Problem, q_index, k_index, sel, d_status, ws, stream=None):
    s = p.c_struct()
    _check(lib.msa_select_topk(ctypes.byref(s), _ptr(q_index), _ptr(k_index), _ptr(sel), _ptr(d_status), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)),
           "msa_select_topk")


def msa_plan_forward(p: Problem, sel, scheduler_metadata, work_count, d_status, ws, stream=None):
    s = p.c_struct()
    _check(lib.msa_plan_forward(ctypes.byref(s), _ptr(sel), _ptr(scheduler_metadata), _ptr(work_count),
                                _ptr(d_status), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "msa_plan_forward")


def msa_fwd_planned(p: Problem, q, k, v, sel, scheduler_metadata, o, lse, d_status, ws, stream=None):
    s = p.c_struct()
    _check(lib.msa_fwd_planned(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(sel), _ptr(scheduler_metadata),
                               _ptr(o), _ptr(lse), _ptr(d_status), _ptr(ws), ws.numel() * ws.element_size(),
                               _stream(stream)),
           "msa_fwd_planned")


def plan_forward(p: Problem, sel, stream=None):
    """msa_plan_forward convenience: returns (scheduler_metadata [Hi*NC, 6],
    work_count [1], status tensor)."""
    import torch
    dev = p.d_cu.device
    meta = torch.empty((p.num_index_heads * p.num_chunks, MSA_TASK_META_COLS), dtype=torch.int32, device=dev)
    wc = torch.zeros(4, dtype=torch.int32, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    ws = torch.empty(msa_workspace_bytes(p, 1, 1, 0), dtype=torch.uint8, device=dev)
    msa_plan_forward(p, sel, meta, wc, st, ws, stream)
    return meta, wc, st


def select_topk(p: Problem, q_index, k_index, stream=None):
    """msa_select_topk convenience: returns (sel int32 [Hi, NC, topk], status tensor)."""
    import torch
    dev = p.d_cu.device
    sel = torch.empty((p.num_index_heads, p.num_chunks, p.topk), dtype=torch.int32, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    ws = torch.empty(msa_workspace_bytes(p, 1, 1, 0), dtype=torch.uint8, device=dev)
    msa_select_topk(p, q_index, k_index, sel, st, ws, stream)
    return sel, st


# ---------------------------------------------------------------------------
# convenience: one problem's buffers and the whole backward sequence
# ---------------------------------------------------------------------------

class Backward:
    """Owns the tables and workspace of one problem and runs the backward.

    ``run(sel, q, k, v, o, do, lse)`` issues msa_build_k2q, msa_build_tasks and
    msa_bwd on the current stream and returns bf16 (dq, dk, dv) tensors.
    """

    def __init__(self, p: Problem, task_tile_chunks: int = 0, num_sms: int = 0, edge_cap=None, task_cap=None,
                 dq_fp32: bool = False):
        import torch
        self.p = p
        dev = p.d_cu.device
        self.tile = int(task_tile_chunks)
        self.num_sms = int(num_sms)
        self.edge_cap = int(edge_cap or p.edge_capacity())
        self.task_cap = int(task_cap or p.task_capacity())
        Hi, NB = p.num_index_heads, p.num_blocks
        i32 = torch.int32
        self.row_ptr = torch.empty((Hi, NB + 1), dtype=i32, device=dev)
        self.q_indices = torch.empty((Hi, self.edge_cap), dtype=i32, device=dev)
        self.task_meta = torch.empty((self.task_cap, MSA_TASK_META_COLS), dtype=i32, device=dev)
        self.task_q_rows = torch.empty((self.task_cap, CHUNK), dtype=i32, device=dev)
        self.task_q_pos = torch.empty((self.task_cap, CHUNK), dtype=i32, device=dev)
        self.walk = torch.zeros(MSA_WALK_LEN, dtype=i32, device=dev)
        self.status = torch.zeros(4, dtype=i32, device=dev)
        self.options = MSA_BWD_DQ_FP32 if dq_fp32 else 0
        nbytes = msa_workspace_bytes_opts(p, self.edge_cap, self.task_cap, self.tile, self.options)
        if nbytes == 0:
            raise MSAError(MSA_ERR_INVALID_ARGUMENT, "msa_workspace_bytes")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        T, Hq, W = p.total_tokens, p.num_q_heads, p.kv_rows
        bf16 = torch.bfloat16
        self.dq = torch.empty((T, Hq, HEAD_DIM), dtype=bf16, device=dev)
        self.dk = torch.empty((W, Hi, HEAD_DIM), dtype=bf16, device=dev)
        self.dv = torch.empty((W, Hi, HEAD_DIM), dtype=bf16, device=dev)

    def build_tables(self, sel, stream=None):
        msa_build_k2q(self.p, sel, self.row_ptr, self.q_indices, self.edge_cap, self.status, self.ws, stream)
        msa_build_tasks(self.p, self.row_ptr, self.q_indices, self.edge_cap, self.tile, self.task_meta,
                        self.task_q_rows, self.task_q_pos, self.walk, self.task_cap, self.num_sms, self.status,
                        self.ws, stream)

    def backward(self, q, k, v, o, do, lse, stream=None):
        if self.options:
            self.backward_stage(MSA_STAGE_ALL, q, k, v, o, do, lse, stream)
        else:
            msa_bwd(self.p, q, k, v, o, do, lse, self.task_meta, self.task_q_rows, self.task_q_pos, self.walk,
                    self.task_cap, self.dq, self.dk, self.dv, self.status, self.ws, stream)
        return self.dq, self.dk, self.dv

    def backward_stage(self, stages, q, k, v, o, do, lse, stream=None):
        msa_bwd_staged(self.p, q, k, v, o, do, lse, self.task_meta, self.task_q_rows, self.task_q_pos, self.walk,
                       self.task_cap, self.dq, self.dk, self.dv, self.status, self.ws, stages | self.options,
                       stream)

    def run(self, sel, q, k, v, o, do, lse, stream=None):
        self.build_tables(sel, stream)
        return self.backward(q, k, v, o, do, lse, stream)

    def check_status(self):
        code = int(self.status[0].item())
        if code != MSA_OK:
            raise MSAError(code, "device status")

    def num_tasks(self) -> int:
        return int(self.walk[0].item())


def forward(p: Problem, sel, q, k, v, stream=None, plan=None):
    """msa_fwd convenience (msa_fwd_planned when plan, a scheduler_metadata
    tensor from plan_forward, is given): returns (o bf16 [T, Hq, 128], lse fp32
    [T, Hq], status tensor)."""
    import torch
    dev = p.d_cu.device
    o = torch.empty((p.total_tokens, p.num_q_heads, HEAD_DIM), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.total_tokens, p.num_q_heads), dtype=torch.float32, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    ws = torch.empty(max(256, 8 * (p.num_docs + 1) + 256), dtype=torch.uint8, device=dev)
    if plan is None:
        msa_fwd(p, q, k, v, sel, o, lse, st, ws, stream)
    else:
        msa_fwd_planned(p, q, k, v, sel, plan, o, lse, st, ws, stream)
    return o, lse, st
