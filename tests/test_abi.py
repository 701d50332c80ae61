"""The C ABI library loads and exports every symbol include/msa.h declares; its
host-only logic (walk rule, argument checks, status strings) matches the oracle
and the header, with no GPU needed."""
import ctypes
import os
import re

import pytest

from oracle import msa_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from block_sparse_top_attn_gb300 import build_lib
    build_lib.build()
    from block_sparse_top_attn_gb300 import binding
    return binding


def _declared():
    src = open(os.path.join(ROOT, "include", "msa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(B):
    names = _declared()
    assert "msa_bwd" in names and "msa_build_k2q" in names and "msa_build_tasks" in names
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_header_constants_match_binding(B):
    src = open(os.path.join(ROOT, "include", "msa.h")).read()
    for name in ("MSA_OK", "MSA_ERR_INVALID_ARGUMENT", "MSA_ERR_UNSUPPORTED_DEVICE", "MSA_ERR_UNSUPPORTED_SHAPE",
                 "MSA_ERR_CAPACITY", "MSA_ERR_INVALID_SELECTION", "MSA_ERR_TIMEOUT", "MSA_ERR_CUDA",
                 "MSA_ERR_INVALID_DOCUMENTS", "MSA_ERR_SCRATCH_TOO_SMALL", "MSA_TASK_META_COLS", "MSA_WALK_LEN",
                 "MSA_STAGE_PREPROCESS", "MSA_STAGE_MAIN", "MSA_STAGE_POSTPROCESS", "MSA_STAGE_ALL"):
        m = re.search(rf"\b{name}\s*=\s*(\d+)", src)
        assert m and int(m.group(1)) == getattr(B, name), name
    for code in range(10):
        assert B.status_string(code) and B.status_string(code) != "unknown status"
    assert B.status_string(99) == "unknown status"


@pytest.mark.parametrize("sms", [1, 7, 148, 152])
def test_host_walk_rule_matches_oracle(B, sms):
    for n in list(range(0, 3000)) + list(range(3000, 200000, 997)):
        R = O.rows_per_cta(n)
        assert B.msa_rows_per_cta(n) == R
        assert B.msa_chunk_map(n, R, sms) == O.chunk_map(n, R, sms)
    for cap in list(range(0, 2600, 7)) + [20000, 65536, 1 << 20, 4162560]:
        assert B.msa_grid_launch_bound(cap, sms) == O.grid_launch_bound(cap, sms), cap


def test_invalid_arguments_rejected_on_host(B):
    lib = B.lib
    p = B.msa_problem()
    # null problem / null pointers are rejected before any device work
    assert lib.msa_build_k2q(None, None, None, None, 1, None, None, 0, None) == B.MSA_ERR_INVALID_ARGUMENT
    assert lib.msa_workspace_bytes(None, 1, 1, 0) == 0
    assert lib.msa_workspace_bytes(ctypes.byref(p), 1, 1, 0) == 0
    # a well-formed struct with fake aligned pointers but an unsupported head_dim
    p.num_docs, p.total_tokens, p.kv_rows = 1, 64, 64
    p.cu_seqlens, p.kv_doc_starts = 4096, 8192
    p.num_q_heads, p.num_index_heads, p.num_kv_heads = 16, 1, 1
    p.head_dim, p.block_size, p.query_chunk, p.topk = 64, 64, 8, 4
    p.num_blocks, p.num_chunks, p.softmax_scale = 1, 8, 0.1
    assert lib.msa_workspace_bytes(ctypes.byref(p), 64, 8, 0) == 0
    p.head_dim = 128
    assert lib.msa_workspace_bytes(ctypes.byref(p), 64, 8, 0) > 0
    p.topk = 33
    assert lib.msa_workspace_bytes(ctypes.byref(p), 64, 8, 0) == 0
    p.topk = 4
    p.num_q_heads = 32  # G must be 16
    assert lib.msa_workspace_bytes(ctypes.byref(p), 64, 8, 0) == 0
    p.num_q_heads = 16
    p.cu_seqlens = 4100  # misaligned
    assert lib.msa_workspace_bytes(ctypes.byref(p), 64, 8, 0) == 0


def test_block_size_and_workspace_options(B):
    """Block sizes 64 and 128 are accepted, others rejected; the fp32 dQ option
    adds one fp32 [T, Hq, 128] accumulator to the workspace; unknown option
    bits are rejected (fake, never dereferenced addresses)."""
    lib = B.lib
    p = B.msa_problem()
    p.num_docs, p.total_tokens, p.kv_rows = 1, 4096, 4096
    p.cu_seqlens, p.kv_doc_starts = 4096, 8192
    p.num_q_heads, p.num_index_heads, p.num_kv_heads = 64, 4, 4
    p.head_dim, p.block_size, p.query_chunk, p.topk = 128, 64, 8, 4
    p.num_blocks, p.num_chunks, p.softmax_scale = 64, 512, 0.1
    base = lib.msa_workspace_bytes(ctypes.byref(p), 64, 8, 0)
    assert base > 0 and lib.msa_workspace_bytes_opts(ctypes.byref(p), 64, 8, 0, 0) == base
    assert lib.msa_workspace_bytes_opts(ctypes.byref(p), 64, 8, 0, B.MSA_BWD_DQ_FP32) == base + 4096 * 64 * 128 * 4
    assert lib.msa_workspace_bytes_opts(ctypes.byref(p), 64, 8, 0, 16) == 0
    p.block_size, p.num_blocks = 128, 32
    assert lib.msa_workspace_bytes(ctypes.byref(p), 64, 8, 0) > 0
    p.block_size, p.num_blocks = 96, 43
    assert lib.msa_workspace_bytes(ctypes.byref(p), 64, 8, 0) == 0
    p.block_size, p.num_blocks = 128, 64     # block count of 64-key blocks with 128-key blocks
    assert lib.msa_workspace_bytes(ctypes.byref(p), 64, 8, 0) == 0


def test_forward_arguments_rejected_on_host(B):
    """msa_fwd rejects a null problem, null or misaligned buffers and a short
    workspace before it touches the device (fake, never dereferenced addresses)."""
    lib = B.lib
    assert lib.msa_fwd(None, *([None] * 8), 0, None) == B.MSA_ERR_INVALID_ARGUMENT
    p = B.msa_problem()
    p.num_docs, p.total_tokens, p.kv_rows = 1, 64, 64
    p.cu_seqlens, p.kv_doc_starts = 4096, 8192
    p.num_q_heads, p.num_index_heads, p.num_kv_heads = 16, 1, 1
    p.head_dim, p.block_size, p.query_chunk, p.topk = 128, 64, 8, 4
    p.num_blocks, p.num_chunks, p.softmax_scale = 1, 8, 0.1
    bufs = [1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20, 6 << 20, 7 << 20, 8 << 20]  # q k v sel o lse status ws
    ws_ok = 256
    for i in range(len(bufs)):
        nulled = list(bufs)
        nulled[i] = None
        assert lib.msa_fwd(ctypes.byref(p), *nulled, ws_ok, None) == B.MSA_ERR_INVALID_ARGUMENT, i
        shifted = list(bufs)
        shifted[i] += 4
        assert lib.msa_fwd(ctypes.byref(p), *shifted, ws_ok, None) == B.MSA_ERR_INVALID_ARGUMENT, i
    assert lib.msa_fwd(ctypes.byref(p), *bufs, 8, None) == B.MSA_ERR_INVALID_ARGUMENT   # ws < 8 (N + 1), rounded
    p.head_dim = 64
    assert lib.msa_fwd(ctypes.byref(p), *bufs, ws_ok, None) == B.MSA_ERR_UNSUPPORTED_SHAPE


def test_selftest_wait_rejects_bad_status_pointer_on_host(B):
    assert B.lib.msa_selftest_wait_timeout(None, None) == B.MSA_ERR_INVALID_ARGUMENT
    assert B.lib.msa_selftest_wait_timeout(4100, None) == B.MSA_ERR_INVALID_ARGUMENT
