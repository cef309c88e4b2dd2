"""deterministic_context_attention_gb300 -- Python binding of librlk_attn.so.

The binding only marshals arguments: every step of the attention path runs
in the library's CUDA kernels for sm_103a (include/rlk_attn.h documents each
entry point).  PyTorch supplies device memory and the current stream.  There
is no fallback: if the library is missing or was built for another GPU, the
calls raise.

Entry points (same names as the C ABI):
    rlk_attn_plan_states, rlk_attn_block_manifest_hash,
    rlk_attn_prefill_states, rlk_attn_merge_states, rlk_attn_merge_states_noalloc,
    rlk_attn_prefill, rlk_attn_prefill_rope,
    rlk_attn_decode_paged, rlk_attn_backward, rlk_attn_workspace_size,
    rlk_attn_check_device_error, rlk_attn_last_error, rlk_attn_core_id
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "librlk_attn.so")

RLK_OK = 0
STATUS_NAMES = {
    0: "RLK_OK", 1: "RLK_ERR_INVALID_ARGUMENT", 2: "RLK_ERR_UNSUPPORTED",
    3: "RLK_ERR_WORKSPACE_TOO_SMALL", 4: "RLK_ERR_DUPLICATE_BLOCK", 5: "RLK_ERR_MISSING_BLOCK",
    6: "RLK_ERR_DEVICE_TIMEOUT", 7: "RLK_ERR_CUDA", 8: "RLK_ERR_BAD_PAGE", 9: "RLK_ERR_BAD_STATE_TABLE",
}
RLK_OP_MERGE, RLK_OP_BACKWARD, RLK_OP_DECODE_SPLIT = 1, 2, 3
CONTIGUOUS, ZIGZAG = 0, 1


class RlkError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {message}")


class rlk_attn_params(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("causal", ctypes.c_int32),
                ("kv_block_size", ctypes.c_int32), ("cp_size", ctypes.c_int32),
                ("cp_layout", ctypes.c_int32)]


# numpy view of rlk_attn_slab (32 bytes)
SLAB_DTYPE = np.dtype([("seq", "<i4"), ("block", "<i4"), ("row_begin", "<i4"), ("row_count", "<i4"),
                       ("offset", "<i8"), ("producer", "<i4"), ("reserved", "<i4")])


def make_params(num_seqs, num_q_heads=32, num_kv_heads=8, kv_block_size=128, cp_size=1,
                cp_layout=ZIGZAG, softmax_scale=None, head_dim=128) -> rlk_attn_params:
    if softmax_scale is None:
        softmax_scale = 1.0 / float(np.sqrt(head_dim))
    return rlk_attn_params(int(num_seqs), int(num_q_heads), int(num_kv_heads), int(head_dim),
                           float(softmax_scale), 1, int(kv_block_size), int(cp_size), int(cp_layout))


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def load():
    """Load librlk_attn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "deterministic_context_attention_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        PP = ctypes.POINTER(rlk_attn_params)
        sig = {
            "rlk_attn_plan_states": [PP, P, P, i32, i64, P, i64, P, P],
            "rlk_attn_block_manifest_hash": [PP, P, P, P],
            "rlk_attn_prefill_states": [PP, P, P, P, P, P, i32, i64, P, P, P],
            "rlk_attn_merge_states": [PP, P, P, P, i64, P, P, i64, P, P, P, P, sz, P],
            "rlk_attn_merge_states_noalloc": [PP, P, P, P, i64, P, P, i64, P, P, P, P],
            "rlk_attn_prefill": [PP, P, P, P, P, P, i32, P, P, P, P],
            "rlk_attn_prefill_rope": [PP, P, P, P, P, P, i32, P, i32, P, P, P, P],
            "rlk_attn_decode_paged": [PP, P, P, P, i32, i32, P, i32, P, P, P, P, P],
            "rlk_attn_decode_paged_splitk": [PP, P, P, P, i32, i32, P, i32, P, i32, P, P, P, P, sz, P],
            "rlk_attn_decode_auto_split": [PP, P, i32],
            "rlk_attn_rope_table": [ctypes.c_double, i32, P],
            "rlk_attn_rope": [PP, P, P, i32, P, P, P, i32, P],
            "rlk_attn_rope_qk": [PP, P, P, P, P, P, P, P, i32, P],
            "rlk_attn_decode_paged_rope": [PP, P, P, P, i32, i32, P, i32, P, P, i32, P, P, P, P],
            "rlk_attn_decode_paged_splitk_rope": [PP, P, P, P, i32, i32, P, i32, P, i32, P, i32, P, P, P, P, sz, P],
            "rlk_attn_backward": [PP, P, P, P, P, P, P, P, i32, P, P, P, P, sz, P],
            "rlk_attn_workspace_size": [PP, i32, P, P],
            "rlk_attn_check_device_error": [P],
            "rlk_attn_selftest_wait_timeout": [P],
            "rlk_attn_last_error": [],
            "rlk_attn_core_id": [],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        lib.rlk_attn_workspace_size.restype = ctypes.c_size_t
        lib.rlk_attn_last_error.restype = ctypes.c_char_p
        lib.rlk_attn_core_id.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _i32_host(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(x):
    """Device pointer of a torch tensor, a numpy array's host pointer, or NULL."""
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return x.ctypes.data_as(ctypes.c_void_p)
    if isinstance(x, int):
        return ctypes.c_void_p(x)
    return ctypes.c_void_p(x.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, where):
    if status != RLK_OK:
        msg = load().rlk_attn_last_error().decode(errors="replace")
        raise RlkError(status, where, msg)


def rlk_attn_core_id() -> str:
    return load().rlk_attn_core_id().decode()


def rlk_attn_last_error() -> str:
    return load().rlk_attn_last_error().decode(errors="replace")


def rlk_attn_plan_states(params, cu_seqlens_q, cu_seqlens_k, cp_rank=-1, pair_base=0):
    """Host-only block plan: returns (slabs as a SLAB_DTYPE array, n_pairs)."""
    lib = load()
    cq, ck = _i32_host(cu_seqlens_q), _i32_host(cu_seqlens_k)
    n_slabs, n_pairs = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib.rlk_attn_plan_states(ctypes.byref(params), _ptr(cq), _ptr(ck), int(cp_rank), int(pair_base),
                                    None, 0, ctypes.byref(n_slabs), ctypes.byref(n_pairs)),
           "rlk_attn_plan_states")
    slabs = np.zeros(n_slabs.value, SLAB_DTYPE)
    _check(lib.rlk_attn_plan_states(ctypes.byref(params), _ptr(cq), _ptr(ck), int(cp_rank), int(pair_base),
                                    _ptr(slabs), n_slabs.value, ctypes.byref(n_slabs),
                                    ctypes.byref(n_pairs)), "rlk_attn_plan_states")
    return slabs, n_pairs.value


def rlk_attn_block_manifest_hash(params, cu_seqlens_q, cu_seqlens_k) -> int:
    lib = load()
    cq, ck = _i32_host(cu_seqlens_q), _i32_host(cu_seqlens_k)
    h = ctypes.c_uint64(0)
    _check(lib.rlk_attn_block_manifest_hash(ctypes.byref(params), _ptr(cq), _ptr(ck), ctypes.byref(h)),
           "rlk_attn_block_manifest_hash")
    return h.value


def rlk_attn_workspace_size(params, op, cu_seqlens_q, cu_seqlens_k=None) -> int:
    """RLK_OP_DECODE_SPLIT: pass the decode context lengths as cu_seqlens_k
    (cu_seqlens_q may be None)."""
    cq = None if cu_seqlens_q is None else _i32_host(cu_seqlens_q)
    ck = _i32_host(cu_seqlens_k if cu_seqlens_k is not None else cu_seqlens_q)
    return int(load().rlk_attn_workspace_size(ctypes.byref(params), int(op), _ptr(cq), _ptr(ck)))


def rlk_attn_prefill_states(params, q, k, v, cu_seqlens_q, cu_seqlens_k, cp_rank, pair_base, state_o,
                            state_lse, stream=None):
    cq, ck = _i32_host(cu_seqlens_q), _i32_host(cu_seqlens_k)
    _check(load().rlk_attn_prefill_states(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(cq), _ptr(ck),
                                          int(cp_rank), int(pair_base), _ptr(state_o), _ptr(state_lse),
                                          _stream(stream)), "rlk_attn_prefill_states")


def _state_pairs(state_lse, n_state_pairs):
    """The state table's (row, head) pair count: given, or the length of the
    state_lse tensor."""
    if n_state_pairs is not None:
        return int(n_state_pairs)
    if not hasattr(state_lse, "numel"):
        raise ValueError("n_state_pairs is required when state_lse is not a tensor")
    return int(state_lse.numel())


def rlk_attn_merge_states(params, cu_seqlens_q, cu_seqlens_k, slabs, n_slabs, state_o, state_lse, out_f32,
                          out_bf16, lse, workspace, workspace_bytes=None, stream=None, n_state_pairs=None):
    cq, ck = _i32_host(cu_seqlens_q), _i32_host(cu_seqlens_k)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().rlk_attn_merge_states(ctypes.byref(params), _ptr(cq), _ptr(ck), _ptr(slabs), int(n_slabs),
                                        _ptr(state_o), _ptr(state_lse), _state_pairs(state_lse, n_state_pairs),
                                        _ptr(out_f32), _ptr(out_bf16), _ptr(lse), _ptr(workspace),
                                        int(workspace_bytes), _stream(stream)),
           "rlk_attn_merge_states")


def rlk_attn_merge_states_noalloc(params, cu_seqlens_q, cu_seqlens_k, slabs, n_slabs, state_o, state_lse,
                                  out_f32, out_bf16, lse, stream=None, n_state_pairs=None):
    """rlk_attn_merge_states for callers that cannot allocate: the index
    scratch is the library's own device array (see the C header for its
    limit and for the rule that overlapping calls race)."""
    cq, ck = _i32_host(cu_seqlens_q), _i32_host(cu_seqlens_k)
    _check(load().rlk_attn_merge_states_noalloc(ctypes.byref(params), _ptr(cq), _ptr(ck), _ptr(slabs),
                                                int(n_slabs), _ptr(state_o), _ptr(state_lse),
                                                _state_pairs(state_lse, n_state_pairs), _ptr(out_f32),
                                                _ptr(out_bf16), _ptr(lse), _stream(stream)),
           "rlk_attn_merge_states_noalloc")


def rlk_attn_prefill(params, q, k, v, cu_seqlens_q, cu_seqlens_k, cp_rank, out_f32, out_bf16, lse,
                     stream=None):
    cq, ck = _i32_host(cu_seqlens_q), _i32_host(cu_seqlens_k)
    _check(load().rlk_attn_prefill(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(cq), _ptr(ck),
                                   int(cp_rank), _ptr(out_f32), _ptr(out_bf16), _ptr(lse), _stream(stream)),
           "rlk_attn_prefill")


def rlk_attn_prefill_rope(params, q, k, v, cu_seqlens_q, cu_seqlens_k, cp_rank, rope_table, rope_max_pos, out_f32,
                          out_bf16, lse, stream=None):
    """rlk_attn_prefill with the pre-RoPE queries rotated inside the kernel."""
    cq, ck = _i32_host(cu_seqlens_q), _i32_host(cu_seqlens_k)
    _check(load().rlk_attn_prefill_rope(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(cq), _ptr(ck),
                                        int(cp_rank), _ptr(rope_table), int(rope_max_pos), _ptr(out_f32),
                                        _ptr(out_bf16), _ptr(lse), _stream(stream)), "rlk_attn_prefill_rope")


def rlk_attn_decode_paged(params, q, k_pool, v_pool, n_pages, page_size, page_table, max_pages, seqlens,
                          out_f32, out_bf16, lse, stream=None):
    sl = _i32_host(seqlens)
    _check(load().rlk_attn_decode_paged(ctypes.byref(params), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                        int(n_pages), int(page_size), _ptr(page_table), int(max_pages),
                                        _ptr(sl), _ptr(out_f32), _ptr(out_bf16), _ptr(lse), _stream(stream)),
           "rlk_attn_decode_paged")


def rlk_attn_decode_paged_splitk(params, q, k_pool, v_pool, n_pages, page_size, page_table, max_pages, seqlens,
                                 split_k, out_f32, out_bf16, lse, workspace, workspace_bytes=None, stream=None):
    sl = _i32_host(seqlens)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().rlk_attn_decode_paged_splitk(ctypes.byref(params), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                               int(n_pages), int(page_size), _ptr(page_table), int(max_pages),
                                               _ptr(sl), int(split_k), _ptr(out_f32), _ptr(out_bf16), _ptr(lse),
                                               _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "rlk_attn_decode_paged_splitk")


def rlk_attn_decode_auto_split(params, seqlens, num_sms) -> int:
    """Split factor rlk_attn_decode_paged_splitk picks for split_k=0 (-1: invalid input)."""
    sl = _i32_host(seqlens)
    return int(load().rlk_attn_decode_auto_split(ctypes.byref(params), _ptr(sl), int(num_sms)))


def rlk_attn_selftest_wait_timeout(stream=None):
    """Launch the bounded-wait self-test (reports a device timeout)."""
    _check(load().rlk_attn_selftest_wait_timeout(_stream(stream)), "rlk_attn_selftest_wait_timeout")


def rlk_attn_rope_table(theta, max_pos):
    """Host RoPE table [max_pos, 128] float32 (cos 64 | sin 64 per position)."""
    table = np.empty((int(max_pos), 128), np.float32)
    _check(load().rlk_attn_rope_table(float(theta), int(max_pos), _ptr(table)), "rlk_attn_rope_table")
    return table


def rlk_attn_rope(params, x, y, num_heads, cu_seqlens, pos_offset, table, max_pos, stream=None):
    cu = _i32_host(cu_seqlens)
    po = None if pos_offset is None else _i32_host(pos_offset)
    _check(load().rlk_attn_rope(ctypes.byref(params), _ptr(x), _ptr(y), int(num_heads), _ptr(cu), _ptr(po),
                                _ptr(table), int(max_pos), _stream(stream)), "rlk_attn_rope")


def rlk_attn_rope_qk(params, q, q_out, k, k_out, cu_seqlens, pos_offset, table, max_pos, stream=None):
    """RoPE of the queries and keys of the same tokens in one launch."""
    cu = _i32_host(cu_seqlens)
    po = None if pos_offset is None else _i32_host(pos_offset)
    _check(load().rlk_attn_rope_qk(ctypes.byref(params), _ptr(q), _ptr(q_out), _ptr(k), _ptr(k_out), _ptr(cu),
                                   _ptr(po), _ptr(table), int(max_pos), _stream(stream)), "rlk_attn_rope_qk")


def rlk_attn_decode_paged_rope(params, q, k_pool, v_pool, n_pages, page_size, page_table, max_pages, seqlens,
                               rope_table, rope_max_pos, out_f32, out_bf16, lse, stream=None):
    sl = _i32_host(seqlens)
    _check(load().rlk_attn_decode_paged_rope(ctypes.byref(params), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                             int(n_pages), int(page_size), _ptr(page_table), int(max_pages),
                                             _ptr(sl), _ptr(rope_table), int(rope_max_pos), _ptr(out_f32),
                                             _ptr(out_bf16), _ptr(lse), _stream(stream)),
           "rlk_attn_decode_paged_rope")


def rlk_attn_decode_paged_splitk_rope(params, q, k_pool, v_pool, n_pages, page_size, page_table, max_pages, seqlens,
                                      split_k, rope_table, rope_max_pos, out_f32, out_bf16, lse, workspace,
                                      workspace_bytes=None, stream=None):
    sl = _i32_host(seqlens)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().rlk_attn_decode_paged_splitk_rope(ctypes.byref(params), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                                    int(n_pages), int(page_size), _ptr(page_table), int(max_pages),
                                                    _ptr(sl), int(split_k), _ptr(rope_table), int(rope_max_pos),
                                                    _ptr(out_f32), _ptr(out_bf16), _ptr(lse), _ptr(workspace),
                                                    int(workspace_bytes), _stream(stream)),
           "rlk_attn_decode_paged_splitk_rope")


def rlk_attn_backward(params, q, k, v, out_f32, dout, lse, cu_seqlens, cp_rank, dq, dk, dv, workspace,
                      workspace_bytes=None, stream=None):
    cu = _i32_host(cu_seqlens)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().rlk_attn_backward(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(out_f32), _ptr(dout),
                                    _ptr(lse), _ptr(cu), int(cp_rank), _ptr(dq), _ptr(dk), _ptr(dv),
                                    _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "rlk_attn_backward")


def rlk_attn_check_device_error(stream=None):
    _check(load().rlk_attn_check_device_error(_stream(stream)), "rlk_attn_check_device_error")
