"""CPU oracle for deterministic context attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never imports, links or runs it, and the two share no code.

The arithmetic lives in ``rlk_oracle.c`` (plain C, FP64 definition, FP32
canonical fold); this module builds it with gcc and wraps it with ctypes and
numpy.  ``cp.py`` holds the oracle's own context-parallel partition
(contiguous and zigzag) and the emulated CP merge.

Citations name the page and section the code follows:
  * "WS2 Attention PR5 Drift Benchmark" (design doc): Scope; the drift-class
    table; Transformer Engine Reuse (state_i = (out_i, lse_i,
    global_block_index_i), sort by global_block_index, then correction
    arithmetic); Report Contract (merge order global_block_index, downcast at
    final write).
  * "[WS2][Attention] H100 validation and reproduction guide" (issue #294):
    Status (FP32 accumulation, Split-KV disabled, fixed merge order) and
    Acceptance (max abs 0.0 across 2/4/8 ranks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rlk_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "librlk_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, EDUP = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile rlk_oracle.c with gcc (OpenMP, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.rlko_attention_f64.argtypes = [i32, P, P, i32, i32, i32, dbl, i32,
                                           P, P, P, i64, P, P, P]
        lib.rlko_row_block_states_f64.argtypes = [i32, P, P, i32, i32, i32, dbl, i32,
                                                  P, P, P, i32, i64, i32, P, P, i32, P]
        lib.rlko_fold_f32.argtypes = [i32, i32, P, P, P, i32, P, P]
        lib.rlko_decode_paged_f64.argtypes = [i32, i32, i32, i32, dbl, P, P, P,
                                              i32, i32, P, i32, P, P, P]
        lib.rlko_backward_f64.argtypes = [i32, P, i32, i32, i32, dbl, P, P, P, P,
                                          i32, i32, P, P, P]
        lib.rlko_rope_f32.argtypes = [i64, i32, i32, dbl, P, P, P]
        lib.rlko_rope_f64.argtypes = [i64, i32, i32, dbl, P, P, P]
        lib.rlko_num_threads.argtypes = []
        for f in (lib.rlko_attention_f64, lib.rlko_row_block_states_f64, lib.rlko_fold_f32,
                  lib.rlko_decode_paged_f64, lib.rlko_backward_f64, lib.rlko_rope_f32,
                  lib.rlko_rope_f64, lib.rlko_num_threads):
            f.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != OK:
        raise OracleError(f"{what} returned {rc}")


def num_threads() -> int:
    return _load().rlko_num_threads()


def attention_f64(q, k, v, cu_q, cu_k, scale, causal=True, rows=None):
    """Causal (bottom-right) GQA attention by definition, FP64.

    q [Tq, Hq, D], k/v [Tk, Hkv, D] (exact BF16 values as float32),
    cu_q / cu_k [B+1].  Returns (out [n, Hq, D] float64, lse [n, Hq] float64)
    for every token, or for the listed token indices ``rows``.
    """
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    tq, hq, d = q.shape
    hkv = k.shape[1]
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows.shape[0]
    else:
        n = tq
    out = np.empty((n, hq, d), np.float64)
    lse = np.empty((n, hq), np.float64)
    rc = lib.rlko_attention_f64(len(cu_q) - 1, _ptr(cu_q), _ptr(cu_k), hq, hkv, d,
                                float(scale), int(causal), _ptr(q), _ptr(k), _ptr(v),
                                n, _ptr(rows), _ptr(out), _ptr(lse))
    _check(rc, "rlko_attention_f64")
    return out, lse


def row_block_states_f64(q, k, v, cu_q, cu_k, scale, block, token, head, causal=True):
    """FP64 partial states (o_b [nb, D], lse_b [nb]) of one (token, head),
    blocks 0..nb-1 in ascending global_block_index."""
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    d = q.shape[2]
    max_nb = (int(np.max(np.diff(cu_k))) + block - 1) // block + 1
    o = np.empty((max_nb, d), np.float64)
    lse = np.empty((max_nb,), np.float64)
    nb = ctypes.c_int(0)
    rc = lib.rlko_row_block_states_f64(len(cu_q) - 1, _ptr(cu_q), _ptr(cu_k), q.shape[1],
                                       k.shape[1], d, float(scale), int(causal), _ptr(q),
                                       _ptr(k), _ptr(v), int(block), int(token), int(head),
                                       _ptr(o), _ptr(lse), max_nb, ctypes.byref(nb))
    _check(rc, "rlko_row_block_states_f64")
    return o[:nb.value].copy(), lse[:nb.value].copy()


def fold_f32(gbi, o, lse, arrival_order=False):
    """Merge FP32 states of one (row, head).  Canonical: sort by
    global_block_index, then fold; ``arrival_order=True`` folds as given."""
    lib = _load()
    gbi = _i32(gbi)
    o = _f32(o)
    lse = _f32(lse)
    n, d = o.shape
    out = np.empty((d,), np.float32)
    lse_out = np.empty((1,), np.float32)
    rc = lib.rlko_fold_f32(n, d, _ptr(gbi), _ptr(o), _ptr(lse), int(bool(arrival_order)),
                           _ptr(out), _ptr(lse_out))
    if rc == EDUP:
        raise OracleError("duplicate global_block_index")
    _check(rc, "rlko_fold_f32")
    return out, float(lse_out[0])


def decode_paged_f64(q, k_pool, v_pool, page_table, seqlens, scale):
    """One decode token per sequence through a paged KV pool, FP64.
    q [n, Hq, D]; pools [n_pages, page_size, Hkv, D]; page_table [n, max_pages]."""
    lib = _load()
    q, k_pool, v_pool = _f32(q), _f32(k_pool), _f32(v_pool)
    page_table, seqlens = _i32(page_table), _i32(seqlens)
    n, hq, d = q.shape
    n_pages, page_size, hkv, _ = k_pool.shape
    out = np.empty((n, hq, d), np.float64)
    lse = np.empty((n, hq), np.float64)
    rc = lib.rlko_decode_paged_f64(n, hq, hkv, d, float(scale), _ptr(q), _ptr(k_pool),
                                   _ptr(v_pool), n_pages, page_size, _ptr(page_table),
                                   page_table.shape[1], _ptr(seqlens), _ptr(out), _ptr(lse))
    _check(rc, "rlko_decode_paged_f64")
    return out, lse


def backward_f64(q, k, v, dout, cu, scale, only_seq=-1, only_group=-1):
    """dQ, dK, dV of causal GQA attention by definition, FP64.  Entries outside
    ``only_seq`` / ``only_group`` (when given) are NaN."""
    lib = _load()
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    cu = _i32(cu)
    t, hq, d = q.shape
    hkv = k.shape[1]
    dq = np.full((t, hq, d), np.nan)
    dk = np.full((t, hkv, d), np.nan)
    dv = np.full((t, hkv, d), np.nan)
    rc = lib.rlko_backward_f64(len(cu) - 1, _ptr(cu), hq, hkv, d, float(scale), _ptr(q),
                               _ptr(k), _ptr(v), _ptr(dout), int(only_seq), int(only_group),
                               _ptr(dq), _ptr(dk), _ptr(dv))
    _check(rc, "rlko_backward_f64")
    return dq, dk, dv


def rope_f32(x, pos, theta):
    """Canonical FP32 RoPE of rows x [T, H, D] (exact BF16 values) at
    positions pos [T]; returns the BF16 results as float32."""
    lib = _load()
    x = _f32(x)
    pos = _i32(pos)
    t, h, d = x.shape
    assert pos.shape == (t,)
    y = np.empty_like(x)
    _check(lib.rlko_rope_f32(t, h, d, float(theta), _ptr(pos), _ptr(x), _ptr(y)), "rlko_rope_f32")
    return y


def rope_f64(x, pos, theta):
    """The exact rotation of rows x [T, H, D] at positions pos [T], float64."""
    lib = _load()
    x = _f32(x)
    pos = _i32(pos)
    t, h, d = x.shape
    assert pos.shape == (t,)
    y = np.empty(x.shape, np.float64)
    _check(lib.rlko_rope_f64(t, h, d, float(theta), _ptr(pos), _ptr(x), _ptr(y)), "rlko_rope_f64")
    return y


def dlogp_f64(out, w, tok):
    """Log-probability of the selected token per row under a linear head
    ("WS2 Attention PR5 Drift Benchmark", the --include-dlogp paragraph: a
    synthetic FP32 lm_head over the attention output and the selected-token
    log-probability; "[WS2][Attention] H100 validation and reproduction
    guide", Status: dlogp max abs 0.0).  FP64 by definition:
        logit_j = sum_i x_i W_ij            (x: the row's outputs of all heads)
        dlogp   = logit_tok - log sum_j exp(logit_j)
    with the sum of exponentials taken relative to the row's largest logit.
    out: [rows, ...] (flattened per row), w: [width, vocab], tok: [rows]."""
    rows = out.shape[0]
    x = np.asarray(out, np.float64).reshape(rows, -1)
    logits = x @ np.asarray(w, np.float64)
    m = logits.max(axis=1)
    lse = m + np.log(np.exp(logits - m[:, None]).sum(axis=1))
    return logits[np.arange(rows), np.asarray(tok)] - lse
