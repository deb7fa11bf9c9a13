"""CPU oracle for sparse shared-KV MLA attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
and reference legs may import this package.  The library itself never does.

The arithmetic lives in ``sfm_oracle.c`` (plain C, fp64); this module compiles
it with gcc, mirrors its struct with ctypes and converts a
``sfm_inputs.Problem`` (tensors on the host) into that struct.

Pinned by the ``-m "not gpu"`` tests against: hand-derived attended sets of
the pages' examples, brute-force dense masked attention on tiny inputs, the
uniform-attention and identical-row closed forms, dense right-down-causal
attention from torch's SDPA, the context-parallel split invariant, layout
equivalence and CSA == HCA when the indices list every visible slot.
Sink semantics and the metadata contents have no printed value on the pages:
parity for the sink term is unpinned beyond the closed forms that assume the
reading documented in ``sfm_oracle.c``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sfm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleProblem(C.Structure):
    _fields_ = [
        ("q_n", C.c_int32), ("d_qk", C.c_int32), ("d_v", C.c_int32), ("rope_dim", C.c_int32),
        ("batch", C.c_int32), ("q_s", C.c_int32), ("q_t", C.c_int32),
        ("ori_s", C.c_int32), ("cmp_s", C.c_int32),
        ("layout_q", C.c_int32), ("layout_kv", C.c_int32),
        ("dtype", C.c_int32), ("kv_packed", C.c_int32),
        ("ori_bs", C.c_int32), ("cmp_bs", C.c_int32), ("ori_bt_stride", C.c_int32), ("cmp_bt_stride", C.c_int32),
        ("ori_row_stride", C.c_int64), ("cmp_row_stride", C.c_int64),
        ("ori_rows", C.c_int64), ("cmp_rows", C.c_int64),
        ("ori_topk", C.c_int32), ("cmp_topk", C.c_int32), ("cmp_ratio", C.c_int32), ("ori_sbs", C.c_int32),
        ("ori_mask_mode", C.c_int32), ("cmp_mask_mode", C.c_int32), ("win_left", C.c_int32),
        ("win_right", C.c_int32),
        ("has_ori", C.c_int32), ("has_cmp", C.c_int32), ("has_sinks", C.c_int32),
        ("softmax_scale", C.c_double),
        ("q", C.c_void_p), ("ori_kv", C.c_void_p), ("cmp_kv", C.c_void_p),
        ("ori_idx", C.c_void_p), ("cmp_idx", C.c_void_p), ("ori_bt", C.c_void_p), ("cmp_bt", C.c_void_p),
        ("cu_q", C.c_void_p), ("cu_ori", C.c_void_p), ("cu_cmp", C.c_void_p), ("used_q", C.c_void_p),
        ("used_ori", C.c_void_p), ("used_cmp", C.c_void_p), ("residual", C.c_void_p),
        ("sinks", C.c_void_p),
    ]


def _configure(l):
    l.oracle_forward.restype = C.c_int
    l.oracle_forward.argtypes = [C.POINTER(OracleProblem), C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p,
                                 C.c_int32]
    l.oracle_attended.restype = C.c_int64
    l.oracle_attended.argtypes = [C.POINTER(OracleProblem), C.c_int32, C.c_void_p, C.c_void_p, C.c_int64]
    l.oracle_token_info.restype = C.c_int
    l.oracle_token_info.argtypes = [C.POINTER(OracleProblem), C.c_int32, C.c_void_p]
    l.oracle_dec_e4m3.restype = C.c_double
    l.oracle_dec_e4m3.argtypes = [C.c_int32]
    return l


class use_library:
    """Temporarily route every oracle call through another build of the
    oracle source (used by the mutation tests, which plant mistakes in a
    copy of ``sfm_oracle.c`` and check that the pins catch them)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.prev = _lib
        _lib = _configure(C.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.prev
        return False


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(C.CDLL(build()))
        return _lib


_LAYOUT = {"BSND": 0, "TND": 1, "PAGED": 2}


def _host(x: Optional[torch.Tensor]):
    if x is None:
        return None
    assert x.device.type == "cpu", "oracle inputs must be host tensors"
    return x.contiguous()


class _Bound:
    """Holds the struct plus references that keep the host buffers alive."""

    def __init__(self, prob):
        t = {k: _host(v) for k, v in prob.t.items()}
        self.keep = t
        s = OracleProblem()
        s.q_n = prob.num_heads_q
        s.d_qk = prob.d_qk
        s.d_v = prob.head_dim
        s.rope_dim = prob.rope_head_dim
        s.batch = prob.batch_size
        s.q_s = prob.max_seqlen_q if prob.layout_q == "BSND" else 0
        s.q_t = prob.total_q
        s.layout_q = _LAYOUT[prob.layout_q]
        s.layout_kv = _LAYOUT[prob.layout_kv]
        s.dtype = 0 if prob.dtype == "bf16" else 1
        s.kv_packed = {"int8_packed": 1, "fp8_packed": 2}.get(prob.kv_format, 0)
        s.ori_bs = prob.ori_block_size
        s.cmp_bs = prob.cmp_block_size
        ori = t["ori_kv"]
        cmp_ = t["cmp_kv"]
        s.ori_row_stride = prob.ori_row_stride
        s.cmp_row_stride = prob.cmp_row_stride
        s.ori_rows = ori.numel() * ori.element_size() // prob.ori_row_stride if ori is not None else 0
        s.cmp_rows = (cmp_.numel() * cmp_.element_size() // prob.cmp_row_stride) if cmp_ is not None else 0
        if prob.layout_kv == "BSND":
            s.ori_s = ori.shape[1]
            s.cmp_s = cmp_.shape[1] if cmp_ is not None else 0
        s.ori_bt_stride = t["ori_block_table"].shape[1] if t["ori_block_table"] is not None else 0
        s.cmp_bt_stride = t["cmp_block_table"].shape[1] if t["cmp_block_table"] is not None else 0
        s.ori_topk = prob.ori_topk
        s.cmp_topk = prob.cmp_topk
        s.cmp_ratio = prob.cmp_ratio
        s.ori_sbs = getattr(prob, "sparse_block_size", 1)
        s.ori_mask_mode = prob.ori_mask_mode
        s.cmp_mask_mode = prob.cmp_mask_mode
        s.win_left = prob.ori_win_left
        s.win_right = prob.ori_win_right
        s.has_ori = int(prob.has_ori_kv)
        s.has_cmp = int(prob.has_cmp_kv)
        s.has_sinks = int(t["sinks"] is not None)
        s.softmax_scale = prob.softmax_scale

        def ptr(name):
            x = t[name]
            return None if x is None else x.data_ptr()

        s.q = ptr("q")
        s.ori_kv = ptr("ori_kv")
        s.cmp_kv = ptr("cmp_kv")
        s.ori_idx = ptr("ori_sparse_indices")
        s.cmp_idx = ptr("cmp_sparse_indices")
        s.ori_bt = ptr("ori_block_table")
        s.cmp_bt = ptr("cmp_block_table")
        s.cu_q = ptr("cu_seqlens_q")
        s.cu_ori = ptr("cu_seqlens_ori_kv")
        s.cu_cmp = ptr("cu_seqlens_cmp_kv")
        s.used_q = ptr("seqused_q")
        s.used_ori = ptr("seqused_ori_kv")
        s.used_cmp = ptr("seqused_cmp_kv")
        s.residual = ptr("cmp_residual_kv")
        s.sinks = ptr("sinks")
        self.s = s


def forward(prob, tokens: Optional[Sequence[int]] = None, nthreads: int = 0):
    """Oracle O (tokens x q_n x 512, fp64) and LSE (tokens x q_n, fp64)."""
    b = _Bound(prob)
    if tokens is None:
        tokens = range(prob.num_tokens)
    tok = np.ascontiguousarray(np.asarray(list(tokens), dtype=np.int32))
    n = tok.size
    O = np.zeros((n, prob.num_heads_q, prob.head_dim), dtype=np.float64)
    lse = np.zeros((n, prob.num_heads_q), dtype=np.float64)
    rc = lib().oracle_forward(C.byref(b.s), tok.ctypes.data, n, O.ctypes.data, lse.ctypes.data, nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_forward failed with code {rc}")
    return O, lse


def attended(prob, token: int, _bound: Optional[_Bound] = None):
    """Attended (src, pos) pairs of one token: src 0 = ori, 1 = cmp."""
    b = _bound or _Bound(prob)
    n = lib().oracle_attended(C.byref(b.s), token, None, None, 0)
    if n < 0:
        raise RuntimeError(f"oracle_attended failed with code {-n}")
    src = np.zeros(max(n, 1), dtype=np.int32)
    pos = np.zeros(max(n, 1), dtype=np.int32)
    lib().oracle_attended(C.byref(b.s), token, src.ctypes.data, pos.ctypes.data, n)
    return src[:n].copy(), pos[:n].copy()


def attended_all(prob):
    b = _Bound(prob)
    return [attended(prob, t, b) for t in range(prob.num_tokens)]


def dec_e4m3(code: int) -> float:
    """The oracle's FLOAT8_E4M3FN decoder for one byte (for its pins)."""
    return lib().oracle_dec_e4m3(int(code))


def token_info(prob, token: int, _bound: Optional[_Bound] = None):
    """(b, i, q_len, kv_len, cmp_len, residual, p, p_cmp, in_range)."""
    b = _bound or _Bound(prob)
    out = np.zeros(9, dtype=np.int32)
    rc = lib().oracle_token_info(C.byref(b.s), token, out.ctypes.data)
    if rc:
        raise RuntimeError(f"oracle_token_info failed with code {rc}")
    return tuple(int(x) for x in out)
