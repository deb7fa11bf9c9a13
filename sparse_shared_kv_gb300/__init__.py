"""Python binding of the sfm C-ABI (``include/sfm.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``_build/libsfm.so``.  torch is used for device memory and streams.
There is no CPU path: if the library is missing or no CUDA device is present
the calls raise.

Two layers:

* ``sfm_metadata_size`` / ``sfm_workspace_size`` / ``sfm_metadata`` /
  ``sfm_forward`` / ``sfm_debug_attended`` / ``sfm_error_string`` -- the C
  entry points with the same names, taking ``SfmParams`` / ``SfmTensors``
  ctypes structs and raw device pointers;
* ``sparse_flash_mla_metadata`` / ``sparse_flash_mla`` -- the two-call torch
  API of the "sparse_flash_mla" doc (函数原型), building those structs from
  tensors and keyword attributes.
"""
from __future__ import annotations

import ctypes as C
import math
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsfm.so")

BSND, TND, PAGED = 0, 1, 2
BF16, FP16 = 0, 1
KV_PLAIN, KV_INT8_PACKED, KV_FP8_PACKED = 0, 1, 2
SPLIT_BATCH_INVARIANT, SPLIT_OCCUPANCY = 0, 1
_LAYOUTS = {"BSND": BSND, "TND": TND, "PAGED": PAGED, "PA_BBND": PAGED, "PA_BSND": PAGED, "PA_ND": PAGED}

STATUS_BAD_INDEX = 0x01
STATUS_BAD_BLOCK = 0x02
STATUS_BAD_LENGTH = 0x04
STATUS_METADATA_MISMATCH = 0x08
STATUS_WORKSPACE_OVERFLOW = 0x10
STATUS_PLAN_OVERFLOW = 0x20


class SfmParams(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "num_heads_q", "num_heads_kv", "head_dim", "rope_head_dim", "batch_size", "max_seqlen_q", "total_q",
        "max_seqlen_ori_kv", "max_seqlen_cmp_kv", "ori_topk", "cmp_topk", "cmp_ratio", "ori_mask_mode",
        "cmp_mask_mode", "ori_win_left", "ori_win_right", "layout_q", "layout_kv", "has_ori_kv", "has_cmp_kv",
        "dtype", "kv_format", "ori_block_size", "cmp_block_size", "return_lse", "kernel_hint", "sparse_block_size",
        "split_policy")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class SfmTensors(C.Structure):
    _fields_ = [
        ("q", C.c_void_p), ("ori_kv", C.c_void_p), ("ori_row_stride", C.c_int64), ("ori_rows", C.c_int64),
        ("cmp_kv", C.c_void_p), ("cmp_row_stride", C.c_int64), ("cmp_rows", C.c_int64),
        ("ori_sparse_indices", C.c_void_p), ("cmp_sparse_indices", C.c_void_p),
        ("ori_block_table", C.c_void_p), ("ori_block_table_stride", C.c_int32),
        ("cmp_block_table", C.c_void_p), ("cmp_block_table_stride", C.c_int32),
        ("cu_seqlens_q", C.c_void_p), ("cu_seqlens_ori_kv", C.c_void_p), ("cu_seqlens_cmp_kv", C.c_void_p),
        ("seqused_q", C.c_void_p), ("seqused_ori_kv", C.c_void_p), ("seqused_cmp_kv", C.c_void_p),
        ("cmp_residual_kv", C.c_void_p), ("sinks", C.c_void_p),
    ]


EXPORTS = ("sfm_metadata_size", "sfm_workspace_size", "sfm_metadata", "sfm_forward", "sfm_forward_noalloc",
           "sfm_debug_attended", "sfm_set_profile_events", "sfm_error_string", "sfm_abi_version")
NOALLOC_WORKSPACE_BYTES = 32 << 20

_lib = None


def build(force: bool = False) -> str:
    from . import buildlib
    return buildlib.build(force=force)


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"sfm CUDA library not built ({LIB_PATH}); run sparse_shared_kv_gb300.build()")
        l = C.CDLL(LIB_PATH)
        P, T = C.POINTER(SfmParams), C.POINTER(SfmTensors)
        l.sfm_metadata_size.argtypes = [P, C.POINTER(C.c_size_t)]
        l.sfm_workspace_size.argtypes = [P, C.POINTER(C.c_size_t)]
        l.sfm_metadata.argtypes = [P, T, C.c_void_p, C.c_size_t, C.c_void_p]
        l.sfm_forward.argtypes = [P, T, C.c_void_p, C.c_size_t, C.c_float, C.c_void_p, C.c_void_p, C.c_void_p,
                                  C.c_size_t, C.c_void_p, C.c_void_p]
        l.sfm_forward_noalloc.argtypes = [P, T, C.c_void_p, C.c_size_t, C.c_float, C.c_void_p, C.c_void_p,
                                          C.c_void_p, C.c_void_p]
        l.sfm_debug_attended.argtypes = [P, T, C.c_void_p, C.c_size_t, C.c_float, C.c_void_p, C.c_void_p,
                                         C.c_void_p, C.c_size_t, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p,
                                         C.c_void_p]
        l.sfm_set_profile_events.argtypes = [C.c_void_p, C.c_void_p]
        l.sfm_error_string.argtypes = [C.c_int]
        l.sfm_error_string.restype = C.c_char_p
        for n in ("sfm_metadata_size", "sfm_workspace_size", "sfm_metadata", "sfm_forward", "sfm_forward_noalloc",
                  "sfm_debug_attended", "sfm_set_profile_events", "sfm_abi_version"):
            getattr(l, n).restype = C.c_int
        _lib = l
    return _lib


class SfmError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {sfm_error_string(code)} ({code})")
        self.code = code


def _check(fn, code):
    if code != 0:
        raise SfmError(fn, code)


def _ptr(x: Optional[torch.Tensor]):
    if x is None:
        return None
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---------------------------------------------------------------------------
# the C entry points
# ---------------------------------------------------------------------------
def sfm_set_profile_events(begin=None, end=None) -> None:
    """Record ``begin`` / ``end`` (torch.cuda.Event) around the main attention
    kernel of the following sfm_forward calls; ``None, None`` turns it off."""
    for ev in (begin, end):
        if ev is not None and ev.cuda_event == 0:
            ev.record()          # torch creates the underlying cudaEvent_t lazily
    b = begin.cuda_event if begin is not None else None
    e = end.cuda_event if end is not None else None
    _check("sfm_set_profile_events", lib().sfm_set_profile_events(b, e))


def sfm_error_string(code: int) -> str:
    return lib().sfm_error_string(code).decode()


def sfm_abi_version() -> int:
    return lib().sfm_abi_version()


def sfm_metadata_size(params: SfmParams) -> int:
    n = C.c_size_t(0)
    _check("sfm_metadata_size", lib().sfm_metadata_size(C.byref(params), C.byref(n)))
    return n.value


def sfm_workspace_size(params: SfmParams) -> int:
    n = C.c_size_t(0)
    _check("sfm_workspace_size", lib().sfm_workspace_size(C.byref(params), C.byref(n)))
    return n.value


def sfm_metadata(params: SfmParams, tensors: SfmTensors, metadata: torch.Tensor, stream=None) -> None:
    assert metadata.dtype == torch.int32 and metadata.is_cuda and metadata.is_contiguous()
    _check("sfm_metadata", lib().sfm_metadata(C.byref(params), C.byref(tensors), metadata.data_ptr(),
                                              metadata.numel(), _stream(stream)))


def sfm_forward(params: SfmParams, tensors: SfmTensors, metadata: torch.Tensor, softmax_scale: float,
                out: torch.Tensor, lse: Optional[torch.Tensor], workspace: Optional[torch.Tensor],
                status: Optional[torch.Tensor] = None, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("sfm_forward", lib().sfm_forward(
        C.byref(params), C.byref(tensors), metadata.data_ptr(), metadata.numel(), C.c_float(softmax_scale),
        out.data_ptr(), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)))


def sfm_forward_noalloc(params: SfmParams, tensors: SfmTensors, metadata: torch.Tensor, softmax_scale: float,
                        out: torch.Tensor, lse: Optional[torch.Tensor], status: Optional[torch.Tensor] = None,
                        stream=None) -> None:
    """sfm_forward with the library's fixed device workspace (no allocation)."""
    _check("sfm_forward_noalloc", lib().sfm_forward_noalloc(
        C.byref(params), C.byref(tensors), metadata.data_ptr(), metadata.numel(), C.c_float(softmax_scale),
        out.data_ptr(), _ptr(lse), _ptr(status), _stream(stream)))


def sfm_debug_attended(params: SfmParams, tensors: SfmTensors, metadata: torch.Tensor, softmax_scale: float,
                       out: torch.Tensor, lse: Optional[torch.Tensor], workspace: Optional[torch.Tensor],
                       rows: torch.Tensor, cap: int, counts: torch.Tensor, status: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """sfm_forward that also records the KV rows the attention kernel's
    resolver hands to its copy warps (rows[t * cap + k], see include/sfm.h)."""
    assert rows.dtype == torch.int32 and counts.dtype == torch.int32
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("sfm_debug_attended", lib().sfm_debug_attended(
        C.byref(params), C.byref(tensors), metadata.data_ptr(), metadata.numel(), C.c_float(softmax_scale),
        out.data_ptr(), _ptr(lse), _ptr(workspace), ws_bytes, rows.data_ptr(), cap, counts.data_ptr(),
        _ptr(status), _stream(stream)))


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _rows_of(kv: Optional[torch.Tensor], row_stride: int) -> int:
    if kv is None:
        return 0
    return kv.numel() * kv.element_size() // row_stride


def make_tensors(q, ori_kv, *, cmp_kv=None, ori_sparse_indices=None, cmp_sparse_indices=None,
                 ori_block_table=None, cmp_block_table=None, cu_seqlens_q=None, cu_seqlens_ori_kv=None,
                 cu_seqlens_cmp_kv=None, seqused_q=None, seqused_ori_kv=None, seqused_cmp_kv=None,
                 cmp_residual_kv=None, sinks=None, ori_row_stride=None, cmp_row_stride=None) -> SfmTensors:
    """SfmTensors from device tensors.  KV row strides default to the
    tensor's last-dim size in bytes (the stride of dim -3 for padded rows)."""
    t = SfmTensors()

    def stride_of(kv, given):
        if given is not None:
            return int(given)
        return kv.stride(-3) * kv.element_size() if kv.dim() >= 3 else kv.stride(0) * kv.element_size()

    for name in ("ori_sparse_indices", "cmp_sparse_indices", "ori_block_table", "cmp_block_table",
                 "cu_seqlens_q", "cu_seqlens_ori_kv", "cu_seqlens_cmp_kv", "seqused_q", "seqused_ori_kv",
                 "seqused_cmp_kv", "cmp_residual_kv"):
        x = locals()[name]
        if x is not None:
            assert x.dtype == torch.int32 and x.is_contiguous(), name
    t.q = _ptr(q)
    t.ori_kv = _ptr(ori_kv)
    t.ori_row_stride = stride_of(ori_kv, ori_row_stride)
    t.ori_rows = _rows_of(ori_kv, t.ori_row_stride)
    if cmp_kv is not None:
        t.cmp_kv = _ptr(cmp_kv)
        t.cmp_row_stride = stride_of(cmp_kv, cmp_row_stride)
        t.cmp_rows = _rows_of(cmp_kv, t.cmp_row_stride)
    t.ori_sparse_indices = _ptr(ori_sparse_indices)
    t.cmp_sparse_indices = _ptr(cmp_sparse_indices)
    t.ori_block_table = _ptr(ori_block_table)
    t.ori_block_table_stride = ori_block_table.shape[-1] if ori_block_table is not None else 0
    t.cmp_block_table = _ptr(cmp_block_table)
    t.cmp_block_table_stride = cmp_block_table.shape[-1] if cmp_block_table is not None else 0
    t.cu_seqlens_q = _ptr(cu_seqlens_q)
    t.cu_seqlens_ori_kv = _ptr(cu_seqlens_ori_kv)
    t.cu_seqlens_cmp_kv = _ptr(cu_seqlens_cmp_kv)
    t.seqused_q = _ptr(seqused_q)
    t.seqused_ori_kv = _ptr(seqused_ori_kv)
    t.seqused_cmp_kv = _ptr(seqused_cmp_kv)
    t.cmp_residual_kv = _ptr(cmp_residual_kv)
    t.sinks = _ptr(sinks)
    return t


def make_params(**kw) -> SfmParams:
    p = SfmParams()
    defaults = dict(num_heads_kv=1, head_dim=512, rope_head_dim=0, total_q=0, max_seqlen_cmp_kv=0, ori_topk=0,
                    cmp_topk=0, cmp_ratio=1, ori_mask_mode=4, cmp_mask_mode=3, ori_win_left=-1, ori_win_right=-1,
                    layout_q=BSND, layout_kv=BSND, has_ori_kv=1, has_cmp_kv=0, dtype=BF16, kv_format=KV_PLAIN,
                    ori_block_size=0, cmp_block_size=0, return_lse=0, kernel_hint=0, sparse_block_size=1,
                    split_policy=SPLIT_BATCH_INVARIANT)
    defaults.update(kw)
    for k, v in defaults.items():
        if k in ("layout_q", "layout_kv") and isinstance(v, str):
            v = _LAYOUTS[v]
        if k == "dtype" and isinstance(v, (str, torch.dtype)):
            v = BF16 if v in ("bf16", torch.bfloat16) else FP16
        setattr(p, k, int(v))
    return p


# ---------------------------------------------------------------------------
# the two-call torch API
# ---------------------------------------------------------------------------
@dataclass
class Metadata:
    """Device int32 plan plus the params it was built for."""
    tensor: torch.Tensor
    params: SfmParams


def sparse_flash_mla_metadata(num_heads_q: int, num_heads_kv: int, head_dim: int, *, cu_seqlens_q=None,
                              cu_seqlens_ori_kv=None, cu_seqlens_cmp_kv=None, seqused_q=None,
                              seqused_ori_kv=None, seqused_cmp_kv=None, cmp_residual_kv=None, batch_size=0,
                              max_seqlen_q=0, max_seqlen_ori_kv=0, max_seqlen_cmp_kv=0, total_q=0, ori_topk=0,
                              cmp_topk=0, cmp_ratio=1, ori_mask_mode=4, cmp_mask_mode=3, ori_win_left=-1,
                              ori_win_right=-1, layout_q="BSND", layout_kv="BSND", has_ori_kv=True,
                              has_cmp_kv=True, dtype=torch.bfloat16, kv_format=KV_PLAIN, rope_head_dim=0,
                              ori_block_size=0, cmp_block_size=0, return_softmax_lse=False,
                              sparse_block_size=1, batch_invariant=True, device=None,
                              stream=None) -> Metadata:
    """Enqueue the device planner and return its plan (two-call contract).

    ``batch_invariant=False`` selects the occupancy split policy: small
    batches are cut into more chunks so they fill the SMs, at the price of a
    row's rounding depending on the batch size."""
    if layout_q == "TND" and cu_seqlens_q is not None:
        batch_size = cu_seqlens_q.numel() - 1
    params = make_params(
        num_heads_q=num_heads_q, num_heads_kv=num_heads_kv, head_dim=head_dim, rope_head_dim=rope_head_dim,
        batch_size=batch_size, max_seqlen_q=max_seqlen_q, total_q=total_q, max_seqlen_ori_kv=max_seqlen_ori_kv,
        max_seqlen_cmp_kv=max_seqlen_cmp_kv, ori_topk=ori_topk, cmp_topk=cmp_topk, cmp_ratio=cmp_ratio,
        ori_mask_mode=ori_mask_mode, cmp_mask_mode=cmp_mask_mode, ori_win_left=ori_win_left,
        ori_win_right=ori_win_right, layout_q=layout_q, layout_kv=layout_kv, has_ori_kv=int(has_ori_kv),
        has_cmp_kv=int(has_cmp_kv), dtype=dtype, kv_format=kv_format, ori_block_size=ori_block_size,
        cmp_block_size=cmp_block_size, return_lse=int(return_softmax_lse), sparse_block_size=sparse_block_size,
        split_policy=SPLIT_BATCH_INVARIANT if batch_invariant else SPLIT_OCCUPANCY)
    lengths = make_tensors(None, None, cu_seqlens_q=cu_seqlens_q, cu_seqlens_ori_kv=cu_seqlens_ori_kv,
                           cu_seqlens_cmp_kv=cu_seqlens_cmp_kv, seqused_q=seqused_q, seqused_ori_kv=seqused_ori_kv,
                           seqused_cmp_kv=seqused_cmp_kv, cmp_residual_kv=cmp_residual_kv, ori_row_stride=0)
    if device is None:
        device = torch.device("cuda", torch.cuda.current_device())
    md = torch.empty(sfm_metadata_size(params), dtype=torch.int32, device=device)
    sfm_metadata(params, lengths, md, stream)
    return Metadata(md, params)


def sparse_flash_mla(q: torch.Tensor, *, metadata: Metadata, ori_kv=None, cmp_kv=None, ori_sparse_indices=None,
                     cmp_sparse_indices=None, ori_block_table=None, cmp_block_table=None, cu_seqlens_q=None,
                     cu_seqlens_ori_kv=None, cu_seqlens_cmp_kv=None, seqused_q=None, seqused_ori_kv=None,
                     seqused_cmp_kv=None, cmp_residual_kv=None, sinks=None, softmax_scale: float = 1.0,
                     ori_row_stride=None, cmp_row_stride=None, out=None, lse=None, workspace=None,
                     status=None, stream=None):
    """Attention output (q's layout, 512 dims per head) and LSE (fp32, or None
    when the plan was made without return_softmax_lse)."""
    params = metadata.params
    tensors = make_tensors(q, ori_kv, cmp_kv=cmp_kv, ori_sparse_indices=ori_sparse_indices,
                           cmp_sparse_indices=cmp_sparse_indices, ori_block_table=ori_block_table,
                           cmp_block_table=cmp_block_table, cu_seqlens_q=cu_seqlens_q,
                           cu_seqlens_ori_kv=cu_seqlens_ori_kv, cu_seqlens_cmp_kv=cu_seqlens_cmp_kv,
                           seqused_q=seqused_q, seqused_ori_kv=seqused_ori_kv, seqused_cmp_kv=seqused_cmp_kv,
                           cmp_residual_kv=cmp_residual_kv, sinks=sinks, ori_row_stride=ori_row_stride,
                           cmp_row_stride=cmp_row_stride)
    if out is None:
        out = torch.empty(q.shape[:-1] + (512,), dtype=q.dtype, device=q.device)
    if lse is None and params.return_lse:
        lse = torch.empty(q.shape[:-1].numel(), dtype=torch.float32, device=q.device)
    if workspace is None:
        nb = sfm_workspace_size(params)
        workspace = torch.empty(max(nb, 1), dtype=torch.uint8, device=q.device) if nb else None
    sfm_forward(params, tensors, metadata.tensor, softmax_scale, out, lse if params.return_lse else None,
                workspace, status, stream)
    return out, lse
