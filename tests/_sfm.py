"""Run a ``sfm_inputs.Problem`` through the CUDA library (C-ABI via ctypes)."""
from __future__ import annotations

import numpy as np
import torch

import sparse_shared_kv_gb300 as sfm


def params_of(prob, **over) -> sfm.SfmParams:
    kw = prob.attrs()
    kw.update(over)
    return sfm.make_params(**kw)


def tensors_of(prob) -> sfm.SfmTensors:
    return sfm.make_tensors(prob.t["q"], prob.t["ori_kv"], **prob.tensor_kwargs())


class Runner:
    """Metadata + workspace + outputs for one problem, reusable across calls."""

    def __init__(self, prob, params=None):
        self.prob = prob
        self.params = params or params_of(prob)
        self.tensors = tensors_of(prob)
        dev = prob.t["q"].device
        self.meta = torch.empty(sfm.sfm_metadata_size(self.params), dtype=torch.int32, device=dev)
        nb = sfm.sfm_workspace_size(self.params)
        self.ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
        self.out = torch.empty(prob.num_tokens, prob.num_heads_q, 512, dtype=prob.torch_dtype, device=dev)
        self.lse = torch.empty(prob.num_tokens, prob.num_heads_q, dtype=torch.float32, device=dev) \
            if self.params.return_lse else None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def plan(self, stream=None):
        sfm.sfm_metadata(self.params, self.tensors, self.meta, stream)

    def forward(self, stream=None):
        sfm.sfm_forward(self.params, self.tensors, self.meta, self.prob.softmax_scale, self.out, self.lse,
                        self.ws, self.status, stream)

    def run(self):
        self.status.zero_()
        self.plan()
        self.forward()
        torch.cuda.synchronize()
        return self.out, self.lse, int(self.status.item())


def run(prob, params=None):
    return Runner(prob, params).run()


def _dump_cap(prob):
    """Upper bound of attended positions per query row."""
    cap = 1
    for name in ("ori_sparse_indices", "cmp_sparse_indices"):
        x = prob.t[name]
        if x is not None:                       # ori entries select sparse_block_size tokens each
            cap += x.shape[-1] * (prob.sparse_block_size if name == "ori_sparse_indices" else 1)
    if prob.ori_topk == 0:
        w = prob.max_seqlen_ori_kv
        if prob.ori_mask_mode == 4 and prob.ori_win_left >= 0 and prob.ori_win_right >= 0:
            w = min(w, prob.ori_win_left + prob.ori_win_right + 1)
        cap += w
    if prob.has_cmp_kv and prob.cmp_topk == 0:
        cap += prob.max_seqlen_cmp_kv
    return cap


UNWRITTEN = -2


def debug_rows(prob, cap=None, params=None):
    """The KV rows the attention kernel's resolver handed to its copy warps,
    per query row, through sfm_debug_attended (the real forward with its dump
    on).  Returns (entries, out, lse, status): entries[t] is the int32 array
    of positions 0..counts[t]-1 (-1 skipped, r an ori pool row, r | 1 << 31 a
    cmp pool row; UNWRITTEN where the kernel wrote nothing)."""
    r = Runner(prob, params)
    cap = cap or _dump_cap(prob)
    dev = prob.t["q"].device
    rows = torch.full((prob.num_tokens, cap), UNWRITTEN, dtype=torch.int32, device=dev)
    counts = torch.zeros(prob.num_tokens, dtype=torch.int32, device=dev)
    r.status.zero_()
    r.plan()
    sfm.sfm_debug_attended(r.params, r.tensors, r.meta, prob.softmax_scale, r.out, r.lse, r.ws, rows, cap, counts,
                           r.status)
    torch.cuda.synchronize()
    rows = rows.cpu().numpy()
    counts = counts.cpu().numpy()
    entries = [rows[t, :counts[t]].copy() for t in range(prob.num_tokens)]
    return entries, r.out, r.lse, int(r.status.item())


def split_entries(e):
    """(src, pool row) of the attended entries of one dump row, skipped ones dropped."""
    e = e[e != -1]
    src = (e < 0).astype(np.int32)                       # bit 31: the compressed pool
    row = (e.astype(np.int64) & 0x7FFFFFFF).astype(np.int64)
    return src, row
