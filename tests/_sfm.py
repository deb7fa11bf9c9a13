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


def run(prob):
    return Runner(prob).run()


def debug_sets(prob, cap=None):
    """Resolved attended rows per token as [(src, pos), ...] in kernel order."""
    params = params_of(prob)
    tens = tensors_of(prob)
    if cap is None:
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
    dev = prob.t["q"].device
    rows = torch.full((prob.num_tokens, cap), -2, dtype=torch.int32, device=dev)
    counts = torch.zeros(prob.num_tokens, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfm.sfm_debug_attended(params, tens, rows, cap, counts, status)
    torch.cuda.synchronize()
    rows = rows.cpu().numpy()
    counts = counts.cpu().numpy()
    out = []
    for t in range(prob.num_tokens):
        r = rows[t, :counts[t]]
        r = r[r >= 0]
        src = (r >> 30) & 1
        pos = r & 0x3FFFFFFF
        out.append((src.astype(np.int32), pos.astype(np.int32)))
    return out, int(status.item())
