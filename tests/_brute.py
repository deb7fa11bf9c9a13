"""Brute-force dense masked attention (test helper, numpy/fp64).

A second formulation of the same definition, structured differently from the
oracle: for one query row it scores *every* ori position in [0, kv_len) and
*every* cmp slot in [0, cmp_len), builds a multiplicity vector from vectorised
mask comparisons and index histograms (no enumeration of an attended list),
and takes the masked softmax over the dense vector.  Element decoding uses
torch/numpy conversions, not the oracle's bit decoders.
"""
from __future__ import annotations

import numpy as np
import torch


def _rows_f64(prob, which: str) -> np.ndarray:
    """All rows of a cache as an (nrows, d_qk) float64 array (packed rows dequantised)."""
    x = prob.t[which]
    stride = prob.ori_row_stride if which == "ori_kv" else prob.cmp_row_stride
    raw = x.contiguous().view(torch.uint8).reshape(-1, stride).numpy()
    if prob.kv_format in ("int8_packed", "fp8_packed"):
        if prob.kv_format == "fp8_packed":
            codes = torch.from_numpy(np.ascontiguousarray(raw[:, :512]))
            nope = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
        else:
            nope = raw[:, :512].view(np.int8).astype(np.float64)
        r = prob.rope_head_dim
        scales = np.ascontiguousarray(raw[:, 512 + 2 * r:512 + 2 * r + 16]).view(np.float32).astype(np.float64)
        k = nope * np.repeat(scales, 128, axis=1)
        if r:
            rope_t = torch.from_numpy(np.ascontiguousarray(raw[:, 512:512 + 2 * r])).view(prob.torch_dtype)
            k = np.concatenate([k, rope_t.to(torch.float64).numpy()], axis=1)
        return k
    vals = torch.from_numpy(np.ascontiguousarray(raw[:, :prob.head_dim * 2])).view(prob.torch_dtype)
    return vals.to(torch.float64).numpy()


def lengths(prob, t: int):
    """(b, i, q_len, kv_len, cmp_len, residual) of token t, from the tensors."""
    T = prob.t
    if prob.layout_q == "BSND":
        b, i = divmod(t, prob.max_seqlen_q)
        qcap = prob.max_seqlen_q
    else:
        cu = T["cu_seqlens_q"].tolist()
        b = max(k for k in range(prob.batch_size) if cu[k] <= t)
        i = t - cu[b]
        qcap = cu[b + 1] - cu[b]
    q_len = int(T["seqused_q"][b]) if T["seqused_q"] is not None else qcap
    if T["seqused_ori_kv"] is not None:
        kv = int(T["seqused_ori_kv"][b])
    elif prob.layout_kv == "TND":
        kv = int(T["cu_seqlens_ori_kv"][b + 1] - T["cu_seqlens_ori_kv"][b])
    else:
        kv = T["ori_kv"].shape[1]
    cl = 0
    if prob.has_cmp_kv:
        if T["seqused_cmp_kv"] is not None:
            cl = int(T["seqused_cmp_kv"][b])
        elif prob.layout_kv == "TND":
            cl = int(T["cu_seqlens_cmp_kv"][b + 1] - T["cu_seqlens_cmp_kv"][b])
        else:
            cl = T["cmp_kv"].shape[1]
    r = int(T["cmp_residual_kv"][b]) if T["cmp_residual_kv"] is not None else 0
    return b, i, q_len, kv, cl, r


def _physical(prob, which: str, b: int, n: int) -> np.ndarray:
    """Physical row numbers of logical positions 0..n-1 of batch b."""
    pos = np.arange(n)
    T = prob.t
    if prob.layout_kv == "BSND":
        return b * T[which].shape[1] + pos
    if prob.layout_kv == "TND":
        cu = T["cu_seqlens_ori_kv" if which == "ori_kv" else "cu_seqlens_cmp_kv"]
        return int(cu[b]) + pos
    bt = T["ori_block_table" if which == "ori_kv" else "cmp_block_table"][b].numpy().astype(np.int64)
    bs = prob.ori_block_size if which == "ori_kv" else prob.cmp_block_size
    return bt[pos // bs] * bs + pos % bs


def dense_reference(prob, t: int, rows_cache=None):
    """O (q_n x 512) and LSE (q_n) of token t by dense masked softmax."""
    if rows_cache is None:
        rows_cache = {}
    b, i, q_len, kv, cl, r = lengths(prob, t)
    qn, dqk = prob.num_heads_q, prob.d_qk
    q = prob.t["q"].reshape(-1, qn, dqk)[t].to(torch.float64).numpy()
    O = np.zeros((qn, 512))
    lse = np.full(qn, -np.inf)
    if i >= q_len:
        return O, lse
    p = kv - q_len + i
    S_parts, M_parts, V_parts = [], [], []
    if kv > 0:
        if "ori_kv" not in rows_cache:
            rows_cache["ori_kv"] = _rows_f64(prob, "ori_kv")
        K = rows_cache["ori_kv"][_physical(prob, "ori_kv", b, kv)]
        pos = np.arange(kv)
        mm = prob.ori_mask_mode
        L, R = prob.ori_win_left, prob.ori_win_right
        if mm == 0:
            mask = np.ones(kv, dtype=bool)
        elif mm == 3:
            mask = pos <= p
        else:
            mask = np.ones(kv, dtype=bool)
            if L >= 0:
                mask &= pos >= p - L
            if R >= 0:
                mask &= pos <= p + R
        if prob.ori_topk > 0:
            # block-wise selection: a histogram over block ids, spread over the
            # sbs tokens of each block, then the token mask
            sbs = max(1, getattr(prob, "sparse_block_size", 1))
            nblk = -(-kv // sbs)
            idx = prob.t["ori_sparse_indices"].reshape(-1, prob.ori_topk)[t].numpy()
            idx = idx[(idx >= 0) & (idx < nblk)]
            per_block = np.bincount(idx, minlength=nblk).astype(np.float64)
            mult = np.repeat(per_block, sbs)[:kv] * mask
        else:
            mult = mask.astype(np.float64)
        S_parts.append(q @ K.T * prob.softmax_scale)
        M_parts.append(mult)
        V_parts.append(K[:, :512])
    if cl > 0:
        if "cmp_kv" not in rows_cache:
            rows_cache["cmp_kv"] = _rows_f64(prob, "cmp_kv")
        K = rows_cache["cmp_kv"][_physical(prob, "cmp_kv", b, cl)]
        j = np.arange(cl)
        p_c = cl * prob.cmp_ratio + r - q_len + i
        vis = ((j + 1) * prob.cmp_ratio <= p_c + 1) if prob.cmp_mask_mode == 3 else np.ones(cl, dtype=bool)
        if prob.cmp_topk > 0:
            idx = prob.t["cmp_sparse_indices"].reshape(-1, prob.cmp_topk)[t].numpy()
            idx = idx[(idx >= 0) & (idx < cl)]
            mult = np.bincount(idx, minlength=cl).astype(np.float64) * vis
        else:
            mult = vis.astype(np.float64)
        S_parts.append(q @ K.T * prob.softmax_scale)
        M_parts.append(mult)
        V_parts.append(K[:, :512])
    if not S_parts:
        return O, lse
    S = np.concatenate(S_parts, axis=1)
    M = np.concatenate(M_parts)
    V = np.concatenate(V_parts, axis=0)
    if M.sum() == 0:
        return O, lse
    Sm = np.where(M > 0, S, -np.inf)
    m = Sm.max(axis=1, keepdims=True)
    W = M * np.exp(Sm - m)
    Z = W.sum(axis=1, keepdims=True)
    den = Z.copy()
    if prob.t["sinks"] is not None:
        den = den + np.exp(prob.t["sinks"].numpy().astype(np.float64)[:, None] - m)
    O = (W @ V) / den
    lse = (m + np.log(Z))[:, 0]
    return O, lse
