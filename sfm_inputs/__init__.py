"""Seeded synthetic inputs for sparse shared-KV MLA attention.

This module only *generates* inputs.  It holds none of the attention
arithmetic: no scores, no softmax, no masking of the attended set.  The same
``Problem`` objects feed both the CUDA library (through the package binding)
and the CPU oracle (through ``oracle``), so neither side ever supplies the
other's inputs.

Shapes and value distributions follow the workloads on the reference pages:

* ``sparse_flash_mla`` doc (CANN ops-transformer), 参数说明 / 调用示例:
  q ``(b, q_s, q_n, d)`` or ``(q_t, q_n, d)``, KV ``(b, s, 1, d)``,
  ``(t, 1, d)`` or paged ``(blocks, block_size, 1, d)``, ``d = 512``,
  int32 ``cmp_sparse_indices`` with ``-1`` at the tail, fp32 ``sinks``.
* ``SparseAttnSharedkv`` README, 调用说明: the block table is a random
  permutation of all cache blocks, reshaped per batch.
* kv_quant_sparse_flash_attention guide, "A2/A3 C8 NoPE" table: a packed KV
  row is 512 int8 NoPE bytes, 64 bf16/fp16 rope values and 4 fp32 scales
  (one per 128-dim tile) = 656 bytes.

Random numbers come from ``torch.Generator`` seeded per problem on the device
the tensors are created on.  Large caches are generated on the GPU in chunks;
the oracle then receives a host copy of exactly the same bytes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import torch

PACKED_ROW_BYTES = 656      # 512 int8 + 64 * 2 rope + 4 * 4 scales
KV_FORMAT_CODES = {"plain": 0, "int8_packed": 1, "fp8_packed": 2}
PACKED_FORMATS = ("int8_packed", "fp8_packed")
PACKED_ROW_BYTES_ROPE0 = 528
HEAD_DIM = 512

LAYOUTS_Q = ("BSND", "TND")
LAYOUTS_KV = ("BSND", "TND", "PAGED")


@dataclass
class Problem:
    """One synthetic invocation: the scalar attributes and the tensors."""

    name: str
    num_heads_q: int
    head_dim: int                 # value / output dim (512)
    rope_head_dim: int            # extra score dims carried by packed rows (0 or 64)
    batch_size: int
    max_seqlen_q: int
    max_seqlen_ori_kv: int
    max_seqlen_cmp_kv: int
    total_q: int
    ori_topk: int
    cmp_topk: int
    cmp_ratio: int
    ori_mask_mode: int
    cmp_mask_mode: int
    ori_win_left: int
    ori_win_right: int
    layout_q: str
    layout_kv: str
    has_ori_kv: bool
    has_cmp_kv: bool
    dtype: str                    # 'bf16' | 'fp16'
    kv_format: str                # 'plain' | 'int8_packed' | 'fp8_packed'
    ori_block_size: int
    cmp_block_size: int
    return_lse: bool
    softmax_scale: float
    seed: int
    t: Dict[str, Optional[torch.Tensor]] = field(default_factory=dict)
    # per-batch effective lengths used to build the problem (host ints)
    q_lens: List[int] = field(default_factory=list)
    kv_lens: List[int] = field(default_factory=list)
    ori_row_stride: int = 0       # bytes between consecutive KV rows
    cmp_row_stride: int = 0
    sparse_block_size: int = 1    # tokens per ori_sparse_indices entry (block-wise selection)

    # ------------------------------------------------------------------
    @property
    def d_qk(self) -> int:
        return self.head_dim + self.rope_head_dim

    @property
    def num_tokens(self) -> int:
        return self.total_q if self.layout_q == "TND" else self.batch_size * self.max_seqlen_q

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    @property
    def packed(self) -> bool:
        return self.kv_format in PACKED_FORMATS

    def kv_row_bytes(self) -> int:
        if self.packed:
            return PACKED_ROW_BYTES if self.rope_head_dim == 64 else PACKED_ROW_BYTES_ROPE0
        return self.head_dim * 2

    def to(self, device) -> "Problem":
        """Copy of the problem with every tensor moved to ``device``."""
        import copy
        p = copy.copy(self)
        p.t = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in self.t.items()}
        return p

    def attrs(self) -> dict:
        """Scalar attributes under the names of the library's sfm_params."""
        return dict(
            num_heads_q=self.num_heads_q, num_heads_kv=1, head_dim=self.head_dim,
            rope_head_dim=self.rope_head_dim, batch_size=self.batch_size, max_seqlen_q=self.max_seqlen_q,
            total_q=self.total_q, max_seqlen_ori_kv=self.max_seqlen_ori_kv,
            max_seqlen_cmp_kv=self.max_seqlen_cmp_kv, ori_topk=self.ori_topk, cmp_topk=self.cmp_topk,
            cmp_ratio=self.cmp_ratio, ori_mask_mode=self.ori_mask_mode, cmp_mask_mode=self.cmp_mask_mode,
            ori_win_left=self.ori_win_left, ori_win_right=self.ori_win_right, layout_q=self.layout_q,
            layout_kv=self.layout_kv, has_ori_kv=1, has_cmp_kv=int(self.has_cmp_kv), dtype=self.dtype,
            kv_format=KV_FORMAT_CODES[self.kv_format], ori_block_size=self.ori_block_size,
            cmp_block_size=self.cmp_block_size, return_lse=int(self.return_lse),
            sparse_block_size=self.sparse_block_size)

    def tensor_kwargs(self) -> dict:
        """Tensors (plus KV row strides) under the names of the library's sfm_tensors."""
        d = {k: v for k, v in self.t.items() if k not in ("q", "ori_kv")}
        d["ori_row_stride"] = self.ori_row_stride
        d["cmp_row_stride"] = self.cmp_row_stride or None
        return d

    def describe(self) -> str:
        return (f"{self.name}: q_n={self.num_heads_q} tokens={self.num_tokens} layout={self.layout_q}/"
                f"{self.layout_kv} topk={self.ori_topk}/{self.cmp_topk} ratio={self.cmp_ratio} "
                f"fmt={self.kv_format} dtype={self.dtype}")


# ----------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------

def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _fill_normal(buf: torch.Tensor, g: torch.Generator, chunk: int = 1 << 27) -> None:
    """Fill a bf16/fp16 tensor with N(0,1) rounded to its dtype, in chunks."""
    flat = buf.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        tmp = torch.randn(e - s, generator=g, device=buf.device, dtype=torch.float32)
        flat[s:e].copy_(tmp)


def _fill_packed(buf: torch.Tensor, g: torch.Generator, rope_dtype: torch.dtype, rope_head_dim: int,
                 fp8: bool = False, chunk_rows: int = 1 << 18) -> None:
    """Fill packed rows.  int8: NoPE ~ U[-127,127], scales ~ lognormal(0,0.5)/127.
    fp8 (E4M3FN): NoPE = N(0,1) * 32 clamped to the finite range [-448, 448]
    and rounded to the nearest E4M3 value (codes span the normal and
    subnormal exponents; no NaN code), scales ~ lognormal(0,0.5)/32.  Rope
    ~ N(0,1) in the input dtype."""
    rows = buf.view(-1, buf.shape[-1])
    n = rows.shape[0]
    rope_bytes = rope_head_dim * 2
    for s in range(0, n, chunk_rows):
        e = min(n, s + chunk_rows)
        r = e - s
        if fp8:
            x = torch.randn(r, 512, generator=g, device=buf.device) * 32.0
            nope = x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
            rows[s:e, :512].copy_(nope)
            div = 32.0
        else:
            nope = torch.randint(-127, 128, (r, 512), generator=g, device=buf.device, dtype=torch.int16)
            rows[s:e, :512].copy_(nope.to(torch.int8).view(torch.uint8))
            div = 127.0
        if rope_bytes:
            rope = torch.randn(r, rope_head_dim, generator=g, device=buf.device).to(rope_dtype)
            rows[s:e, 512:512 + rope_bytes].copy_(rope.view(torch.uint8))
        scales = (torch.randn(r, 4, generator=g, device=buf.device) * 0.5).exp() / div
        rows[s:e, 512 + rope_bytes:512 + rope_bytes + 16].copy_(scales.to(torch.float32).view(torch.uint8))


def _cu(lengths: Sequence[int], device) -> torch.Tensor:
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + int(x))
    return torch.tensor(cu, dtype=torch.int32, device=device)


def sample_sorted_subsets(counts: torch.Tensor, k: int, g: torch.Generator) -> torch.Tensor:
    """For each row r, draw min(k, counts[r]) distinct values of [0, counts[r])
    uniformly without replacement, sort them ascending and pad with -1.

    This is the index recipe of the workloads (top-k picks among the slots a
    query may see, valid entries first, -1 tail); it is input generation only.
    """
    device = counts.device
    rows = counts.numel()
    out = torch.full((rows, k), -1, dtype=torch.int32, device=device)
    if rows == 0:
        return out
    nmax = int(counts.max().item()) if rows else 0
    if nmax <= 0:
        return out
    step = max(1, (1 << 26) // max(nmax, 1))
    for s in range(0, rows, step):
        e = min(rows, s + step)
        c = counts[s:e].to(torch.int64)
        keys = torch.rand(e - s, nmax, generator=g, device=device)
        col = torch.arange(nmax, device=device).unsqueeze(0)
        keys = torch.where(col < c.unsqueeze(1), keys, torch.full_like(keys, 2.0))
        kk = min(k, nmax)
        _, idx = torch.topk(keys, kk, dim=1, largest=False, sorted=False)
        valid = idx < c.unsqueeze(1)
        big = torch.full_like(idx, 1 << 40)
        idx = torch.where(valid, idx, big)
        idx, _ = torch.sort(idx, dim=1)
        idx = torch.where(idx >= (1 << 40), torch.full_like(idx, -1), idx)
        out[s:e, :kk] = idx.to(torch.int32)
    return out


def _block_table_tail(lengths: Sequence[int], bs: int, tail: int, g: torch.Generator, device):
    """Block table that stores only the last `tail` logical blocks of each
    sequence (in a random permutation of physical blocks 1..); every other
    logical block maps to physical block 0, which holds no row any query
    reads.  For workloads whose queries read only the end of each sequence."""
    nblk = [max(1, math.ceil(int(L) / bs)) for L in lengths]
    keep = [min(tail, n) for n in nblk]
    total = 1 + sum(keep)
    perm = (torch.randperm(total - 1, generator=g, device=device) + 1).to(torch.int32)
    table = torch.zeros(len(lengths), max(nblk), dtype=torch.int32, device=device)
    o = 0
    for b, (n, k) in enumerate(zip(nblk, keep)):
        table[b, n - k:n] = perm[o:o + k]
        o += k
    return table, total


def _block_table(lengths: Sequence[int], bs: int, g: torch.Generator, device, min_cols: int = 1):
    nblk = [max(1, math.ceil(int(L) / bs)) for L in lengths]
    total = sum(nblk)
    perm = torch.randperm(total, generator=g, device=device).to(torch.int32)
    cols = max(max(nblk), min_cols)
    table = torch.zeros(len(lengths), cols, dtype=torch.int32, device=device)
    o = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[o:o + n]
        o += n
    return table, total


# ----------------------------------------------------------------------
# generic builder
# ----------------------------------------------------------------------

def build(name: str, *, seed: int, device="cpu", q_n: int, q_lens: Sequence[int], kv_lens: Sequence[int],
          layout_q: str = "BSND", layout_kv: str = "BSND", dtype: str = "bf16", mode: str = "swa",
          cmp_ratio: int = 1, cmp_topk: int = 0, ori_topk: int = 0, win_left: int = 127, win_right: int = 0,
          ori_mask_mode: Optional[int] = None, cmp_mask_mode: Optional[int] = None,
          kv_format: str = "plain", rope_head_dim: int = 0, ori_block_size: int = 128,
          cmp_block_size: int = 128, sinks: bool = False, return_lse: bool = True,
          softmax_scale: Optional[float] = None, q_capacity: Optional[int] = None,
          kv_capacity: Optional[int] = None, seqused_q: Optional[Sequence[int]] = None,
          pass_seqused_ori: Optional[bool] = None, pass_seqused_cmp: Optional[bool] = None,
          residuals: Optional[Sequence[int]] = None, cmp_lens: Optional[Sequence[int]] = None,
          index_mode: str = "visible", kv_row_pad: int = 0, sparse_block_size: int = 1,
          ori_tail_blocks: Optional[int] = None) -> Problem:
    """Build a problem.

    mode: 'swa' (ori window only), 'csa' (window + top-k compressed),
          'hca' (window + all visible compressed), 'ori_sparse' (token-wise
          top-k over ori, the packed-KV decode form; no window, no cmp).
    index_mode: 'visible' samples from the slots each query may see;
          'all_visible' lists every visible slot in order (the form the
          context-parallel example builds); 'any' samples from [0, len).
    kv_row_pad: extra bytes between consecutive KV rows (inter-row padding).
    sparse_block_size: 'ori_sparse' only; each index selects a block of that
          many tokens (sampled among the blocks holding a visible token).
    ori_tail_blocks: PAGED ori caches only: store just the last that many
          blocks of each sequence (the rest of the block table points at one
          shared block no query reads) -- a small device footprint for
          workloads that read only the end of each sequence.
    """
    assert layout_q in LAYOUTS_Q and layout_kv in LAYOUTS_KV
    B = len(q_lens)
    assert len(kv_lens) == B
    g = _gen(seed, device)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    assert kv_format in KV_FORMAT_CODES
    packed = kv_format in PACKED_FORMATS
    d_v = HEAD_DIM
    d_qk = d_v + (rope_head_dim if packed else 0)
    has_cmp = mode in ("csa", "hca")
    if ori_mask_mode is None:
        ori_mask_mode = 3 if mode == "ori_sparse" else 4
    if cmp_mask_mode is None:
        cmp_mask_mode = 3 if has_cmp else 0
    if not has_cmp:
        cmp_ratio = 1 if mode != "ori_sparse" else cmp_ratio
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d_qk)

    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    if cmp_lens is None:
        cmp_lens = [L // cmp_ratio for L in kv_lens] if has_cmp else [0] * B
    if residuals is None:
        residuals = [L % cmp_ratio for L in kv_lens] if has_cmp else [0] * B
    cmp_lens = [int(x) for x in cmp_lens]
    residuals = [int(x) for x in residuals]

    t: Dict[str, Optional[torch.Tensor]] = {k: None for k in (
        "q", "ori_kv", "cmp_kv", "ori_sparse_indices", "cmp_sparse_indices", "ori_block_table",
        "cmp_block_table", "cu_seqlens_q", "cu_seqlens_ori_kv", "cu_seqlens_cmp_kv", "seqused_q",
        "seqused_ori_kv", "seqused_cmp_kv", "cmp_residual_kv", "sinks")}

    # ---------------- q ----------------
    if layout_q == "BSND":
        q_s = q_capacity if q_capacity is not None else max(q_lens)
        q = torch.empty(B, q_s, q_n, d_qk, dtype=tdt, device=device)
        n_tok = B * q_s
        max_q = q_s
    else:
        q_s = max(q_lens)
        n_tok = sum(q_lens)
        q = torch.empty(n_tok, q_n, d_qk, dtype=tdt, device=device)
        t["cu_seqlens_q"] = _cu(q_lens, device)
        max_q = max(q_lens)
    _fill_normal(q, g)
    t["q"] = q
    if seqused_q is not None:
        t["seqused_q"] = torch.tensor(list(seqused_q), dtype=torch.int32, device=device)

    # ---------------- caches ----------------
    def make_cache(lengths, bs, capacity, tail=None):
        row_bytes = (PACKED_ROW_BYTES if rope_head_dim == 64 else PACKED_ROW_BYTES_ROPE0) if packed else d_v * 2
        stride_bytes = row_bytes + kv_row_pad
        table = None
        if layout_kv == "PAGED":
            if tail is not None:
                table, nblk = _block_table_tail(lengths, bs, tail, g, device)
            else:
                table, nblk = _block_table(lengths, bs, g, device)
            nrows = nblk * bs
            shape = (nblk, bs, 1)
        elif layout_kv == "TND":
            nrows = max(1, sum(lengths))
            shape = (nrows, 1)
        else:
            cap = capacity if capacity is not None else max(max(lengths), 1)
            nrows = B * cap
            shape = (B, cap, 1)
        raw = torch.empty(nrows, stride_bytes, dtype=torch.uint8, device=device)
        if packed:
            _fill_packed(raw[:, :row_bytes], g, tdt, rope_head_dim, fp8=kv_format == "fp8_packed")
        else:
            vals = torch.empty(nrows, d_v, dtype=tdt, device=device)
            _fill_normal(vals, g)
            raw[:, :row_bytes].copy_(vals.view(torch.uint8).view(nrows, row_bytes))
            del vals
        if kv_row_pad:
            raw[:, row_bytes:].fill_(0xAB)   # padding bytes must never be read
        if packed or kv_row_pad:
            cache = raw.view(*shape, stride_bytes)          # uint8 rows (possibly padded)
        else:
            cache = raw.view(tdt).view(*shape, d_v)
        return cache, table, stride_bytes

    ori_kv, ori_table, ori_stride = make_cache(kv_lens, ori_block_size, kv_capacity, ori_tail_blocks)
    t["ori_kv"] = ori_kv
    t["ori_block_table"] = ori_table
    if layout_kv == "TND":
        t["cu_seqlens_ori_kv"] = _cu(kv_lens, device)
    kv_cap = kv_capacity if kv_capacity is not None else max(kv_lens)
    if pass_seqused_ori is None:
        pass_seqused_ori = layout_kv == "PAGED" or (layout_kv == "BSND" and any(L != kv_cap for L in kv_lens))
    if pass_seqused_ori:
        t["seqused_ori_kv"] = torch.tensor(kv_lens, dtype=torch.int32, device=device)

    cmp_stride = 0
    if has_cmp:
        cmp_cap = max(max(cmp_lens), 1)
        cmp_kv, cmp_table, cmp_stride = make_cache([max(c, 0) for c in cmp_lens], cmp_block_size, cmp_cap)
        t["cmp_kv"] = cmp_kv
        t["cmp_block_table"] = cmp_table
        if layout_kv == "TND":
            t["cu_seqlens_cmp_kv"] = _cu(cmp_lens, device)
        if pass_seqused_cmp is None:
            pass_seqused_cmp = layout_kv == "PAGED" or (layout_kv == "BSND" and any(c != cmp_cap for c in cmp_lens))
        if pass_seqused_cmp:
            t["seqused_cmp_kv"] = torch.tensor(cmp_lens, dtype=torch.int32, device=device)
        if cmp_mask_mode == 3 or residuals is not None:
            t["cmp_residual_kv"] = torch.tensor(residuals, dtype=torch.int32, device=device)
        max_cmp = cmp_cap
    else:
        max_cmp = 0

    # ---------------- indices ----------------
    # query row i of batch b sits at position kv_len - q_len + i (right-down
    # alignment, sparse_flash_mla doc CP example); the recipe samples among the
    # slots such a row may see.
    qlen_eff = list(seqused_q) if seqused_q is not None else q_lens
    tok_b: List[int] = []
    tok_i: List[int] = []
    if layout_q == "BSND":
        for b in range(B):
            for i in range(q_s):
                tok_b.append(b)
                tok_i.append(i)
    else:
        for b in range(B):
            for i in range(q_lens[b]):
                tok_b.append(b)
                tok_i.append(i)

    def vis_counts_cmp():
        c = []
        for b, i in zip(tok_b, tok_i):
            ql = qlen_eff[b]
            if index_mode == "any":
                c.append(max(cmp_lens[b], 0))
                continue
            p_c = cmp_lens[b] * cmp_ratio + residuals[b] - ql + i
            c.append(max(0, min(cmp_lens[b], (p_c + 1) // cmp_ratio)) if cmp_mask_mode == 3 else max(cmp_lens[b], 0))
        return torch.tensor(c, dtype=torch.int64, device=device)

    if mode == "csa":
        counts = vis_counts_cmp()
        if index_mode == "all_visible":
            idx = torch.full((len(tok_b), cmp_topk), -1, dtype=torch.int32, device=device)
            for r, c in enumerate(counts.tolist()):
                c = min(c, cmp_topk)
                if c > 0:
                    idx[r, :c] = torch.arange(c, dtype=torch.int32, device=device)
        else:
            idx = sample_sorted_subsets(counts, cmp_topk, g)
        if layout_q == "BSND":
            idx = idx.view(B, q_s, 1, cmp_topk)
        else:
            idx = idx.view(n_tok, 1, cmp_topk)
        t["cmp_sparse_indices"] = idx
    if mode == "ori_sparse":
        c = []
        for b, i in zip(tok_b, tok_i):
            ql = qlen_eff[b]
            p = kv_lens[b] - ql + i
            if index_mode == "any" or ori_mask_mode == 0:
                c.append(kv_lens[b])
            else:
                c.append(max(0, min(kv_lens[b], p + 1)))
        c = [-(-x // sparse_block_size) for x in c]          # blocks holding a candidate token
        counts = torch.tensor(c, dtype=torch.int64, device=device)
        idx = sample_sorted_subsets(counts, ori_topk, g)
        if layout_q == "BSND":
            idx = idx.view(B, q_s, 1, ori_topk)
        else:
            idx = idx.view(n_tok, 1, ori_topk)
        t["ori_sparse_indices"] = idx

    if sinks:
        t["sinks"] = torch.randn(q_n, generator=g, device=device, dtype=torch.float32)

    p = Problem(
        name=name, num_heads_q=q_n, head_dim=d_v, rope_head_dim=(rope_head_dim if packed else 0),
        batch_size=B, max_seqlen_q=max_q, max_seqlen_ori_kv=kv_cap if layout_kv == "BSND" else max(kv_lens),
        max_seqlen_cmp_kv=max_cmp, total_q=n_tok, ori_topk=(ori_topk if mode == "ori_sparse" else 0),
        cmp_topk=(cmp_topk if mode == "csa" else 0), cmp_ratio=cmp_ratio, ori_mask_mode=ori_mask_mode,
        cmp_mask_mode=cmp_mask_mode, ori_win_left=win_left, ori_win_right=win_right, layout_q=layout_q,
        layout_kv=layout_kv, has_ori_kv=True, has_cmp_kv=has_cmp, dtype=dtype, kv_format=kv_format,
        ori_block_size=ori_block_size if layout_kv == "PAGED" else 0,
        cmp_block_size=cmp_block_size if (layout_kv == "PAGED" and has_cmp) else 0,
        return_lse=return_lse, softmax_scale=float(softmax_scale), seed=seed, t=t,
        q_lens=q_lens, kv_lens=kv_lens, sparse_block_size=sparse_block_size)
    p.ori_row_stride = ori_stride
    p.cmp_row_stride = cmp_stride
    return p


# ----------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------

def _uniform_ints(lo: int, hi: int, n: int, seed: int) -> List[int]:
    g = _gen(seed, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g).tolist()]


def swa_decode_tiny(device="cpu", seed: int = 0) -> Problem:
    """SWA-only decode: B=2, q_n=16, BSND contiguous ori with kv_len=256,
    window 127/0, no cmp, no sinks, scale 1/sqrt(512), O and LSE returned."""
    return build("swa_decode_tiny", seed=seed, device=device, q_n=16, q_lens=[1, 1], kv_lens=[256, 256],
                 layout_q="BSND", layout_kv="BSND", mode="swa", win_left=127, win_right=0,
                 ori_mask_mode=4, cmp_mask_mode=0, sinks=False, return_lse=True)


def csa_decode(device="cpu", seed: int = 1, batch: int = 32, cmp_topk: int = 512) -> Problem:
    """CSA decode: q_n=64, paged ori (block 128, random permutation),
    kv_len ~ U[4096, 32768], window 127/0, cmp_ratio 4 paged, top-512 (or
    top-1024, the other size the pages allow) visible compressed slots per
    query, fp32 sinks."""
    kv = _uniform_ints(4096, 32768, batch, seed * 7919 + 11)
    return build("csa_decode", seed=seed, device=device, q_n=64, q_lens=[1] * batch, kv_lens=kv,
                 layout_q="BSND", layout_kv="PAGED", mode="csa", cmp_ratio=4, cmp_topk=cmp_topk,
                 win_left=127, win_right=0, sinks=True, return_lse=True)


def hca_decode(device="cpu", seed: int = 2, batch: int = 64, kv_len: int = 131072, compact_pool: bool = False) -> Problem:
    """HCA decode: q_n=128, paged ori (block 128) with kv_len=131072, window
    127/0, cmp_ratio 128 with all 1024 visible slots, fp32 sinks.
    compact_pool stores only the two last ori blocks of each sequence (the
    window reads nothing else): the same attended rows and bytes in a small
    device footprint (for profiler captures)."""
    return build("hca_decode", seed=seed, device=device, q_n=128, q_lens=[1] * batch, kv_lens=[kv_len] * batch,
                 layout_q="BSND", layout_kv="PAGED", mode="hca", cmp_ratio=128, win_left=127, win_right=0,
                 sinks=True, return_lse=True, ori_tail_blocks=2 if compact_pool else None)


def csa_prefill(device="cpu", seed: int = 3, nseq: int = 8, qmin: int = 512, qmax: int = 4096,
                prefix_max: int = 8192) -> Problem:
    """CSA varlen prefill (TND): q lengths ~ U[512, 4096], kv = q + U[0, 8192]
    prefix, q_n=64, window 127/0, cmp_ratio 4, top-2048 visible slots per
    token, sinks, LSE returned."""
    ql = _uniform_ints(qmin, qmax, nseq, seed * 7919 + 13)
    pre = _uniform_ints(0, prefix_max, nseq, seed * 7919 + 17)
    kv = [a + b for a, b in zip(ql, pre)]
    return build("csa_prefill", seed=seed, device=device, q_n=64, q_lens=ql, kv_lens=kv, layout_q="TND",
                 layout_kv="TND", mode="csa", cmp_ratio=4, cmp_topk=2048, win_left=127, win_right=0,
                 sinks=True, return_lse=True)


def packed_decode(device="cpu", seed: int = 4, batch: int = 64, kv_len: int = 65536) -> Problem:
    """Quantized packed-KV sparse decode: q_n=128, Q_D=576 bf16, paged block
    64, 656-byte rows, token-wise top-2048 indices from [0, kv_len), right-down
    causal, scale 1/sqrt(576), no sinks."""
    return build("packed_decode", seed=seed, device=device, q_n=128, q_lens=[1] * batch,
                 kv_lens=[kv_len] * batch, layout_q="BSND", layout_kv="PAGED", mode="ori_sparse",
                 ori_topk=2048, ori_mask_mode=3, cmp_mask_mode=0, kv_format="int8_packed",
                 rope_head_dim=64, ori_block_size=64, sinks=False, return_lse=True,
                 softmax_scale=1.0 / math.sqrt(576))


def packed_fp8_decode(device="cpu", seed: int = 5, batch: int = 64, kv_len: int = 65536) -> Problem:
    """The packed decode workload with FLOAT8_E4M3FN NoPE bytes (the A5 rows
    of the kv_quant guide): same shapes, 656-byte rows, top-2048 indices."""
    return build("packed_fp8_decode", seed=seed, device=device, q_n=128, q_lens=[1] * batch,
                 kv_lens=[kv_len] * batch, layout_q="BSND", layout_kv="PAGED", mode="ori_sparse",
                 ori_topk=2048, ori_mask_mode=3, cmp_mask_mode=0, kv_format="fp8_packed",
                 rope_head_dim=64, ori_block_size=64, sinks=False, return_lse=True,
                 softmax_scale=1.0 / math.sqrt(576))


WORKLOADS = {
    "swa_decode_tiny": swa_decode_tiny,
    "csa_decode": csa_decode,
    "hca_decode": hca_decode,
    "csa_prefill": csa_prefill,
    "packed_decode": packed_decode,
    "packed_fp8_decode": packed_fp8_decode,
}
