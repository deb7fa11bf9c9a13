"""Pins for the CPU oracle: it is checked against things other than itself.

* hand-derived attended sets of the pages' worked examples (tests/golden),
* a brute-force dense masked formulation on tiny random inputs (all modes,
  layouts, dtypes, the packed format, padding rows, invalid and duplicate
  indices),
* closed forms: uniform attention (Q = 0) and identical KV rows, with and
  without sinks,
* a library routine: torch SDPA (fp64) for the dense right-down causal case,
  plus a naive log-sum-exp without max subtraction,
* invariants: the context-parallel split of the sparse_flash_mla doc, layout
  equivalence BSND / TND / paged, CSA == HCA when the indices list every
  visible slot, packed rows with power-of-two scales == plain rows.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import sfm_inputs as S
from tests import _brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")


def _set_of(prob, t):
    src, pos = oracle.attended(prob, t)
    ori = sorted(int(p) for s, p in zip(src, pos) if s == 0)
    cmp_ = sorted(int(p) for s, p in zip(src, pos) if s == 1)
    return ori, cmp_


# ---------------------------------------------------------------------------
# worked examples of the pages
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("key", ["swa_bsnd", "hca_bsnd", "csa_tnd", "cp_global", "cp_rank1"])
def test_page_example_sets(key):
    ex = json.load(open(GOLDEN))[key]
    pr = dict(ex["params"])
    mode = pr.pop("mode")
    prob = S.build(key, seed=5, q_n=2, mode=mode, win_left=127, win_right=0, sinks=False, **pr)
    assert prob.num_tokens == len(ex["tokens"])
    for t, (lo, hi, cmp_slots) in enumerate(ex["tokens"]):
        ori, cmp_ = _set_of(prob, t)
        assert ori == list(range(lo, hi + 1)), (key, t)
        assert cmp_ == cmp_slots, (key, t)


# ---------------------------------------------------------------------------
# brute force on tiny random inputs
# ---------------------------------------------------------------------------
def _tiny_cases():
    cases = []
    # (name, kwargs)
    cases.append(("swa_bsnd", dict(q_lens=[3, 2], kv_lens=[40, 9], layout_q="BSND", layout_kv="BSND", mode="swa",
                                   win_left=5, win_right=2, q_capacity=3)))
    cases.append(("swa_tnd_unbounded", dict(q_lens=[4, 1], kv_lens=[7, 30], layout_q="TND", layout_kv="TND",
                                            mode="swa", win_left=-1, win_right=1)))
    cases.append(("causal_mode3_paged", dict(q_lens=[3, 5], kv_lens=[20, 37], layout_q="TND", layout_kv="PAGED",
                                             mode="swa", ori_mask_mode=3, ori_block_size=16)))
    cases.append(("nomask_mode0_bsnd", dict(q_lens=[2, 2], kv_lens=[11, 6], layout_q="BSND", layout_kv="BSND",
                                            mode="swa", ori_mask_mode=0)))
    cases.append(("hca_paged", dict(q_lens=[2, 3], kv_lens=[50, 70], layout_q="BSND", layout_kv="PAGED",
                                    mode="hca", cmp_ratio=4, win_left=6, win_right=0, ori_block_size=16,
                                    cmp_block_size=16, sinks=True, q_capacity=3)))
    cases.append(("csa_tnd_any_idx", dict(q_lens=[3, 2], kv_lens=[45, 33], layout_q="TND", layout_kv="TND",
                                          mode="csa", cmp_ratio=4, cmp_topk=8, win_left=4, win_right=0,
                                          index_mode="any", sinks=True)))
    cases.append(("csa_paged_fp16", dict(q_lens=[1, 1, 1], kv_lens=[64, 100, 17], layout_q="BSND",
                                         layout_kv="PAGED", mode="csa", cmp_ratio=4, cmp_topk=16, win_left=9,
                                         win_right=0, dtype="fp16", ori_block_size=32, cmp_block_size=16,
                                         sinks=True)))
    cases.append(("csa_paged_odd_blocks", dict(q_lens=[1, 1], kv_lens=[150, 333], layout_q="BSND",
                                               layout_kv="PAGED", mode="csa", cmp_ratio=4, cmp_topk=32,
                                               win_left=20, win_right=0, ori_block_size=48, cmp_block_size=80,
                                               sinks=True)))
    cases.append(("hca_mode0_bsnd", dict(q_lens=[2], kv_lens=[24], layout_q="BSND", layout_kv="BSND", mode="hca",
                                         cmp_ratio=8, cmp_mask_mode=0, win_left=3, win_right=0)))
    cases.append(("packed_paged", dict(q_lens=[1, 2], kv_lens=[90, 40], layout_q="TND", layout_kv="PAGED",
                                       mode="ori_sparse", ori_topk=12, kv_format="int8_packed", rope_head_dim=64,
                                       ori_block_size=16)))
    cases.append(("packed_rope0_bsnd_any", dict(q_lens=[2], kv_lens=[33], layout_q="BSND", layout_kv="BSND",
                                                mode="ori_sparse", ori_topk=10, kv_format="int8_packed",
                                                rope_head_dim=0, index_mode="any", sinks=True)))
    cases.append(("packed_fp8_paged", dict(q_lens=[1, 2], kv_lens=[90, 40], layout_q="TND", layout_kv="PAGED",
                                           mode="ori_sparse", ori_topk=12, kv_format="fp8_packed", rope_head_dim=64,
                                           ori_block_size=16, sinks=True)))
    cases.append(("packed_fp8_rope0_bsnd", dict(q_lens=[2], kv_lens=[33], layout_q="BSND", layout_kv="BSND",
                                                mode="ori_sparse", ori_topk=10, kv_format="fp8_packed",
                                                rope_head_dim=0, index_mode="any")))
    cases.append(("packed_blockwise4_paged", dict(q_lens=[1, 2], kv_lens=[90, 45], layout_q="TND",
                                                  layout_kv="PAGED", mode="ori_sparse", ori_topk=6,
                                                  kv_format="int8_packed", rope_head_dim=64, ori_block_size=16,
                                                  sparse_block_size=4, sinks=True)))
    cases.append(("plain_blockwise16_any", dict(q_lens=[2, 1], kv_lens=[70, 40], layout_q="BSND",
                                                layout_kv="BSND", mode="ori_sparse", ori_topk=3,
                                                sparse_block_size=16, index_mode="any")))
    cases.append(("swa_rowpad_tnd", dict(q_lens=[2, 3], kv_lens=[10, 12], layout_q="TND", layout_kv="TND",
                                         mode="swa", win_left=3, win_right=1, kv_row_pad=48)))
    cases.append(("csa_q_longer_than_kv", dict(q_lens=[6], kv_lens=[4], layout_q="TND", layout_kv="TND",
                                               mode="csa", cmp_ratio=2, cmp_topk=4, win_left=2, win_right=0)))
    cases.append(("seqused_q_short", dict(q_lens=[4, 4], kv_lens=[30, 30], layout_q="BSND", layout_kv="BSND",
                                          mode="swa", win_left=7, win_right=0, seqused_q=[2, 4])))
    return cases


@pytest.mark.parametrize("name,kw", _tiny_cases(), ids=[c[0] for c in _tiny_cases()])
def test_oracle_matches_brute_force(name, kw):
    prob = S.build(name, seed=11, q_n=4, **kw)
    if name == "csa_tnd_any_idx":
        # plant duplicates and out-of-range / negative entries in the middle
        idx = prob.t["cmp_sparse_indices"]
        idx[0, 0, 1] = idx[0, 0, 0]
        idx[1, 0, 2] = 10_000
        idx[2, 0, 0] = -7
    O, lse = oracle.forward(prob)
    cache = {}
    for t in range(prob.num_tokens):
        Ob, lb = _brute.dense_reference(prob, t, cache)
        np.testing.assert_allclose(O[t], Ob, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[t], lb, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("sinks", [False, True])
def test_uniform_attention_closed_form(sinks):
    """Q = 0: every score is 0, so O = sum(V_attended) / (|A| + [sink] e^sink)
    and LSE = log |A| (the uniform-attention strategy of the
    kv_quant_sparse_flash_attention guide's test list)."""
    B, kv, topk = 2, 300, 16
    prob = S.build("uniform", seed=3, q_n=3, q_lens=[1] * B, kv_lens=[kv] * B, layout_q="BSND",
                   layout_kv="BSND", mode="csa", cmp_ratio=4, cmp_topk=topk, sinks=sinks)
    prob.t["q"].zero_()
    O, lse = oracle.forward(prob)
    ori = prob.t["ori_kv"].to(torch.float64)
    cmp_ = prob.t["cmp_kv"].to(torch.float64)
    idx = prob.t["cmp_sparse_indices"].reshape(B, topk)
    for b in range(B):
        win = ori[b, kv - 128:kv, 0]          # positions p-127 .. p with p = kv - 1
        sel = cmp_[b, idx[b].long(), 0]       # every sampled index is visible
        n = 128 + topk
        tot = (win.sum(0) + sel.sum(0)).numpy()
        for h in range(3):
            den = n + (math.exp(float(prob.t["sinks"][h])) if sinks else 0.0)
            np.testing.assert_allclose(O[b, h], tot / den, rtol=1e-12, atol=1e-14)
            assert abs(lse[b, h] - math.log(n)) < 1e-12


@pytest.mark.parametrize("sinks", [False, True])
def test_identical_rows_closed_form(sinks):
    prob = S.build("identical", seed=4, q_n=4, q_lens=[2, 1], kv_lens=[40, 70], layout_q="TND",
                   layout_kv="PAGED", mode="hca", cmp_ratio=8, win_left=9, ori_block_size=16,
                   cmp_block_size=16, sinks=sinks)
    v = prob.t["ori_kv"].reshape(-1, 512)[0].clone()
    prob.t["ori_kv"].reshape(-1, 512)[:] = v
    prob.t["cmp_kv"].reshape(-1, 512)[:] = v
    O, lse = oracle.forward(prob)
    vd = v.to(torch.float64).numpy()
    q = prob.t["q"].to(torch.float64)
    for t in range(prob.num_tokens):
        src, pos = oracle.attended(prob, t)
        n = len(src)
        for h in range(4):
            s = float(q[t, h] @ torch.from_numpy(vd)) * prob.softmax_scale
            f = n / (n + math.exp(float(prob.t["sinks"][h]) - s)) if sinks else 1.0
            np.testing.assert_allclose(O[t, h], vd * f, rtol=1e-12, atol=1e-13)
            assert abs(lse[t, h] - (s + math.log(n))) < 1e-9


def test_dense_causal_matches_sdpa_and_naive_lse():
    """Window unbounded on the left and closed on the right (mode 4, -1/0) and
    mode 3 both reduce to dense right-down causal attention; compare with
    torch's SDPA in fp64 and with a naive log(sum(exp(S)))."""
    q_lens, kv_lens = [5, 3], [9, 3]
    for mode, wl in ((4, -1), (3, 127)):
        prob = S.build("dense", seed=8, q_n=2, q_lens=q_lens, kv_lens=kv_lens, layout_q="TND", layout_kv="TND",
                       mode="swa", ori_mask_mode=mode, win_left=wl, win_right=0)
        prob.t["q"].mul_(0.05)  # small scores so the naive LSE stays exact enough
        O, lse = oracle.forward(prob)
        q = prob.t["q"].to(torch.float64)
        kvt = prob.t["ori_kv"].to(torch.float64)[:, 0]
        cq = prob.t["cu_seqlens_q"].tolist()
        ck = prob.t["cu_seqlens_ori_kv"].tolist()
        for b in range(2):
            Qb = q[cq[b]:cq[b + 1]].transpose(0, 1)          # heads x q_len x d
            Kb = kvt[ck[b]:ck[b + 1]]                        # kv_len x d
            ql, kl = q_lens[b], kv_lens[b]
            i = torch.arange(ql)[:, None]
            j = torch.arange(kl)[None, :]
            mask = j <= (kl - ql + i)                        # right-down causal
            ref = torch.nn.functional.scaled_dot_product_attention(
                Qb, Kb[None].expand(2, -1, -1), Kb[None].expand(2, -1, -1), attn_mask=mask,
                scale=prob.softmax_scale)
            np.testing.assert_allclose(O[cq[b]:cq[b + 1]], ref.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)
            Sm = (Qb @ Kb.T) * prob.softmax_scale
            naive = torch.log(torch.where(mask, torch.exp(Sm), torch.zeros_like(Sm)).sum(-1))
            np.testing.assert_allclose(lse[cq[b]:cq[b + 1]], naive.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
def _cp_slice(prob, q_rows, ori_rows, cmp_rows, q_lens, kv_lens, cmp_lens, residuals):
    """Problem for one simulated context-parallel rank, sliced from ``prob``."""
    r = S.build("cp_rank", seed=0, q_n=prob.num_heads_q, q_lens=q_lens, kv_lens=kv_lens, cmp_lens=cmp_lens,
                residuals=residuals, layout_q="TND", layout_kv="TND", mode="csa", cmp_ratio=4,
                cmp_topk=prob.cmp_topk, index_mode="all_visible", sinks=True)
    r.t["q"] = torch.cat([prob.t["q"][a:b] for a, b in q_rows])
    r.t["ori_kv"] = torch.cat([prob.t["ori_kv"][a:b] for a, b in ori_rows])
    r.t["cmp_kv"] = torch.cat([prob.t["cmp_kv"][a:b] for a, b in cmp_rows])
    r.t["sinks"] = prob.t["sinks"]
    return r


def test_context_parallel_split_invariant():
    """The two-rank split of the sparse_flash_mla doc's CP example, run rank by
    rank, concatenates to the global result exactly."""
    g = S.build("cp_global", seed=21, q_n=4, q_lens=[16, 18], kv_lens=[16, 18], cmp_lens=[4, 4],
                residuals=[0, 2], layout_q="TND", layout_kv="TND", mode="csa", cmp_ratio=4, cmp_topk=512,
                index_mode="all_visible", sinks=True)
    Og, lg = oracle.forward(g)
    r0 = _cp_slice(g, [(0, 16), (16, 24)], [(0, 16), (16, 24)], [(0, 4), (4, 6)], [16, 8], [16, 8], [4, 2], [0, 0])
    r1 = _cp_slice(g, [(24, 34)], [(16, 34)], [(4, 8)], [10], [18], [4], [2])
    O0, l0 = oracle.forward(r0)
    O1, l1 = oracle.forward(r1)
    np.testing.assert_array_equal(np.concatenate([O0, O1]), Og)
    np.testing.assert_array_equal(np.concatenate([l0, l1]), lg)


def test_csa_with_all_visible_indices_equals_hca():
    kw = dict(seed=6, q_n=3, q_lens=[3, 2], kv_lens=[41, 64], layout_q="TND", layout_kv="TND", cmp_ratio=4,
              win_left=5, sinks=True)
    hca = S.build("hca", mode="hca", **kw)
    csa = S.build("csa", mode="csa", cmp_topk=32, index_mode="all_visible", **kw)
    for k in ("q", "ori_kv", "cmp_kv", "sinks"):
        csa.t[k] = hca.t[k]
    Oh, lh = oracle.forward(hca)
    Oc, lc = oracle.forward(csa)
    np.testing.assert_array_equal(Oh, Oc)
    np.testing.assert_array_equal(lh, lc)


def _bsnd_to(prob, layout_kv, bs=16, seed=0):
    """Same logical problem with the caches re-laid out as TND or paged."""
    import copy
    B = prob.batch_size
    out = copy.copy(prob)
    out.t = dict(prob.t)
    out.layout_kv = layout_kv
    g = torch.Generator().manual_seed(seed)
    kv_lens = prob.kv_lens
    cmp_lens = [L // prob.cmp_ratio for L in kv_lens] if prob.has_cmp_kv else None
    for which, lens, bt_name, cu_name, used_name in (
            ("ori_kv", kv_lens, "ori_block_table", "cu_seqlens_ori_kv", "seqused_ori_kv"),
            ("cmp_kv", cmp_lens, "cmp_block_table", "cu_seqlens_cmp_kv", "seqused_cmp_kv")):
        if lens is None:
            continue
        src = prob.t[which]
        if layout_kv == "TND":
            out.t[which] = torch.cat([src[b, :lens[b]] for b in range(B)])
            cu = [0]
            for L in lens:
                cu.append(cu[-1] + L)
            out.t[cu_name] = torch.tensor(cu, dtype=torch.int32)
            out.t[used_name] = None
        else:
            nblk = [max(1, math.ceil(L / bs)) for L in lens]
            perm = torch.randperm(sum(nblk), generator=g)
            cache = torch.zeros(sum(nblk), bs, 1, 512, dtype=src.dtype)
            table = torch.zeros(B, max(nblk), dtype=torch.int32)
            o = 0
            for b in range(B):
                for k in range(nblk[b]):
                    blk = int(perm[o + k])
                    table[b, k] = blk
                    n = min(bs, lens[b] - k * bs)
                    if n > 0:
                        cache[blk, :n] = src[b, k * bs:k * bs + n]
                o += nblk[b]
            out.t[which] = cache
            out.t[bt_name] = table
            out.t[used_name] = torch.tensor(lens, dtype=torch.int32)
            if which == "ori_kv":
                out.ori_block_size = bs
            else:
                out.cmp_block_size = bs
    return out


@pytest.mark.parametrize("mode", ["swa", "hca", "csa"])
def test_layout_equivalence(mode):
    kw = dict(cmp_ratio=4, cmp_topk=8) if mode == "csa" else (dict(cmp_ratio=4) if mode == "hca" else {})
    prob = S.build("lay", seed=9, q_n=3, q_lens=[1, 1, 1], kv_lens=[37, 64, 21], layout_q="BSND",
                   layout_kv="BSND", mode=mode, win_left=6, win_right=0, sinks=True, **kw)
    O, l = oracle.forward(prob)
    for lay in ("TND", "PAGED"):
        if lay == "TND":
            # TND kv needs TND q as well; q_s = 1 so the token order is unchanged
            p2 = _bsnd_to(prob, "TND")
            p2.layout_q = "TND"
            p2.t["q"] = prob.t["q"].reshape(-1, 3, 512)
            p2.t["cu_seqlens_q"] = torch.arange(0, 4, dtype=torch.int32)
            if mode == "csa":
                p2.t["cmp_sparse_indices"] = prob.t["cmp_sparse_indices"].reshape(3, 1, -1)
        else:
            p2 = _bsnd_to(prob, "PAGED", bs=16, seed=3)
        O2, l2 = oracle.forward(p2)
        np.testing.assert_array_equal(O2, O)
        np.testing.assert_array_equal(l2, l)


def test_packed_pow2_scales_equal_plain_rows():
    """Packed rows whose scales are powers of two dequantise exactly; with a
    zero rope they must give the plain-row result bit for bit, which pins the
    tile -> scale mapping and the byte offsets of the 656-byte row."""
    pk = S.build("pk", seed=12, q_n=4, q_lens=[1, 1], kv_lens=[80, 50], layout_q="BSND", layout_kv="BSND",
                 mode="ori_sparse", ori_topk=20, kv_format="int8_packed", rope_head_dim=64, sinks=True)
    rows = pk.t["ori_kv"].view(-1, 656)
    nrows = rows.shape[0]
    exps = torch.tensor([-7.0, -5.0, -9.0, -6.0])
    scales = torch.pow(2.0, exps).to(torch.float32).repeat(nrows, 1)
    rows[:, 640:656] = scales.view(torch.uint8).view(nrows, 16)
    rows[:, 512:640] = 0
    deq = rows[:, :512].view(torch.int8).to(torch.float32) * scales.repeat_interleave(128, dim=1)
    plain = S.build("pl", seed=12, q_n=4, q_lens=[1, 1], kv_lens=[80, 50], layout_q="BSND", layout_kv="BSND",
                    mode="ori_sparse", ori_topk=20, sinks=True)
    plain.t["ori_kv"] = deq.to(torch.bfloat16).view(pk.t["ori_kv"].shape[:-1] + (512,))
    assert torch.equal(plain.t["ori_kv"].float().view(-1, 512), deq)      # exact in bf16
    plain.t["q"] = pk.t["q"][..., :512].contiguous()
    plain.t["ori_sparse_indices"] = pk.t["ori_sparse_indices"]
    plain.t["sinks"] = pk.t["sinks"]
    plain.softmax_scale = pk.softmax_scale
    Op, lp = oracle.forward(pk)
    Ol, ll = oracle.forward(plain)
    np.testing.assert_array_equal(Op, Ol)
    np.testing.assert_array_equal(lp, ll)


def test_e4m3_decoder_matches_library_and_definition():
    """The oracle's FLOAT8_E4M3FN decoder, all 256 codes, against torch's
    float8_e4m3fn dtype and against values the format's definition fixes
    (bias 7, subnormals m * 2^-9, largest finite 448, S.1111.111 = NaN)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.dec_e4m3(c) for c in range(256)])
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    fixed = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5,
             0x40: 2.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in fixed.items():
        assert oracle.dec_e4m3(c) == v, hex(c)
    assert math.copysign(1.0, oracle.dec_e4m3(0x80)) == -1.0


def test_fp8_pow2_scales_are_exact_products():
    """An FP8 packed row with power-of-two scales dequantises exactly, so the
    oracle must equal the plain-row oracle on rows holding those products
    (bf16 holds every E4M3 value times a power of two in range)."""
    pk = S.build("pk8", seed=13, q_n=4, q_lens=[1, 1], kv_lens=[80, 50], layout_q="BSND", layout_kv="BSND",
                 mode="ori_sparse", ori_topk=20, kv_format="fp8_packed", rope_head_dim=64, sinks=True)
    rows = pk.t["ori_kv"].view(-1, 656)
    nrows = rows.shape[0]
    scales = torch.pow(2.0, torch.tensor([-4.0, -6.0, -3.0, -5.0])).to(torch.float32).repeat(nrows, 1)
    rows[:, 640:656] = scales.view(torch.uint8).view(nrows, 16)
    rows[:, 512:640] = 0
    deq = rows[:, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float32) * scales.repeat_interleave(128, dim=1)
    plain = S.build("pl8", seed=13, q_n=4, q_lens=[1, 1], kv_lens=[80, 50], layout_q="BSND", layout_kv="BSND",
                    mode="ori_sparse", ori_topk=20, sinks=True)
    plain.t["ori_kv"] = deq.to(torch.bfloat16).view(pk.t["ori_kv"].shape[:-1] + (512,))
    assert torch.equal(plain.t["ori_kv"].float().view(-1, 512), deq)      # exact in bf16
    plain.t["q"] = pk.t["q"][..., :512].contiguous()
    plain.t["ori_sparse_indices"] = pk.t["ori_sparse_indices"]
    plain.t["sinks"] = pk.t["sinks"]
    plain.softmax_scale = pk.softmax_scale
    Op, lp = oracle.forward(pk)
    Ol, ll = oracle.forward(plain)
    np.testing.assert_array_equal(Op, Ol)
    np.testing.assert_array_equal(lp, ll)


def test_empty_rows_give_zero_and_neg_inf():
    prob = S.build("empty", seed=2, q_n=2, q_lens=[5, 3], kv_lens=[3, 20], layout_q="BSND", layout_kv="BSND",
                   mode="swa", win_left=1, win_right=0, ori_mask_mode=4, q_capacity=5, seqused_q=[5, 2])
    O, l = oracle.forward(prob)
    # batch 0: p = 3 - 5 + i < 0 for i < 2 -> empty; batch 1 rows i >= 2 are beyond seqused_q
    for t in (0, 1, 7, 8, 9):
        assert np.all(O[t] == 0) and np.all(np.isneginf(l[t])), t
    for t in (2, 3, 4, 5, 6):
        assert np.all(np.isfinite(l[t])), t
