"""GPU parity: the CUDA library (through its C-ABI) against the CPU oracle.

Tolerances (bf16 / fp16 inputs, fp32 accumulation, bf16 / fp16 output):
|O_gpu - O_ref| <= 2e-2 + 2e-2 |O_ref| element-wise and |LSE_gpu - LSE_ref| <=
1e-3 (packed int8 / FP8 rows included: their scores are exact products of
the unscaled values, scaled in fp32); rows with an empty attended set must
give exactly 0 and -inf.  Attended
row sets are compared exactly: the attention kernel's resolver records every
KV row it hands to its copy warps (sfm_debug_attended) and the sequence must
equal the oracle's attended set mapped to pool rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sfm_inputs as S
import sparse_shared_kv_gb300 as sfm
from tests import _brute, _sfm
from tests.test_oracle_pins import _tiny_cases

pytestmark = pytest.mark.gpu

ATOL = 2e-2
RTOL = 2e-2
LSE_ATOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    sfm.build()
    torch.cuda.init()


def assert_parity(prob, out, lse, tokens=None, host=None):
    host = host or prob.to("cpu")
    if tokens is None:
        tokens = list(range(prob.num_tokens))
    O_ref, L_ref = oracle.forward(host, tokens)
    got = out.reshape(prob.num_tokens, prob.num_heads_q, 512)[tokens].float().cpu().numpy().astype(np.float64)
    err = np.abs(got - O_ref)
    bound = ATOL + RTOL * np.abs(O_ref)
    bad = err > bound
    assert not bad.any(), (f"{prob.name}: {bad.sum()} O elements out of tolerance, max err "
                           f"{err.max():.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}")
    if lse is not None:
        gl = lse.reshape(prob.num_tokens, prob.num_heads_q)[tokens].cpu().numpy().astype(np.float64)
        assert np.array_equal(np.isneginf(gl), np.isneginf(L_ref)), f"{prob.name}: -inf LSE pattern differs"
        fin = np.isfinite(L_ref)
        if fin.any():
            tol = np.broadcast_to(LSE_ATOL, L_ref.shape)
            with np.errstate(invalid="ignore"):          # -inf - -inf on empty rows, masked below
                d = np.abs(gl - L_ref)
            assert (d[fin] <= tol[fin]).all(), (f"{prob.name}: LSE max err {d[fin].max():.3e}, "
                                                f"worst over tolerance {(d[fin] - tol[fin]).max():.3e}")
        empty = np.isneginf(L_ref)
        if empty.any():
            assert np.all(got[empty] == 0.0)
    return err.max()


def _pool_rows(host, t, src, pos):
    """Pool rows of the oracle's attended (src, pos) of token t, through the
    layout (and block table) by the test's own mapping."""
    b = _brute.lengths(host, t)[0]
    rows = np.zeros(len(pos), dtype=np.int64)
    for s_, which in ((0, "ori_kv"), (1, "cmp_kv")):
        m = src == s_
        if m.any():
            rows[m] = _brute._physical(host, which, b, int(pos[m].max()) + 1)[pos[m]]
    return rows


def assert_sets(prob, tokens=None, host=None, out=None, lse=None, params=None):
    """Exact attended sets of the attention kernel itself: the rows its
    resolver handed to the copy warps (sfm_debug_attended), in position
    order, against the oracle's attended set mapped to pool rows; every
    attended position must have been written.  With out / lse given, the
    dump call's outputs must equal them bit for bit (the dump does not change
    the computation)."""
    host = host or prob.to("cpu")
    entries, o_dbg, l_dbg, status = _sfm.debug_rows(prob, params=params)
    assert status & ~sfm.STATUS_BAD_INDEX == 0, hex(status)
    if out is not None:
        assert torch.equal(o_dbg, out), f"{prob.name}: output of the dump call differs"
    if lse is not None:
        assert torch.equal(l_dbg, lse), f"{prob.name}: LSE of the dump call differs"
    if tokens is None:
        tokens = range(prob.num_tokens)
    b = oracle._Bound(host)
    for t in tokens:
        src, pos = oracle.attended(host, t, b)
        e = entries[t]
        assert (e != _sfm.UNWRITTEN).all(), f"{prob.name}: token {t}: attended positions the resolver never wrote"
        gs, gr = _sfm.split_entries(e)
        want = _pool_rows(host, t, src, pos)
        assert np.array_equal(gs, src) and np.array_equal(gr, want), \
            f"{prob.name}: token {t}: resolved rows differ from the oracle's attended set"


# ---------------------------------------------------------------------------
# tiny cases: every mode, layout, dtype, padded rows, packed rows, bad indices
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name,kw", _tiny_cases(), ids=[c[0] for c in _tiny_cases()])
def test_tiny_parity_and_sets(name, kw):
    prob = S.build(name, seed=11, q_n=4, device="cuda", **kw)
    if name == "csa_tnd_any_idx":
        idx = prob.t["cmp_sparse_indices"]
        idx[0, 0, 1] = idx[0, 0, 0]
        idx[1, 0, 2] = 10_000
        idx[2, 0, 0] = -7
    out, lse, status = _sfm.run(prob)
    expected = sfm.STATUS_BAD_INDEX if name == "csa_tnd_any_idx" else 0
    assert status == expected, hex(status)
    assert_parity(prob, out, lse)
    assert_sets(prob, out=out, lse=lse)


@pytest.mark.parametrize("q_n", [1, 2, 8, 16, 32, 48, 64, 128])
def test_head_counts(q_n):
    prob = S.build(f"heads{q_n}", seed=q_n, device="cuda", q_n=q_n, q_lens=[1, 1, 1], kv_lens=[700, 1500, 300],
                   layout_q="BSND", layout_kv="PAGED", mode="csa", cmp_ratio=4, cmp_topk=96, sinks=True)
    out, lse, status = _sfm.run(prob)
    assert status == 0
    assert_parity(prob, out, lse)


# ---------------------------------------------------------------------------
# the five workloads, reduced so the oracle checks every row
# ---------------------------------------------------------------------------
REDUCED = {
    "swa_decode_tiny": lambda: S.swa_decode_tiny(device="cuda"),
    "csa_decode_b4": lambda: S.csa_decode(device="cuda", batch=4),
    "hca_decode_b2": lambda: S.hca_decode(device="cuda", batch=2),
    "hca_decode_b2_compact_pool": lambda: S.hca_decode(device="cuda", batch=2, compact_pool=True),
    "csa_prefill_small": lambda: S.csa_prefill(device="cuda", nseq=3, qmin=40, qmax=300, prefix_max=700),
    "packed_decode_b3": lambda: S.packed_decode(device="cuda", batch=3, kv_len=8192),
}


@pytest.mark.parametrize("key", list(REDUCED))
def test_reduced_workloads(key):
    prob = REDUCED[key]()
    out, lse, status = _sfm.run(prob)
    assert status == 0, hex(status)
    host = prob.to("cpu")
    assert_parity(prob, out, lse, host=host)
    assert_sets(prob, host=host, out=out, lse=lse)


@pytest.mark.parametrize("batch", [4, 32], ids=["reduced", "full_size"])
def test_csa_topk_1024(batch):
    """CSA with 1024 compressed indices per query, the second top-k size the
    pages allow for cmp_sparse_indices (512 or 1024): every row of a reduced
    batch, sampled rows of the full-size decode batch, sets exactly."""
    prob = S.csa_decode(device="cuda", batch=batch, cmp_topk=1024, seed=9)
    out, lse, status = _sfm.run(prob)
    assert status == 0, hex(status)
    host = prob.to("cpu")
    tokens = None if batch <= 4 else _sample(prob, 12)
    assert_parity(prob, out, lse, tokens=tokens, host=host)
    assert_sets(prob, tokens=tokens, host=host, out=out, lse=lse)


@pytest.mark.parametrize("mode", ["csa", "hca"])
def test_largest_pages(mode):
    """Paged ori and cmp caches with the largest page the parameter rules
    allow (1024 rows per block): windows and compressed rows that straddle
    page boundaries, every row against the oracle, attended sets exact."""
    kw = dict(q_n=64, q_lens=[1, 1, 1], kv_lens=[5000, 2100, 9000], layout_q="BSND", layout_kv="PAGED",
              mode=mode, cmp_ratio=4 if mode == "csa" else 16, ori_block_size=1024, cmp_block_size=1024,
              sinks=True)
    if mode == "csa":
        kw["cmp_topk"] = 512
    prob = S.build(f"pages1024_{mode}", seed=23, device="cuda", **kw)
    out, lse, status = _sfm.run(prob)
    assert status == 0, hex(status)
    host = prob.to("cpu")
    assert_parity(prob, out, lse, host=host)
    assert_sets(prob, host=host, out=out, lse=lse)


def test_fp16_and_lse_off():
    prob = S.build("fp16_nolse", seed=5, device="cuda", q_n=64, q_lens=[1, 1], kv_lens=[900, 4000],
                   layout_q="BSND", layout_kv="PAGED", mode="hca", cmp_ratio=16, dtype="fp16", sinks=True,
                   return_lse=False)
    out, lse, status = _sfm.run(prob)
    assert lse is None and status == 0
    assert_parity(prob, out, None)


# ---------------------------------------------------------------------------
# full sizes, sampled rows (the launch configuration the benchmark times)
# ---------------------------------------------------------------------------
def _sample(prob, n, extra=()):
    g = torch.Generator().manual_seed(123)
    T = prob.num_tokens
    pick = set(torch.randperm(T, generator=g)[:n].tolist()) | {0, T - 1} | set(extra)
    return sorted(t for t in pick if 0 <= t < T)


@pytest.mark.parametrize("key", ["csa_decode", "hca_decode", "csa_prefill", "packed_decode", "packed_fp8_decode"])
def test_full_size_sampled(key):
    prob = S.WORKLOADS[key](device="cuda")
    out, lse, status = _sfm.run(prob)
    assert status == 0, hex(status)
    extra = ()
    if key == "csa_prefill":
        cu = prob.t["cu_seqlens_q"].tolist()
        extra = [c + d for c in cu[:-1] for d in (0, 1, 129)] + [c - 1 for c in cu[1:]]
    tokens = _sample(prob, 24 if key != "csa_prefill" else 64, extra)
    host = prob.to("cpu")
    assert_parity(prob, out, lse, tokens=tokens, host=host)
    assert_sets(prob, tokens=tokens, host=host, out=out, lse=lse)
    # properties that hold at any size: finite outputs, LSE finite where rows attend something
    assert torch.isfinite(out.float()).all()


# ---------------------------------------------------------------------------
# properties of the library itself
# ---------------------------------------------------------------------------
def test_deterministic():
    prob = S.csa_decode(device="cuda", batch=8)
    r = _sfm.Runner(prob)
    o1, l1, _ = r.run()
    o1, l1 = o1.clone(), l1.clone()
    o2, l2, _ = r.run()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_batch_invariance():
    """A sequence's result is bitwise the same alone and inside a batch."""
    prob = S.csa_decode(device="cuda", batch=6)
    out, lse, _ = _sfm.run(prob)
    out, lse = out.clone(), lse.clone()
    for b in (0, 3, 5):
        single = S.build("single", seed=0, device="cuda", q_n=64, q_lens=[1], kv_lens=[prob.kv_lens[b]],
                         layout_q="BSND", layout_kv="PAGED", mode="csa", cmp_ratio=4, cmp_topk=512, sinks=True)
        for k in ("ori_kv", "cmp_kv", "sinks"):
            single.t[k] = prob.t[k]
        single.t["q"] = prob.t["q"][b:b + 1].clone()
        single.t["cmp_sparse_indices"] = prob.t["cmp_sparse_indices"][b:b + 1].clone()
        single.t["ori_block_table"] = prob.t["ori_block_table"][b:b + 1].clone()
        single.t["cmp_block_table"] = prob.t["cmp_block_table"][b:b + 1].clone()
        for k in ("seqused_ori_kv", "seqused_cmp_kv", "cmp_residual_kv"):
            single.t[k] = prob.t[k][b:b + 1].clone()
        o1, l1, st = _sfm.run(single)
        assert st == 0
        assert torch.equal(o1[0], out[b]) and torch.equal(l1[0], lse[b]), b


# ---------------------------------------------------------------------------
# occupancy split policy: batches too small to fill the SMs are cut finer
# ---------------------------------------------------------------------------
OCCUPANCY = {
    "csa_decode_b4": lambda: S.csa_decode(device="cuda", batch=4),
    "hca_decode_b8": lambda: S.hca_decode(device="cuda", batch=8, compact_pool=True),
    "packed_decode_b3": lambda: S.packed_decode(device="cuda", batch=3, kv_len=8192),
    "packed_fp8_decode_b2": lambda: S.packed_fp8_decode(device="cuda", batch=2, kv_len=8192),
    # prefill-shaped (more than 16 query rows per sequence: one split per row
    # by default): 2 sequences of 17-24 rows
    "csa_prefill_tiny": lambda: S.csa_prefill(device="cuda", nseq=2, qmin=17, qmax=24, prefix_max=3000),
}


def _units(meta, q_n):
    m = meta.cpu().numpy()
    return int(m[6]) * ((q_n + 63) // 64), int(m[4])


@pytest.mark.parametrize("key", list(OCCUPANCY))
def test_occupancy_policy(key):
    """SFM_SPLIT_OCCUPANCY: the plan of a small batch has more work units than
    the batch-invariant one (at least 64 for eight 128-head HCA rows, which
    the batch-invariant plan runs as 16), the outputs match the oracle on
    every row, the attended sets are exact, and two calls give the same
    bits."""
    prob = OCCUPANCY[key]()
    inv = _sfm.Runner(prob)
    inv.plan()
    occ = _sfm.Runner(prob, _sfm.params_of(prob, split_policy=sfm.SPLIT_OCCUPANCY))
    out, lse, status = occ.run()
    assert status == 0, hex(status)
    u_inv, s_inv = _units(inv.meta, prob.num_heads_q)
    u_occ, s_occ = _units(occ.meta, prob.num_heads_q)
    assert u_occ > u_inv and s_occ < s_inv, (u_inv, u_occ, s_inv, s_occ)
    if key == "hca_decode_b8":
        assert u_inv == 16 and u_occ >= 64, (u_inv, u_occ)
    out, lse = out.clone(), lse.clone()
    host = prob.to("cpu")
    assert_parity(prob, out, lse, host=host)
    assert_sets(prob, host=host, out=out, lse=lse, params=occ.params)
    o2, l2, _ = occ.run()
    assert torch.equal(o2, out) and torch.equal(l2, lse)


def test_occupancy_policy_keeps_full_batches_invariant():
    """Where the batch-invariant plan already gives every CTA a unit, the
    occupancy policy leaves the plan (and so the bits) unchanged."""
    prob = S.csa_decode(device="cuda", batch=64, seed=3)
    a = _sfm.Runner(prob)
    b = _sfm.Runner(prob, _sfm.params_of(prob, split_policy=sfm.SPLIT_OCCUPANCY))
    oa, la, sa = a.run()
    ob, lb, sb = b.run()
    assert sa == 0 and sb == 0
    assert _units(a.meta, 64) == _units(b.meta, 64)
    assert torch.equal(oa, ob) and torch.equal(la, lb)


def test_plan_sees_lengths_written_just_before():
    """sfm_metadata reads the length tensors before it waits for the kernel
    before it in the stream; a kernel that does not release its dependents
    early (torch's, like most) still orders its writes first: lengths
    shortened by a torch kernel right before the plan, on the same stream
    with no synchronisation, are the ones the plan and the forward use."""
    prob = S.csa_decode(device="cuda", batch=4, seed=17)
    r = _sfm.Runner(prob)
    _, _, status = r.run()
    assert status == 0
    torch.cuda.synchronize()
    prob.t["seqused_ori_kv"].sub_(3)        # the window moves back three rows
    r.status.zero_()
    r.plan()
    r.forward()
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    host = prob.to("cpu")
    assert_parity(prob, r.out, r.lse, host=host)


def test_context_parallel_split_on_gpu():
    from tests.test_oracle_pins import _cp_slice
    g = S.build("cp_global", seed=21, q_n=64, q_lens=[16, 18], kv_lens=[16, 18], cmp_lens=[4, 4],
                residuals=[0, 2], layout_q="TND", layout_kv="TND", mode="csa", cmp_ratio=4, cmp_topk=512,
                index_mode="all_visible", sinks=True)
    r0 = _cp_slice(g, [(0, 16), (16, 24)], [(0, 16), (16, 24)], [(0, 4), (4, 6)], [16, 8], [16, 8], [4, 2], [0, 0])
    r1 = _cp_slice(g, [(24, 34)], [(16, 34)], [(4, 8)], [10], [18], [4], [2])
    outs = []
    for p in (g, r0, r1):
        pg = p.to("cuda")
        o, l, st = _sfm.run(pg)
        assert st == 0
        assert_parity(pg, o, l, host=p)
        outs.append(o.cpu())
    # the global call is prefill-shaped (one split per row) and the rank calls are
    # decode-shaped (fixed-size splits merged by the combine), so the two agree
    # to rounding, not bit for bit
    d = (torch.cat([outs[1], outs[2]]).float() - outs[0].float()).abs()
    assert d.max().item() <= ATOL


def test_bad_values_are_flagged_not_faulted():
    prob = S.build("bad", seed=3, device="cuda", q_n=8, q_lens=[1, 1], kv_lens=[300, 500], layout_q="BSND",
                   layout_kv="PAGED", mode="csa", cmp_ratio=4, cmp_topk=16, sinks=True)
    prob.t["cmp_sparse_indices"][0, 0, 0, 3] = 1 << 20            # beyond cmp_len
    prob.t["ori_block_table"][1, 2] = 1 << 24                     # beyond the cache
    out, lse, status = _sfm.run(prob)
    assert status & sfm.STATUS_BAD_INDEX and status & sfm.STATUS_BAD_BLOCK
    assert torch.isfinite(out.float()).all()
    # the rows that stayed valid still match the oracle (which skips the same entries)
    host = prob.to("cpu")
    host.t["ori_block_table"][1, 2] = 0
    O_ref, _ = oracle.forward(host, [0])
    got = out[0].float().cpu().numpy()
    assert np.all(np.abs(got - O_ref[0]) <= ATOL + RTOL * np.abs(O_ref[0]))


def test_metadata_mismatch_zeroes_outputs():
    prob = S.csa_decode(device="cuda", batch=2)
    r = _sfm.Runner(prob)
    r.run()
    other = _sfm.params_of(prob, ori_win_left=63)
    md = torch.empty(sfm.sfm_metadata_size(other), dtype=torch.int32, device="cuda")
    sfm.sfm_metadata(other, r.tensors, md)
    r.status.zero_()
    sfm.sfm_forward(r.params, r.tensors, md, prob.softmax_scale, r.out, r.lse, r.ws, r.status)
    torch.cuda.synchronize()
    assert int(r.status.item()) & sfm.STATUS_METADATA_MISMATCH
    assert torch.count_nonzero(r.out.float()) == 0 and torch.isneginf(r.lse).all()


def test_metadata_mismatch_zeroes_outputs_without_combine():
    # 128 heads: one split per row, so no combine kernel runs and the
    # attention kernel itself reports the mismatch and zeroes every row
    prob = S.build("mismatch128", seed=5, device="cuda", q_n=128, q_lens=[1, 1, 1], kv_lens=[700, 0, 1500],
                   layout_kv="PAGED", mode="hca", cmp_ratio=128, sinks=True)
    r = _sfm.Runner(prob)
    assert sfm.sfm_workspace_size(r.params) == 0
    out, lse, status = r.run()
    assert status == 0
    assert_parity(prob, out, lse)          # the empty row: O = 0, LSE = -inf
    other = _sfm.params_of(prob, ori_win_left=63)
    md = torch.empty(sfm.sfm_metadata_size(other), dtype=torch.int32, device="cuda")
    sfm.sfm_metadata(other, r.tensors, md)
    r.status.zero_()
    sfm.sfm_forward(r.params, r.tensors, md, prob.softmax_scale, r.out, r.lse, r.ws, r.status)
    torch.cuda.synchronize()
    assert int(r.status.item()) & sfm.STATUS_METADATA_MISMATCH
    assert torch.count_nonzero(r.out.float()) == 0 and torch.isneginf(r.lse).all()


@pytest.mark.parametrize("return_lse", [False, True], ids=["lse_off", "lse_on"])
@pytest.mark.parametrize("fmt", ["int8_packed", "fp8_packed"])
def test_packed_128_heads_row_without_positions(fmt, return_lse):
    """128-head packed decode plans have at most one split per row, so no
    combine kernel runs: the attention kernel itself must write the row with
    no attended position (kv_len 0) as O = 0 (and LSE = -inf when returned)
    and leave the status clean."""
    prob = S.build("packed_empty", seed=88, device="cuda", q_n=128, q_lens=[1, 1, 1], kv_lens=[900, 0, 1500],
                   layout_q="BSND", layout_kv="PAGED", mode="ori_sparse", ori_topk=256, ori_mask_mode=3,
                   cmp_mask_mode=0, kv_format=fmt, rope_head_dim=64, ori_block_size=64, sinks=True,
                   return_lse=return_lse)
    r = _sfm.Runner(prob)
    assert sfm.sfm_workspace_size(r.params) == 0          # one split per row: no combine launch
    r.out.fill_(float("nan"))
    if r.lse is not None:
        r.lse.fill_(float("nan"))
    out, lse, status = r.run()
    assert status == 0, hex(status)
    assert (lse is None) == (not return_lse)
    assert torch.count_nonzero(out[1].float()) == 0
    if lse is not None:
        assert torch.isneginf(lse[1]).all()
    assert_parity(prob, out, lse)
    assert_sets(prob, out=out, lse=lse)


@pytest.mark.parametrize("batch_invariant", [True, False], ids=["invariant", "occupancy"])
def test_public_two_call_api(batch_invariant):
    prob = S.csa_decode(device="cuda", batch=3)
    T = prob.t
    md = sfm.sparse_flash_mla_metadata(
        64, 1, 512, seqused_ori_kv=T["seqused_ori_kv"], seqused_cmp_kv=T["seqused_cmp_kv"],
        cmp_residual_kv=T["cmp_residual_kv"], batch_size=3, max_seqlen_q=1, max_seqlen_ori_kv=prob.max_seqlen_ori_kv,
        max_seqlen_cmp_kv=prob.max_seqlen_cmp_kv, cmp_topk=512, cmp_ratio=4, ori_mask_mode=4, cmp_mask_mode=3,
        ori_win_left=127, ori_win_right=0, layout_q="BSND", layout_kv="PAGED", ori_block_size=128,
        cmp_block_size=128, return_softmax_lse=True, batch_invariant=batch_invariant)
    assert md.params.split_policy == (sfm.SPLIT_BATCH_INVARIANT if batch_invariant else sfm.SPLIT_OCCUPANCY)
    out, lse = sfm.sparse_flash_mla(
        T["q"], metadata=md, ori_kv=T["ori_kv"], cmp_kv=T["cmp_kv"], cmp_sparse_indices=T["cmp_sparse_indices"],
        ori_block_table=T["ori_block_table"], cmp_block_table=T["cmp_block_table"],
        seqused_ori_kv=T["seqused_ori_kv"], seqused_cmp_kv=T["seqused_cmp_kv"],
        cmp_residual_kv=T["cmp_residual_kv"], sinks=T["sinks"], softmax_scale=1 / math.sqrt(512))
    torch.cuda.synchronize()
    assert out.shape == T["q"].shape
    assert_parity(prob, out, lse)


def _api_call(prob, T, out, lse, stream):
    md = sfm.sparse_flash_mla_metadata(
        prob.num_heads_q, 1, 512, seqused_ori_kv=T["seqused_ori_kv"], seqused_cmp_kv=T["seqused_cmp_kv"],
        cmp_residual_kv=T["cmp_residual_kv"], batch_size=prob.batch_size, max_seqlen_q=1,
        max_seqlen_ori_kv=prob.max_seqlen_ori_kv, max_seqlen_cmp_kv=prob.max_seqlen_cmp_kv,
        cmp_topk=prob.cmp_topk, cmp_ratio=prob.cmp_ratio, ori_mask_mode=prob.ori_mask_mode,
        cmp_mask_mode=prob.cmp_mask_mode, ori_win_left=prob.ori_win_left, ori_win_right=prob.ori_win_right,
        layout_q="BSND", layout_kv="PAGED", ori_block_size=prob.ori_block_size,
        cmp_block_size=prob.cmp_block_size, return_softmax_lse=True, stream=stream)
    sfm.sparse_flash_mla(
        T["q"], metadata=md, ori_kv=T["ori_kv"], cmp_kv=T["cmp_kv"], cmp_sparse_indices=T["cmp_sparse_indices"],
        ori_block_table=T["ori_block_table"], cmp_block_table=T["cmp_block_table"],
        seqused_ori_kv=T["seqused_ori_kv"], seqused_cmp_kv=T["seqused_cmp_kv"],
        cmp_residual_kv=T["cmp_residual_kv"], sinks=T["sinks"], softmax_scale=prob.softmax_scale, out=out,
        lse=lse, stream=stream)


def test_two_call_api_in_cuda_graphs_on_two_streams():
    """Both calls captured in a CUDA graph (planner, attention and combine
    chained by programmatic dependent launch), two independent problems
    replayed alternately on two streams: results equal the eager calls bit
    for bit and meet the oracle."""
    probs = [S.csa_decode(device="cuda", batch=5, seed=71), S.csa_decode(device="cuda", batch=7, seed=72)]
    eager, graphs, outs = [], [], []
    for prob in probs:
        T = prob.t
        out = torch.empty(T["q"].shape, dtype=T["q"].dtype, device="cuda")
        lse = torch.empty(prob.num_tokens * prob.num_heads_q, dtype=torch.float32, device="cuda")
        _api_call(prob, T, out, lse, torch.cuda.current_stream())
        torch.cuda.synchronize()
        eager.append((out.clone(), lse.clone()))
        out.zero_()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            _api_call(prob, T, out, lse, side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            _api_call(prob, T, out, lse, torch.cuda.current_stream())
        graphs.append(g)
        outs.append((out, lse))
    for o, l in outs:
        o.zero_()
        l.zero_()
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for k in range(8):
        with torch.cuda.stream(streams[k % 2]):
            graphs[k % 2].replay()
    torch.cuda.synchronize()
    for prob, (o, l), (eo, el) in zip(probs, outs, eager):
        assert torch.equal(o, eo) and torch.equal(l, el)
        assert_parity(prob, o, l)


def test_independent_problems_on_eight_streams():
    """Independent problems (CSA decode, HCA decode, packed INT8 decode, CSA
    prefill, each with its own plan, workspace and outputs) dealt round robin
    over eight streams for several rounds, a problem's next step ordered
    after its previous one by an event, so kernels of different problems run
    at the same time: every result equals the problem's eager result bit for
    bit and meets the oracle."""
    probs = [S.csa_decode(device="cuda", batch=4, seed=81), S.csa_decode(device="cuda", batch=9, seed=82),
             S.hca_decode(device="cuda", batch=2, compact_pool=True, seed=83),
             S.packed_decode(device="cuda", batch=2, kv_len=4096, seed=84),
             S.csa_prefill(device="cuda", nseq=2, qmin=40, qmax=120, prefix_max=500, seed=85),
             S.csa_decode(device="cuda", batch=3, cmp_topk=1024, seed=86)]
    runners = [_sfm.Runner(p) for p in probs]
    eager = []
    for r in runners:
        out, lse, status = r.run()
        assert status == 0, hex(status)
        eager.append((out.clone(), lse.clone()))
        r.out.zero_()
        r.lse.zero_()
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(8)]
    done = [None] * len(runners)
    cur = torch.cuda.current_stream()
    for st in streams:
        st.wait_stream(cur)
    for k in range(4 * len(runners)):
        i = k % len(runners)
        st = streams[k % len(streams)]
        if done[i] is not None:
            st.wait_event(done[i])
        runners[i].plan(st)
        runners[i].forward(st)
        done[i] = torch.cuda.Event()
        done[i].record(st)
    for st in streams:
        cur.wait_stream(st)
    torch.cuda.synchronize()
    for prob, r, (eo, el) in zip(probs, runners, eager):
        assert int(r.status.item()) == 0
        assert torch.equal(r.out, eo) and torch.equal(r.lse, el), prob.name
        assert_parity(prob, r.out, r.lse)


# ---------------------------------------------------------------------------
# the attention kernel's code paths: head counts, split counts, dtypes,
# block-wise selection, packed formats
# ---------------------------------------------------------------------------
def _plain_cases():
    return [c for c in _tiny_cases() if "packed" not in c[0]]


@pytest.mark.parametrize("name,kw", _plain_cases(), ids=[c[0] for c in _plain_cases()])
def test_kernel_paths_tiny(name, kw):
    prob = S.build(name, seed=17, q_n=4, device="cuda", **kw)
    out, lse, status = _sfm.run(prob)
    assert status == 0, hex(status)
    assert_parity(prob, out, lse)
    assert_sets(prob, out=out, lse=lse)


@pytest.mark.parametrize("q_n", [1, 8, 16, 32, 40, 64, 65, 96, 128])
def test_kernel_paths_heads(q_n):
    prob = S.build(f"heads{q_n}", seed=100 + q_n, device="cuda", q_n=q_n, q_lens=[1, 1, 1, 1],
                   kv_lens=[700, 1500, 300, 20000], layout_q="BSND", layout_kv="PAGED", mode="csa", cmp_ratio=4,
                   cmp_topk=384, sinks=True)
    out, lse, status = _sfm.run(prob)
    assert status == 0, hex(status)
    assert_parity(prob, out, lse)
    assert_sets(prob, out=out, lse=lse)


def test_many_splits_and_single_split_rows():
    # a causal decode batch mixing a row of 6000 positions (dozens of splits:
    # the combine's looped merge past its unrolled case), a row of one split
    # (written directly by the attention kernel) and rows in between
    prob = S.build("many_splits", seed=61, device="cuda", q_n=64, q_lens=[1, 1, 1, 1],
                   kv_lens=[6000, 100, 1300, 2600], layout_q="BSND", layout_kv="PAGED", mode="swa",
                   ori_mask_mode=3, win_left=-1, win_right=-1, sinks=True)
    out, lse, status = _sfm.run(prob)
    assert status == 0, hex(status)
    assert_parity(prob, out, lse)
    assert_sets(prob, out=out, lse=lse)


def test_kernel_paths_prefill_fp16():
    prob = S.build("prefill_fp16", seed=23, device="cuda", q_n=64, q_lens=[70, 130], kv_lens=[200, 900],
                   layout_q="TND", layout_kv="PAGED", mode="hca", cmp_ratio=4, dtype="fp16", sinks=True,
                   ori_block_size=64, cmp_block_size=32)
    out, lse, status = _sfm.run(prob)
    assert status == 0, hex(status)
    assert_parity(prob, out, lse)
    assert_sets(prob, out=out, lse=lse)


@pytest.mark.parametrize("sbs", [2, 16, 64])
def test_blockwise_selection(sbs):
    # block-wise top-k over a paged packed pool (each index selects sbs
    # consecutive tokens, masked per token by right-down causality); indices
    # include masked (-1), partly visible and out-of-range blocks
    prob = S.build(f"blockwise{sbs}", seed=400 + sbs, device="cuda", q_n=64, q_lens=[1, 2, 1],
                   kv_lens=[1500, 3000, 200], layout_q="BSND", layout_kv="PAGED", mode="ori_sparse",
                   ori_topk=2048 // sbs, ori_mask_mode=3, cmp_mask_mode=0, kv_format="int8_packed",
                   rope_head_dim=64, ori_block_size=64, sparse_block_size=sbs, index_mode="any",
                   softmax_scale=1.0 / 24.0)
    out, lse, status = _sfm.run(prob)
    assert status in (0, 1), hex(status)
    assert_parity(prob, out, lse)
    assert_sets(prob, out=out, lse=lse)


@pytest.mark.parametrize("fmt", ["int8_packed", "fp8_packed"])
def test_rope0_rows_equal_zero_padded_rows(fmt):
    """Compact 528-byte rows (rope_head_dim 0, q of 512 dims) against the same
    NoPE bytes and scales in 656-byte rows with a zero rope part and q's rope
    part zero: bit for bit the same output and LSE
    (the kv_quant guide's rope-0 test compares the two with torch.equal)."""
    kw = dict(seed=77, device="cuda", q_n=64, q_lens=[1, 1], kv_lens=[1200, 700], layout_q="BSND",
              layout_kv="PAGED", mode="ori_sparse", ori_topk=256, ori_mask_mode=3, cmp_mask_mode=0,
              kv_format=fmt, ori_block_size=64, sinks=True)
    p64 = S.build("pad", rope_head_dim=64, **kw)
    p0 = S.build("compact", rope_head_dim=0, **kw)
    r64 = p64.t["ori_kv"].view(-1, 656)
    r0 = p0.t["ori_kv"].view(-1, 528)
    r64[:, 512:640] = 0                           # zero rope part
    r64[:, 640:656] = r0[:, 512:528]              # the compact rows' scales
    r64[:, :512] = r0[:, :512]                    # the compact rows' NoPE bytes
    p64.t["ori_block_table"] = p0.t["ori_block_table"]
    p64.t["ori_sparse_indices"] = p0.t["ori_sparse_indices"]
    p64.t["sinks"] = p0.t["sinks"]
    q = p64.t["q"]
    q[..., :512] = p0.t["q"]
    q[..., 512:] = 0
    p64.softmax_scale = p0.softmax_scale
    o64, l64, st64 = _sfm.run(p64)
    o0, l0, st0 = _sfm.run(p0)
    assert st64 == 0 and st0 == 0
    assert torch.equal(o64, o0) and torch.equal(l64, l0)
    assert_parity(p0, o0, l0)


@pytest.mark.parametrize("rope", [0, 64])
@pytest.mark.parametrize("fmt", ["int8_packed", "fp8_packed"])
@pytest.mark.parametrize("q_n", [16, 64, 128])
def test_kernel_paths_packed(q_n, fmt, rope):
    # packed int8 / E4M3 rows (656 bytes) with token-wise top-k over a paged
    # pool; the index lists include masked (-1) and future entries
    prob = S.build(f"packed{q_n}", seed=300 + q_n, device="cuda", q_n=q_n, q_lens=[1, 1, 1], kv_lens=[900, 3000, 200],
                   layout_q="BSND", layout_kv="PAGED", mode="ori_sparse", ori_topk=256, ori_mask_mode=3,
                   cmp_mask_mode=0, kv_format=fmt, rope_head_dim=rope, ori_block_size=64,
                   index_mode="any", softmax_scale=1.0 / 24.0)
    out, lse, status = _sfm.run(prob)
    assert status in (0, 1), hex(status)       # out-of-range indices are flagged (BAD_INDEX) and skipped
    assert_parity(prob, out, lse)
    assert_sets(prob, out=out, lse=lse)
