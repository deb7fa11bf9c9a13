"""GPU: the device planner's metadata, word by word, against the plan's
definition recomputed on the host.

The plan ("sparse_flash_mla_metadata": the task split of the main call)
is: per query row t its attended-position count n_t = n_ori + n_cmp, cut
into ns_t = ceil(n_t / S) equal splits of size ceil(n_t / ns_t) rounded up to
32 rows; the split table sp = exclusive prefix of ns; per split a record
(row, first split, split count, size | batch, kv_len, cmp_len, p_cmp | window
lo, hi, n_ori, n_cmp); units = (split, head group), group-major in a row; and
worker c starting at the unit whose modelled-cost span holds floor(c total /
G), a unit costing its split size plus a fixed 128 rows.  The row words are
checked against the oracle's lengths and positions, the window and counts
against the mask rules written out here.  Batches of at most 64 rows and more
than 64 rows go through the planner's two kernels.
"""
import numpy as np
import pytest
import torch

import oracle
import sfm_inputs as S
import sparse_shared_kv_gb300 as sfm
from tests import _sfm

pytestmark = pytest.mark.gpu

HDR = 16
OVERHEAD = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    sfm.build()
    torch.cuda.init()


def _expected_rows(prob):
    """Per row: (b, kv_len, cmp_len, p_cmp, lo, hi, n_ori, n_cmp)."""
    rows = []
    host = prob.to("cpu")
    bound = oracle._Bound(host)
    for t in range(prob.num_tokens):
        b, i, q_len, kv_len, cmp_len, _res, p, p_cmp, in_range = oracle.token_info(host, t, bound)
        assert p == kv_len - q_len + i
        lo, hi = 0, kv_len - 1
        if prob.ori_mask_mode == 3:
            hi = min(hi, p)
        elif prob.ori_mask_mode == 4:
            if prob.ori_win_left >= 0:
                lo = max(lo, p - prob.ori_win_left)
            if prob.ori_win_right >= 0:
                hi = min(hi, p + prob.ori_win_right)
        if hi < lo:
            lo, hi = 0, -1
        n_ori = n_cmp = 0
        if in_range and kv_len > 0:
            n_ori = prob.ori_topk * prob.sparse_block_size if prob.ori_topk > 0 else hi - lo + 1
        if in_range and prob.has_cmp_kv and cmp_len > 0:
            if prob.cmp_topk > 0:
                n_cmp = prob.cmp_topk
            elif prob.cmp_mask_mode == 3:
                n_cmp = min(cmp_len, max(0, (p_cmp + 1) // prob.cmp_ratio))
            else:
                n_cmp = cmp_len
        rows.append((b, kv_len, cmp_len, p_cmp, lo, hi, n_ori, n_cmp))
    return rows


def _shape(n, S_):
    if n <= 0:
        return 0, S_
    ns = -(-n // S_)
    size = n if ns == 1 else -(-n // ns)
    return ns, (size + 31) // 32 * 32


def check_plan(prob, meta, q_n):
    m = meta.cpu().numpy().astype(np.int64)
    T, G, S_, path = int(m[2]), int(m[3]), int(m[4]), int(m[5])
    assert T == prob.num_tokens
    assert m[7] == 0 and m[8] == 0, (m[7], m[8])       # plan flags, length flags
    wcap = int(m[9])
    HG = (q_n + 63) // 64 if path == 2 else 1
    rows = _expected_rows(prob)
    shapes = [_shape(r[6] + r[7], S_) for r in rows]
    ns = np.array([s[0] for s in shapes], dtype=np.int64)
    sp_exp = np.concatenate([[0], np.cumsum(ns)])
    W = int(sp_exp[-1])
    assert m[6] == W and W <= wcap

    ws_off = HDR
    sp_off = HDR + G + 1
    rec_off = sp_off + 2 * (T + 1)
    srec_off = (rec_off + 8 * T + 15) & ~15
    wrec_off = srec_off + 16 * wcap
    np.testing.assert_array_equal(m[sp_off:sp_off + T + 1], sp_exp)

    srec = m[srec_off:srec_off + 16 * W].reshape(W, 16)[:, :12]
    for t, (r, (nst, size)) in enumerate(zip(rows, shapes)):
        for j in range(nst):
            w = int(sp_exp[t]) + j
            assert list(srec[w]) == [t, sp_exp[t], nst, size, *r], (t, j, list(srec[w]))

    # worker starts from the modelled cost
    ucost = np.array([s[1] + OVERHEAD for s in shapes], dtype=np.int64)
    cost = ns * HG * ucost
    incl = np.cumsum(cost)
    total = int(incl[-1]) if T else 0
    ws_exp = np.zeros(G + 1, dtype=np.int64)
    ws_exp[G] = W * HG
    if total > 0:
        for c in range(G):
            tgt = c * total // G
            t = int(np.searchsorted(incl, tgt, side="right"))
            c0 = int(incl[t] - cost[t])
            j = min(int(ns[t]) * HG - 1, (tgt - c0) // int(ucost[t]))
            ws_exp[c] = int(sp_exp[t]) * HG + j
    ws = m[ws_off:ws_off + G + 1]
    np.testing.assert_array_equal(ws, ws_exp)
    assert np.all(np.diff(ws) >= 0)

    wrec = m[wrec_off:wrec_off + 16 * G].reshape(G, 16)
    for c in range(G):
        assert list(wrec[c, :4]) == [ws[c], ws[c + 1], 0, 0], c
        if ws[c] < ws[c + 1]:
            assert list(wrec[c, 4:16]) == list(srec[ws[c] // HG]), c
    return W, G


CASES = {
    # at most 64 rows
    "csa_decode_32": dict(q_n=64, q_lens=[1] * 32, kv_lens=list(range(300, 300 + 32 * 97, 97)), layout_kv="PAGED",
                          mode="csa", cmp_ratio=4, cmp_topk=128, sinks=True),
    "hca_decode_64_heads128": dict(q_n=128, q_lens=[1] * 64, kv_lens=[2000 + 13 * b for b in range(64)],
                                   layout_kv="PAGED", mode="hca", cmp_ratio=128),
    "hca_decode_8_heads128": dict(q_n=128, q_lens=[1] * 8, kv_lens=[1500 + 977 * b for b in range(8)],
                                  layout_kv="PAGED", mode="hca", cmp_ratio=128),
    "swa_empty_rows": dict(q_n=16, q_lens=[1] * 6, kv_lens=[0, 500, 0, 1000, 3, 0], layout_kv="PAGED", mode="swa"),
    "causal_many_splits": dict(q_n=64, q_lens=[1, 1, 1, 1], kv_lens=[6000, 100, 1300, 2600], layout_kv="PAGED",
                               mode="swa", ori_mask_mode=3, win_left=-1, win_right=-1),
    "csa_decode_40_rows": dict(q_n=32, q_lens=[1] * 40, kv_lens=[100 + 211 * b for b in range(40)],
                               layout_kv="PAGED", mode="csa", cmp_ratio=4, cmp_topk=64),
    "mtp_q2": dict(q_n=32, q_lens=[2, 1, 2], kv_lens=[900, 40, 2500], mode="csa", cmp_ratio=4, cmp_topk=64,
                   seqused_q=[2, 1, 2]),
    # more than 64 rows
    "swa_decode_100": dict(q_n=16, q_lens=[1] * 100, kv_lens=[50 + 37 * b for b in range(100)], layout_kv="PAGED",
                           mode="swa", ori_mask_mode=3, win_left=-1, win_right=-1),
    "prefill_tnd": dict(q_n=64, q_lens=[70, 130, 33], kv_lens=[200, 900, 33], layout_q="TND", layout_kv="TND",
                        mode="csa", cmp_ratio=4, cmp_topk=32),
}


@pytest.mark.parametrize("name", list(CASES))
def test_plan_words(name):
    kw = dict(CASES[name])
    q_n = kw.pop("q_n")
    prob = S.build(name, seed=71, device="cuda", q_n=q_n, **kw)
    r = _sfm.Runner(prob)
    r.plan()
    torch.cuda.synchronize()
    W, G = check_plan(prob, r.meta, q_n)
    assert G >= 1


def _occupancy_split(T, q_n, mp, G, S_inv):
    """The occupancy policy's chunk size, written out: keep the batch-invariant
    cut when its units already reach G; otherwise take the k (chunks per row)
    that minimises 2 waves (max(tiles per chunk, 3) + 1), plus 2 + k when a
    row is split, the smallest k on ties."""
    hg = (q_n + 63) // 64
    ms = -(-mp // S_inv)
    if T * hg * ms >= G:
        return S_inv
    tiles = -(-mp // 32)
    def cost(k):
        return 2 * -(-(T * hg * k) // G) * (max(-(-tiles // k), 3) + 1) + (2 + k if k > 1 else 0)
    best = min(range(ms, min(tiles, G) + 1), key=lambda k: (cost(k), k))
    return S_inv if best == ms else 32 * -(-tiles // best)


def _max_positions(p):
    """Upper bound of a row's attended positions from the params alone."""
    if p.ori_topk > 0:
        ori = p.ori_topk * max(1, p.sparse_block_size)
    else:
        ori = p.max_seqlen_ori_kv
        if p.ori_mask_mode == 4 and p.ori_win_left >= 0 and p.ori_win_right >= 0:
            ori = min(ori, p.ori_win_left + p.ori_win_right + 1)
    cmp = (p.cmp_topk if p.cmp_topk > 0 else p.max_seqlen_cmp_kv) if p.has_cmp_kv else 0
    return ori + cmp


OCC_CASES = ["csa_decode_32", "hca_decode_8_heads128", "mtp_q2", "swa_empty_rows", "causal_many_splits",
             "prefill_tnd"]


@pytest.mark.parametrize("name", OCC_CASES)
def test_plan_words_occupancy_policy(name):
    """The occupancy policy's plan: the same plan words for its chunk size,
    the chunk size the policy's cost model picks, and never fewer work units
    than the batch-invariant plan."""
    kw = dict(CASES[name])
    q_n = kw.pop("q_n")
    prob = S.build(name, seed=71, device="cuda", q_n=q_n, **kw)
    inv = _sfm.Runner(prob)
    inv.plan()
    occ = _sfm.Runner(prob, _sfm.params_of(prob, split_policy=sfm.SPLIT_OCCUPANCY))
    occ.plan()
    torch.cuda.synchronize()
    W_inv, G = check_plan(prob, inv.meta, q_n)
    W_occ, _ = check_plan(prob, occ.meta, q_n)
    S_inv, S_occ = int(inv.meta[4]), int(occ.meta[4])
    mp = _max_positions(occ.params)
    assert S_occ == _occupancy_split(prob.num_tokens, q_n, mp, G, S_inv), (S_inv, S_occ)
    assert W_occ >= W_inv
