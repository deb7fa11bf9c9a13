"""Plant plausible mistakes in a copy of the oracle and check the pins catch
every one of them.  Each mutant is compiled from a textual edit of
``oracle/sfm_oracle.c`` into a temporary library; the real oracle is never
modified.  A mutant that passes every pin would mean a part of the oracle is
not pinned."""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sfm_oracle.c")

MUTATIONS = [
    ("query position ignores right-down alignment",
     "o->p = o->kv_len - o->q_len + i;", "o->p = i;"),
    ("window one row short on the left",
     "p - P->win_left > *lo) *lo = p - P->win_left;", "p - P->win_left + 1 > *lo) *lo = p - P->win_left + 1;"),
    ("window right bound dropped",
     "if (P->win_right >= 0 && p + P->win_right < *hi) *hi = p + P->win_right;", ""),
    ("causal mode 3 off by one",
     "if (p < *hi) *hi = p;", "if (p - 1 < *hi) *hi = p - 1;"),
    ("cmp visibility off by one",
     "return (j + 1) * (int64_t)P->cmp_ratio <= (int64_t)ti->p_cmp + 1;",
     "return (j + 1) * (int64_t)P->cmp_ratio <= (int64_t)ti->p_cmp;"),
    ("cmp residual ignored",
     "o->p_cmp = o->cmp_len * P->cmp_ratio + o->residual - o->q_len + i;",
     "o->p_cmp = o->cmp_len * P->cmp_ratio - o->q_len + i;"),
    ("csa keeps out-of-range entries",
     "if (e < 0 || e >= ti->cmp_len || !cmp_visible(P, ti, e)) continue;",
     "if (e < 0 || !cmp_visible(P, ti, e)) { if (e >= ti->cmp_len) e = ti->cmp_len - 1; }"),
    ("sink with the wrong sign",
     "denom += exp((double)P->sinks[h] - m);", "denom += exp(m - (double)P->sinks[h]);"),
    ("sink of head 0 for every head",
     "denom += exp((double)P->sinks[h] - m);", "denom += exp((double)P->sinks[0] - m);"),
    ("LSE includes the sink",
     "lse[task] = m + log(Z);", "lse[task] = m + log(denom);"),
    ("softmax scale dropped",
     "s[a] = acc * P->softmax_scale;", "s[a] = acc;"),
    ("dequant scale tile index wrong",
     "k[d] = (double)(int8_t)r[d] * (double)scale[d / 128];",
     "k[d] = (double)(int8_t)r[d] * (double)scale[d % 4];"),
    ("rope read at the wrong byte offset",
     "memcpy(&h, r + 512 + 2 * j, 2);", "memcpy(&h, r + 512 + j, 2);"),
    ("paged row offset wrong",
     "row = blk * bs + pos % bs;", "row = blk * bs + (pos + 1) % bs;"),
    ("value rows taken from the score tail",
     "for (int d = 0; d < P->d_v; ++d) o[d] += w * k[d];",
     "for (int d = 0; d < P->d_v; ++d) o[d] += w * k[d + P->d_qk - P->d_v];"),
    ("e4m3 exponent bias wrong",
     "else v = ldexp((double)(m + 8), e - 10);", "else v = ldexp((double)(m + 8), e - 9);"),
    ("e4m3 subnormals decoded as normals",
     "if (e == 0) v = ldexp((double)m, -9);", "if (e == 0) v = ldexp((double)(m + 8), -10);"),
    ("fp8 rows decoded as int8",
     "if (P->kv_packed == 2)", "if (P->kv_packed == 3)"),
    ("block-wise selection ignored",
     "const int64_t sbs = P->ori_sbs > 1 ? P->ori_sbs : 1;", "const int64_t sbs = 1;"),
    ("block-wise tokens not masked",
     "if (e >= ti->kv_len || e < lo || e > hi) continue;", "if (e >= ti->kv_len) continue;"),
    ("fp16 exponent bias wrong",
     "else v = ldexp((double)(m + 1024), e - 25);", "else v = ldexp((double)(m + 1024), e - 24);"),
]


def _pin_calls():
    calls = []
    for key in ["swa_bsnd", "hca_bsnd", "csa_tnd", "cp_global", "cp_rank1"]:
        calls.append(lambda key=key: pins.test_page_example_sets(key))
    for name, kw in pins._tiny_cases():
        calls.append(lambda name=name, kw=kw: pins.test_oracle_matches_brute_force(name, kw))
    for s in (False, True):
        calls.append(lambda s=s: pins.test_uniform_attention_closed_form(s))
        calls.append(lambda s=s: pins.test_identical_rows_closed_form(s))
    calls.append(pins.test_dense_causal_matches_sdpa_and_naive_lse)
    calls.append(pins.test_context_parallel_split_invariant)
    calls.append(pins.test_csa_with_all_visible_indices_equals_hca)
    for m in ("swa", "hca", "csa"):
        calls.append(lambda m=m: pins.test_layout_equivalence(m))
    calls.append(pins.test_packed_pow2_scales_equal_plain_rows)
    calls.append(pins.test_e4m3_decoder_matches_library_and_definition)
    calls.append(pins.test_fp8_pow2_scales_are_exact_products)
    calls.append(pins.test_empty_rows_give_zero_and_neg_inf)
    return calls


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(tmp_path, what, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-fopenmp", "-o", str(so), str(mut), "-lm"],
                   check=True, capture_output=True)
    caught = False
    with oracle.use_library(str(so)):
        for call in _pin_calls():
            try:
                call()
            except Exception:
                caught = True
                break
    assert caught, f"no pin caught the planted mistake: {what}"
