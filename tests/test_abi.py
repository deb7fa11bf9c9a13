"""CPU checks of the C-ABI library: it builds for sm_103a, loads, exports every
entry point ``include/sfm.h`` declares, and rejects bad scalar attributes on
the host (no compute call: validation runs before any device query)."""
import ctypes as C
import os
import re

import pytest

import sparse_shared_kv_gb300 as sfm

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "sfm.h")


@pytest.fixture(scope="module")
def lib():
    sfm.build()
    return sfm.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sfm_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert set(names) == set(sfm.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sfm.sfm_abi_version() == 4


def test_error_strings(lib):
    for code in range(6):
        assert sfm.sfm_error_string(code)
    assert sfm.sfm_error_string(99) == "unknown error"


def _p(**kw):
    base = dict(num_heads_q=64, batch_size=2, max_seqlen_q=1, max_seqlen_ori_kv=1024, ori_mask_mode=4,
                ori_win_left=127, ori_win_right=0, cmp_mask_mode=0, has_cmp_kv=0, cmp_ratio=1)
    base.update(kw)
    return sfm.make_params(**base)


BAD = [
    ("q_n zero", dict(num_heads_q=0), 1),
    ("q_n above 128", dict(num_heads_q=129), 1),
    ("kv_n 2", dict(num_heads_kv=2), 2),
    ("d 256", dict(head_dim=256), 2),
    ("plain rows with rope", dict(rope_head_dim=64), 1),
    ("packed rope 32", dict(kv_format=sfm.KV_INT8_PACKED, rope_head_dim=32), 1),
    ("BSND q with TND kv", dict(layout_q=sfm.BSND, layout_kv=sfm.TND), 3),
    ("paged block 20", dict(layout_kv=sfm.PAGED, ori_block_size=20), 3),
    ("paged block 2048", dict(layout_kv=sfm.PAGED, ori_block_size=2048), 3),
    ("no ori_kv", dict(has_ori_kv=0), 2),
    ("mask mode 2", dict(ori_mask_mode=2), 1),
    ("cmp mask mode 4", dict(cmp_mask_mode=4), 1),
    ("window -2", dict(ori_win_left=-2), 1),
    ("SWA with cmp_topk", dict(cmp_topk=512), 1),
    ("SWA with cmp_ratio 4", dict(cmp_ratio=4), 1),
    ("CSA ratio 0", dict(has_cmp_kv=1, cmp_ratio=0, cmp_topk=512, cmp_mask_mode=3), 1),
    ("TND without total_q", dict(layout_q=sfm.TND, layout_kv=sfm.TND, total_q=0), 1),
    ("dtype 7", dict(dtype=7), 1),
    ("return_lse 2", dict(return_lse=2), 1),
    ("fp8 packed rope 32", dict(kv_format=sfm.KV_FP8_PACKED, rope_head_dim=32), 1),
    ("kv format 3", dict(kv_format=3), 1),
    ("block-wise without ori_topk", dict(sparse_block_size=4), 1),
    ("block-wise 3", dict(ori_topk=64, ori_mask_mode=3, sparse_block_size=3), 1),
    ("block-wise 256", dict(ori_topk=64, ori_mask_mode=3, sparse_block_size=256), 1),
    ("block-wise not dividing the page", dict(ori_topk=64, ori_mask_mode=3, sparse_block_size=32,
                                              layout_kv=sfm.PAGED, ori_block_size=16), 3),
    ("kernel hint 3", dict(kernel_hint=3), 1),
    ("kernel hint 1 (retired CUDA-core kernel)", dict(kernel_hint=1), 2),
    ("kernel hint -1", dict(kernel_hint=-1), 1),
    ("split policy 2", dict(split_policy=2), 1),
    ("split policy -1", dict(split_policy=-1), 1),
    ("window right -2", dict(ori_win_right=-2), 1),
    ("paged cmp block 8", dict(layout_kv=sfm.PAGED, ori_block_size=128, has_cmp_kv=1, cmp_ratio=4, cmp_topk=64,
                               cmp_mask_mode=3, cmp_block_size=8), 3),
]


@pytest.mark.parametrize("what,kw,code", BAD, ids=[b[0] for b in BAD])
def test_host_rejects_bad_attributes(lib, what, kw, code):
    p = _p(**kw)
    n = C.c_size_t(0)
    assert lib.sfm_metadata_size(C.byref(p), C.byref(n)) == code
    assert lib.sfm_workspace_size(C.byref(p), C.byref(n)) == code


def test_valid_attributes_reach_the_device_query(lib):
    """Valid params pass validation; without a GPU the SM-count query then
    fails with SFM_ERR_CUDA (on a GPU machine it succeeds)."""
    import torch
    p = _p()
    n = C.c_size_t(0)
    rc = lib.sfm_metadata_size(C.byref(p), C.byref(n))
    if torch.cuda.is_available():
        assert rc == 0 and n.value >= 1024
    else:
        assert rc == 5


def test_null_params_rejected(lib):
    n = C.c_size_t(0)
    assert lib.sfm_metadata_size(None, C.byref(n)) == 1
    assert lib.sfm_forward(None, None, None, 0, C.c_float(1.0), None, None, None, 0, None, None) == 1
