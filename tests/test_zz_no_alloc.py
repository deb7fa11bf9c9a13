"""sfm_forward_noalloc: the attention entry point for callers that cannot
allocate device memory (a captured graph replayed with frozen memory, a
plug-in whose host framework owns all allocations, a path that must not
allocate).  It takes its split-KV scratch from a fixed device array inside
the library instead of a caller workspace.

Checked through the C-ABI against sfm_forward with a caller-allocated
workspace, within the parity tolerance and bit for bit (both run the same
deterministic kernels), on two calls in a row (the second call reuses the
array the first one left behind).  This file is collected
last so that a run stopping at the first failure has run everything else.
"""
import numpy as np
import pytest
import torch

import sfm_inputs as S
import sparse_shared_kv_gb300 as sfm
from tests import _sfm

pytestmark = pytest.mark.gpu

ATOL = 2e-2
RTOL = 2e-2


def _close(a, b):
    a = a.float().cpu().numpy()
    b = b.float().cpu().numpy()
    return np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b))


def test_noalloc_matches_forward_twice():
    sfm.build()
    prob = S.csa_decode(device="cuda", batch=6, seed=31)
    r = _sfm.Runner(prob)
    need = sfm.sfm_workspace_size(r.params)
    assert 0 < need <= sfm.NOALLOC_WORKSPACE_BYTES      # the case really uses scratch
    ref_out, ref_lse, st = r.run()
    assert st == 0
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        sfm.sfm_forward_noalloc(r.params, r.tensors, r.meta, prob.softmax_scale, out, lse, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, (call, hex(int(status.item())))
        assert _close(out, ref_out), call
        assert _close(lse, ref_lse), call
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), call


def test_noalloc_rejects_oversized_workspace():
    sfm.build()
    # 128 heads, causal rows of up to 131072 positions (dozens of splits per
    # row): the split-KV partials need more than the fixed array
    p = sfm.make_params(num_heads_q=128, batch_size=256, max_seqlen_q=1, max_seqlen_ori_kv=131072,
                        max_seqlen_cmp_kv=1024, cmp_ratio=128, ori_mask_mode=3, cmp_mask_mode=3,
                        ori_win_left=-1, ori_win_right=-1, layout_q="BSND", layout_kv="PAGED", has_cmp_kv=1,
                        ori_block_size=128, cmp_block_size=128, return_lse=1)
    assert sfm.sfm_workspace_size(p) > sfm.NOALLOC_WORKSPACE_BYTES
    out = torch.empty(1, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sfm.SfmError) as e:
        sfm.sfm_forward_noalloc(p, sfm.SfmTensors(), torch.empty(1, dtype=torch.int32, device="cuda"), 1.0, out, None)
    assert e.value.code == 4   # SFM_ERR_WORKSPACE
