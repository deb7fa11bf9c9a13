"""GPU parity on seeded random configurations (every mode, layout pair, mask
mode, dtype, head count, packed format and block-wise selection size the
parameter rules allow): the attention kernel through the C-ABI against the
oracle, element by element, and its resolved rows exactly, under the
batch-invariant split policy and under the occupancy policy (which re-cuts
these small batches into more splits)."""
import pytest
import torch

import sfm_inputs as S
import sparse_shared_kv_gb300 as sfm
from tests import _sfm
from tests._random_cases import SEEDS, random_case
from tests.test_gpu_parity import assert_parity, assert_sets

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    sfm.build()
    torch.cuda.init()


@pytest.mark.parametrize("policy", ["invariant", "occupancy"])
@pytest.mark.parametrize("seed", SEEDS)
def test_random_case_parity(seed, policy):
    name, q_n, kw = random_case(seed)
    prob = S.build(name, seed=seed, device="cuda", q_n=q_n, **kw)
    host = prob.to("cpu")
    params = _sfm.params_of(prob, split_policy=sfm.SPLIT_OCCUPANCY if policy == "occupancy" else
                            sfm.SPLIT_BATCH_INVARIANT)
    out, lse, status = _sfm.run(prob, params)
    assert status == 0, hex(status)
    assert_parity(prob, out, lse, host=host)
    assert_sets(prob, host=host, out=out, lse=lse, params=params)
