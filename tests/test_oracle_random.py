"""The oracle against the brute-force restatement (dense score matrix over the
explicitly listed attended rows, fp64) on seeded random configurations that
cover every mode, layout pair, mask mode, packed format and block-wise
selection size the parameter rules allow."""
import ctypes as C

import numpy as np
import pytest

import oracle
import sfm_inputs as S
import sparse_shared_kv_gb300 as sfm
from tests import _brute, _sfm
from tests._random_cases import SEEDS, random_case


@pytest.mark.parametrize("seed", SEEDS)
def test_random_case_oracle_matches_brute_force(seed):
    name, q_n, kw = random_case(seed)
    prob = S.build(name, seed=seed, q_n=q_n, **kw)
    # the configuration passes the library's host validation (without a GPU
    # the SM-count query that follows it fails with SFM_ERR_CUDA)
    sfm.build()
    n = C.c_size_t(0)
    assert sfm.lib().sfm_metadata_size(C.byref(_sfm.params_of(prob)), C.byref(n)) in (0, 5)
    O, lse = oracle.forward(prob)
    cache = {}
    for t in range(prob.num_tokens):
        Ob, lb = _brute.dense_reference(prob, t, cache)
        np.testing.assert_allclose(O[t], Ob, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[t], lb, rtol=1e-12, atol=1e-12)
