"""The forward kernel with the FMA-pipe exp2 option (bsa_set_forward_options
exp2_fma = 2: two of every eight exponentials by a polynomial instead of
ex2.approx) against the oracle."""
import numpy as np
import pytest

import long_context_mask_gb300 as bsa
import synth
from gpu_util import compare, cuda, gpu_index, run_forward, status_ok

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
def test_fma_exp2_option_matches_oracle(D):
    prob = synth.tiny(seed=70 + D, H=2, N=2048, D=D, density=0.4)
    idx, cnt, _ = gpu_index(prob)
    lw = cuda(np.random.default_rng(D).normal(0.0, 2.0, idx.shape).astype(np.float32))
    bsa.set_forward_options(exp2_fma=2)
    try:
        o, lse = run_forward(prob, idx, cnt, lw=lw)
        status_ok()
    finally:
        bsa.set_forward_options()
    compare(prob, o, lse, idx, cnt, lw=lw)
