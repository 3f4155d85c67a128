"""The forward kernel with the FMA-pipe exp2 option (BSA_EXP2_POLY=2: two of
every eight exponentials by a polynomial instead of ex2.approx) against the
oracle.  The option is read once per process, so the check runs in a child
process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
import numpy as np, synth
from gpu_util import compare, cuda, gpu_index, run_forward, status_ok
for D in (64, 128):
    prob = synth.tiny(seed=70 + D, H=2, N=2048, D=D, density=0.4)
    idx, cnt, _ = gpu_index(prob)
    lw = cuda(np.random.default_rng(D).normal(0.0, 2.0, idx.shape).astype(np.float32))
    o, lse = run_forward(prob, idx, cnt, lw=lw)
    status_ok()
    print(D, compare(prob, o, lse, idx, cnt, lw=lw))
"""


def test_fma_exp2_option_matches_oracle():
    env = dict(os.environ, BSA_EXP2_POLY="2")
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
