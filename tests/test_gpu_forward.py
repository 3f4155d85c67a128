"""GPU block-sparse attention forward vs the fp64 oracle.

Small problems are compared on every row; the full-size workloads on a
seeded sample of query blocks (the first and last block and random blocks of
head 0 and the last head)."""
import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import oracle
import synth
from gpu_util import DEV, compare, cuda, gpu_index, run_forward, sample_rows, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    bsa.device_status()


def _mask_problem(seed, H, N, D, density, empty_rows=0):
    p = synth.tiny(seed=seed, H=H, N=N, D=D, density=density)
    if empty_rows:
        p.mask[:empty_rows] = 0
    return p


@pytest.mark.parametrize("D", [64, 128])
def test_tiny_config_all_rows(D):
    prob = synth.tiny(seed=1, D=D)  # B1 H2 N2048, Bernoulli(0.25) + diagonal
    idx, cnt, _ = gpu_index(prob)
    o, lse = run_forward(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt)


@pytest.mark.parametrize("D", [64, 128])
def test_dense_mask_equals_all_blocks(D):
    prob = _mask_problem(3, 2, 1024, D, 1.0)
    idx, cnt, _ = gpu_index(prob)
    o, lse = run_forward(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt)


def test_single_block_sequence():
    prob = _mask_problem(4, 3, 128, 128, 1.0)
    idx, cnt, _ = gpu_index(prob)
    o, lse = run_forward(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt)


def test_ragged_lists_empty_rows_and_short_capacity():
    """Counts from 0 to nKB, a capacity below nKB (short lists only), empty rows."""
    prob = _mask_problem(5, 2, 3072, 128, 0.2, empty_rows=3)
    nkb = prob.nqb
    g = np.random.default_rng(0)
    prob.mask[5] = 1
    prob.mask[6, : nkb // 2] = 1
    idx, cnt, _ = gpu_index(prob)
    o, lse = run_forward(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt)
    # capacity smaller than nKB with lists that fit
    prob.mask[5] = 0
    prob.mask[6] = 0
    prob.mask[:, :] &= (g.random(prob.mask.shape) < 0.5).astype(np.uint8)
    cap = int(prob.mask.astype(bool).sum(1).max())
    idx, cnt, _ = gpu_index(prob, max_kv=max(cap, 1))
    o, lse = run_forward(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt)


def test_log_weights():
    prob = _mask_problem(6, 2, 2048, 128, 0.3)
    idx, cnt, _ = gpu_index(prob)
    g = np.random.default_rng(1)
    lw = cuda(g.uniform(-3, 3, idx.shape).astype(np.float32))
    o, lse = run_forward(prob, idx, cnt, lw=lw)
    status_ok()
    compare(prob, o, lse, idx, cnt, lw=lw)


@pytest.mark.parametrize("D", [64, 128])
def test_gather_and_scatter_maps(D):
    prob = _mask_problem(7, 2, 2048, D, 0.3)
    g = np.random.default_rng(2)
    prob.q_map = np.stack([g.permutation(prob.N) for _ in range(2)]).astype(np.int32)
    prob.kv_map = np.stack([g.permutation(prob.N) for _ in range(2)]).astype(np.int32)
    idx, cnt, _ = gpu_index(prob)
    o, lse = run_forward(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt)


def test_query_map_only_and_key_map_only():
    prob = _mask_problem(8, 1, 1024, 128, 0.5)
    g = np.random.default_rng(3)
    perm = g.permutation(prob.N).astype(np.int32)[None]
    idx, cnt, _ = gpu_index(prob)
    for qm, km in ((perm, None), (None, perm)):
        prob.q_map, prob.kv_map = qm, km
        o, lse = run_forward(prob, idx, cnt)
        status_ok()
        compare(prob, o, lse, idx, cnt)


def test_row_order_changes_nothing():
    """Any execution order (row_perm) gives bit-identical O and LSE."""
    prob = _mask_problem(9, 3, 4096, 128, 0.25)
    idx, cnt, _ = gpu_index(prob)
    o0, l0 = run_forward(prob, idx, cnt)
    g = np.random.default_rng(4)
    perm = cuda(np.stack([g.permutation(prob.nqb) for _ in range(3)]).astype(np.int32))
    o1, l1 = run_forward(prob, idx, cnt, row_perm=perm)
    wave = bsa.resident_ctas(128)
    rp = torch.empty((3, prob.nqb), dtype=torch.int32, device=DEV)
    bsa.reorder_rows(cnt.reshape(3, prob.nqb), wave, rp)
    o2, l2 = run_forward(prob, idx, cnt, row_perm=rp)
    status_ok()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert torch.equal(o0, o2) and torch.equal(l0, l2)


def test_bad_entries_are_flagged_not_faulted():
    prob = _mask_problem(10, 1, 1024, 128, 0.5)
    idx, cnt, _ = gpu_index(prob)
    bad = idx.clone()
    bad[0, 0] = 1000            # KV block out of range: skipped, BOUNDS
    o, lse = run_forward(prob, bad, cnt)
    assert bsa.device_status() == 6
    over = cnt.clone()
    over[1] = idx.shape[1] + 5  # count above capacity: clamped, OVERFLOW
    o, lse = run_forward(prob, idx, over)
    assert bsa.device_status() == 3
    status_ok()


# ------------------------------------------------------------------ full-size workloads
def test_threshold_config_full_size_sampled_rows():
    prob = synth.threshold(seed=2)  # H12 N32768 D128, p = 0.15
    idx, cnt, _ = gpu_index(prob)
    o, lse = run_forward(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt, sel=sample_rows(prob, 3))


@pytest.mark.parametrize("layer", ["scatter", "gather"])
def test_scatter_gather_config_full_size(layer):
    prob = synth.scatter(seed=3, layer=layer)  # H24 N16384 D128, one block per query block
    idx, cnt, _ = gpu_index(prob)
    o, lse = run_forward(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt, sel=sample_rows(prob, 6))


def test_sampled_config_full_size():
    prob = synth.sampled(seed=4)  # H40 N75776: top-16 exact + 8 PPS-sampled, random perms
    idx, cnt, lw = gpu_index(prob)
    assert int(cnt.min()) == 24 and int(cnt.max()) == 24
    o, lse = run_forward(prob, idx, cnt, lw=lw)
    status_ok()
    compare(prob, o, lse, idx, cnt, lw=lw, sel=sample_rows(prob, 3))


def test_dynamic_config_full_size_reordered_equals_identity():
    prob = synth.dynamic(seed=5)  # H24 N118784, per-row top-k of cluster-structured scores
    idx, cnt, _ = gpu_index(prob)
    heads = prob.B * prob.H
    rp = torch.empty((heads, prob.nqb), dtype=torch.int32, device=DEV)
    bsa.reorder_rows(cnt.reshape(heads, prob.nqb), bsa.resident_ctas(128), rp)
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    o1, l1 = run_forward(prob, idx, cnt, row_perm=rp, q=q, k=k, v=v)
    o0, l0 = run_forward(prob, idx, cnt, q=q, k=k, v=v)
    status_ok()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    compare(prob, o1, l1, idx, cnt, sel=sample_rows(prob, 2))
