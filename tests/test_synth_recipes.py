"""The seeded workloads have the structure the input recipe states (no GPU):
densities, per-row block counts, the dynamic workload's clusters, the Scatter
map, and bit-identical regeneration from a seed."""
import numpy as np
import torch

import oracle
import synth


def test_threshold_density_and_band():
    p = synth.threshold(H=2)
    nb = p.nqb
    keep = p.T <= np.float32(p.p)
    assert abs(keep.mean() - 0.268) < 0.005
    band = synth.frame_band(nb)
    T = p.T.reshape(2, nb, nb)
    assert np.all(T[:, band] == 0.0)   # same / adjacent latent frames always kept


def test_dynamic_density_and_clusters():
    p = synth.dynamic(H=2)
    nb = p.nqb
    assert p.k_per_row.min() >= int(np.ceil(0.10 * nb)) and p.k_per_row.max() <= int(np.floor(0.20 * nb))
    idx, cnt, _ = oracle.index_topk(p.scores, p.k_per_row)
    assert abs(cnt.sum() / (p.rows * nb) - 0.150) < 0.005
    cl = p.extra["clusters"]
    # rows of one cluster share most of their blocks; rows of different clusters few
    rng = np.random.default_rng(0)
    same, diff = [], []
    for _ in range(300):
        a, b = rng.integers(0, nb, 2)
        if a == b:
            continue
        sa, sb = set(idx[a, :cnt[a]].tolist()), set(idx[b, :cnt[b]].tolist())
        j = len(sa & sb) / min(len(sa), len(sb))
        (same if cl[0, a] == cl[0, b] else diff).append(j)
    assert np.mean(same) > 0.8 and np.mean(diff) < 0.3


def test_llm_window_rows_hold_six_or_seven_blocks():
    p = synth.llm_window(H=2, H_kv=1, N=16384)
    cnt = p.mask.reshape(2, p.nqb, p.nqb).sum(2)[0]
    assert set(cnt[8:].tolist()) <= {6, 7}


def test_scatter_map_is_a_permutation_with_stride_R():
    m = synth.scatter_map(16384, 128)
    assert np.array_equal(np.sort(m), np.arange(16384))
    assert np.array_equal(m[:128], np.arange(128) * 128)


def test_same_seed_same_bytes():
    a, b = synth.sampled(H=1), synth.sampled(H=1)
    assert torch.equal(a.q, b.q) and np.array_equal(a.scores, b.scores) and np.array_equal(a.u, b.u)
    assert np.array_equal(a.q_map, b.q_map)
    c = synth.sampled(seed=99, H=1)
    assert not torch.equal(a.q, c.q)
