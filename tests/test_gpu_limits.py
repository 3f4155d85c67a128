"""Size limits of the boundary: the longest sequences and the most heads a
launch allows, the widest sampled row, and long index rows, against the oracle
on sampled rows (index arithmetic and grid limits at their extremes)."""
import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import oracle
import synth
from gpu_util import DEV, compare, cuda, run_forward, status_ok

pytestmark = pytest.mark.gpu


def _lists(rows, nqb, per_row, seed):
    """Ascending distinct KV-block lists: the diagonal, the last block and
    random others."""
    g = np.random.default_rng(seed)
    idx = np.full((rows, per_row), -1, np.int32)
    cnt = np.zeros(rows, np.int32)
    for r in range(rows):
        qb = r % nqb
        s = {qb, nqb - 1} | set(g.choice(nqb, size=per_row - 2, replace=False).tolist())
        s = sorted(s)[:per_row]
        idx[r, :len(s)] = s
        cnt[r] = len(s)
    return idx, cnt


def test_long_sequence_two_million_tokens():
    # 2^21 tokens (16384 blocks) per head: token offsets beyond 2^31 bytes
    B, H, N, D = 1, 2, 1 << 21, 128
    g = synth._gen(41)
    prob = synth.Problem("long", B, H, N, D, *(synth.normal_bf16(g, (B, H, N, D)) for _ in range(3)))
    idx, cnt = _lists(prob.rows, prob.nqb, 4, 41)
    o, lse = run_forward(prob, cuda(idx), cuda(cnt))
    status_ok()
    nqb = prob.nqb
    sel = np.array([0, 1, nqb // 2, nqb - 1, nqb, 2 * nqb - 1], np.int64)
    compare(prob, o, lse, cuda(idx), cuda(cnt), sel=sel)


def test_most_heads_one_block_each():
    # B*H = 65535, the grid limit of one launch
    B, H, N, D = 5, 13107, 128, 64
    g = synth._gen(42)
    prob = synth.Problem("heads", B, H, N, D, *(synth.normal_bf16(g, (B, H, N, D)) for _ in range(3)))
    idx = np.zeros((prob.rows, 1), np.int32)
    cnt = np.ones(prob.rows, np.int32)
    o, lse = run_forward(prob, cuda(idx), cuda(cnt))
    status_ok()
    sel = np.array([0, 1, 17, 40000, prob.rows - 1], np.int64)
    compare(prob, o, lse, cuda(idx), cuda(cnt), sel=sel)


def test_widest_sampled_row():
    # nKB = 4096, the sampler's limit: the drawn set matches the oracle bit for bit
    nkb, rows, m = 4096, 64, 37
    g = np.random.default_rng(43)
    scores = np.maximum(g.random((rows, nkb)).astype(np.float32), np.float32(2.0 ** -24))
    ex_idx = np.sort(g.choice(nkb, size=(rows, 50), replace=True), axis=1).astype(np.int32)
    ex_idx = np.stack([np.unique(r)[:40] for r in ex_idx]).astype(np.int32)
    ex_cnt = np.full(rows, ex_idx.shape[1], np.int32)
    u = g.random(rows)
    cap = ex_idx.shape[1] + m
    idx = torch.empty((rows, cap), dtype=torch.int32, device=DEV)
    cnt = torch.empty(rows, dtype=torch.int32, device=DEV)
    lw = torch.empty((rows, cap), dtype=torch.float32, device=DEV)
    bsa.sample_blocks(cuda(scores), cuda(ex_idx), cuda(ex_cnt), m, cuda(u), idx, cnt, lw)
    status_ok()
    ridx, rcnt, rlw, ov = oracle.sample_blocks(scores, ex_idx, ex_cnt, m, u, cap)
    assert ov == 0
    np.testing.assert_array_equal(cnt.cpu().numpy(), rcnt)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(lw.cpu().numpy(), rlw, rtol=1e-6, atol=0)


def test_long_index_rows():
    # 65536 blocks per row, the index builder's limit (an 8M-token sequence):
    # threshold compaction and top-k
    rows, nkb = 4, 65536
    g = np.random.default_rng(44)
    T = g.random((rows, nkb)).astype(np.float32)
    idx = torch.empty((rows, nkb), dtype=torch.int32, device=DEV)
    cnt = torch.empty(rows, dtype=torch.int32, device=DEV)
    bsa.build_index(bsa.IDX_THRESHOLD_F32, cuda(T), idx, cnt, p=0.3)
    status_ok()
    ridx, rcnt, _ = oracle.index_threshold(T, 0.3)
    np.testing.assert_array_equal(cnt.cpu().numpy(), rcnt)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    k = 777
    tidx = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    tcnt = torch.empty(rows, dtype=torch.int32, device=DEV)
    bsa.build_index(bsa.IDX_TOPK_F32, cuda(T), tidx, tcnt, k_const=k)
    status_ok()
    ridx, rcnt, _ = oracle.index_topk(T, k)
    np.testing.assert_array_equal(tcnt.cpu().numpy(), rcnt)
    np.testing.assert_array_equal(tidx.cpu().numpy(), ridx)
