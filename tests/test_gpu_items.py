"""The per-item forward blocks against one block per row, bit for bit.

The launch chooses per-item blocks for the Scatter and Gather 0 layers and
for windowed token masks (short rows); bsa_set_forward_options switches the
choice for the calling thread.  The per-row arithmetic is the same in both
kernels, so the outputs must be identical.  Parity with the oracle is covered
by the Scatter, Gather 0 and masked test files, which run the default choice.
"""
import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import synth

pytestmark = pytest.mark.gpu


def _run(case, schedule):
    bsa.set_forward_options(schedule=schedule)
    try:
        if case == "scatter":
            prob = synth.scatter(H=4)
            rows, nqb = prob.rows, prob.nqb
            idx = torch.from_numpy((np.arange(rows) % nqb).astype(np.int32)[:, None]).cuda()
            cnt = torch.ones(rows, dtype=torch.int32, device="cuda")
            q, k, v = prob.q.cuda(), prob.k.cuda(), prob.v.cuda()
            o = torch.empty_like(q)
            lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
            perm = torch.empty((4, nqb), dtype=torch.int32, device="cuda")
            bsa.reorder_rows(cnt.view(4, -1), 7, perm)
            bsa.forward_scatter(q, k, v, 128, idx, cnt, o, lse, row_perm=perm)
        elif case == "gather0":
            prob = synth.image_gather0(H=3, img_h=64, img_w=48, n_text=256, groups=8)
            q_map, kv_map, idx, cnt, qm = bsa.gather0_layout(prob.img_h, prob.img_w, prob.n_text,
                                                             prob.groups, 3)
            q, k, v = prob.q.cuda(), prob.k.cuda(), prob.v.cuda()
            o = torch.empty_like(q)
            lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
            bsa.forward_gather0(q, k, v, prob.img_h, prob.img_w, prob.n_text, prob.groups, idx, cnt, o,
                                lse, quad_mask=qm)
        elif case == "window":
            prob = synth.llm_window(H=8, H_kv=2, N=4096)
            mask = torch.from_numpy(prob.mask).cuda()
            idx = torch.empty((prob.rows, prob.nqb), dtype=torch.int32, device="cuda")
            cnt = torch.empty(prob.rows, dtype=torch.int32, device="cuda")
            bsa.build_index(bsa.IDX_MASK_U8, mask, idx, cnt)
            q, k, v = prob.q.cuda(), prob.k.cuda(), prob.v.cuda()
            o = torch.empty_like(q)
            lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
            bsa.forward_masked(q, k, v, idx, cnt, o, lse, causal=True, window=prob.window,
                               sinks=prob.sinks)
        else:  # the plain tile path (long rows), per-item blocks forced
            prob = synth.threshold(H=2, N=8192)
            T = torch.from_numpy(prob.T).cuda()
            idx = torch.empty((prob.rows, prob.nqb), dtype=torch.int32, device="cuda")
            cnt = torch.empty(prob.rows, dtype=torch.int32, device="cuda")
            bsa.build_index(bsa.IDX_THRESHOLD_F32, T, idx, cnt, p=prob.p)
            q, k, v = prob.q.cuda(), prob.k.cuda(), prob.v.cuda()
            o = torch.empty_like(q)
            lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
            bsa.forward(q, k, v, idx, cnt, o, lse)
        torch.cuda.synchronize()
        assert bsa.device_status() == 0
        return o.view(torch.int16).cpu().numpy(), lse.cpu().numpy()
    finally:
        bsa.set_forward_options()


@pytest.mark.parametrize("case", ["scatter", "gather0", "window", "tile"])
def test_items_match_one_block_per_row(case):
    o1, l1 = _run(case, "per_item")
    o2, l2 = _run(case, "per_row")
    assert np.array_equal(o1, o2)
    assert np.array_equal(l1.view(np.int32), l2.view(np.int32))


def test_items_flag_bad_entries():
    """Per-item blocks meet bad list entries, counts and row-order entries the
    way one block per row does: the status word says which, nothing faults,
    and the next launch runs clean."""
    prob = synth.threshold(H=2, N=8192)
    T = torch.from_numpy(prob.T).cuda()
    idx = torch.empty((prob.rows, prob.nqb), dtype=torch.int32, device="cuda")
    cnt = torch.empty(prob.rows, dtype=torch.int32, device="cuda")
    bsa.build_index(bsa.IDX_THRESHOLD_F32, T, idx, cnt, p=prob.p)
    q, k, v = prob.q.cuda(), prob.k.cuda(), prob.v.cuda()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    bsa.set_forward_options(schedule="per_item")
    try:
        bad = idx.clone()
        bad[5, 0] = prob.nqb + 7                 # a KV block out of range
        bsa.forward(q, k, v, bad, cnt, o, lse)
        torch.cuda.synchronize()
        assert bsa.device_status() == 6          # BSA_ERR_BOUNDS
        over = cnt.clone()
        over[3] = idx.shape[1] + 5               # a count above the list capacity
        bsa.forward(q, k, v, idx, over, o, lse)
        torch.cuda.synchronize()
        assert bsa.device_status() == 3          # BSA_ERR_OVERFLOW
        perm = torch.arange(prob.nqb, dtype=torch.int32, device="cuda").repeat(2, 1)
        perm[1, 4] = prob.nqb                    # a row-order entry out of range
        bsa.forward(q, k, v, idx, cnt, o, lse, row_perm=perm)
        torch.cuda.synchronize()
        assert bsa.device_status() == 6
        bsa.forward(q, k, v, idx, cnt, o, lse)
        torch.cuda.synchronize()
        assert bsa.device_status() == 0
    finally:
        bsa.set_forward_options()
