"""Shared helpers for the GPU parity tests (test infrastructure)."""
from __future__ import annotations

import numpy as np
import torch

import long_context_mask_gb300 as bsa
import oracle

# Float tolerances of the parity bar: O max-abs and mean-relative error,
# LSE max-abs (finite entries; -inf must match exactly).
O_MAX_ABS = 1e-2
O_MEAN_REL = 5e-3
LSE_MAX_ABS = 1e-3

DEV = "cuda"


def cuda(x, dtype=None):
    if x is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(x)) if isinstance(x, np.ndarray) else x
    if dtype is not None:
        t = t.to(dtype)
    return t.to(DEV).contiguous()


def gpu_index(prob, max_kv=None):
    """Index lists for a synthetic problem on the GPU (returns device tensors)."""
    rows, nqb = prob.rows, prob.nqb
    if prob.diag_list:
        idx = torch.from_numpy((np.arange(rows) % nqb).astype(np.int32)[:, None]).to(DEV)
        cnt = torch.ones(rows, dtype=torch.int32, device=DEV)
        return idx, cnt, None
    if prob.mask is not None:
        src, mode = cuda(prob.mask), bsa.IDX_MASK_U8
    elif prob.T is not None:
        src, mode = cuda(prob.T), bsa.IDX_THRESHOLD_F32
    else:
        src, mode = cuda(prob.scores), bsa.IDX_TOPK_F32
    nkb = src.shape[1]
    if max_kv is None:
        if mode == bsa.IDX_TOPK_F32:
            max_kv = int(prob.k_const if prob.k_per_row is None else prob.k_per_row.max())
        else:
            max_kv = nkb
    kpr = cuda(prob.k_per_row) if prob.k_per_row is not None else None
    kk = prob.k_const or 0
    if prob.m_sample:
        ex_idx = torch.empty((rows, max_kv), dtype=torch.int32, device=DEV)
        ex_cnt = torch.empty(rows, dtype=torch.int32, device=DEV)
        bsa.build_index(mode, src, ex_idx, ex_cnt, k_per_row=kpr, k_const=kk)
        cap = max_kv + prob.m_sample
        idx = torch.empty((rows, cap), dtype=torch.int32, device=DEV)
        cnt = torch.empty(rows, dtype=torch.int32, device=DEV)
        lw = torch.empty((rows, cap), dtype=torch.float32, device=DEV)
        bsa.sample_blocks(src, ex_idx, ex_cnt, prob.m_sample, cuda(prob.u), idx, cnt, lw)
        return idx, cnt, lw
    idx = torch.empty((rows, max_kv), dtype=torch.int32, device=DEV)
    cnt = torch.empty(rows, dtype=torch.int32, device=DEV)
    bsa.build_index(mode, src, idx, cnt, p=prob.p or 0.0, k_per_row=kpr, k_const=kk)
    return idx, cnt, None


def run_forward(prob, idx, cnt, lw=None, row_perm=None, q=None, k=None, v=None):
    q = cuda(prob.q) if q is None else q
    k = cuda(prob.k) if k is None else k
    v = cuda(prob.v) if v is None else v
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    bsa.forward(q, k, v, idx, cnt, o, lse, log_w=lw, q_map=cuda(prob.q_map),
                kv_map=cuda(prob.kv_map), row_perm=row_perm)
    return o, lse


def few_key_o_bound(v):
    """Max-abs O bound for rows that see only a few keys (token masks).

    P is rounded to bf16 before PV (relative error <= 2^-8 per weight) and O
    is rounded to bf16 (<= 2^-8 |O|), so |O_gpu - O| <= 2^-8 (|O| + max_j
    |v_j - O|) <= 3 * 2^-8 * max|v|.  A row averaging hundreds of keys stays
    far below it; a row that sees two keys can reach a sizeable part of it."""
    return 3 * 2.0 ** -8 * float(torch.as_tensor(v).float().abs().max())


def compare(prob, o, lse, idx, cnt, lw=None, sel=None, o_max_abs=O_MAX_ABS, **mask):
    """Check GPU O / LSE against the oracle on the query blocks `sel` (all when None).
    ``mask`` (causal, n_valid, window, sinks) goes to the oracle unchanged.

    Returns (max-abs O, mean-rel O, max-abs LSE)."""
    idx_h = idx.cpu().numpy()
    cnt_h = cnt.cpu().numpy()
    lw_h = None if lw is None else lw.cpu().numpy()
    O, L, tok = oracle.attention(prob.q, prob.k, prob.v, idx_h, cnt_h, log_w=lw_h,
                                 q_map=prob.q_map, kv_map=prob.kv_map, sel=sel, **mask)
    nqb = prob.nqb
    sel_arr = np.arange(prob.rows) if sel is None else np.asarray(sel)
    bh = np.repeat(sel_arr // nqb, 128)
    flat = bh * prob.N + tok
    og = o.reshape(-1, prob.D)[torch.from_numpy(flat).to(o.device)].float().cpu().numpy()
    lg = lse.reshape(-1)[torch.from_numpy(flat).to(o.device)].cpu().numpy().astype(np.float64)
    diff = np.abs(og - O)
    max_abs = float(diff.max()) if diff.size else 0.0
    denom = float(np.abs(O).sum())
    mean_rel = float(diff.sum() / denom) if denom > 0 else float(diff.sum())
    fin = np.isfinite(L)
    assert np.array_equal(np.isneginf(lg), np.isneginf(L)), "-inf LSE rows differ"
    lse_abs = float(np.abs(lg[fin] - L[fin]).max()) if fin.any() else 0.0
    assert max_abs <= o_max_abs, f"O max-abs {max_abs} > {o_max_abs}"
    assert mean_rel <= O_MEAN_REL, f"O mean-rel {mean_rel}"
    assert lse_abs <= LSE_MAX_ABS, f"LSE max-abs {lse_abs}"
    return max_abs, mean_rel, lse_abs


def sample_rows(prob, n_per_head=3, heads=None, seed=0):
    """A seeded subset of query blocks: the first, last and random blocks of the
    chosen heads (head 0 and the last head by default)."""
    g = np.random.default_rng(seed)
    nqb = prob.nqb
    BH = prob.B * prob.H
    heads = [0, BH - 1] if heads is None else heads
    out = []
    for h in heads:
        blocks = {0, nqb - 1} | set(g.choice(nqb, size=min(n_per_head, nqb), replace=False).tolist())
        out += [h * nqb + b for b in sorted(blocks)]
    return np.array(out, np.int64)


def status_ok():
    st = bsa.device_status()
    assert st == 0, f"device status {st}"
