"""bsa_forward_masked: grouped key/value heads and the token mask (causal,
sliding window + sinks, tail) against the oracle, and bit-identity with
bsa_forward when nothing is masked.

Causal rows near the start of the sequence see only a few keys, so their O
is close to single value rows and the bf16 rounding of P and O is not
averaged away: O is held to the bound of gpu_util.few_key_o_bound (mean
relative error and LSE keep the usual bar)."""
import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import synth
from gpu_util import DEV, compare, cuda, few_key_o_bound, gpu_index, sample_rows, status_ok

pytestmark = pytest.mark.gpu


def run_masked(prob, idx, cnt, lw=None, **over):
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    kw = dict(causal=prob.causal, n_valid=prob.n_valid, window=prob.window, sinks=prob.sinks)
    kw.update(over)
    bsa.forward_masked(q, k, v, idx, cnt, o, lse, log_w=lw, q_map=cuda(prob.q_map),
                       kv_map=cuda(prob.kv_map), **kw)
    return o, lse, kw


@pytest.mark.parametrize("D", [64, 128])
def test_causal_block_layer_grouped_heads(D):
    prob = synth.llm(seed=31, H=4, H_kv=2, N=2048, D=D)
    idx, cnt, _ = gpu_index(prob)
    o, lse, kw = run_masked(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt, o_max_abs=few_key_o_bound(prob.v), **kw)


def test_sliding_window_with_sinks():
    prob = synth.llm_window(seed=32, H=4, H_kv=1, N=2048, window=300, sinks=64)
    idx, cnt, _ = gpu_index(prob)
    o, lse, kw = run_masked(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt, o_max_abs=few_key_o_bound(prob.v), **kw)


def test_causal_through_maps_with_log_weights():
    prob = synth.llm(seed=33, H=4, H_kv=2, N=2048)
    g = np.random.default_rng(33)
    prob.q_map = np.stack([g.permutation(prob.N) for _ in range(4)]).astype(np.int32)
    prob.kv_map = np.stack([g.permutation(prob.N) for _ in range(2)]).astype(np.int32)
    prob.mask[:] = 1  # every block listed: the mask decides, on original tokens
    idx, cnt, _ = gpu_index(prob)
    lw = cuda(g.uniform(-2, 2, idx.shape).astype(np.float32))
    o, lse, kw = run_masked(prob, idx, cnt, lw=lw)
    status_ok()
    compare(prob, o, lse, idx, cnt, lw=lw, o_max_abs=few_key_o_bound(prob.v), **kw)


def test_tail_padding_without_causal():
    prob = synth.tiny(seed=34, H=2, N=2048, D=128, density=0.4)
    prob.n_valid = 1900
    idx, cnt, _ = gpu_index(prob)
    o, lse, kw = run_masked(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt, **kw)


def test_fully_masked_rows_are_empty():
    prob = synth.llm(seed=35, H=2, H_kv=2, N=1024)
    m = prob.mask.reshape(2, 8, 8)
    m[0, 2] = 0
    m[0, 2, 5] = 1  # query block 2 lists only a later block: every key dropped
    idx, cnt, _ = gpu_index(prob)
    o, lse, kw = run_masked(prob, idx, cnt)
    status_ok()
    rows = slice(2 * 128, 3 * 128)
    assert torch.all(torch.isneginf(lse[0, 0, rows])) and not torch.any(o[0, 0, rows].float())
    compare(prob, o, lse, idx, cnt, o_max_abs=few_key_o_bound(prob.v), **kw)


def test_no_mask_is_bit_identical_to_forward():
    prob = synth.tiny(seed=36, H=4, N=2048, D=128, density=0.3)
    idx, cnt, _ = gpu_index(prob)
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    o1, l1 = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    bsa.forward(q, k, v, idx, cnt, o1, l1)
    o2, l2, _ = run_masked(prob, idx, cnt, causal=False, n_valid=0, window=0, sinks=0)
    o3, l3 = torch.empty_like(q), torch.empty_like(l1)  # the masked kernel, nothing dropped
    bsa.forward_masked(q, k, v, idx, cnt, o3, l3, n_valid=prob.N - 1)
    status_ok()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    # grouped heads = forward on K/V repeated per query head
    kg, vg = k[:, ::2].contiguous(), v[:, ::2].contiguous()
    o4, l4 = torch.empty_like(q), torch.empty_like(l1)
    bsa.forward_masked(q, kg, vg, idx, cnt, o4, l4)
    o5, l5 = torch.empty_like(q), torch.empty_like(l1)
    bsa.forward(q, kg.repeat_interleave(2, 1), vg.repeat_interleave(2, 1), idx, cnt, o5, l5)
    status_ok()
    assert torch.equal(o4.view(torch.int16), o5.view(torch.int16)) and torch.equal(l4, l5)
    # n_valid = N - 1 drops one key: rows that list the last block differ, compare to the oracle
    compare(prob, o3, l3, idx, cnt, n_valid=prob.N - 1)


@pytest.mark.parametrize("cfg", [7, 8])
def test_llm_configs_full_size_sampled_rows(cfg):
    prob = synth.CONFIGS[cfg]()
    idx, cnt, _ = gpu_index(prob)
    o, lse, kw = run_masked(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt, sel=sample_rows(prob, 3), o_max_abs=few_key_o_bound(prob.v), **kw)
