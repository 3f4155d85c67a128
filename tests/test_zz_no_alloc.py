"""The allocation-free spectral order against the ordinary entry point.

bsa_spectral_order_noalloc is for callers that cannot allocate device memory
while they run (a serving loop or host framework that owns the device memory
pool, or an interface with no room for a workspace buffer).  It takes its
scratch from a fixed array inside the library.  This file is collected last
so that a run stopping at its first failure has already run every other
test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    bsa.device_status()  # clear anything an earlier test left behind
    return bsa.load_library()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _problem(seed):
    """Lists of the dynamic workload (2 heads, 928 query blocks) and a start."""
    prob = synth.dynamic(seed=seed, H=2)
    idx, cnt, _ = oracle.index_topk(prob.scores, prob.k_per_row)
    x0 = synth.spectral_start(seed + 1, 2, prob.nqb).astype(np.float32)
    return (torch.from_numpy(idx).to(DEV), torch.from_numpy(cnt).to(DEV),
            torch.from_numpy(x0).to(DEV), prob.nqb)


def test_noalloc_matches_ordinary_entry_point_twice_in_a_row(lib):
    idx, cnt, x0, nqb = _problem(31)
    heads = 2
    assert bsa.spectral_order_workspace_size(heads, nqb, nqb) <= bsa.NOALLOC_SCRATCH_BYTES
    ref_o = torch.empty((heads, nqb), dtype=torch.int32, device=DEV)
    ref_x = torch.empty((heads, nqb, 2), dtype=torch.float32, device=DEV)
    ref_a = torch.empty((heads, nqb), dtype=torch.float32, device=DEV)
    bsa.spectral_order(idx, cnt, nqb, x0, ref_o, x_out=ref_x, angle=ref_a, iters=10)
    assert bsa.device_status() == 0
    rx, ra = ref_x.cpu().numpy(), ref_a.cpu().numpy()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        order = torch.full((heads, nqb), -1, dtype=torch.int32, device=DEV)
        x_out = torch.full((heads, nqb, 2), float("nan"), dtype=torch.float32, device=DEV)
        angle = torch.full((heads, nqb), float("nan"), dtype=torch.float32, device=DEV)
        code = lib.bsa_spectral_order_noalloc(_ptr(idx), _ptr(cnt), idx.shape[1], heads, nqb, nqb,
                                              10, _ptr(x0), _ptr(x_out), _ptr(angle), _ptr(order),
                                              stream)
        assert code == 0, (call, code)
        assert bsa.device_status() == 0
        o, x, a = order.cpu().numpy(), x_out.cpu().numpy(), angle.cpu().numpy()
        for h in range(heads):
            assert sorted(o[h]) == list(range(nqb))
            # the order sorts this call's own angles, ties to the lower query block
            assert np.array_equal(o[h], np.lexsort((np.arange(nqb), a[h])))
            # same embedding and angles as the ordinary call, within the tolerance
            # the order tests use against the fp64 oracle
            assert np.abs(x[h] - rx[h]).max() <= 2e-3 * np.abs(rx[h]).max()
            assert np.all(np.diff(ra[h][o[h]]) >= -2e-3)


def test_noalloc_allocates_nothing_after_the_first_call(lib):
    """After one zero-size call (the per-device set-up), two full calls leave
    the device's free memory and torch's allocator untouched."""
    idx, cnt, x0, nqb = _problem(37)
    heads = 2
    order = torch.empty((heads, nqb), dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.bsa_spectral_order_noalloc(None, None, 1, 0, nqb, nqb, 10, None, None, None, None,
                                          stream) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for _ in range(2):
        assert lib.bsa_spectral_order_noalloc(_ptr(idx), _ptr(cnt), idx.shape[1], heads, nqb, nqb, 10,
                                              _ptr(x0), None, None, _ptr(order), stream) == 0
    torch.cuda.synchronize()
    assert bsa.device_status() == 0
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0
    for key in ("allocation.all.allocated", "reserved_bytes.all.current", "allocated_bytes.all.current"):
        assert stats1.get(key) == stats0.get(key), key


def test_noalloc_checks_arguments_like_the_ordinary_call(lib):
    """Sizes the ordinary entry point rejects are rejected here too, even with
    heads = 0 (nQB = 1 is below the minimum of 2)."""
    assert lib.bsa_spectral_order_noalloc(None, None, 1, 0, 1, 5, 10, None, None, None, None, None) == 1
    assert lib.bsa_spectral_order(None, None, 1, 0, 1, 5, 10, None, None, ctypes.c_size_t(0), None, None,
                                  None, None) == 1


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    heads, nqb, nkb = 4096, 4096, 4096  # needs far more than the fixed scratch
    assert bsa.spectral_order_workspace_size(heads, nqb, nkb) > bsa.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: rejected before any launch
    code = lib.bsa_spectral_order_noalloc(fake, fake, 8, heads, nqb, nkb, 10, fake, None, None,
                                          fake, None)
    assert code == 2  # BSA_ERR_UNSUPPORTED
