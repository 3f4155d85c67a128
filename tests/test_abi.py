"""The C-ABI library: it loads without a GPU, exports every symbol bsa.h
declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

import long_context_mask_gb300 as bsa
from long_context_mask_gb300 import build as bsa_build
from long_context_mask_gb300.binding import EXPORTS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    bsa_build.build()
    return bsa.load_library()


def _declared():
    src = "".join(open(os.path.join(ROOT, "include", h)).read() for h in ("bsa.h", "bsa_selftest.h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(bsa_[a-z_0-9]+)\s*\(", src))


def test_header_declarations_match_binding_exports():
    assert _declared() == set(EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.bsa_status_string(0) == b"BSA_OK"
    assert lib.bsa_status_string(6) == b"BSA_ERR_BOUNDS"
    assert lib.bsa_status_string(99) == b"BSA_ERR_UNKNOWN"


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: the calls below fail validation first
FAKE_ODD = ctypes.c_void_p(0x10002)


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, B=1, H=1, N=256, D=128, kv_idx=FAKE, kv_cnt=FAKE, max_kv=2,
             log_w=None, q_map=None, kv_map=None, row_perm=None, scale=0.0, o=FAKE, lse=FAKE,
             stream=None)
    a.update(kw)
    return lib.bsa_forward(*a.values())


def test_forward_host_validation(lib):
    assert _fwd(lib, D=96) == 2                    # unsupported head dim
    assert _fwd(lib, N=200) == 1                   # not a multiple of 128
    assert _fwd(lib, N=0) == 1
    assert _fwd(lib, max_kv=3) == 1                # > nKB
    assert _fwd(lib, max_kv=0) == 1
    assert _fwd(lib, q=None) == 1                  # null required pointer
    assert _fwd(lib, lse=None) == 1
    assert _fwd(lib, k=FAKE_ODD) == 1              # 16-byte alignment
    assert _fwd(lib, q_map=ctypes.c_void_p(0x10004)) == 1
    assert _fwd(lib, B=70000, H=1) == 1            # grid limits
    assert _fwd(lib, B=1, H=1, N=1 << 25) == 1


def test_index_host_validation(lib):
    f = lib.bsa_build_index
    assert f(7, FAKE, 4, 8, 0.5, None, 1, FAKE, FAKE, 8, None) == 1     # bad mode
    assert f(0, FAKE, 4, 8, 0.5, None, 1, FAKE, FAKE, 9, None) == 1     # max_kv > nKB
    assert f(0, None, 4, 8, 0.5, None, 1, FAKE, FAKE, 8, None) == 1     # null src
    assert f(1, FAKE_ODD, 4, 8, 0.5, None, 1, FAKE, FAKE, 8, None) == 1  # misaligned fp32 src
    assert f(2, FAKE, 4, 8, 0.5, None, -1, FAKE, FAKE, 8, None) == 1    # negative k
    assert f(0, None, 0, 8, 0.5, None, 1, None, None, 8, None) == 0     # empty: nothing to do


def test_reorder_and_sample_host_validation(lib):
    assert lib.bsa_reorder_rows(FAKE, None, 2, 16, 0, FAKE, None) == 1
    assert lib.bsa_reorder_rows(FAKE, None, 2, 16, 9000, FAKE, None) == 1
    assert lib.bsa_reorder_rows(None, None, 2, 16, 4, FAKE, None) == 1
    assert lib.bsa_reorder_rows(None, None, 0, 16, 4, None, None) == 0
    s = lib.bsa_sample_blocks
    assert s(FAKE, 4, 5000, FAKE, FAKE, 1, 2, FAKE, FAKE, FAKE, FAKE, 4, None) == 1  # nKB > 4096
    assert s(FAKE, 4, 16, FAKE, FAKE, 1, -1, FAKE, FAKE, FAKE, FAKE, 4, None) == 1   # m < 0
    assert s(FAKE, 4, 16, FAKE, FAKE, 1, 2, ctypes.c_void_p(0x10004), FAKE, FAKE, FAKE, 4,
             None) == 1                                                           # u not 8-aligned


def test_spectral_order_workspace_and_validation(lib):
    ws = lib.bsa_spectral_order_workspace_size
    assert ws(2, 100, 80) == 2 * (5 * 80 + 2 * 100 + 16) * 4
    assert ws(2, 1, 80) == 0 and ws(2, 9000, 80) == 0
    f = lib.bsa_spectral_order
    assert f(FAKE, FAKE, 8, 2, 100, 80, 10, FAKE, FAKE, 10, None, None, FAKE, None) == 1  # too small
    assert f(FAKE, FAKE, 8, 2, 100, 80, 10, FAKE, None, 1 << 20, None, None, FAKE, None) == 1


def test_gather_rows_host_validation(lib):
    g = lib.bsa_gather_rows
    far = ctypes.c_void_p(0x40000000)
    assert g(FAKE, FAKE, 2, 256, 96, far, None) == 2            # unsupported head dim
    assert g(FAKE, FAKE, 2, 0, 128, far, None) == 1             # N < 1
    assert g(FAKE, FAKE, 70000, 256, 128, far, None) == 1       # heads > 65535
    assert g(FAKE, FAKE, 200, 1 << 24, 128, far, None) == 1     # heads * N >= 2^31
    assert g(None, FAKE, 2, 256, 128, far, None) == 1           # null src
    assert g(FAKE_ODD, FAKE, 2, 256, 128, far, None) == 1       # src not 16-byte aligned
    assert g(FAKE, FAKE, 2, 256, 128, FAKE, None) == 1          # dst overlaps src
    assert g(None, None, 0, 256, 128, None, None) == 0          # empty: nothing to do


def test_forward_masked_host_validation(lib):
    f = lib.bsa_forward_masked

    def call(H=4, H_kv=2, N=256, D=128, causal=1, n_valid=0, window=0, sinks=0, k=FAKE):
        return f(FAKE, k, FAKE, 1, H, H_kv, N, D, FAKE, FAKE, 2, None, None, None, None,
                 causal, n_valid, window, sinks, 0.0, FAKE, FAKE, None)
    assert call(D=96) == 2
    assert call(H_kv=3) == 1           # H not a multiple of H_kv
    assert call(H_kv=0) == 1
    assert call(H_kv=8) == 1           # more key/value heads than query heads
    assert call(causal=2) == 1
    assert call(n_valid=257) == 1      # beyond N
    assert call(n_valid=-1) == 1
    assert call(window=-5) == 1
    assert call(sinks=-1) == 1
    assert call(k=FAKE_ODD) == 1


def test_forward_packed_host_validation(lib):
    f = lib.bsa_forward_packed

    def call(N=256, N_kv=1024, max_kv=2, kv_map=FAKE, causal=0, H_kv=2):
        return f(FAKE, FAKE, FAKE, 1, 4, H_kv, N, 128, FAKE, FAKE, max_kv, None, None, kv_map, N_kv,
                 FAKE, None, causal, 0, 0, 0, 0.0, FAKE, FAKE, None)
    assert call(kv_map=None) == 1      # the packed tiles need a map
    assert call(N_kv=0) == 1
    assert call(N_kv=1000) == 1        # not a multiple of 128
    assert call(N_kv=1 << 27) == 1     # beyond 2^26
    assert call(max_kv=9) == 1         # more entries than packed tiles (8)
    assert call(H_kv=3) == 1
    assert call(causal=2) == 1
    assert call(kv_map=FAKE_ODD) == 1  # kv_map not 16-byte aligned


def test_gather0_sizes_and_layout_validation(lib):
    i32 = ctypes.c_int32
    N, N_kv, mk = i32(0), i32(0), i32(0)

    def sizes(h, w, nt, g):
        return lib.bsa_gather0_sizes(h, w, nt, g, ctypes.byref(N), ctypes.byref(N_kv), ctypes.byref(mk))
    # FLUX.1-dev shapes (INTRA, "Sparse Pattern Index Function", Gather 0):
    # 512 text tokens, 128 x 128 or 64 x 64 image, 8 Scatter groups
    assert sizes(128, 128, 512, 8) == 0
    assert (N.value, N_kv.value, mk.value) == (16896, 512 + 5 * 16384, 4 + 2 * 16)
    assert sizes(64, 64, 512, 8) == 0
    assert (N.value, N_kv.value, mk.value) == (4608, 512 + 5 * 4096, 4 + 2 * 4)
    assert sizes(16, 24, 0, 1) == 0                     # one row of tile pairs: two bands each
    assert (N.value, N_kv.value, mk.value) == (384, 4 * 384, 2)
    assert sizes(48, 16, 256, 2) == 0                   # 128 text queries per group
    assert (N.value, N_kv.value, mk.value) == (1024, 256 + 5 * 768, 2 + 4)  # edge pairs: 4 bands
    assert sizes(24, 16, 0, 1) == 1                     # height not a multiple of 16
    assert sizes(32, 12, 0, 1) == 1                     # width not a multiple of 8
    assert sizes(8, 16, 0, 1) == 1                      # smaller than a window
    assert sizes(32, 32, 100, 1) == 1                   # text not a multiple of 128
    assert sizes(32, 32, 128, 8) == 1                   # 16 text queries per group
    assert sizes(32, 32, 128, 3) == 1
    assert sizes(16, 16, 128, 4) == 1                   # 64 image tokens per group
    lay = lib.bsa_gather0_layout
    assert lay(32, 32, 0, 1, 2, FAKE, FAKE, FAKE, FAKE, FAKE, 3, None) == 1      # max_kv < 4
    assert lay(32, 32, 0, 1, 70000, FAKE, FAKE, FAKE, FAKE, FAKE, 4, None) == 1  # heads > 65535
    assert lay(32, 32, 0, 1, 2, None, FAKE, FAKE, FAKE, FAKE, 4, None) == 1
    assert lay(32, 32, 0, 1, 2, FAKE_ODD, FAKE, FAKE, FAKE, FAKE, 4, None) == 1
    assert lay(32, 32, 0, 1, 0, None, None, None, None, None, 4, None) == 0      # nothing to do


def test_forward_gather0_host_validation(lib):
    f = lib.bsa_forward_gather0

    def call(img_h=32, img_w=32, n_text=128, groups=2, max_kv=9, H_kv=2, D=128, q=FAKE):
        return f(q, FAKE, FAKE, 1, 4, H_kv, D, img_h, img_w, n_text, groups, FAKE, FAKE, FAKE, max_kv,
                 None, 0.0, FAKE, FAKE, None)
    assert call(D=96) == 2
    assert call(img_h=24) == 1          # not a multiple of 16
    assert call(n_text=100) == 1
    assert call(groups=3) == 1
    assert call(max_kv=0) == 1
    assert call(max_kv=42) == 1         # beyond the 41 packed tiles
    assert call(H_kv=3) == 1
    assert call(q=FAKE_ODD) == 1


def test_forward_scatter_host_validation(lib):
    f = lib.bsa_forward_scatter

    def call(N=2048, R=16, max_kv=2, H_kv=2, D=128):
        return f(FAKE, FAKE, FAKE, 1, 4, H_kv, N, D, R, FAKE, FAKE, max_kv, None, None, 0.0, FAKE, FAKE, None)
    assert call(D=96) == 2
    assert call(R=0) == 1
    assert call(R=3) == 1               # does not divide N
    assert call(R=32) == 1              # N / R = 64 is not a multiple of 128
    assert call(N=2000) == 1
    assert call(max_kv=17) == 1         # more entries than blocks
    assert call(H_kv=3) == 1


def test_device_status_rejects_null_output(lib):
    assert lib.bsa_device_status(None, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from long_context_mask_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="libbsa.so not found"):
        binding.load_library()


def test_row_counts_beyond_one_launch_are_rejected(lib):
    """Row counts a single launch cannot cover (grid.x <= 2^31 - 1 blocks of
    8 rows for the list kernels, of 64 rows for the sampler; grid.y <= 65535
    target rows for the upscale) are refused on the host instead of being
    truncated; the calls return before any pointer is touched."""
    grid_x = (1 << 31) - 1
    assert lib.bsa_build_index(0, FAKE, 8 * grid_x + 1, 8, 0.5, None, 1, FAKE, FAKE, 8, None) == 1
    assert lib.bsa_build_index(2, FAKE, 8 * grid_x + 1, 8, 0.5, None, 1, FAKE, FAKE, 8, None) == 1
    assert lib.bsa_build_crm(0, FAKE, 8 * grid_x + 1, 8, 0.5, FAKE, 1, None) == 1
    assert lib.bsa_sample_blocks(FAKE, 64 * grid_x + 1, 16, FAKE, FAKE, 1, 2, FAKE, FAKE, FAKE, FAKE, 4,
                                 None) == 1
    assert lib.bsa_upscale_threshold(FAKE, 1, 4, 4, 65536, 4, FAKE, None) == 1
    assert lib.bsa_upscale_threshold(FAKE, 65536, 4, 4, 4, 4, FAKE, None) == 1


def test_plain_c_client_builds_links_and_runs(lib, tmp_path):
    """The headers compile as C99 and a C program links libbsa.so and calls
    it (only calls that need no GPU)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "client")
    libdir = os.path.dirname(bsa.lib_path())
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_client.c"),
                    "-L", libdir, "-lbsa", "-Wl,-rpath," + libdir, "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    assert out[0] == "BSA_ERR_BOUNDS"
    assert out[1] == "0"
    N, N_kv, max_kv = (int(x) for x in out[2].split())
    assert (N, N_kv) == (512 + 128 * 128, 512 + 5 * 128 * 128) and max_kv > 0
    assert out[3] == "2"  # BSA_ERR_UNSUPPORTED
    assert out[4] == "0"


def test_forward_options_are_checked(lib):
    O = bsa.binding.ForwardOptions
    assert lib.bsa_set_forward_options(ctypes.byref(O(3, 0))) == 1   # no such schedule
    assert lib.bsa_set_forward_options(ctypes.byref(O(0, 1))) == 1   # exp2_fma must be 0 or 2
    assert lib.bsa_set_forward_options(ctypes.byref(O(2, 2))) == 0
    assert lib.bsa_set_forward_options(None) == 0                   # back to the defaults
    with pytest.raises(bsa.BsaError):
        bsa.set_forward_options(exp2_fma=3)
    bsa.set_forward_options()


def test_non_finite_scale_is_rejected(lib):
    for bad in (float("inf"), float("-inf"), float("nan")):
        assert _fwd(lib, scale=bad) == 1
        args = [FAKE, FAKE, 1, 1, 256, 64, None, None, ctypes.c_float(bad), 0, FAKE, ctypes.c_size_t(1 << 20),
                FAKE, None]
        assert lib.bsa_block_scores(*args) == 1


def test_spectral_entry_points_share_their_argument_checks(lib):
    """With heads = 0 and nQB = 1 (below the minimum of 2) both the ordinary
    and the allocation-free spectral order refuse, on the host."""
    assert lib.bsa_spectral_order(None, None, 1, 0, 1, 5, 10, None, None, ctypes.c_size_t(0), None, None,
                                  None, None) == 1
    assert lib.bsa_spectral_order_noalloc(None, None, 1, 0, 1, 5, 10, None, None, None, None, None) == 1
    assert lib.bsa_spectral_order_noalloc(None, None, 6, 0, 4, 5, 10, None, None, None, None, None) == 1  # max_kv > nKB


def test_block_scores_want_16_byte_aligned_tokens(lib):
    args = [FAKE_ODD, FAKE, 1, 1, 256, 64, None, None, ctypes.c_float(0.0), 0, FAKE, ctypes.c_size_t(1 << 20),
            FAKE, None]
    assert lib.bsa_block_scores(*args) == 1
    args[0], args[1] = FAKE, ctypes.c_void_p(0x10008)
    assert lib.bsa_block_scores(*args) == 1
