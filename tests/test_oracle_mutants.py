"""Planted mistakes in the oracle are caught by its pins (no GPU).

Each mutant is one plausible slip in ``oracle/bsa_oracle.c``: a flipped
comparison, a dropped term, a wrong index or a transposed operand.  It is
compiled into a scratch library, and the pins that should notice it run
against that library in a child process.  The child must fail an
assertion.  The unaltered source, built and run the same way, passes the
same pins.  The mistakes are planted in the oracle on the CPU and nowhere
else.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
O = "tests/test_oracle.py::"
G = "tests/test_oracle_gather0.py::"

# (name, original text, planted text, pins that must catch it)
MUTANTS = [
    ("threshold exclusive", "keep[kb] = T[r * nKB + kb] <= p;", "keep[kb] = T[r * nKB + kb] < p;",
     [O + "test_threshold_is_inclusive_and_compared_in_fp32"]),
    ("top-k ties to the higher block", "return (x->kb > y->kb) - (x->kb < y->kb);",
     "return (x->kb < y->kb) - (x->kb > y->kb);",
     [O + "test_topk_matches_rank_counting_brute_force_with_ties"]),
    ("reorder ascending", "while (j >= b0 && cnt[ord[j]] < cnt[q])", "while (j >= b0 && cnt[ord[j]] > cnt[q])",
     [O + "test_reorder_hand_worked_example"]),
    ("reorder unstable ties", "while (j >= b0 && cnt[ord[j]] < cnt[q])",
     "while (j >= b0 && cnt[ord[j]] <= cnt[q])", [O + "test_reorder_hand_worked_example"]),
    ("sampler interval closed on the right", "ceilf(C - ur) > ceilf(C_prev - ur)",
     "floorf(C - ur) > floorf(C_prev - ur)", [O + "test_sampler_hand_worked_draws"]),
    ("sampler lambda not renormalised after capping", "lambda = (float)(m - n_cap) / sum;",
     "lambda = (float)m / sum;", [O + "test_sampler_hand_worked_draws"]),
    ("sampler weight sign", "(float)(-log((double)pi[kb]))", "(float)(log((double)pi[kb]))",
     [O + "test_sample_size_inclusion_probabilities_and_promotion"]),
    ("attention scale 1/D", "if (scale <= 0.0) scale = 1.0 / sqrt((double)D);\n    if (n_valid <= 0)",
     "if (scale <= 0.0) scale = 1.0 / (double)D;\n    if (n_valid <= 0)",
     [O + "test_all_ones_mask_is_dense_softmax_attention"]),
    ("caller scale ignored", "if (scale <= 0.0) scale = 1.0 / sqrt((double)D);\n    if (n_valid <= 0)",
     "scale = 1.0 / sqrt((double)D);\n    if (n_valid <= 0)", [O + "test_caller_scale_is_the_logit_factor"]),
    ("attention log-weight dropped", "visible ? dot * scale + lw : -INFINITY", "visible ? dot * scale : -INFINITY",
     [O + "test_log_weight_is_a_multiplicative_key_weight"]),
    ("attention log-weight subtracted", "visible ? dot * scale + lw : -INFINITY",
     "visible ? dot * scale - lw : -INFINITY", [O + "test_log_weight_is_a_multiplicative_key_weight"]),
    ("LSE in base 2", "const double lse = mx + log(z);\n        for (int64_t x = 0; x < nkeys",
     "const double lse = mx + log2(z);\n        for (int64_t x = 0; x < nkeys",
     [O + "test_block_of_identical_keys_gives_its_value_exactly"]),
    ("empty row LSE 0", "if (cnt <= 0) {\n            LSE[w] = -INFINITY;", "if (cnt <= 0) {\n            LSE[w] = 0.0;",
     [O + "test_empty_list_gives_zero_output_and_minus_inf_lse"]),
    ("causal strict", "(!causal || j <= i)", "(!causal || j < i)",
     [O + "test_token_mask_all_blocks_equals_matrix_form"]),
    ("window one key wider", "(window <= 0 || j > i - window || j < sinks)",
     "(window <= 0 || j >= i - window || j < sinks)",
     [O + "test_token_mask_all_blocks_equals_matrix_form"]),
    ("sinks dropped", "|| j > i - window || j < sinks)", "|| j > i - window)",
     [O + "test_token_mask_all_blocks_equals_matrix_form"]),
    ("tail mask ignored", "const int visible = j < n_valid &&", "const int visible = 1 &&",
     [O + "test_token_mask_all_blocks_equals_matrix_form"]),
    ("grouped heads interleaved", "const int64_t kvh = (bh / H) * H_kv + (bh % H) / group;",
     "const int64_t kvh = (bh / H) * H_kv + (bh % H) % H_kv;",
     [O + "test_grouped_heads_equal_repeated_heads_and_matrix_form"]),
    ("key map ignored", "const int32_t j = kv_map ? kv_map[kvh * N + pos] : pos;", "const int32_t j = pos;",
     [O + "test_maps_equal_physically_gathered_tensors"]),
    ("query map ignored", "const int32_t i = q_map ? q_map[bh * N + p] : p;\n        const int64_t kvh",
     "const int32_t i = p;\n        const int64_t kvh", [O + "test_maps_equal_physically_gathered_tensors"]),
    ("Gather 0 window one row low", "clamp64(8 * r - 4, 0, img_h - 16)", "clamp64(8 * r - 3, 0, img_h - 16)",
     [G + "test_window_corners_hand_worked"]),
    ("Gather 0 window not clamped", "clamp64(8 * c - 4, 0, img_w - 16)", "(8 * c - 4 < 0 ? 0 : 8 * c - 4)",
     [G + "test_window_geometry"]),
    ("Scatter groups contiguous", "k_tok[nk++] = (int32_t)(n_text + t * groups + g);",
     "k_tok[nk++] = (int32_t)(n_text + g * (hw / groups) + t);", [G + "test_window_geometry"]),
    ("text queries interleaved across groups", "q_tok[i] = (int32_t)(g * per + i);",
     "q_tok[i] = (int32_t)(i * groups + g);", [G + "test_attention_against_masked_sdpa"]),
    ("image-layer scale 1/D", "if (scale <= 0.0) scale = 1.0 / sqrt((double)D);\n#pragma omp parallel for "
     "schedule(dynamic, 1)\n    for (int64_t x = 0; x < nq; ++x)",
     "if (scale <= 0.0) scale = 1.0 / (double)D;\n#pragma omp parallel for schedule(dynamic, 1)\n"
     "    for (int64_t x = 0; x < nq; ++x)", [G + "test_attention_against_masked_sdpa"]),
    ("CRM bit order reversed", "|= 1u << (kb % 32);", "|= 1u << (31 - kb % 32);",
     [O + "test_crm_rows_encode_the_same_blocks_as_the_lists"]),
    ("upscale takes a maximum", "if (b[(int64_t)i1 * Vb + j1] < m)", "if (b[(int64_t)i1 * Vb + j1] > m)",
     [O + "test_upscale_hand_worked_example"]),
    ("upscale ignores the second neighbour", "const int32_t i1 = (xu % Ut != 0 && i0 + 1 < Ub) ? i0 + 1 : i0;",
     "const int32_t i1 = i0;", [O + "test_upscale_hand_worked_example"]),
    ("block score of sums, not means", "qm[(int64_t)b * D + d] = sq / ORACLE_BLOCK;", "qm[(int64_t)b * D + d] = sq;",
     [O + "test_block_scores_closed_form_for_constant_blocks_and_attention_logit"]),
    ("block scores read Q through the key map",
     "const int32_t i = q_map ? q_map[bh * N + p] : p;\n                    const int32_t j",
     "const int32_t i = kv_map ? kv_map[bh * N + p] : p;\n                    const int32_t j",
     [O + "test_block_scores_ignore_order_inside_a_block_and_follow_maps"]),
    # (centring the key-side product is redundant once the iterate is
    # orthogonal to the ones vector, so only the row-side centring is planted)
    ("spectral rows not centred", "X[2 * r] = y0 - m0;\n                X[2 * r + 1] = y1 - m1;",
     "X[2 * r] = y0;\n                X[2 * r + 1] = y1;", [O + "test_spectral_subspace_matches_svd_of_centered_mask"]),
    ("spectral ties to the higher row", "return (p->r > q->r) - (p->r < q->r);",
     "return (p->r < q->r) - (p->r > q->r);", [O + "test_spectral_angle_and_ties_to_the_lower_row"]),
    ("spectral angle arguments swapped", "srt[r].a = atan2(X[2 * r + 1], X[2 * r]);",
     "srt[r].a = atan2(X[2 * r], X[2 * r + 1]);", [O + "test_spectral_angle_and_ties_to_the_lower_row"]),
    ("spectral order by descending angle", "if (p->a < q->a) return -1;\n    if (p->a > q->a) return 1;",
     "if (p->a < q->a) return 1;\n    if (p->a > q->a) return -1;",
     [O + "test_spectral_order_groups_planted_clusters_and_is_a_permutation"]),
]


def _build(src_text, path):
    src = path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *oracle.CFLAGS, src, "-o", path, "-lm"], check=True, capture_output=True)
    return path


def _run_pins(lib, pins):
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=lib, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "not gpu",
                        *pins], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-1500:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    d = tmp_path_factory.mktemp("mutants")
    with open(oracle._SRC) as f:
        src = f.read()
    jobs = {"unaltered": (src, sorted({p for m in MUTANTS for p in m[3]}))}
    for name, old, new, pins in MUTANTS:
        assert src.count(old) == 1, f"{name}: the text to alter must occur once"
        jobs[name] = (src.replace(old, new), pins)

    def work(item):
        i, (name, (text, pins)) = item
        lib = _build(text, str(d / f"mutant{i}.so"))
        return name, _run_pins(lib, pins)

    with cf.ThreadPoolExecutor(max_workers=max(2, min(8, (os.cpu_count() or 2)))) as ex:
        return dict(ex.map(work, enumerate(jobs.items())))


def test_unaltered_oracle_passes_every_pin(outcomes):
    code, out = outcomes["unaltered"]
    assert code == 0, out


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(outcomes, name):
    code, out = outcomes[name]
    # pytest exit code 1: tests ran and at least one failed (not a crash,
    # not a collection error)
    assert code == 1, f"{name}: pins exit {code}\n{out}"
