#!/usr/bin/env python
"""Benchmark: block-sparse attention forward on one GB300 (per rank).

One step = one pass of the whole path over one synthetic workload resident
in HBM: block scoring (mean-pooled Q/K blocks, for the dynamic workloads) ->
index-list construction (threshold map, mask or top-k scores, plus sampling
where the workload has it) -> query-row reordering (when the reorder guard
says it pays) -> block-sparse attention forward.  The default workload is the
dynamic one (B1 H24 N118784 D128, top-k of mean-pooled QK^T at 10-20 %
density), the largest that the benchmark configurations give one GPU.  The metric is effective TFLOP/s: 4 * 128 * 128 * D FLOPs
per computed (query block, KV block) pair, divided by the step time; for the
Gather 0 image layer (config 9) 4 * D FLOPs per attended query-key pair.  The
roofline object reports the forward kernel against the measured bf16 peak,
or against the measured HBM copy bandwidth when the workload's FLOPs per
compulsory byte fall below the ridge (the one-pair Scatter layer).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 5]
                    [--order auto|identity|reordered|spectral] [--scores auto|pooled|given]
                    [--impl ours|reference]

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (the reference arm of this comparison).  Under torchrun each rank
runs its own copy of the workload on its own GPU (weak scaling); timing is
the max over ranks.  One JSON line is printed by rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "block-sparse attn fwd effective TFLOP/s (% of GB300 BF16 TC peak); ms/call"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# A kernel launched back to back for at least this long runs under the
# board's power limit (its clock samples show sw_power_cap); it is compared
# with the GEMM rate sustained under that limit, a shorter run with the burst
# rate.
SUSTAINED_AFTER_MS = 100.0
L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2


# ---------------------------------------------------------------- helpers
def tensor_peak(peaks: dict, launches: int, avg_ms: float):
    """(peak TFLOP/s, which) for a kernel timed over `launches` back-to-back
    launches of `avg_ms` each: the sustained bf16 GEMM rate once the sequence
    lasts SUSTAINED_AFTER_MS, else the burst rate."""
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    if launches * avg_ms >= SUSTAINED_AFTER_MS:
        return sustained, "sustained"
    return burst, "burst"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    """Hash of the forward kernel's code: comments and whitespace are dropped,
    so that a comment edit does not orphan the recorded ncu counters."""
    h = hashlib.sha256()
    for f in ("bsa_attn.cu", "bsa_ptx.cuh", "bsa_math.cuh", "bsa_gather0.cuh"):
        with open(os.path.join(ROOT, "long_context_mask_gb300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(args, order: str):
    """DRAM bytes per forward launch from a committed ncu capture, if it was
    taken on the current kernel source, on this exact workload (the default
    options of that configuration) and in the row order this run uses; else
    None."""
    p = os.path.join(ROOT, "profiles", "forward_traffic.json")
    if not os.path.exists(p):
        return None
    default_run = (args.heads is None and not args.dense and not args.crm and args.scores == "auto"
                   and args.order == "auto" and args.kv_gather == "auto")
    if not default_run:
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"config{args.config}")
    if not e or e.get("kernel_hash") != kernel_source_hash() or e.get("order") != order:
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        busy = [s for s in sm if mx is None or s >= 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- the path
class Path:
    """Device buffers and the per-step launch sequence for one workload."""

    def __init__(self, prob, dev, order: str, scores_on_gpu: bool = False, crm: bool = False,
                 kv_gather: str = "auto"):
        import long_context_mask_gb300 as bsa
        self.bsa = bsa
        self.prob = prob
        self.dev = dev
        self.order = order
        cu = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(dev)  # noqa: E731
        self.q, self.k, self.v = (t.to(dev) for t in (prob.q, prob.k, prob.v))
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:3], dtype=torch.float32, device=dev)
        self.q_map, self.kv_map = cu(prob.q_map), cu(prob.kv_map)
        rows, nqb = prob.rows, prob.nqb
        self.heads = prob.B * prob.H
        self.image = is_image_layer(prob)
        self.quad_mask = None
        if self.image:
            # the static Gather 0 pattern: maps, lists and quadrant masks built
            # once on the GPU (the layer's fixed index functions)
            self.q_map, self.kv_map, self.idx, self.cnt, self.quad_mask = bsa.gather0_layout(
                prob.img_h, prob.img_w, prob.n_text, prob.groups, self.heads, device=dev)
            self.mode, self.src, self.max_kv = None, None, self.idx.shape[1]
        elif prob.mask is not None:
            self.mode, self.src, self.max_kv = bsa.IDX_MASK_U8, cu(prob.mask), nqb
        elif prob.T is not None:
            self.mode, self.src, self.max_kv = bsa.IDX_THRESHOLD_F32, cu(prob.T), nqb
        elif prob.scores is not None:
            self.mode, self.src = bsa.IDX_TOPK_F32, cu(prob.scores)
            self.max_kv = int(prob.k_const if prob.k_per_row is None else prob.k_per_row.max())
        else:
            self.mode, self.src, self.max_kv = None, None, 1
        self.k_per_row = cu(prob.k_per_row)
        self.scores_on_gpu = scores_on_gpu and prob.scores is not None
        if self.scores_on_gpu:
            self.score_mode = bsa.SCORE_CENTROID_EXP if prob.m_sample else bsa.SCORE_MEAN_DOT
            self.score_ws = torch.empty(max(1, bsa.load_library().bsa_block_scores_workspace_size(
                prob.B, prob.H, prob.N, prob.D)), dtype=torch.uint8, device=dev)
        self.u = cu(prob.u)
        if not self.image:
            self.idx = torch.empty((rows, self.max_kv), dtype=torch.int32, device=dev)
            self.cnt = torch.empty(rows, dtype=torch.int32, device=dev)
        if self.mode is None and not self.image:  # one KV block per query block (Scatter / Gather layers)
            self.idx.copy_(torch.arange(rows, device=dev, dtype=torch.int32).remainder(nqb)[:, None])
            self.cnt.fill_(1)
        self.lw = None
        if prob.m_sample:
            cap = self.max_kv + prob.m_sample
            self.s_idx = torch.empty((rows, cap), dtype=torch.int32, device=dev)
            self.s_cnt = torch.empty(rows, dtype=torch.int32, device=dev)
            self.lw = torch.empty((rows, cap), dtype=torch.float32, device=dev)
        self.crm = crm and self.mode in (bsa.IDX_MASK_U8, bsa.IDX_THRESHOLD_F32)
        if self.crm:
            self.words = torch.empty((rows, (nqb + 31) // 32), dtype=torch.int32, device=dev)
            order = self.order = "identity"
        self.row_perm = torch.empty((self.heads, nqb), dtype=torch.int32, device=dev)
        self.wave = bsa.resident_ctas(prob.D)
        if order == "spectral":
            self.x0 = torch.from_numpy(synth.spectral_start(7, self.heads, nqb)).float().to(dev)
            self.spec = torch.empty((self.heads, nqb), dtype=torch.int32, device=dev)
            self.spec_ws = torch.empty(bsa.spectral_order_workspace_size(self.heads, nqb, nqb),
                                       dtype=torch.uint8, device=dev)
        # Gathered keys/values: copy them into gathered order once per step
        # (one HBM pass) when blocks are listed by many query blocks each, or
        # gather rows inside the forward kernel when each block is used once
        # (the Scatter layer's one block per query block).
        self.image_boxes = False
        # the Scatter layer: tiles as strided boxes (auto), or rows through the maps
        self.scatter_boxes = prob.scatter_R > 0 and kv_gather == "auto"
        if self.image:
            # packed key tiles overlap (no N-row gathered copy exists): fetch
            # them as boxes of the image (auto), or row by row through kv_map
            if kv_gather == "hbm":
                raise SystemExit("--kv-gather hbm does not apply to the image layer")
            self.image_boxes = kv_gather == "auto"
            kv_gather = "kernel"
        if kv_gather == "auto":
            kv_gather = "kernel" if prob.diag_list else "hbm"
        self.pregather = self.kv_map is not None and kv_gather == "hbm" and not self.crm
        self.masked = uses_masked_forward(prob)
        if self.pregather:
            self.kg, self.vg = torch.empty_like(self.k), torch.empty_like(self.v)
        self.launches_per_step = (1 + 2 * self.pregather + (self.mode is not None) + bool(prob.m_sample)
                                  + (order != "identity") + (order == "spectral")
                                  + 2 * self.scores_on_gpu)

    def lists(self):
        return (self.s_idx, self.s_cnt) if self.prob.m_sample else (self.idx, self.cnt)

    def build_lists(self):
        bsa, p = self.bsa, self.prob
        if self.crm:
            bsa.build_crm(self.mode, self.src, self.words, p=p.p or 0.0)
            return
        if self.scores_on_gpu:
            bsa.block_scores(self.q, self.k, self.src, q_map=self.q_map, kv_map=self.kv_map,
                             mode=self.score_mode, workspace=self.score_ws)
        if self.mode is not None:
            bsa.build_index(self.mode, self.src, self.idx, self.cnt, p=p.p or 0.0,
                            k_per_row=self.k_per_row, k_const=p.k_const or 0)
        if p.m_sample:
            bsa.sample_blocks(self.src, self.idx, self.cnt, p.m_sample, self.u, self.s_idx,
                              self.s_cnt, self.lw)
        if self.order == "spectral":
            idx, cnt = self.lists()
            bsa.spectral_order(idx, cnt, p.nqb, self.x0, self.spec, workspace=self.spec_ws, iters=10)
            bsa.reorder_rows(cnt.reshape(self.heads, p.nqb), self.wave, self.row_perm,
                             order_in=self.spec)
        elif self.order == "reordered":
            _, cnt = self.lists()
            bsa.reorder_rows(cnt.reshape(self.heads, p.nqb), self.wave, self.row_perm)

    def host_inputs(self):
        """Tensors a step takes from the host (end-to-end leg); the static
        patterns of the image and Scatter layers (layout, maps) stay on the
        device, and their geometry modes do not read maps at all.  Block
        scores computed inside the step are not inputs."""
        ts = (self.q, self.k, self.v) if (self.image or self.scatter_boxes) else (
            self.q, self.k, self.v, None if self.scores_on_gpu else self.src, self.q_map, self.kv_map,
            self.k_per_row, self.u)
        return [t for t in ts if t is not None]

    def attend(self, row_perm="auto"):
        """The forward launch; row_perm overrides the path's row order (None:
        input order) for the order comparison."""
        if isinstance(row_perm, str):
            row_perm = None if self.order == "identity" else self.row_perm
        if self.scatter_boxes:
            idx, cnt = self.lists()
            self.bsa.forward_scatter(self.q, self.k, self.v, self.prob.scatter_R, idx, cnt, self.o, self.lse,
                                     log_w=self.lw, row_perm=row_perm)
            return
        if self.image:
            perm = row_perm
            p = self.prob
            if self.image_boxes:
                self.bsa.forward_gather0(self.q, self.k, self.v, p.img_h, p.img_w, p.n_text, p.groups,
                                         self.idx, self.cnt, self.o, self.lse, quad_mask=self.quad_mask,
                                         row_perm=perm)
            else:
                self.bsa.forward_packed(self.q, self.k, self.v, self.idx, self.cnt, self.kv_map, self.o,
                                        self.lse, quad_mask=self.quad_mask, q_map=self.q_map, row_perm=perm)
            return
        if self.crm:
            self.bsa.forward_crm(self.q, self.k, self.v, self.words, self.o, self.lse,
                                 q_map=self.q_map, kv_map=self.kv_map)
            return
        idx, cnt = self.lists()
        k, v, kv_map = self.k, self.v, self.kv_map
        if self.pregather:
            k, v, kv_map = self.kg, self.vg, None
        if self.masked:
            self.bsa.forward_masked(self.q, k, v, idx, cnt, self.o, self.lse, log_w=self.lw,
                                    q_map=self.q_map, kv_map=kv_map, row_perm=row_perm,
                                    **token_mask(self.prob))
            return
        self.bsa.forward(self.q, k, v, idx, cnt, self.o, self.lse, log_w=self.lw,
                         q_map=self.q_map, kv_map=kv_map, row_perm=row_perm)

    def wave_order(self, out):
        """The NNZ wave sort of the current lists into `out` (for the order
        comparison and the guard's cost measurement)."""
        _, cnt = self.lists()
        self.bsa.reorder_rows(cnt.reshape(self.heads, self.prob.nqb), self.wave, out)

    def prepare_kv(self):
        """Keys/values into gathered order in HBM (only when pre-gathering)."""
        if self.pregather:
            self.bsa.gather_rows(self.k, self.kv_map, self.kg)
            self.bsa.gather_rows(self.v, self.kv_map, self.vg)

    def step(self):
        self.build_lists()
        self.prepare_kv()
        self.attend()

    def effective_flops(self):
        if self.image:
            return image_useful_flops(self.prob)
        if self.crm:
            self.bsa.build_index(self.mode, self.src, self.idx, self.cnt, p=self.prob.p or 0.0)
        _, cnt = self.lists()
        return self.bsa.effective_flops(cnt, self.prob.D)


def make_problem(config: int, heads: int | None, dense: bool = False):
    kw = {} if heads is None else {"H": heads}
    prob = synth.CONFIGS[config](**kw)
    if dense:
        prob.mask = np.ones((prob.rows, prob.nqb), np.uint8)
        prob.T = prob.scores = prob.k_per_row = prob.k_const = prob.m_sample = prob.u = None
        prob.diag_list = False
        prob.name += "+dense"
    return prob


# ---------------------------------------------------------------- CPU oracle timing
def sample_heads(prob):
    """Heads the oracle samples: every head of the small workloads; the first
    and the last head of those whose heads take the oracle a minute or more
    each (the per-head rate is the same for every head)."""
    bh = prob.B * prob.H
    per_head_flops = float(prob.nqb) * prob.nqb * 4 * 128 * 128 * prob.D * 0.3
    return None if per_head_flops < 2e12 or bh <= 2 else (0, bh - 1)


def time_oracle(prob, lists, budget_s: float, max_blocks: int | None = None, seed: int = 0,
                full_heads: bool = False):
    """Oracle on a bounded sample of query blocks (seeded, spread over the
    heads of sample_heads()), or with full_heads every query block of those
    heads.  Returns (effective TFLOP/s, seconds, blocks, threads)."""
    import oracle
    if is_image_layer(prob):
        return time_oracle_image(prob, budget_s, seed)
    idx, cnt, lw = lists
    g = np.random.default_rng(seed)
    heads = sample_heads(prob)
    if heads is None:
        order = g.permutation(prob.rows)
    else:
        rows = np.concatenate([np.arange(h * prob.nqb, (h + 1) * prob.nqb) for h in heads])
        order = rows[g.permutation(len(rows))]
    done, fl, t_total = 0, 0.0, 0.0
    chunk = 8
    while done < len(order):
        sel = order[done:done + chunk]
        t0 = time.perf_counter()
        oracle.attention(prob.q, prob.k, prob.v, idx, cnt, log_w=lw, q_map=prob.q_map,
                         kv_map=prob.kv_map, sel=sel, **token_mask(prob))
        t_total += time.perf_counter() - t0
        fl += float(cnt[sel].sum()) * 4 * 128 * 128 * prob.D
        done += len(sel)
        if not (full_heads and heads is not None) and (t_total >= budget_s or (max_blocks and done >= max_blocks)):
            break
    return fl / t_total / 1e12, t_total, done, oracle.num_threads()


def is_image_layer(prob):
    return prob.img_h > 0


def image_visible_pairs(prob):
    """Query-key pairs the Gather 0 layer attends, per head: every image query
    sees the text keys and its 16 x 16 window; every text query the text keys
    and its Scatter group's image tokens."""
    hw = prob.img_h * prob.img_w
    text = prob.n_text * (prob.n_text + hw // prob.groups) if prob.n_text else 0
    return hw * (prob.n_text + 256) + text


def image_useful_flops(prob):
    return 4.0 * prob.D * prob.B * prob.H * image_visible_pairs(prob)


def time_oracle_image(prob, budget_s: float, seed: int = 0):
    """The Gather 0 oracle on a bounded, seeded sample of (head, CQS) pairs.
    Returns (TFLOP/s over visible pairs, seconds, sets, threads)."""
    import oracle
    sets = oracle.gather0_sets(prob.img_h, prob.img_w, prob.n_text, prob.groups)
    order = np.random.default_rng(seed).permutation(prob.B * prob.H * len(sets))
    done, fl, t_total = 0, 0.0, 0.0
    for x in order:
        bh, si = divmod(int(x), len(sets))
        qt, kt = sets[si]
        t0 = time.perf_counter()
        oracle.attention_set(prob.q, prob.k, prob.v, bh, qt, kt)
        t_total += time.perf_counter() - t0
        fl += 4.0 * prob.D * len(qt) * len(kt)
        done += 1
        if t_total >= budget_s:
            break
    return fl / t_total / 1e12, t_total, done, oracle.num_threads()


def token_mask(prob):
    return dict(causal=prob.causal, n_valid=prob.n_valid, window=prob.window, sinks=prob.sinks)


def uses_masked_forward(prob):
    return ((prob.H_kv not in (None, prob.H)) or prob.causal or prob.window > 0 or prob.n_valid > 0
            or is_image_layer(prob))


def uses_pooled_scores(prob, scores_arg: str, config: int) -> bool:
    """Block scores from the tokens inside the step: the dynamic workloads by
    default (top-k of mean-pooled QK^T), any scored workload on request."""
    if prob.scores is None:
        return False
    return scores_arg == "pooled" or (scores_arg == "auto" and config in (5, 6))


def host_lists(prob, pooled: bool = False):
    """Index lists for the oracle, from the oracle (reference arm / CPU leg
    only); with pooled scores the oracle scores the blocks itself."""
    import oracle
    if is_image_layer(prob):
        return None  # the Gather 0 oracle works from the layer's definition
    if prob.diag_list:
        idx, cnt = synth.diag_lists(prob.rows, prob.nqb)
        return idx, cnt, None
    if prob.mask is not None:
        idx, cnt, _ = oracle.index_mask(prob.mask)
    elif prob.T is not None:
        idx, cnt, _ = oracle.index_threshold(prob.T, prob.p)
    else:
        k = prob.k_per_row if prob.k_per_row is not None else prob.k_const
        scores = prob.scores
        if pooled:
            scores = oracle.block_scores(prob.q, prob.k, prob.q_map, prob.kv_map,
                                         mode=1 if prob.m_sample else 0).astype(np.float32)
        idx, cnt, _ = oracle.index_topk(scores, k)
    if prob.m_sample:
        idx, cnt, lw, _ = oracle.sample_blocks(prob.scores, idx, cnt, prob.m_sample, prob.u,
                                               idx.shape[1] + prob.m_sample)
        return idx, cnt, lw
    return idx, cnt, None


# ---------------------------------------------------------------- main
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5, 6, 7, 8, 9])
    ap.add_argument("--heads", type=int, default=None, help="override H (smaller profiling case)")
    ap.add_argument("--order", default="auto", choices=["auto", "reordered", "identity", "spectral"],
                    help="row order: as the reorder guard decides (auto), NNZ-guided wave sort, "
                         "identity, or spectral (stage 1) + wave sort")
    ap.add_argument("--crm", action="store_true",
                    help="mask / threshold workloads: CRM bitmask rows instead of index lists "
                         "(identity row order)")
    ap.add_argument("--scores", default="auto", choices=["auto", "pooled", "given"],
                    help="top-k / sampling scores: from Q/K inside the step (pooled: mean-pooled "
                         "QK^T, centroid scores for --config 4) or the generator's (given); auto: "
                         "pooled for the dynamic workloads 5 and 6")
    ap.add_argument("--dense", action="store_true",
                    help="every query block attends to every KV block (the in-build dense ceiling)")
    ap.add_argument("--kv-gather", default="auto", choices=["auto", "kernel", "hbm"],
                    help="index-mapped K/V: gather rows inside the forward kernel, or copy them "
                         "into gathered order in HBM first (auto: HBM unless each block is "
                         "listed once; the image layer: tiles as boxes of the image, 'kernel' "
                         "rows through kv_map)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle CPU time")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-once", action="store_true",
                    help="build inputs, run one step, exit (for ncu captures)")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def config_dict(prob, config, density, world):
    name = synth.CONFIG_NAMES[config] + (" [dense: all blocks listed]" if prob.name.endswith("+dense") else "")
    return {"workload": name, "config_id": config, "B": prob.B, "H": prob.H,
            "N": prob.N, "D": prob.D, "block": 128, "density": round(density, 4),
            "l2": "flushed between timed steps (256 MiB write)",
            "parallelism": "one independent workload per GPU" if world > 1 else "single GPU",
            "scores": (("centroid scores of Q/K blocks" if prob.m_sample else "mean-pooled Q/K blocks")
                       + ", inside the step") if getattr(prob, "_scores_on_gpu", False) else "given",
            "kv_sets": "CRM bitmask rows" if getattr(prob, "_crm", False) else "index lists",
            "kv_rows": getattr(prob, "_kv_rows", "contiguous"),
            **({"H_kv": prob.H_kv or prob.H, "token_mask": token_mask(prob),
                "flops": "listed blocks in full (masked keys inside a listed block are computed)"}
               if uses_masked_forward(prob) and not is_image_layer(prob) else {}),
            **({"image": f"{prob.img_h}x{prob.img_w}", "n_text": prob.n_text,
                "scatter_groups": prob.groups,
                "layout": "two 8x8 query patches per 128-row tile; 16x16 windows as packed "
                          "8x16 key bands; 32-row quadrant masks (built once on the GPU)",
                "flops": "attended query-key pairs only (4 D per pair); products of tiles "
                         "hidden from a quadrant are extra work, not counted"}
               if is_image_layer(prob) else {})}


def compulsory_bytes(prob):
    """Bytes a forward launch must move: Q, K, V read once, O and LSE written."""
    H_kv = prob.H_kv or prob.H
    qo = 2 * prob.B * prob.H * prob.N * prob.D * 2
    kv = 2 * prob.B * H_kv * prob.N * prob.D * 2
    return float(qo + kv + prob.B * prob.H * prob.N * 4)


def sample_text(prob):
    heads = sample_heads(prob)
    if is_image_layer(prob):
        return "seeded sample over all heads"
    if heads is None:
        return "seeded sample over all heads"
    return f"seeded sample of heads {heads[0]} and {heads[1]}; the rate is per query block, the same for every head"


def sample_unit(prob):
    return "(head, CQS) query sets" if is_image_layer(prob) else "query blocks"


def workload_density(prob, listed_blocks):
    """Fraction of the dense attention computed: listed blocks over all
    blocks, or (image layer) attended query-key pairs over N^2."""
    if is_image_layer(prob):
        return image_visible_pairs(prob) / float(prob.N) ** 2
    return float(listed_blocks) / (prob.rows * prob.nqb)


def run_reference(args, world, rank):
    if rank != 0:
        return
    prob = make_problem(args.config, args.heads, args.dense)
    pooled = uses_pooled_scores(prob, args.scores, args.config)
    prob._scores_on_gpu = pooled
    lists = host_lists(prob, pooled)
    density = workload_density(prob, None if lists is None else lists[1].sum())
    # each step: the oracle on a bounded sample (about 1 s of CPU work)
    budget = 1.0
    for _ in range(args.warmup):
        time_oracle(prob, lists, budget / 4, seed=1)
    vals, secs, blocks = [], 0.0, 0
    for k in range(args.steps):
        v, s, b, threads = time_oracle(prob, lists, budget, seed=100 + k)
        vals.append(v)
        secs += s
        blocks += b
    value = statistics.median(vals)
    ms = secs / args.steps * 1e3
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": config_dict(prob, args.config, density, 1),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"{blocks} {sample_unit(prob)} ({sample_text(prob)}) over "
                                       f"{args.steps} steps (~{budget:.0f} s of oracle CPU time per step)"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


ORDER_OF_GUARD = {"input": "identity", "wave": "reordered", "spectral": "spectral"}


def event_ms(fn, reps: int, flush=None) -> float:
    """Mean device time of fn() over reps launches (CUDA events on the current
    stream, L2 flushed before each when a flush buffer is given)."""
    stream = torch.cuda.current_stream()
    total = 0.0
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        total += a.elapsed_time(b)
    return total / reps


def choose_order(prob, dev, args, pooled: bool, peaks: dict, flush):
    """The row order the reorder guard picks for this workload, and the guard's
    inputs and estimates.  The inputs are measured on this GPU: the listed
    block pairs, the forward's rate in the input order, and what the NNZ wave
    sort and the spectral stage cost on these lists."""
    import long_context_mask_gb300 as bsa
    path = Path(prob, dev, "identity", pooled, args.crm, args.kv_gather)
    path.step()
    torch.cuda.synchronize()
    _, cnt = path.lists()
    listed = int(cnt.sum().item())
    fwd_ms = event_ms(path.attend, 3, flush)
    rate = listed * 4.0 * 128 * 128 * prob.D / (fwd_ms * 1e-3) / 1e12 if listed else 0.0
    perm = torch.empty_like(path.row_perm)
    wave_ms = event_ms(lambda: path.wave_order(perm), 3)
    idx, cnt = path.lists()
    nqb = prob.nqb
    # key tiles a list entry may name: blocks of the sequence, or packed tiles of the image layer
    nkb = path.kv_map.shape[-1] // 128 if path.image else nqb
    spectral_ms = -1.0  # the guard's estimate where the spectral stage does not apply
    if nqb >= 2:
        x0 = torch.from_numpy(synth.spectral_start(7, path.heads, nqb)).float().to(dev)
        spec = torch.empty((path.heads, nqb), dtype=torch.int32, device=dev)
        ws = torch.empty(max(1, bsa.spectral_order_workspace_size(path.heads, nqb, nkb)),
                         dtype=torch.uint8, device=dev)
        spectral_ms = event_ms(lambda: bsa.spectral_order(idx, cnt, nkb, x0, spec, workspace=ws, iters=10), 3)
        del x0, spec, ws
    g = bsa.reorder_guard(heads=path.heads, kv_heads=prob.B * (prob.H_kv or prob.H), nqb=nqb, nkb=nkb,
                          D=prob.D, listed_blocks=listed, tensor_tflops=rate,
                          hbm_gbs=float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                          wave_ms=wave_ms, spectral_ms=spectral_ms)
    del path, perm
    torch.cuda.empty_cache()
    g.update({"measured_forward_ms_input_order": fwd_ms, "measured_wave_ms": wave_ms,
              "measured_spectral_ms": spectral_ms, "listed_blocks": listed})
    return ORDER_OF_GUARD[g["order"]], g


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py --impl ours needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    import long_context_mask_gb300 as bsa

    peaks, peak_src = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    prob = make_problem(args.config, args.heads, args.dense)
    pooled = uses_pooled_scores(prob, args.scores, args.config)
    prob._scores_on_gpu = pooled
    prob._crm = args.crm and (prob.mask is not None or prob.T is not None)
    guard = None
    order = args.order
    if prob._crm:
        order = "identity"
    elif order == "auto":
        order, guard = choose_order(prob, dev, args, pooled, peaks, flush)
    path = Path(prob, dev, order, pooled, args.crm, args.kv_gather)
    if path.image:
        prob._kv_rows = ("tiles fetched as TMA boxes of the image / Scatter-group views "
                         "(bsa_forward_gather0)" if path.image_boxes else
                         "gathered through kv_map inside the forward kernel (bsa_forward_packed)")
    elif path.scatter_boxes:
        prob._kv_rows = "Scatter tiles fetched as strided TMA boxes (bsa_forward_scatter)"
    elif path.kv_map is not None:
        prob._kv_rows = ("copied into gathered order in HBM each step (bsa_gather_rows)"
                         if path.pregather else "gathered through kv_map inside the forward kernel")
    path.step()
    torch.cuda.synchronize()
    if args.profile_once:
        st = bsa.device_status()
        print(json.dumps({"profile_once": True, "status": st, "order": path.order}))
        return

    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        path.step()
    torch.cuda.synchronize()
    flops = path.effective_flops()
    density = workload_density(prob, path.lists()[1].sum())

    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    fwd_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with ClockSampler(gpu_id) as clk:
        # ---- timed region: K steps (L2 flushed before each, outside the events)
        barrier(world)
        torch.cuda.synchronize()
        # extra flushes ahead of the loop keep the GPU busy while the host
        # enqueues the first steps, so that no step's events span host time
        for _ in range(3):
            flush.zero_()
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            path.step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        step_ms = [a.elapsed_time(b) for a, b in ev]
        # ---- the dominant kernel alone (same inputs, L2 flushed before each launch)
        path.build_lists()
        path.prepare_kv()
        for i in range(K):
            flush.zero_()
            fwd_ev[i][0].record(stream)
            path.attend()
            fwd_ev[i][1].record(stream)
        torch.cuda.synchronize()
        fwd_ms = [a.elapsed_time(b) for a, b in fwd_ev]
    # ---- the forward under the input order and under the NNZ wave sort (same lists)
    orders_ms = None
    if not path.crm:
        perm = torch.empty_like(path.row_perm)
        path.wave_order(perm)
        reps = max(3, min(K, 10))
        orders_ms = {"identity": event_ms(lambda: path.attend(None), reps, flush),
                     "reordered": event_ms(lambda: path.attend(perm), reps, flush)}
        del perm
    status = bsa.device_status()
    if status != 0:
        raise SystemExit(f"device status {status} after the timed region")

    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / K
    value = world * flops / (ms_per_step * 1e-3) / 1e12

    # ---- end to end: host (pinned) inputs -> device -> path -> host outputs.
    # Every step copies its inputs in and its O / LSE out inside the timed
    # region.  Two device buffer sets and separate copy streams let step k+1's
    # inputs travel (and step k-1's outputs come back) while step k computes.
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    paths = [path, Path(prob, dev, path.order, pooled, args.crm, args.kv_gather)]

    d_ins = [pth.host_inputs() for pth in paths]
    h_in = [pin(t) for t in d_ins[0]]
    h_o = [torch.empty_like(path.o, device="cpu").pin_memory() for _ in range(2)]
    h_l = [torch.empty_like(path.lse, device="cpu").pin_memory() for _ in range(2)]
    bi = sum(t.numel() * t.element_size() for t in h_in)
    bo = h_o[0].numel() * h_o[0].element_size() + h_l[0].numel() * h_l[0].element_size()
    # the first copies from freshly pinned pages run at a fraction of the link
    # rate, and the first few steps of the pipeline still meet stalls of tens
    # of ms in the host copies: once-per-buffer costs that a serving process
    # pays when it sets up.  The pipelined loop below therefore runs its
    # warm-up steps untimed first, like the device-timed region.
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_loop(E, timed):
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_done, comp_done, out_done = [ev() for _ in range(E)], [ev() for _ in range(E)], [ev() for _ in range(E)]
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if timed:
            barrier(world)
        torch.cuda.synchronize()
        e_start.record(stream)
        s_in.wait_event(e_start)
        s_out.wait_event(e_start)
        for k in range(E):
            b = k % 2
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(comp_done[k - 2])  # buffer set b no longer read
                for h, d in zip(h_in, d_ins[b]):
                    d.copy_(h, non_blocking=True)
                in_done[k].record(s_in)
            stream.wait_event(in_done[k])
            if k >= 2:
                stream.wait_event(out_done[k - 2])  # O / LSE of buffer set b copied out
            paths[b].step()
            comp_done[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[k])
                h_o[b].copy_(paths[b].o, non_blocking=True)
                h_l[b].copy_(paths[b].lse, non_blocking=True)
                out_done[k].record(s_out)
        stream.wait_event(out_done[E - 1])
        stream.wait_event(in_done[E - 1])
        e_end.record(stream)
        torch.cuda.synchronize()
        if timed:
            barrier(world)
        return e_start.elapsed_time(e_end)

    e2e_loop(max(args.warmup, 3) + 2, timed=False)
    E = max(4, K)
    e2e_total_ms = e2e_loop(E, timed=True)
    e2e_ms = max_over_ranks(e2e_total_ms / E, world, dev)
    e2e_value = world * flops / (e2e_ms * 1e-3) / 1e12
    del paths

    fwd_avg_ms = sum(fwd_ms) / len(fwd_ms)
    achieved = flops / (fwd_avg_ms * 1e-3) / 1e12
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak, which = tensor_peak(peaks, len(fwd_ms), fwd_avg_ms)
    traffic = recorded_traffic(args, path.order)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": "k_bsa_forward",
                "peak_source": (f"{peak_src} bf16 {which} ({len(fwd_ms)} launches back to back, "
                                f"{len(fwd_ms) * fwd_avg_ms:.0f} ms)"),
                "ms_per_launch": fwd_avg_ms, "frac_of_burst": achieved / burst,
                "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained",
                                                                FALLBACK_PEAKS["bf16_tflops_sustained"]))}
    # A workload whose FLOPs per compulsory byte (Q, K, V read once, O and LSE
    # written once) fall below the measured ridge is bounded by HBM instead.
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    alg_bytes = compulsory_bytes(prob)
    if flops / alg_bytes < burst * 1e12 / (hbm * 1e9):
        gbs = alg_bytes / (fwd_avg_ms * 1e-3) / 1e9
        roofline.update({"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "peak_source": f"{peak_src} HBM copy", "algorithmic_bytes": alg_bytes,
                         "tensor_tflops": achieved})
        roofline.pop("frac_of_sustained")
        roofline.pop("frac_of_burst")

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        heads = sample_heads(prob)
        full = heads is not None and not is_image_layer(prob)
        v, s, b, threads = time_oracle(prob, host_lists(prob, pooled), args.cpu_budget, full_heads=full)
        if full:
            # the CPU plan's subset for workloads too large for the oracle:
            # whole heads (the first and the last), then a labelled linear
            # extrapolation to every head
            sample = (f"{len(heads)} full heads ({heads[0]} and {heads[1]}): {b} {sample_unit(prob)}, "
                      f"{s:.1f} s fp64 on host cores; full workload extrapolated as per-head time x "
                      f"{prob.B * prob.H} heads")
            extrapolated = s / len(heads) * prob.B * prob.H
        else:
            sample = f"{b} {sample_unit(prob)} ({sample_text(prob)}), {s:.1f} s fp64 on host cores"
            extrapolated = flops / (v * 1e12) if v else None
        cpu = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample,
               "full_workload_s_extrapolated": extrapolated}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
            "ms_per_step_median": statistics.median(step_ms) if world == 1 else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_dict(prob, args.config, density, world),
            "row_order": {"order": path.order, "chosen_by": "reorder guard" if guard else "--order",
                          "guard": guard, "forward_ms": orders_ms},
            "pct_of_peak": 100.0 * value / world / burst,
            "roofline": roofline, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": bi,
                    "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms},
            "gpu_launches": K * path.launches_per_step,
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
