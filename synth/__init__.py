"""Seeded synthetic inputs for block-sparse attention.

This module only draws random numbers and lays out input structure (shapes,
distributions, sparsity patterns, index maps).  It holds none of the
attention, selection, sampling or reordering arithmetic: the CUDA library
and the oracle each implement that on their own, and both are fed the arrays
made here.  Everything is produced on the CPU from a seeded
``torch.Generator`` so that the two sides see identical bytes.

Workload shapes (the pages measure on trained video/image models that are not
available here; these synthetic inputs stand in for them, with the shapes and
structure the pages describe):

* ``tiny``       B1 H2 N2048 D64, Bernoulli(0.25) 16x16 block mask + diagonal.
* ``threshold``  Wan-1.3B 480p shape: H12 N32768 D128, per-head threshold map
                 T ~ U(0,1) with same/adjacent-frame blocks forced to 0
                 (1560 tokens per latent frame), mask T <= p at p = 0.15
                 (ScalingAttention section 5.2).
* ``scatter``    2K-image DiT shape: H24 N16384 D128, T = R = 128; Scatter
                 groups {t*128 + r : t} gathered through index maps, one KV
                 block per query block; Gather groups are the neighbourhoods
                 (INTRA, "Why Scatter Is Uniform and Non-Contiguous").
* ``sampled``    Wan-14B 720p shape: H40 N75776 D128, a random token
                 permutation per head into 592 clusters, U(0,1) block scores,
                 one U[0,1) draw per query block for systematic sampling
                 (InstaGen section 3.2.1).
* ``dynamic``    long-video shape: H24 N118784 D128; Q/K carry per-cluster /
                 per-block offsets so that query blocks fall into 8 shuffled
                 low-rank access clusters; per-row k ~ U{ceil(0.10 nB) ..
                 floor(0.20 nB)}.  The benchmark scores blocks from these
                 tokens (mean-pooled QK^T, in the library); ``scores`` holds a
                 planted alternative, the cluster-block affinity plus seeded
                 noise (drawn, not pooled), for the index-build tests.
* ``long_video`` the same at N401408 (401 latent frames), H2: one head's K/V
                 exceeds the L2 (WaveAlign's longest Wan2.1 workload).
* ``llm``, ``llm_window``  LLaMA-3.1-8B prefill shapes (32 query heads over 8
                 key/value heads, causal): every second 256-token block, or a
                 575-token sliding window with 64 sinks (INTRA section 4.7).
* ``image_gather0`` FLUX.1-dev image layer: H24 D128, 512 text tokens and a
                 128 x 128 latent image (INTRA appendix, Gather 0).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 128
FRAME_TOKENS_480P = 1560  # 30 x 52 latent tokens per frame (Wan 1.3B, 480p)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def normal_bf16(g: torch.Generator, shape) -> torch.Tensor:
    """i.i.d. N(0,1) rounded to bf16 (CPU tensor)."""
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


@dataclass
class Problem:
    """One synthetic block-sparse attention problem (all CPU tensors)."""
    name: str
    B: int
    H: int
    N: int
    D: int
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    # index source, one of:
    mask: np.ndarray | None = None          # uint8 [B*H*nQB, nKB]
    T: np.ndarray | None = None             # fp32 [B*H*nQB, nKB]
    p: float | None = None
    scores: np.ndarray | None = None        # fp32 [B*H*nQB, nKB]
    k_per_row: np.ndarray | None = None     # int32 [B*H*nQB]
    k_const: int | None = None
    m_sample: int | None = None             # sampled blocks per row
    u: np.ndarray | None = None             # fp64 [B*H*nQB], systematic-PPS draw
    diag_list: bool = False                 # one KV block per query block: kb = qb
    q_map: np.ndarray | None = None         # int32 [B*H, N]
    kv_map: np.ndarray | None = None        # int32 [B*H_kv, N]
    # grouped key/value heads (k, v are [B, H_kv, N, D]) and the token mask
    H_kv: int | None = None                 # None: H
    causal: bool = False
    n_valid: int = 0                        # 0: N
    window: int = 0
    sinks: int = 0
    # image layer (INTRA Gather 0): n_text text tokens, then an img_h x img_w
    # image; the maps and lists come from the layout, not from here
    img_h: int = 0
    img_w: int = 0
    n_text: int = 0
    groups: int = 1
    scatter_R: int = 0                      # > 0: q_map = kv_map = scatter_map(N, scatter_R)
    extra: dict = field(default_factory=dict)

    @property
    def nqb(self) -> int:
        return self.N // BLOCK

    @property
    def rows(self) -> int:
        return self.B * self.H * self.nqb


def tiny(seed: int = 1, B: int = 1, H: int = 2, N: int = 2048, D: int = 64,
         density: float = 0.25) -> Problem:
    g = _gen(seed)
    q, k, v = (normal_bf16(g, (B, H, N, D)) for _ in range(3))
    nb = N // BLOCK
    m = (torch.rand((B * H, nb, nb), generator=g) < density).to(torch.uint8)
    idx = torch.arange(nb)
    m[:, idx, idx] = 1
    return Problem("tiny", B, H, N, D, q, k, v, mask=m.reshape(B * H * nb, nb).numpy())


def frame_band(nb: int, frame_tokens: int = FRAME_TOKENS_480P) -> np.ndarray:
    """[nb, nb] bool: blocks whose latent frames are the same or adjacent."""
    fr = (np.arange(nb) * BLOCK) // frame_tokens
    return np.abs(fr[:, None] - fr[None, :]) <= 1


def threshold(seed: int = 2, B: int = 1, H: int = 12, N: int = 32768, D: int = 128,
              p: float = 0.15, frame_tokens: int = FRAME_TOKENS_480P) -> Problem:
    g = _gen(seed)
    q, k, v = (normal_bf16(g, (B, H, N, D)) for _ in range(3))
    nb = N // BLOCK
    T = torch.rand((B * H, nb, nb), generator=g, dtype=torch.float32).numpy()
    T[:, frame_band(nb, frame_tokens)] = 0.0
    return Problem("threshold", B, H, N, D, q, k, v, T=T.reshape(B * H * nb, nb), p=p)


def scatter_map(N: int, R: int = BLOCK) -> np.ndarray:
    """Scatter gather map for N = T*R tokens in T neighbourhoods of R tokens.

    Token (t, r) = t*R + r.  Scatter group S_r = {(t, r) : t} is laid out
    contiguously: gathered position p = r*T + t holds token t*R + r."""
    T = N // R
    p = np.arange(N)
    r, t = p // T, p % T
    return (t * R + r).astype(np.int32)


def scatter(seed: int = 3, B: int = 1, H: int = 24, N: int = 16384, D: int = 128,
            layer: str = "scatter") -> Problem:
    """Scatter layer (maps) or Gather layer (neighbourhoods, no maps); one block per row."""
    g = _gen(seed)
    q, k, v = (normal_bf16(g, (B, H, N, D)) for _ in range(3))
    prob = Problem(layer, B, H, N, D, q, k, v, diag_list=True)
    if layer == "scatter":
        m = np.broadcast_to(scatter_map(N), (B * H, N)).copy()
        prob.q_map, prob.kv_map = m, m
        prob.scatter_R = BLOCK
    return prob


def sampled(seed: int = 4, B: int = 1, H: int = 40, N: int = 75776, D: int = 128,
            k_exact: int = 16, m_sample: int = 8) -> Problem:
    g = _gen(seed)
    q, k, v = (normal_bf16(g, (B, H, N, D)) for _ in range(3))
    nb = N // BLOCK
    perm = np.stack([torch.randperm(N, generator=g).numpy() for _ in range(B * H)]).astype(np.int32)
    scores = torch.rand((B * H * nb, nb), generator=g, dtype=torch.float32).numpy()
    # strictly positive scores (the sampling design needs s_j > 0)
    scores = np.maximum(scores, np.float32(2.0 ** -24))
    u = torch.rand(B * H * nb, generator=g, dtype=torch.float64).numpy()
    return Problem("sampled", B, H, N, D, q, k, v, scores=scores, k_const=k_exact,
                   m_sample=m_sample, u=u, q_map=perm, kv_map=perm)


def dynamic(seed: int = 5, B: int = 1, H: int = 24, N: int = 118784, D: int = 128,
            n_clusters: int = 8, lo: float = 0.10, hi: float = 0.20) -> Problem:
    g = _gen(seed)
    nb = N // BLOCK
    BH = B * H
    # cluster of each query block: a seeded shuffle of (qb mod n_clusters)
    cl = np.stack([(np.arange(nb) % n_clusters)[torch.randperm(nb, generator=g).numpy()]
                   for _ in range(BH)])
    a = torch.randn((BH, n_clusters, D), generator=g)
    b = torch.randn((BH, nb, D), generator=g)
    qf = torch.randn((BH, nb, BLOCK, D), generator=g)
    qf += a[torch.arange(BH)[:, None], torch.from_numpy(cl)][:, :, None, :]
    q = qf.to(torch.bfloat16).reshape(B, H, N, D)
    del qf
    kf = torch.randn((BH, nb, BLOCK, D), generator=g)
    kf += b[:, :, None, :]
    k = kf.to(torch.bfloat16).reshape(B, H, N, D)
    del kf
    v = normal_bf16(g, (B, H, N, D))
    k_lo, k_hi = math.ceil(lo * nb), math.floor(hi * nb)
    kpr = torch.randint(k_lo, k_hi + 1, (BH * nb,), generator=g, dtype=torch.int32).numpy()
    # Block scores, an input of the top-k selection: the planted affinity
    # a_c(qb) . b_kb / sqrt(D) of the query block's cluster offset with the key
    # block's offset, plus N(0, 1/64) noise, about the spread that the token
    # noise of a 128-row block adds to its mean (fp64, rounded to fp32).
    # Scoring blocks from the tokens themselves is the library's block-score
    # step and the oracle's, not the generator's.
    a_q = a.double()[torch.arange(BH)[:, None], torch.from_numpy(cl)]
    affinity = torch.bmm(a_q, b.double().transpose(1, 2)) / math.sqrt(D)
    noise = torch.randn((BH, nb, nb), generator=g, dtype=torch.float64) / 8
    scores = (affinity + noise).to(torch.float32)
    prob = Problem("dynamic", B, H, N, D, q, k, v, scores=scores.reshape(BH * nb, nb).numpy(),
                   k_per_row=kpr)
    prob.extra["clusters"] = cl
    return prob


def long_video(seed: int = 6, B: int = 1, H: int = 2, N: int = 401408, D: int = 128) -> Problem:
    """The dynamic workload at 401K tokens (3136 blocks per head): one head's
    K/V (205 MB) no longer fits in a 129 MB L2, the regime where the order in
    which query rows run decides K/V reuse (WaveAlign's 401-frame Wan2.1 case)."""
    p = dynamic(seed=seed, B=B, H=H, N=N, D=D)
    p.name = "long_video"
    return p


def spectral_start(seed: int, heads: int, nqb: int) -> np.ndarray:
    """Random starting vectors [heads, nQB, 2] for the subspace iteration."""
    g = _gen(seed)
    return torch.randn((heads, nqb, 2), generator=g, dtype=torch.float64).numpy()


def diag_lists(rows: int, nqb: int):
    """kv_idx [rows, 1] = qb, kv_cnt = 1: each query block attends to its own block."""
    idx = (np.arange(rows) % nqb).astype(np.int32)[:, None]
    return idx, np.ones(rows, np.int32)


def llm(seed: int = 7, B: int = 1, H: int = 32, H_kv: int = 8, N: int = 16384, D: int = 128,
        layer: str = "block", window: int = 575, sinks: int = 64) -> Problem:
    """Language-model prefill shapes (32 query heads over 8 key/value heads,
    causal).  layer "block": every second 256-token block (128-blocks kb
    with floor(kb / 2) even) up to the query block, plus the query's own
    block; layer "window": the blocks that hold some key of the sliding
    window of `window` tokens or of the first `sinks` tokens."""
    g = _gen(seed)
    q = normal_bf16(g, (B, H, N, D))
    k, v = (normal_bf16(g, (B, H_kv, N, D)) for _ in range(2))
    nb = N // BLOCK
    qb = np.arange(nb)[:, None]
    kb = np.arange(nb)[None, :]
    if layer == "block":
        keep = (kb <= qb) & (((kb // 2) % 2 == 0) | (kb == qb))
        w = s_ = 0
    else:
        # rows 128 qb .. 128 qb + 127 see keys (128 qb - window, 128 qb + 127]
        lo = (BLOCK * qb - window + 1) // BLOCK
        keep = ((kb >= lo) & (kb <= qb)) | (kb * BLOCK < sinks)
        w, s_ = window, sinks
    m = np.broadcast_to(keep.astype(np.uint8), (B * H, nb, nb)).reshape(B * H * nb, nb).copy()
    return Problem(f"llm-{layer}", B, H, N, D, q, k, v, mask=m, H_kv=H_kv, causal=True,
                   window=w, sinks=s_)


def llm_window(seed: int = 8, **kw) -> Problem:
    return llm(seed=seed, layer="window", **kw)


def image_gather0(seed: int = 9, B: int = 1, H: int = 24, img_h: int = 128, img_w: int = 128,
                  n_text: int = 512, groups: int = 8, D: int = 128) -> Problem:
    """FLUX.1-dev image layer shape: 24 heads of 128, 512 text tokens ahead of
    a 128 x 128 latent image (2048 x 2048 pixels), N(0,1) bf16 Q/K/V; the
    Gather 0 pattern itself is built by the library's layout call."""
    g = _gen(seed)
    N = n_text + img_h * img_w
    q, k, v = (normal_bf16(g, (B, H, N, D)) for _ in range(3))
    return Problem("image-gather0", B, H, N, D, q, k, v, img_h=img_h, img_w=img_w, n_text=n_text,
                   groups=groups)


CONFIGS = {1: tiny, 2: threshold, 3: scatter, 4: sampled, 5: dynamic, 6: long_video, 7: llm,
           8: llm_window, 9: image_gather0}
CONFIG_NAMES = {
    1: "tiny B1 H2 N2048 D64, Bernoulli(0.25) block mask + diagonal",
    2: "threshold-map mask B1 H12 N32768 D128, T~U(0,1) + frame band, p=0.15",
    3: "Scatter/Gather maps B1 H24 N16384 D128, T=R=128, one block per query block",
    4: "permuted exact top-16 + 8 PPS-sampled blocks B1 H40 N75776 D128",
    5: "dynamic top-k (10-20%) of mean-pooled QK^T block scores, 8 shuffled access clusters, B1 H24 N118784 D128",
    6: "dynamic top-k (10-20%) of mean-pooled QK^T, 8 shuffled access clusters, long video B1 H2 N401408 D128",
    7: "causal block-level layer (every second 256-token block) B1 H32 H_kv8 N16384 D128",
    8: "causal sliding window 575 + 64 sinks B1 H32 H_kv8 N16384 D128",
    9: "INTRA Gather 0 image layer: 512 text + 128x128 image, 16x16 windows, B1 H24 N16896 D128",
}
