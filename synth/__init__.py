"""Seeded synthetic inputs for large-beam Gated DeltaNet decoding.

This module is shared by the CPU oracle and by the harness that drives the
CUDA library. It holds no step of the decoding method: only the workload
shapes and the random draws that fill them (embedding table, projection
weights, gate vectors, codebook head, prompts, per-parent score bias and
forced beam lineages), rounded to the storage precision both sides consume.

Recipe (stated once here so both sides read the same numbers):
  * generator: numpy PCG64 seeded with the workload's seed;
  * parameter stream PCG64(seed), draw order: E, then per layer (W_q, W_k,
    W_v, w_alpha, w_beta), then W_o; prompt tokens from PCG64([seed, 1]);
    per-parent bias from PCG64([seed, 2]); forced lineages from
    PCG64([seed, 3, k]);
  * E[V, d_model] ~ N(0, 1); W_q, W_k [H*d_k, d_model], W_v [H*d_v, d_model]
    and w_alpha, w_beta [H, d_model] ~ N(0, 1/d_model) (fan-in scaled);
    W_o [V, F] ~ N(0, 1/F) with F the width of the feature the head reads;
  * prompt tokens uniform over [0, V);
  * bias (skewed workload only) ~ N(0, bias_var) per (decode call, request,
    parent beam);
  * bf16 workloads: every stored parameter is rounded to bf16 (round to
    nearest even) and kept as float32 holding bf16-representable values, so
    both sides see bit-identical inputs.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, Optional, Sequence, Tuple

import numpy as np


@dataclass(frozen=True)
class Workload:
    """Shape of one large-beam GDN decode job.

    W lists the beam counts after each selection: W[0] is the number of beams
    the root selection keeps from the prefill row, W[t] (t >= 1) the number
    kept after decode call t-1. Decode call t (0 <= t <= T-2) therefore runs
    on W[t] beams per request, and the final beam set has W[T-1] beams.
    """

    name: str
    R: int                 # requests
    layers: int            # stacked GDN layers
    H: int                 # heads
    d_k: int
    d_v: int
    d_model: int
    V: int                 # codebook size
    T: int                 # SID length = number of selections
    W: Tuple[int, ...]     # beams after each selection (len T)
    L: int                 # prompt length
    dtype: str             # "f32" or "bf16" storage
    seed: int
    residual: bool = False # residual stream + RMSNorm glue between layers
    bias_var: float = 0.0  # variance of the per-parent score bias (0 = none)
    H_k: int = 0           # key heads (0: one per value head); H is a multiple

    @property
    def Hk(self) -> int:
        """Key (query/key) heads; value head h reads key head h // (H // Hk)."""
        return self.H_k or self.H

    @property
    def W_max(self) -> int:
        return max(self.W)

    @property
    def feat_dim(self) -> int:
        """Width of the feature the codebook head reads."""
        return self.d_model if self.residual else self.H * self.d_v

    @property
    def beam_steps(self) -> int:
        """Beams advanced through all decode calls, over all requests."""
        return sum(self.R * self.W[t] for t in range(self.T - 1))

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _sched(first: int, rest: int, T: int, V: int) -> Tuple[int, ...]:
    w = [min(first, V)]
    for _ in range(1, T):
        w.append(min(rest, w[-1] * V))
    return tuple(w)


# The five workloads. Sizes follow the decode shape of the OneLA paper
# (long shared prompt, short SID suffix, beam width much larger than T) and
# its largest operator geometry (16 heads, d_k = d_v = 128, W up to 512).
TINY = Workload("tiny_f32", R=1, layers=1, H=1, d_k=16, d_v=16, d_model=16,
                V=16, T=3, W=_sched(8, 8, 3, 16), L=32, dtype="f32", seed=0)
SINGLE = Workload("single_w256", R=1, layers=1, H=16, d_k=128, d_v=128,
                  d_model=2048, V=8192, T=3, W=_sched(256, 256, 3, 8192),
                  L=4096, dtype="bf16", seed=1)
BATCHED = Workload("batched_r64_w512", R=64, layers=1, H=16, d_k=128, d_v=128,
                   d_model=2048, V=8192, T=4, W=_sched(512, 512, 4, 8192),
                   L=2048, dtype="bf16", seed=2)
DEEP = Workload("deep4_w1024", R=32, layers=4, H=8, d_k=128, d_v=128,
                d_model=1024, V=4096, T=4, W=_sched(1024, 1024, 4, 4096),
                L=8192, dtype="bf16", seed=3, residual=True)
SKEWED = Workload("skewed_r128", R=128, layers=1, H=16, d_k=128, d_v=128,
                  d_model=2048, V=8192, T=4, W=(256, 1024, 1024, 1024),
                  L=2048, dtype="bf16", seed=4, bias_var=4.0)

# Grouped key heads on the tensor-core path: 8 value heads reading 4 key heads.
GQA = Workload("gqa_w128", R=2, layers=1, H=8, d_k=128, d_v=128, d_model=1024, V=2048, T=3,
               W=(128, 128, 128), L=256, dtype="bf16", seed=4, H_k=4)

WORKLOADS: Dict[str, Workload] = {w.name: w for w in (TINY, SINGLE, BATCHED, DEEP, SKEWED, GQA)}

# Operator sweep (OneLA §3, operator experiments; results in §4.2): R in
# {4, 8, 16}, W in {128, 256, 512}, T = 2..6 decode calls (there T = O - 1,
# so the replay depths of a shape are 0 .. T-1), and nine recurrent
# geometries spanning H_K 4-32, H_V 4-64, K 128-256, V 128-512: 405 shapes.
# The pages give only those ranges and the largest "Qwen" geometry
# (H_K = H_V = 16, K = V = 128); the other eight below are chosen to reach
# the ends of every range, with grouped key heads and wide heads.
SWEEP_R = (4, 8, 16)
SWEEP_W = (128, 256, 512)
SWEEP_T = (2, 3, 4, 5, 6)
SWEEP_GEOMETRIES = (  # (H_K, H_V, K, V)
    (16, 16, 128, 128),
    (4, 4, 128, 128),
    (32, 32, 128, 128),
    (8, 16, 128, 128),
    (16, 64, 128, 128),
    (8, 8, 256, 256),
    (4, 8, 256, 256),
    (8, 8, 128, 512),
    (4, 16, 256, 512),
)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float values to the nearest bf16 (ties to even); float32 result."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    return round_bf16(x) if dtype == "bf16" else x


@dataclass
class Params:
    E: np.ndarray                    # [V, d_model]
    Wq: Sequence[np.ndarray]         # per layer [H*d_k, d_model]
    Wk: Sequence[np.ndarray]
    Wv: Sequence[np.ndarray]         # per layer [H*d_v, d_model]
    w_alpha: Sequence[np.ndarray]    # per layer [H, d_model]
    w_beta: Sequence[np.ndarray]
    Wo: np.ndarray                   # [V, feat_dim]


def make_params(wl: Workload) -> Params:
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    st = lambda a: to_storage(a, wl.dtype)
    E = st(rng.standard_normal((wl.V, wl.d_model), dtype=np.float32))
    s_in = np.float32(1.0 / np.sqrt(wl.d_model))
    Wq, Wk, Wv, wa, wb = [], [], [], [], []
    for _ in range(wl.layers):
        Wq.append(st(rng.standard_normal((wl.Hk * wl.d_k, wl.d_model), dtype=np.float32) * s_in))
        Wk.append(st(rng.standard_normal((wl.Hk * wl.d_k, wl.d_model), dtype=np.float32) * s_in))
        Wv.append(st(rng.standard_normal((wl.H * wl.d_v, wl.d_model), dtype=np.float32) * s_in))
        wa.append(st(rng.standard_normal((wl.H, wl.d_model), dtype=np.float32) * s_in))
        wb.append(st(rng.standard_normal((wl.H, wl.d_model), dtype=np.float32) * s_in))
    s_o = np.float32(1.0 / np.sqrt(wl.feat_dim))
    Wo = st(rng.standard_normal((wl.V, wl.feat_dim), dtype=np.float32) * s_o)
    return Params(E, Wq, Wk, Wv, wa, wb, Wo)


def make_prompt(wl: Workload) -> np.ndarray:
    """Prompt tokens [R, L] int32."""
    rng = np.random.Generator(np.random.PCG64([wl.seed, 1]))
    return rng.integers(0, wl.V, size=(wl.R, wl.L), dtype=np.int64).astype(np.int32)


def make_bias(wl: Workload) -> Optional[np.ndarray]:
    """Per-parent score bias [T-1, R, W_max] float32, or None."""
    if wl.bias_var <= 0.0:
        return None
    rng = np.random.Generator(np.random.PCG64([wl.seed, 2]))
    b = rng.standard_normal((wl.T - 1, wl.R, wl.W_max)) * np.sqrt(wl.bias_var)
    return b.astype(np.float32)


def random_lineage(wl: Workload, seed: int) -> Tuple[list, list]:
    """A random but valid beam lineage for every request.

    Returns (parents, tokens): parents[s] and tokens[s] are int32 [R, W[s]]
    for selection s = 0..T-1; parents[0] is all zero (the root row). Used to
    force both sides along the same beam tree where the oracle's own
    selection is not computed (requests outside a sampled subset).
    """
    rng = np.random.Generator(np.random.PCG64([wl.seed, 3, seed]))
    parents, tokens = [], []
    prev = 1
    for s in range(wl.T):
        n = wl.W[s]
        parents.append(rng.integers(0, prev, size=(wl.R, n)).astype(np.int32))
        tokens.append(rng.integers(0, wl.V, size=(wl.R, n)).astype(np.int32))
        prev = n
    parents[0][:] = 0
    return parents, tokens


def tiny_workload(d=4, V=3, T=3, W=(3, 9, 27), H=1, layers=1, d_model=None,
                  residual=False, seed=11, L=5, dtype="f32", R=1, H_k=0, d_v=None) -> Workload:
    """Small shapes for brute-force checks (d_v defaults to d = d_k)."""
    d_v = d_v or d
    d_model = d_model or H * d_v
    return Workload(f"tiny_d{d}_V{V}_T{T}", R=R, layers=layers, H=H, d_k=d, d_v=d_v,
                    d_model=d_model, V=V, T=T, W=tuple(W), L=L, dtype=dtype,
                    seed=seed, residual=residual, H_k=H_k)
