"""Stage checks of one decode call on the values the GPU itself stored.

Test code. The end-to-end comparison against the fp64 oracle inherits every
bf16 rounding the GPU makes between stages; here each stage is instead fed,
through the oracle's own functions, exactly the stored values the kernel
read, so the bound that applies is the kernels' own arithmetic (fp32
accumulation over bf16 or fp32 operands):

  projections  oracle.gdn_inputs on the stored layer input (the embedding row,
               or the RMS-normalised residual stream rounded to storage);
  replay       oracle.step_from_records on S_ctx as read back (fp32) and the
               stored q, k, v, alpha, beta of the call plus the stored records
               (k_j, delta_j, alpha_j) of the beam's ancestors, found by
               walking the parent maps (OneLA §2.3 eqs. 6-8 against the
               FullState step of §1.2 eq. 3);
  logits       oracle.codebook_logits and log_normalizer on the stored
               feature (concat_h o, or RMSNorm of the residual stream).

The GPU's fp32 dumps are its values before storage rounding; what it stored
is that value rounded to the storage type (round to nearest even), which is
how the stored inputs are rebuilt here. Only numpy, the oracle and the seeded
generators are used, so the helper itself is checked on the CPU against the
oracle's own decode (tests/test_stored_parity_host.py).
"""
from __future__ import annotations

from typing import Dict, List, Sequence

import numpy as np

import oracle
import synth

F64 = np.float64
FIELDS = ("q", "k", "v", "alpha", "beta", "delta", "o")


def stored(a, wl) -> np.ndarray:
    """A value as the GPU stored it: fp32, rounded to bf16 on bf16 workloads."""
    return synth.to_storage(np.asarray(a, F64).astype(np.float32), wl.dtype).astype(F64)


class ErrMax:
    """Per tensor max|gpu - oracle| / max|oracle|, accumulated over rows."""

    def __init__(self):
        self.num: Dict[str, float] = {}
        self.den: Dict[str, float] = {}

    def add(self, key, gpu, ref):
        g = np.asarray(gpu, F64)
        r = np.asarray(ref, F64)
        self.num[key] = max(self.num.get(key, 0.0), float(np.abs(g - r).max()))
        self.den[key] = max(self.den.get(key, 0.0), float(np.abs(r).max()))

    def add_scaled(self, key, err, scale):
        self.num[key] = max(self.num.get(key, 0.0), float(err))
        self.den[key] = max(self.den.get(key, 0.0), float(scale))

    def result(self) -> Dict[str, float]:
        return {k: (self.num[k] / self.den[k] if self.den[k] > 0 else self.num[k]) for k in self.num}


def call_rows(wl, dumps: Dict[str, np.ndarray], n: int) -> Dict[str, np.ndarray]:
    """Reshapes one request's dump rows of a call to per-head arrays:
    q, k [layers, n, Hk, d_k]; v, delta, o [layers, n, H, d_v];
    alpha, beta [layers, n, H]; logits [n, V]."""
    L, H, Hk, dk, dv = wl.layers, wl.H, wl.Hk, wl.d_k, wl.d_v
    shape = {"q": (L, n, Hk, dk), "k": (L, n, Hk, dk), "v": (L, n, H, dv),
             "delta": (L, n, H, dv), "o": (L, n, H, dv), "alpha": (L, n, H), "beta": (L, n, H),
             "logits": (n, wl.V)}
    return {f: np.asarray(dumps[f], F64).reshape(shape[f]) for f in shape if f in dumps}


def stage_errors(wl, params, S_ctx: np.ndarray, calls: Sequence[Dict[str, np.ndarray]],
                 anc: np.ndarray, t: int, beams: Sequence[int], chunk: int = 32) -> Dict[str, float]:
    """Errors of decode call t's stages for the given beams of one request.

    S_ctx [layers, H, d_v, d_k] as read back; calls[j] (j <= t) holds the
    request's rows of call j: the fields of call_rows plus "tokens" [n_j]
    and "lse" [n_j]; anc [n_t, t] the ancestor slots of call t's beams.
    """
    err = ErrMax()
    beams = list(beams)
    c = calls[t]
    for s0 in range(0, len(beams), chunk):
        bb = np.asarray(beams[s0:s0 + chunk])
        m = len(bb)
        x = params.E[np.asarray(c["tokens"])[bb]].astype(F64)   # [m, d_model]
        feat = None
        for layer in range(wl.layers):
            # projections on the stored layer input
            u = stored(oracle.rms_normalize(x), wl) if wl.residual else x
            q, k, v, a, b = oracle.gdn_inputs(wl, params, layer, u)
            for f, ref in (("q", q), ("k", k), ("v", v), ("alpha", a), ("beta", b)):
                err.add(f, c[f][layer][bb], ref)
            # replay on the stored step inputs and the ancestors' stored records
            recs = []
            for j in range(t):
                sj = anc[bb, j]
                recs.append((calls[j]["alpha"][layer][sj], stored(calls[j]["delta"][layer][sj], wl),
                             oracle.per_value_head(wl, stored(calls[j]["k"][layer][sj], wl))))
            delta, o = oracle.step_from_records(
                S_ctx[layer], recs,
                oracle.per_value_head(wl, stored(c["q"][layer][bb], wl)),
                oracle.per_value_head(wl, stored(c["k"][layer][bb], wl)),
                stored(c["v"][layer][bb], wl), c["alpha"][layer][bb], c["beta"][layer][bb])
            err.add("delta", c["delta"][layer][bb], delta)
            err.add("o", c["o"][layer][bb], o)
            if wl.residual:
                x = x + c["o"][layer][bb].reshape(m, -1)
            else:
                feat = stored(c["o"][layer][bb].reshape(m, -1), wl)
        if wl.residual:
            feat = stored(oracle.rms_normalize(x), wl)
        z = oracle.codebook_logits(params, feat)
        lse = oracle.log_normalizer(z)
        err.add("logits", c["logits"][bb], z)
        err.add_scaled("lse", np.abs(np.asarray(c["lse"], F64)[bb] - lse).max(), np.abs(z).max())
    return err.result()


def selection_matches(z_stored, lse, cum, W_next: int, bias, parents, tokens, cum_next) -> None:
    """The GPU's selection of one request equals the oracle's contract on the
    same stored logits, lse, cumulative scores and bias (bit for bit)."""
    z32 = np.asarray(z_stored, np.float32)
    n = z32.shape[0]
    c32 = np.zeros(n, np.float32) if cum is None else np.asarray(cum, np.float32)
    b32 = None if bias is None else np.asarray(bias, np.float32)
    p, tk, s = oracle.select_top(z32, np.asarray(lse, np.float32), c32, W_next, b32)
    np.testing.assert_array_equal(np.asarray(parents), p)
    np.testing.assert_array_equal(np.asarray(tokens), tk)
    np.testing.assert_array_equal(np.asarray(cum_next, np.float32), s)


def ancestry(parents: List[np.ndarray], t: int) -> np.ndarray:
    return oracle.ancestry_slots(parents, t)
