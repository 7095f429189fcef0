"""Helpers shared by the GPU parity tests (test code, not product code)."""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

import linear_attention_beam_gb300 as gb
from linear_attention_beam_gb300.decoder import BeamDecoder, pack_weights

DEV = "cuda"

# Tolerances, as max|gpu - oracle| / max|oracle| over a tensor.
TOL_F32 = 1e-5   # fp32 storage run
TOL_BF16 = 2e-3  # bf16 storage, fp32 accumulation, same stored inputs on both sides


def maxrel(g, o) -> float:
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    den = np.abs(o).max()
    return float(np.abs(g - o).max() / den) if den > 0 else float(np.abs(g - o).max())


# Device tensors made by to_dev stay referenced until the test ends, so a
# pointer handed to the library is never freed (and reused) before the
# asynchronous kernel that reads it has run.
_LIVE = []


def to_dev(a, dtype=torch.float32):
    t = torch.as_tensor(np.ascontiguousarray(a)).to(DEV, dtype=dtype)
    _LIVE.append(t)
    return t


def release():
    if _LIVE:
        torch.cuda.synchronize()
        _LIVE.clear()


def dt(wl):
    return gb.BF16 if wl.dtype == "bf16" else gb.F32


def tdt(wl):
    return torch.bfloat16 if wl.dtype == "bf16" else torch.float32


def store(a, wl):
    """Values rounded to the workload's storage type, as float64."""
    import synth
    return synth.to_storage(np.asarray(a, np.float64).astype(np.float32), wl.dtype).astype(np.float64)


def host(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def decoder_for(wl, params, L_max=None, state_path=0):
    w = pack_weights(params.E, params.Wq, params.Wk, params.Wv, params.w_alpha, params.w_beta,
                     params.Wo, dt(wl), DEV)
    return BeamDecoder.for_workload(wl, w, L_max=L_max, state_path=state_path)


def cfg_for(wl, **over) -> gb.Config:
    d = dict(R=wl.R, layers=wl.layers, H=wl.H, d_k=wl.d_k, d_v=wl.d_v, d_model=wl.d_model,
             V=wl.V, T=wl.T, W_max=wl.W_max, L_max=wl.L, dtype=dt(wl), residual=int(wl.residual),
             H_k=wl.Hk)
    d.update(over)
    return gb.Config(**d)


def device_status_clear() -> int:
    torch.cuda.synchronize()
    return gb.load().gdnbeam_device_status(1)
