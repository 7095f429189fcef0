"""BeamDecoder: the decode loop of large-beam GDN decoding over the C ABI.

Holds one gdnbeam context and the device buffers of a decode job. Each method
is one or two ABI calls; all arithmetic runs in the library's CUDA kernels.
Torch provides device memory and streams.

A decode job (OneLA §1.1 and §3: prefill selects the first SID token, then
T-1 decode calls each feed one selection):
    prefill -> select(t=-1) -> [step(t) -> select(t)] for t = 0..T-2 -> paths
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import BF16, F32, Config, Dumps, Footprint, Weights, check, load, ptr, stream_handle

TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


def pack_weights(E, Wq: Sequence, Wk: Sequence, Wv: Sequence, w_alpha: Sequence,
                 w_beta: Sequence, Wo, dtype: int, device) -> Dict[str, torch.Tensor]:
    """Lays weights out as the ABI expects (see gdnbeam_weights).

    W_proj[layer] stacks, row-wise, the query, key and value projections and
    then the decay- and write-gate vectors of that layer.
    """
    td = TORCH_DTYPE[dtype]
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(device=device, dtype=td)
    W_proj = torch.stack([torch.cat([t(Wq[i]), t(Wk[i]), t(Wv[i]), t(w_alpha[i]), t(w_beta[i])])
                          for i in range(len(Wq))]).contiguous()
    return {"E": t(E).contiguous(), "W_proj": W_proj, "W_o": t(Wo).contiguous()}


@dataclass
class DecodeResult:
    parents: List[torch.Tensor]   # per selection [R, W_s] int32
    tokens: List[torch.Tensor]
    cum: List[torch.Tensor]       # per selection [R, W_s] fp32
    sid: torch.Tensor             # [R, W_final, T] int32
    logits: List[torch.Tensor]    # per decode call [R*W_t, V] (storage) — kept only if asked
    lse: List[torch.Tensor]
    dumps: List[Dict[str, torch.Tensor]]


class BeamDecoder:
    def __init__(self, *, R: int, layers: int, H: int, d_k: int, d_v: int, d_model: int, V: int,
                 T: int, W_max: int, L_max: int, dtype: int, residual: bool,
                 weights: Dict[str, torch.Tensor], device="cuda", state_path: int = 0,
                 H_k: int = 0):
        self.lib = load()
        self.cfg = Config(R=R, layers=layers, H=H, d_k=d_k, d_v=d_v, d_model=d_model, V=V, T=T,
                          W_max=W_max, L_max=L_max, dtype=dtype, residual=int(residual),
                          state_path=int(state_path), H_k=int(H_k))
        self.device = torch.device(device)
        self.dtype = dtype
        self.tdtype = TORCH_DTYPE[dtype]
        fp = Footprint()
        check(self.lib.gdnbeam_footprint_of(C.byref(self.cfg), C.byref(fp)), "footprint")
        self.footprint = fp
        self.weights = weights
        self.workspace = torch.empty(fp.workspace_bytes, dtype=torch.uint8, device=self.device)
        w = Weights(E=ptr(weights["E"]), W_proj=ptr(weights["W_proj"]), W_o=ptr(weights["W_o"]))
        h = C.c_void_p()
        check(self.lib.gdnbeam_create(C.byref(self.cfg), C.byref(w), ptr(self.workspace),
                                      fp.workspace_bytes, C.byref(h)), "create")
        self.ctx = h
        W, R_ = W_max, R
        dev = self.device
        # caller-owned buffers of the decode loop
        self.logits = torch.empty(R_ * W, V, dtype=self.tdtype, device=dev)
        self.lse = torch.empty(R_ * W, dtype=torch.float32, device=dev)
        self.root_logits = torch.empty(R_, V, dtype=self.tdtype, device=dev)
        self.root_lse = torch.empty(R_, dtype=torch.float32, device=dev)
        self.sid = torch.empty(R_, W, T, dtype=torch.int32, device=dev)
        self._serve = {}  # per served shape: its buffers and captured graph

    @classmethod
    def for_workload(cls, wl, weights, L_max: Optional[int] = None, device="cuda",
                     state_path: int = 0):
        """state_path 0: shared context + records + replay; 1: FullState baseline;
        2: ReplaySSM baseline."""
        return cls(R=wl.R, layers=wl.layers, H=wl.H, d_k=wl.d_k, d_v=wl.d_v, d_model=wl.d_model,
                   V=wl.V, T=wl.T, W_max=wl.W_max, L_max=L_max or wl.L,
                   dtype=BF16 if wl.dtype == "bf16" else F32, residual=wl.residual,
                   weights=weights, device=device, state_path=state_path, H_k=wl.Hk)

    def __del__(self):
        try:
            if getattr(self, "ctx", None) and self.ctx.value:
                self.lib.gdnbeam_destroy(self.ctx)
                self.ctx = C.c_void_p()
        except Exception:
            pass

    @property
    def variant(self) -> str:
        return self.lib.gdnbeam_variant(self.ctx).decode()

    # ---------------------------------------------------------------- calls
    def prefill(self, prompt: torch.Tensor, stream=None):
        R, L = prompt.shape
        check(self.lib.gdnbeam_prefill_state(self.ctx, ptr(prompt), L, ptr(self.root_logits),
                                             ptr(self.root_lse), stream_handle(stream)), "prefill")
        return self.root_logits, self.root_lse

    def select(self, t: int, W_t: int, W_next: int, logits, lse, cum=None, bias=None,
               out=None, stream=None):
        R = self.cfg.R
        if out is None:
            out = (torch.empty(R, W_next, dtype=torch.int32, device=self.device),
                   torch.empty(R, W_next, dtype=torch.int32, device=self.device),
                   torch.empty(R, W_next, dtype=torch.float32, device=self.device))
        par, tok, cn = out
        check(self.lib.gdnbeam_select(self.ctx, t, W_t, W_next, ptr(logits), ptr(lse), ptr(cum),
                                      ptr(bias), ptr(par), ptr(tok), ptr(cn),
                                      stream_handle(stream)), f"select t={t}")
        return par, tok, cn

    def step(self, t: int, W_t: int, parents, tokens, logits=None, lse=None, dumps=None,
             stream=None):
        n = self.cfg.R * W_t
        logits = self.logits[:n] if logits is None else logits
        lse = self.lse[:n] if lse is None else lse
        d = None
        if dumps is not None:
            d = Dumps()
            for k, v in dumps.items():
                setattr(d, k, ptr(v))
        check(self.lib.gdnbeam_step(self.ctx, t, W_t, ptr(parents), ptr(tokens), ptr(logits),
                                    ptr(lse), C.byref(d) if d is not None else None,
                                    stream_handle(stream)), f"step t={t}")
        return logits, lse

    def get_paths(self, W_final: int, parents, tokens, sid=None, stream=None):
        sid = self.sid[:, :W_final] if sid is None else sid
        if sid.shape[1] != W_final or not sid.is_contiguous():
            sid = torch.empty(self.cfg.R, W_final, self.cfg.T, dtype=torch.int32, device=self.device)
        check(self.lib.gdnbeam_get_paths(self.ctx, W_final, ptr(parents), ptr(tokens), ptr(sid),
                                         stream_handle(stream)), "get_paths")
        return sid

    def read_sctx(self) -> torch.Tensor:
        c = self.cfg
        out = torch.empty(c.R, c.layers, c.H, c.d_v, c.d_k, dtype=torch.float32, device=self.device)
        check(self.lib.gdnbeam_read_sctx(self.ctx, ptr(out), None), "read_sctx")
        return out

    def status(self, stream=None) -> int:
        return self.lib.gdnbeam_status(self.ctx, stream_handle(stream))

    def reset(self, requests: Optional[Sequence[int]] = None):
        """Releases the listed requests' contexts (all when None)."""
        mask = None
        if requests is not None:
            m = np.zeros(self.cfg.R, dtype=np.int32)
            m[list(requests)] = 1
            mask = m.ctypes.data_as(C.POINTER(C.c_int32))
        check(self.lib.gdnbeam_reset(self.ctx, mask), "reset")

    def prefill_requests(self, requests: Sequence[int], prompts: torch.Tensor, stream=None):
        """Prefills only the listed requests (prompt row i for requests[i])
        into their slots; the others keep their contexts and root rows."""
        ids = np.ascontiguousarray(np.asarray(requests, dtype=np.int32))
        count, L = prompts.shape
        check(self.lib.gdnbeam_prefill_requests(
            self.ctx, ids.ctypes.data_as(C.POINTER(C.c_int32)), count, ptr(prompts), L,
            ptr(self.root_logits), ptr(self.root_lse), stream_handle(stream)), "prefill_requests")
        return self.root_logits, self.root_lse

    # ---------------------------------------------------------------- loop
    def decode(self, W: Sequence[int], bias: Optional[torch.Tensor] = None, forced=None,
               keep_logits: bool = False, dump: bool = False, stream=None) -> DecodeResult:
        """Runs root selection, the T-1 decode calls and their selections.

        W[s]: beams kept by selection s. bias: optional [T-1, R, W_max] fp32
        per-parent bias. forced: optional (parents, tokens) lists of device
        int32 [R, W[s]] tensors; when given, every decode call follows them
        (the selections still run and are returned).
        """
        c = self.cfg
        T, R = c.T, c.R
        parents, tokens, cums, logits_k, lse_k, dumps_k = [], [], [], [], [], []
        p, tk, cm = self.select(-1, 1, W[0], self.root_logits, self.root_lse, None, None,
                                stream=stream)
        parents.append(p); tokens.append(tk); cums.append(cm)
        for t in range(T - 1):
            W_t = W[t]
            fp_ = forced[0][t] if forced is not None else parents[t]
            ft = forced[1][t] if forced is not None else tokens[t]
            n = R * W_t
            dd = None
            if dump:
                dd = self._dump_buffers(n)
            lg = torch.empty(n, c.V, dtype=self.tdtype, device=self.device) if keep_logits else None
            ls = torch.empty(n, dtype=torch.float32, device=self.device) if keep_logits else None
            lg, ls = self.step(t, W_t, fp_ if t > 0 else None, ft, lg, ls, dd, stream=stream)
            cum_in = cums[t]
            if forced is not None:
                cum_in = self._forced_cum(t, forced)
            b = None
            if bias is not None:
                b = bias[t, :, :W_t].contiguous()
            p, tk, cm = self.select(t, W_t, W[t + 1], lg, ls, cum_in, b, stream=stream)
            parents.append(p); tokens.append(tk); cums.append(cm)
            if keep_logits:
                logits_k.append(lg); lse_k.append(ls)
            if dump:
                dumps_k.append(dd)
        fp_ = forced[0][T - 1] if forced is not None else parents[T - 1]
        ft = forced[1][T - 1] if forced is not None else tokens[T - 1]
        sid = self.get_paths(W[T - 1], fp_ if T > 1 else None, ft, stream=stream)
        return DecodeResult(parents, tokens, cums, sid, logits_k, lse_k, dumps_k)

    # ---------------------------------------------------------------- serving
    def serve(self, prompts, W: Sequence[int], bias: Optional[torch.Tensor] = None, *,
              graph: bool = True):
        """One batch of requests end to end: prompts (host int32 [R, L]) go to
        the device, then prefill, the root selection, the T-1 decode calls and
        their selections, and the SID paths [R, W[-1], T] and final cumulative
        scores [R, W[-1]] come back to host memory. W and bias as in decode.

        Returns (sid, cum) as pinned host tensors owned by the decoder and
        overwritten by the next call of the same shape; the call returns once
        they hold the results, after checking the device error word.

        With graph=True the sequence, its two host copies included, is
        captured into a CUDA graph the first time a (prompt length, W, bias)
        shape is served (after one ordinary run of it) and replayed from then
        on: one graph launch instead of some thirty kernel launches, with the
        gaps between dependent kernels gone. Prompts and bias are first copied
        into the buffers the captured work reads."""
        c = self.cfg
        W = tuple(int(w) for w in W)
        prompts = torch.as_tensor(prompts)
        if prompts.device.type != "cpu" or prompts.dim() != 2 or prompts.shape[0] != c.R:
            raise ValueError("prompts: host tensor [R, L]")
        if len(W) != c.T or max(W) > c.W_max:
            raise ValueError("W: one width per selection, at most W_max")
        key = (int(prompts.shape[1]), W, bias is not None)
        st = self._serve.get(key)
        fresh = st is None
        if fresh:
            st = self._serve_buffers(key[0], W, bias is not None)
            self._serve[key] = st
        st["h_prompt"].copy_(prompts)
        stream = st["stream"]
        with torch.cuda.stream(stream):
            if bias is not None:
                for t in range(c.T - 1):
                    st["bias"][t].copy_(bias[t, :, :W[t]], non_blocking=True)
            if not graph:
                self._serve_run(st, W, stream)
            elif fresh or st["graph"] is None:
                # one ordinary run (first-use set-up, the results of this
                # call), then the capture
                self._serve_run(st, W, stream)
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    self._serve_run(st, W, stream)
                st["graph"] = g
            else:
                st["graph"].replay()
        check(self.status(stream), "serve")
        return st["h_sid"], st["h_cum"]

    def _serve_buffers(self, L: int, W: Sequence[int], with_bias: bool):
        c = self.cfg
        dev = self.device
        T, R = c.T, c.R
        i32 = dict(dtype=torch.int32, device=dev)
        return {
            "h_prompt": torch.empty(R, L, dtype=torch.int32).pin_memory(),
            "d_prompt": torch.empty(R, L, **i32),
            "sel": [(torch.empty(R, W[s], **i32), torch.empty(R, W[s], **i32),
                     torch.empty(R, W[s], dtype=torch.float32, device=dev)) for s in range(T)],
            "bias": ([torch.empty(R, W[t], dtype=torch.float32, device=dev) for t in range(T - 1)]
                     if with_bias else None),
            "d_sid": torch.empty(R, W[T - 1], T, **i32),
            "h_sid": torch.empty(R, W[T - 1], T, dtype=torch.int32).pin_memory(),
            "h_cum": torch.empty(R, W[T - 1], dtype=torch.float32).pin_memory(),
            "stream": torch.cuda.Stream(dev),
            "graph": None,
        }

    def _serve_run(self, st, W: Sequence[int], stream):
        T = self.cfg.T
        st["d_prompt"].copy_(st["h_prompt"], non_blocking=True)
        self.prefill(st["d_prompt"], stream=stream)
        par, tok, cum = self.select(-1, 1, W[0], self.root_logits, self.root_lse, out=st["sel"][0],
                                    stream=stream)
        for t in range(T - 1):
            lg, ls = self.step(t, W[t], par if t else None, tok, stream=stream)
            b = st["bias"][t] if st["bias"] is not None else None
            par, tok, cum = self.select(t, W[t], W[t + 1], lg, ls, cum, b, out=st["sel"][t + 1],
                                        stream=stream)
        sid = self.get_paths(W[T - 1], par if T > 1 else None, tok, sid=st["d_sid"], stream=stream)
        st["h_sid"].copy_(sid, non_blocking=True)
        st["h_cum"].copy_(cum, non_blocking=True)

    def _forced_cum(self, t, forced):
        # under a forced lineage the cumulative scores of the forced beams are
        # supplied by the caller alongside the lineage (forced[2][t]), if given
        if len(forced) > 2 and forced[2] is not None:
            return forced[2][t]
        return None

    def _dump_buffers(self, n: int) -> Dict[str, torch.Tensor]:
        c = self.cfg
        f = lambda *s: torch.zeros(*s, dtype=torch.float32, device=self.device)
        hk = c.H_k or c.H
        return {"q": f(c.layers, n, hk * c.d_k), "k": f(c.layers, n, hk * c.d_k),
                "v": f(c.layers, n, c.H * c.d_v), "alpha": f(c.layers, n, c.H),
                "beta": f(c.layers, n, c.H), "delta": f(c.layers, n, c.H * c.d_v),
                "o": f(c.layers, n, c.H * c.d_v), "logits": f(n, c.V)}
