"""FullState Gated DeltaNet large-beam decoder in float64 — the CPU oracle.

TEST INFRASTRUCTURE. Only the tests, the package smoke check and the bench's
CPU-baseline / reference leg may import this module; the product path never
does. It shares no code with the CUDA library: it reads parameters and prompts
from the seeded `synth` module and nothing else.

It is the plain definition the GPU method must reproduce: every beam carries
its own d_v x d_k recurrent state, advanced by the GDN recurrence, copied when
the beam tree is reordered. Sources are named by page title:

  OneLA   "OneLA: Scaling Linear-Attention Decoding to Large Beams in
           Generative Recommendation" (paper-archivist review page)
  RecoGEM "RecoGEM: A Serving System for Production-Scale Generative
           Recommendation" (conceptio page)

Readings taken where the pages are silent (each also tested):
  * prefill starts from S = 0;
  * q and k are L2-normalised with eps = 1e-6 inside the square root, q is not
    scaled by 1/sqrt(d);
  * alpha = exp(-softplus(w_alpha . x)), beta = sigmoid(w_beta . x);
  * single-layer workloads read logits off concat_h(o); stacked workloads use
    a residual stream with unit-gain RMSNorm (eps = 1e-6) before every layer
    and before the codebook head;
  * T counts selections: the prefill row feeds selection 0 and decode calls
    t = 0..T-2 each feed selection t+1;
  * the per-parent bias is added to the parent's cumulative score;
  * equal scores are ordered by lower flat index b*V + v.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
from scipy.special import expit, logsumexp

F64 = np.float64
F32 = np.float32
EPS = 1e-6


# --------------------------------------------------------------------------
# Per-token GDN inputs (OneLA §1.2, eq. 3 and the tiny workload's recipe)
# --------------------------------------------------------------------------

def l2_normalize(y: np.ndarray) -> np.ndarray:
    """y / sqrt(sum(y^2) + eps) over the last axis."""
    return y / np.sqrt(np.sum(y * y, axis=-1, keepdims=True) + EPS)


def rms_normalize(x: np.ndarray) -> np.ndarray:
    """Unit-gain RMSNorm over the last axis: x / sqrt(mean(x^2) + eps)."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + EPS)


def decay_gate(z: np.ndarray) -> np.ndarray:
    """alpha = exp(-softplus(z)); softplus(z) = log(1 + e^z), evaluated stably."""
    return np.exp(-np.logaddexp(0.0, z))


def write_gate(z: np.ndarray) -> np.ndarray:
    """beta = sigmoid(z)."""
    return expit(z)


def gdn_inputs(wl, params, layer: int, u: np.ndarray):
    """Projections of layer inputs u [n, d_model] for every head.

    Returns q_hat, k_hat [n, Hk, d_k] (one per key head), v [n, H, d_v],
    alpha, beta [n, H] (one per value head).
    """
    n = u.shape[0]
    u = np.asarray(u, dtype=F64)
    q = u @ params.Wq[layer].astype(F64).T
    k = u @ params.Wk[layer].astype(F64).T
    v = u @ params.Wv[layer].astype(F64).T
    za = u @ params.w_alpha[layer].astype(F64).T
    zb = u @ params.w_beta[layer].astype(F64).T
    q_hat = l2_normalize(q.reshape(n, wl.Hk, wl.d_k))
    k_hat = l2_normalize(k.reshape(n, wl.Hk, wl.d_k))
    return q_hat, k_hat, v.reshape(n, wl.H, wl.d_v), decay_gate(za), write_gate(zb)


def per_value_head(wl, x: np.ndarray) -> np.ndarray:
    """Key-head arrays [n, Hk, d_k] seen from the value heads [n, H, d_k]:
    grouped query attention with consecutive value heads sharing a key head
    (value head h reads key head h // (H // Hk))."""
    return np.repeat(x, wl.H // wl.Hk, axis=1)


# --------------------------------------------------------------------------
# The recurrence (OneLA §1.2 eq. 3; the record of §2.2 eqs. 4-5)
# --------------------------------------------------------------------------

def gdn_transition(S, q, k, v, alpha, beta):
    """One GDN transition on a batch of states.

    S [..., d_v, d_k]; q, k [..., d_k]; v [..., d_v]; alpha, beta [...].
    S_next = alpha*S + beta*(v - alpha*S k) k^T and o = S_next q (eq. 3).
    Also returns the bracketed correction delta = beta*(v - alpha*S k), the
    vector OneLA stores in a transition record (eq. 4).
    """
    Sk = np.einsum("...ij,...j->...i", S, k)
    correction = v - alpha[..., None] * Sk
    S_next = alpha[..., None, None] * S + beta[..., None, None] * np.einsum(
        "...i,...j->...ij", correction, k)
    o = np.einsum("...ij,...j->...i", S_next, q)
    delta = beta[..., None] * correction
    return S_next, delta, o


def state_from_records(S_ctx, records):
    """Materialise a beam's state from the shared context state and its chain.

    records: sequence of (alpha [...], delta [..., d_v], k [..., d_k]) in
    depth order; each applies S <- alpha*S + delta k^T (eq. 4).
    """
    S = np.array(S_ctx, dtype=F64, copy=True)
    for a, d, k in records:
        S = np.asarray(a, F64)[..., None, None] * S + np.einsum(
            "...i,...j->...ij", np.asarray(d, F64), np.asarray(k, F64))
    return S


def step_from_records(S_ctx, records, q, k, v, alpha, beta):
    """FullState step of a beam whose parent chain is given as records.

    The parent state is rebuilt explicitly (eq. 4 applied along the chain),
    then eq. 3 is applied. Returns (delta, o). Used to check the GPU's
    replay kernel on exactly the stored values it reads.
    """
    S_par = state_from_records(S_ctx, records)
    _, delta, o = gdn_transition(S_par, np.asarray(q, F64), np.asarray(k, F64),
                                 np.asarray(v, F64), np.asarray(alpha, F64),
                                 np.asarray(beta, F64))
    return delta, o


def prefill_scan(q, k, v, alpha, beta):
    """Run eq. 3 over a prompt from S = 0 for every head.

    q, k [L, H, d_k]; v [L, H, d_v]; alpha, beta [L, H].
    Returns (S after the last token [H, d_v, d_k], o [L, H, d_v]).
    """
    L, H, dk = q.shape
    dv = v.shape[-1]
    S = np.zeros((H, dv, dk), dtype=F64)
    o = np.empty((L, H, dv), dtype=F64)
    for i in range(L):
        S, _, o[i] = gdn_transition(S, q[i], k[i], v[i], alpha[i], beta[i])
    return S, o


# --------------------------------------------------------------------------
# Codebook head and log-softmax
# --------------------------------------------------------------------------

def codebook_logits(params, feat: np.ndarray) -> np.ndarray:
    """z = W_o . feat for rows of feat [n, F] -> [n, V]."""
    return np.asarray(feat, F64) @ params.Wo.astype(F64).T


def log_normalizer(z: np.ndarray) -> np.ndarray:
    """lse = log sum_v exp(z_v) per row."""
    return logsumexp(np.asarray(z, F64), axis=-1)


def layer_feature(wl, x_or_o: np.ndarray) -> np.ndarray:
    """Feature the codebook head reads: RMSNorm(x) for stacked workloads,
    concat_h(o) for single-layer ones."""
    return rms_normalize(x_or_o) if wl.residual else x_or_o


# --------------------------------------------------------------------------
# Selection contract (OneLA §1.1 global top-k; RecoGEM §4.3)
# --------------------------------------------------------------------------

def scores_f32(z32, lse32, cum32, bias32=None):
    """s = fl32(cum' + fl32(z - lse)), cum' = fl32(cum + bias), in IEEE fp32."""
    z32 = np.asarray(z32, F32)
    lse32 = np.asarray(lse32, F32)
    cum32 = np.asarray(cum32, F32)
    cum_p = cum32 if bias32 is None else (cum32 + np.asarray(bias32, F32)).astype(F32)
    return (cum_p[:, None] + (z32 - lse32[:, None]).astype(F32)).astype(F32)


def select_top(z32, lse32, cum32, W_next: int, bias32=None):
    """Global top-W_next of all n x V candidate scores of one request.

    Order: score descending, then flat index b*V + v ascending. Returns
    parents [W_next] (row b), tokens [W_next] (v) and the kept scores.
    """
    s = scores_f32(z32, lse32, cum32, bias32)
    n, V = s.shape
    flat = np.arange(n * V, dtype=np.int64)
    order = np.lexsort((flat, -s.ravel()))[:W_next]
    return ((order // V).astype(np.int32), (order % V).astype(np.int32),
            s.ravel()[order].astype(F32))


def kept_scores_f32(z, dtype: str):
    """Round logits to the storage precision the selection is taken in.

    The GPU accumulates in fp32 and stores z in the workload's storage type;
    the oracle's fp64 z is brought through fp32 to the same type.
    """
    z32 = np.asarray(z, dtype=F64).astype(F32)
    if dtype == "bf16":
        u = z32.view(np.uint32)
        lsb = (u >> np.uint32(16)) & np.uint32(1)
        z32 = ((u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)).view(F32)
    return z32


# --------------------------------------------------------------------------
# Ancestry (by walking parent maps, not by the eq. 9 recursion)
# --------------------------------------------------------------------------

def ancestry_slots(parents: Sequence[np.ndarray], t: int) -> np.ndarray:
    """Slots of beam b's ancestors at decode call t: h[b, j] for j < t.

    parents[s] maps each beam after selection s to its row at the previous
    call (s >= 1). The ancestor of b at call j is found by following the
    parent maps back from call t.
    """
    n_t = len(parents[t])
    h = np.zeros((n_t, t), dtype=np.int32)
    for b in range(n_t):
        cur = b
        for j in range(t - 1, -1, -1):
            cur = int(parents[j + 1][cur])
            h[b, j] = cur
    return h


def token_paths(parents: Sequence[np.ndarray], tokens: Sequence[np.ndarray]) -> np.ndarray:
    """SID sequence of every final beam, [W_final, T], by walking back."""
    T = len(tokens)
    n = len(tokens[-1])
    sid = np.zeros((n, T), dtype=np.int32)
    for b in range(n):
        cur = b
        for s in range(T - 1, -1, -1):
            sid[b, s] = tokens[s][cur]
            if s > 0:
                cur = int(parents[s][cur])
    return sid


# --------------------------------------------------------------------------
# The decoder
# --------------------------------------------------------------------------

@dataclass
class CallTrace:
    """Everything decode call t computed for one request (fp64 unless noted)."""
    tokens: np.ndarray                 # [n] input tokens of the beams
    q: List[np.ndarray] = field(default_factory=list)      # per layer [n,Hk,dk]
    k: List[np.ndarray] = field(default_factory=list)
    v: List[np.ndarray] = field(default_factory=list)
    alpha: List[np.ndarray] = field(default_factory=list)  # per layer [n,H]
    beta: List[np.ndarray] = field(default_factory=list)
    delta: List[np.ndarray] = field(default_factory=list)  # per layer [n,H,dv]
    o: List[np.ndarray] = field(default_factory=list)
    feat: Optional[np.ndarray] = None  # [n, F]
    z: Optional[np.ndarray] = None     # [n, V]
    lse: Optional[np.ndarray] = None   # [n]


@dataclass
class RequestTrace:
    S_ctx: np.ndarray                  # [layers, H, dv, dk]
    root_feat: np.ndarray              # [F]
    root_z: np.ndarray                 # [V]
    root_lse: float
    parents: List[np.ndarray]          # per selection s: [W[s]]
    tokens: List[np.ndarray]
    cum: List[np.ndarray]              # fp32 kept scores per selection
    calls: List[CallTrace]
    sid: np.ndarray                    # [W[T-1], T]


def prefill(wl, params, prompt: np.ndarray):
    """Compress one request's prompt into S_ctx and its last-position feature.

    Returns (S_ctx [layers, H, dv, dk], feature [F]).
    """
    x = params.E[np.asarray(prompt)].astype(F64)
    S_ctx = np.zeros((wl.layers, wl.H, wl.d_v, wl.d_k), dtype=F64)
    o_last = None
    for layer in range(wl.layers):
        u = rms_normalize(x) if wl.residual else x
        q, k, v, a, b = gdn_inputs(wl, params, layer, u)
        S_ctx[layer], o = prefill_scan(per_value_head(wl, q), per_value_head(wl, k), v, a, b)
        if wl.residual:
            x = x + o.reshape(len(x), wl.H * wl.d_v)
        else:
            assert wl.layers == 1, "without the residual glue only one layer is defined"
            o_last = o[-1].reshape(wl.H * wl.d_v)
    feat = rms_normalize(x[-1]) if wl.residual else o_last
    return S_ctx, feat


def decode_request(wl, params, prompt: np.ndarray, bias: Optional[np.ndarray] = None,
                   forced=None, context=None) -> RequestTrace:
    """Large-beam FullState decode of one request.

    bias: [T-1, W_max] per-parent bias for this request, or None.
    forced: optional (parents, tokens) lists indexed by selection; when given,
    the beam tree follows them instead of the oracle's own selections (both
    sides then run on the same lineage). Scores kept are still the oracle's.
    context: optional (S_ctx, root feature) from an earlier prefill() of the
    same prompt, to skip recomputing it.
    """
    S_ctx, root_feat = context if context is not None else prefill(wl, params, prompt)
    root_z = codebook_logits(params, root_feat[None, :])[0]
    root_lse = float(log_normalizer(root_z[None, :])[0])

    z32 = kept_scores_f32(root_z[None, :], wl.dtype)
    lse32 = np.array([root_lse], dtype=F32)
    par, tok, cum = select_top(z32, lse32, np.zeros(1, F32), wl.W[0])
    if forced is not None:
        par, tok = forced[0][0].astype(np.int32), forced[1][0].astype(np.int32)
        cum = scores_f32(z32, lse32, np.zeros(1, F32))[par, tok]
    parents, tokens, cums = [par], [tok], [cum]

    # Per-beam full states: [n, layers, H, dv, dk], all starting at S_ctx.
    n = wl.W[0]
    states = np.broadcast_to(S_ctx, (n,) + S_ctx.shape).copy()
    calls: List[CallTrace] = []
    for t in range(wl.T - 1):
        tr = CallTrace(tokens=tokens[t].copy())
        x = params.E[tokens[t]].astype(F64)
        feat_in = x
        for layer in range(wl.layers):
            u = rms_normalize(x) if wl.residual else x
            q, k, v, a, b = gdn_inputs(wl, params, layer, u)
            states[:, layer], delta, o = gdn_transition(
                states[:, layer], per_value_head(wl, q), per_value_head(wl, k), v, a, b)
            tr.q.append(q); tr.k.append(k); tr.v.append(v)
            tr.alpha.append(a); tr.beta.append(b)
            tr.delta.append(delta); tr.o.append(o)
            if wl.residual:
                x = x + o.reshape(n, wl.H * wl.d_v)
            else:
                feat_in = o.reshape(n, wl.H * wl.d_v)
        tr.feat = layer_feature(wl, x if wl.residual else feat_in)
        tr.z = codebook_logits(params, tr.feat)
        tr.lse = log_normalizer(tr.z)
        calls.append(tr)

        zs = kept_scores_f32(tr.z, wl.dtype)
        ls = tr.lse.astype(F32)
        bs = None if bias is None else bias[t][:n]
        W_next = wl.W[t + 1]
        par, tok, cum = select_top(zs, ls, cums[-1], W_next, bs)
        if forced is not None:
            par = forced[0][t + 1].astype(np.int32)
            tok = forced[1][t + 1].astype(np.int32)
            cum = scores_f32(zs, ls, cums[-1], bs)[par, tok]
        parents.append(par); tokens.append(tok); cums.append(cum)
        # Copy-on-reorder: the new beam order takes its parents' states.
        states = states[par]
        n = W_next

    sid = token_paths(parents, tokens)
    return RequestTrace(S_ctx, root_feat, root_z, root_lse, parents, tokens, cums,
                        calls, sid)


def chain_trace(wl, params, S_ctx: np.ndarray, path: Sequence[int]) -> List[CallTrace]:
    """Decode one SID path sequentially (a single beam, no beam tree).

    path: tokens fed at decode calls 0..len(path)-1 (the beam's ancestors'
    tokens, root first). Returns one single-row CallTrace per call. A beam's
    values at call t depend only on S_ctx and its own path, so this gives the
    FullState result for sampled beams of a large beam tree.
    """
    S = np.array(S_ctx, dtype=F64, copy=True)
    out: List[CallTrace] = []
    for tok in path:
        tr = CallTrace(tokens=np.array([tok], dtype=np.int32))
        x = params.E[[tok]].astype(F64)
        feat_in = x
        for layer in range(wl.layers):
            u = rms_normalize(x) if wl.residual else x
            q, k, v, a, b = gdn_inputs(wl, params, layer, u)
            S[layer], delta, o = gdn_transition(S[layer], per_value_head(wl, q)[0],
                                                per_value_head(wl, k)[0], v[0], a[0], b[0])
            tr.q.append(q); tr.k.append(k); tr.v.append(v); tr.alpha.append(a); tr.beta.append(b)
            tr.delta.append(delta[None]); tr.o.append(o[None])
            if wl.residual:
                x = x + o.reshape(1, -1)
            else:
                feat_in = o.reshape(1, -1)
        tr.feat = layer_feature(wl, x if wl.residual else feat_in)
        tr.z = codebook_logits(params, tr.feat)
        tr.lse = log_normalizer(tr.z)
        out.append(tr)
    return out


def chain_decode(wl, params, S_ctx: np.ndarray, path: Sequence[int]):
    """Per-call (feature [F], z [V], lse) of one sequentially decoded path."""
    tr = chain_trace(wl, params, S_ctx, path)
    return ([c.feat[0] for c in tr], [c.z[0] for c in tr], [float(c.lse[0]) for c in tr])
