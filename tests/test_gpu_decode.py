"""The whole decode path (prefill, decode calls, selections, paths) through the
context-level C ABI, against the oracle.

Both sides run the same beam tree: the GPU's decode calls are forced along a
lineage the oracle chose (small workloads) or a seeded random lineage
(full-size workloads, checked on sampled requests and beams). The paths are
compared bit for bit.

Three comparisons per decode call:
  * selection, bit for bit: the decode's own selection outputs (parents,
    tokens, cumulative scores; the production path, which bounds the search
    with the logits GEMM's tile maxima) against the oracle's selection
    contract on the GPU's own stored logits, lse, input scores and bias, for
    the root selection and every decode call;
  * every stage on the values the GPU stored (tests/stored_parity.py):
    projections, replay and logits recomputed by the oracle from the stored
    inputs of that call, within 2e-3 (bf16 storage, fp32 accumulation) or
    1e-5 (fp32 storage), max|gpu - oracle| / max|oracle| per tensor;
  * end to end against the fp64 oracle: with bf16 storage the GPU rounds
    S_ctx, q, k, v, delta and o between stages while the oracle keeps fp64,
    so each value inherits up to three storage roundings of its inputs; that
    derived bound, E2E_BF16 = 3 * 2^-8, applies here (1e-5 in fp32).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
import linear_attention_beam_gb300 as gb
from gpu_util import DEV, TOL_BF16, TOL_F32, decoder_for, device_status_clear, host, maxrel, to_dev
from stored_parity import ancestry, call_rows, selection_matches, stage_errors

pytestmark = pytest.mark.gpu

E2E_BF16 = {"sctx": 1.2e-2, "q": 1.2e-2, "k": 1.2e-2, "v": 1.2e-2, "alpha": 1.2e-2, "beta": 1.2e-2,
            "delta": 1.2e-2, "o": 1.2e-2, "logits": 1.2e-2, "lse": 1.2e-2, "root": 1.2e-2}
FIELDS = ("q", "k", "v", "alpha", "beta", "delta", "o")
REPORT = {}


def _tol(wl, key):
    return TOL_F32 if wl.dtype == "f32" else E2E_BF16[key]


def _stage_tol(wl):
    return TOL_F32 if wl.dtype == "f32" else TOL_BF16


def _check_stages(name, wl, p, sctx_r, calls, anc, t, beams):
    e = stage_errors(wl, p, sctx_r, calls, anc, t, beams)
    for k, v in e.items():
        _record(name, "stored_" + k, v)
    bad = {k: v for k, v in e.items() if v > _stage_tol(wl)}
    assert not bad, (t, bad)


def _i32(a):
    return to_dev(np.asarray(a), torch.int32)


def _record(name, key, val):
    REPORT.setdefault(name, {})
    REPORT[name][key] = max(REPORT[name].get(key, 0.0), val)


def _select_identical(wl, z, lse, cum, W_next, bias=None):
    """GPU selection on the oracle's stored logits for one request."""
    lib = gb.load()
    n, V = z.shape
    zs = oracle.kept_scores_f32(z, wl.dtype)
    ls = lse.astype(np.float32)
    scratch = torch.empty(lib.gdnbeam_select_scratch_bytes(1, n, W_next, V), dtype=torch.uint8, device=DEV)
    par = torch.empty(1, W_next, dtype=torch.int32, device=DEV)
    tok = torch.empty_like(par)
    cn = torch.empty(1, W_next, device=DEV)
    td = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    assert lib.gdnbeam_select_topw(1, n, W_next, V, gb.BF16 if wl.dtype == "bf16" else gb.F32,
                                   gb.ptr(to_dev(zs, td)), gb.ptr(to_dev(ls)), gb.ptr(to_dev(cum)),
                                   gb.ptr(to_dev(bias) if bias is not None else None), gb.ptr(par),
                                   gb.ptr(tok), gb.ptr(cn), gb.ptr(scratch), scratch.numel(), None) == 0
    p, t, s = oracle.select_top(zs, ls, cum, W_next, bias)
    np.testing.assert_array_equal(par[0].cpu().numpy(), p)
    np.testing.assert_array_equal(tok[0].cpu().numpy(), t)
    np.testing.assert_array_equal(cn[0].cpu().numpy(), s)


SMALL = {
    "tiny_f32": synth.TINY,
    "single_w256": synth.SINGLE,
    "single_w256_f32": synth.SINGLE.with_(name="single_w256_f32", dtype="f32"),
    # grouped key heads (value heads 2h, 2h + 1 read key head h) with d_v != d_k
    "tiny_gqa_f32": synth.tiny_workload(d=16, d_v=32, H=4, H_k=2, V=24, T=3, W=(8, 12, 10),
                                        d_model=64, L=40, seed=3),
    # the same grouping on the tensor-core paths (d = 128, bf16); one request,
    # as the forced lineage is one request's
    "gqa_w128": synth.GQA.with_(R=1),
    # wide heads: d_k 256, d_v 512 on the CUDA-core paths (fp32), and d_v 256
    # through the tensor-core replay (bf16)
    "wide_f32": synth.tiny_workload(d=256, d_v=512, H=2, H_k=1, V=40, T=3, W=(6, 9, 7),
                                    d_model=96, L=24, seed=12),
    "wide_v256": synth.Workload("wide_v256", R=1, layers=1, H=4, d_k=128, d_v=256, d_model=512,
                                V=1024, T=3, W=(64, 64, 64), L=96, dtype="bf16", seed=13, H_k=2),
    # stacked layers with a residual stream: the embedding rows and the first
    # layer's RMS norm in one pass (d_model a multiple of 128), or as a gather
    # then a norm (d_model = 96); and one request of the four-layer bf16 model
    "resid_f32": synth.tiny_workload(d=16, H=8, layers=3, residual=True, V=24, T=3, W=(8, 12, 10),
                                     d_model=128, L=40, seed=5),
    "resid96_f32": synth.tiny_workload(d=16, H=6, layers=3, residual=True, V=24, T=3, W=(8, 12, 10),
                                       d_model=96, L=40, seed=6),
    "deep_r1": synth.DEEP.with_(name="deep_r1", R=1, W=(32, 64, 64, 64), L=130),
}


@pytest.mark.parametrize("state_path", [0, 1, 2], ids=["replay", "fullstate", "replayssm"])
@pytest.mark.parametrize("name", list(SMALL))
def test_decode_forced_on_oracle_lineage(name, state_path):
    if state_path and max(SMALL[name].d_k, SMALL[name].d_v) > 128:
        pytest.skip("the state-path baselines keep heads of width <= 128")
    # state_path 1 is the FullState baseline (per-beam states copied on
    # reorder), 2 the ReplaySSM baseline (states rebuilt from S_ctx and the
    # ancestors' records every call): the same comparisons hold for both
    wl = SMALL[name]
    p = synth.make_params(wl)
    prompt = synth.make_prompt(wl)
    tr = oracle.decode_request(wl, p, prompt[0])
    dec = decoder_for(wl, p, state_path=state_path)
    dec.prefill(_i32(prompt))
    sctx = host(dec.read_sctx())[0]
    e = maxrel(sctx, tr.S_ctx); _record(name, "sctx", e)
    assert e <= _tol(wl, "sctx")
    e = maxrel(host(dec.root_logits)[0], tr.root_z); _record(name, "root", e)
    assert e <= _tol(wl, "root")
    forced = ([_i32(x[None]) for x in tr.parents], [_i32(x[None]) for x in tr.tokens],
              [to_dev(x[None]) for x in tr.cum])
    res = dec.decode(wl.W, forced=forced, keep_logits=True, dump=True)
    assert dec.status() == 0
    # the root selection the decode made, on its own root row
    selection_matches(host(dec.root_logits)[:1], host(dec.root_lse)[:1], None, wl.W[0], None,
                      host(res.parents[0][0]).astype(np.int32), host(res.tokens[0][0]).astype(np.int32),
                      host(res.cum[0][0]))
    sctx_r = host(dec.read_sctx())[0]
    calls = []
    for t, call in enumerate(tr.calls):
        n = wl.W[t]
        dd = res.dumps[t]
        # the decode's own selection (GEMM tile maxima as its bound) on the
        # logits, lse and input scores it was given
        selection_matches(host(res.logits[t]), host(res.lse[t]), tr.cum[t], wl.W[t + 1], None,
                          res.parents[t + 1][0].cpu().numpy(), res.tokens[t + 1][0].cpu().numpy(),
                          res.cum[t + 1][0].cpu().numpy())
        if state_path == 0:
            rows = call_rows(wl, {f: host(dd[f]) for f in FIELDS + ("logits",)}, n)
            rows.update(tokens=tr.tokens[t], lse=host(res.lse[t]))
            calls.append(rows)
            _check_stages(name, wl, p, sctx_r, calls, ancestry(tr.parents, t), t, range(n))
        for f in FIELDS:
            for layer in range(wl.layers):
                e = maxrel(host(dd[f][layer]).reshape(n, -1), getattr(call, f)[layer].reshape(n, -1))
                _record(name, f, e)
                assert e <= _tol(wl, f), (t, f, layer, e)
        e = maxrel(host(dd["logits"]), call.z); _record(name, "logits", e)
        assert e <= _tol(wl, "logits")
        e = np.abs(host(res.lse[t]) - call.lse).max() / np.abs(call.z).max(); _record(name, "lse", e)
        assert e <= _tol(wl, "lse")
        _select_identical(wl, call.z, call.lse, tr.cum[t], wl.W[t + 1])
    np.testing.assert_array_equal(res.sid[0].cpu().numpy(), tr.sid)
    print("\nmax rel errors", name, {k: f"{v:.2e}" for k, v in REPORT[name].items()})


def test_decode_free_running_tiny():
    # fp32 run: the GPU's own selections reproduce the oracle's beam tree
    wl = synth.TINY
    p = synth.make_params(wl)
    prompt = synth.make_prompt(wl)
    tr = oracle.decode_request(wl, p, prompt[0])
    dec = decoder_for(wl, p)
    dec.prefill(_i32(prompt))
    res = dec.decode(wl.W)
    assert dec.status() == 0
    for s in range(wl.T):
        np.testing.assert_array_equal(res.parents[s][0].cpu().numpy(), tr.parents[s])
        np.testing.assert_array_equal(res.tokens[s][0].cpu().numpy(), tr.tokens[s])
        assert maxrel(res.cum[s][0].cpu().numpy(), tr.cum[s]) <= TOL_F32
    np.testing.assert_array_equal(res.sid[0].cpu().numpy(), tr.sid)


def test_exhaustive_small_tree_on_gpu():
    # V = 3, T = 3, W = 27: every SID survives and paths are a permutation of all
    wl = synth.tiny_workload(d=16, V=3, T=3, W=(3, 9, 27), H=2, d_model=32, L=6, seed=31)
    p = synth.make_params(wl)
    dec = decoder_for(wl, p)
    dec.prefill(_i32(synth.make_prompt(wl)))
    res = dec.decode(wl.W)
    assert dec.status() == 0
    seqs = sorted(map(tuple, res.sid[0].cpu().numpy().tolist()))
    import itertools
    assert seqs == sorted(itertools.product(range(3), repeat=3))


FULL = {
    "single_w256": (synth.SINGLE, (0,)),
    "batched_r64_w512": (synth.BATCHED, (0, 63)),
    "deep4_w1024": (synth.DEEP, (5,)),
    "skewed_r128": (synth.SKEWED, (127,)),
    "gqa_w128": (synth.GQA, (0, 1)),
}


@pytest.mark.parametrize("name", list(FULL))
def test_decode_full_size_sampled(name):
    wl, sample = FULL[name]
    p = synth.make_params(wl)
    prompts = synth.make_prompt(wl)
    bias = synth.make_bias(wl)
    lin_par, lin_tok = synth.random_lineage(wl, seed=0)
    dec = decoder_for(wl, p)
    dec.prefill(_i32(prompts))
    sctx = dec.read_sctx()
    ctx_host = {r: oracle.prefill(wl, p, prompts[r]) for r in sample}
    for r in sample:
        S_r, feat_r = ctx_host[r]
        e = maxrel(host(sctx[r]), S_r); _record(name, "sctx", e)
        assert e <= _tol(wl, "sctx")
        z_r = oracle.codebook_logits(p, feat_r[None])[0]
        e = maxrel(host(dec.root_logits[r]), z_r); _record(name, "root", e)
        assert e <= _tol(wl, "root")
    # the root selection, bit for bit, on the GPU's own root rows
    par0, tok0, cum0 = dec.select(-1, 1, wl.W[0], dec.root_logits, dec.root_lse)
    for r in sample:
        selection_matches(host(dec.root_logits[r:r + 1]), host(dec.root_lse[r:r + 1]), None, wl.W[0],
                          None, par0[r].cpu().numpy(), tok0[r].cpu().numpy(), cum0[r].cpu().numpy())
    sctx_h = {r: host(sctx[r]) for r in sample}
    calls = {r: [] for r in sample}
    cum = cum0
    for t in range(wl.T - 1):
        W_t = wl.W[t]
        n = wl.R * W_t
        f = lambda *s: torch.zeros(*s, device=DEV)
        dd = {"q": f(wl.layers, n, wl.Hk * wl.d_k), "k": f(wl.layers, n, wl.Hk * wl.d_k),
              "v": f(wl.layers, n, wl.H * wl.d_v), "alpha": f(wl.layers, n, wl.H),
              "beta": f(wl.layers, n, wl.H), "delta": f(wl.layers, n, wl.H * wl.d_v),
              "o": f(wl.layers, n, wl.H * wl.d_v), "logits": f(n, wl.V)}
        lg, ls = dec.step(t, W_t, _i32(lin_par[t]) if t else None, _i32(lin_tok[t]), dumps=dd)
        b = to_dev(bias[t, :, :W_t]) if bias is not None else None
        # the decode's own selection: input scores are the previous
        # selection's output, the bound comes from the logits GEMM's tiles
        p_, t_, c_ = dec.select(t, W_t, wl.W[t + 1], lg, ls, cum, b)
        assert dec.status() == 0, f"device error after call {t}"
        for r in sample:
            rows = slice(r * W_t, (r + 1) * W_t)
            selection_matches(host(lg[rows]), host(ls[rows]), host(cum[r]), wl.W[t + 1],
                              None if bias is None else bias[t, r, :W_t],
                              p_[r].cpu().numpy(), t_[r].cpu().numpy(), c_[r].cpu().numpy())
            # every stage on the values the GPU stored, for sampled beams
            d = call_rows(wl, {k: host(v[:, rows]) if k != "logits" else host(v[rows])
                               for k, v in dd.items()}, W_t)
            d.update(tokens=lin_tok[t][r], lse=host(ls[rows]))
            calls[r].append(d)
            pars = [x[r] for x in lin_par]
            h = oracle.ancestry_slots(pars, t)
            # (W_t - 65, W_t - 64: the boundary when a request's beams are
            # split over two unequal blocks in the replay)
            beams = sorted({0, 1, W_t // 3, W_t // 2, max(W_t - 65, 0), max(W_t - 64, 0), W_t - 1})
            _check_stages(name, wl, p, sctx_h[r], calls[r], h, t, beams)
            # end to end against an fp64 single-path decode (derived bound)
            for bb in sorted({0, W_t // 2, W_t - 1}):
                path = [int(lin_tok[j][r][h[bb, j]]) for j in range(t)] + [int(lin_tok[t][r][bb])]
                ch = oracle.chain_trace(wl, p, ctx_host[r][0], path)[-1]
                row = r * W_t + bb
                for fld in FIELDS:
                    for layer in range(wl.layers):
                        e = maxrel(host(dd[fld][layer, row]), getattr(ch, fld)[layer].reshape(-1))
                        _record(name, fld, e)
                        assert e <= _tol(wl, fld), (t, r, bb, fld, layer, e)
                e = maxrel(host(dd["logits"][row]), ch.z[0]); _record(name, "logits", e)
                assert e <= _tol(wl, "logits")
                e = abs(float(ls[row]) - float(ch.lse[0])) / np.abs(ch.z).max(); _record(name, "lse", e)
                assert e <= _tol(wl, "lse")
        cum = c_
        del dd
    print("\nmax rel errors", name, {k: f"{v:.2e}" for k, v in REPORT[name].items()})


def test_step_before_prefill_is_rejected():
    wl = synth.TINY
    dec = decoder_for(wl, synth.make_params(wl))
    tok = _i32(np.zeros((1, 8)))
    with pytest.raises(gb.GdnbeamError) as ei:
        dec.step(0, 8, None, tok)
    assert ei.value.status == gb.ESTATE


@pytest.mark.parametrize("wl", [synth.TINY, synth.GQA.with_(name="gqa_r1", R=1, L=64)],
                         ids=["tiny_f32", "gqa_bf16"])
def test_bad_token_sets_device_error(wl):
    # a token outside [0, V) is reported through the status word, whether
    # the embedding rows are copied out (CUDA-core path) or gathered by the
    # tensor-core projection's own loads
    dec = decoder_for(wl, synth.make_params(wl))
    dec.prefill(_i32(synth.make_prompt(wl)))
    assert dec.status() == 0
    W = wl.W[0]
    tok = np.zeros((wl.R, W), dtype=np.int32)
    tok[0, W // 2] = wl.V + 3
    dec.step(0, W, None, _i32(tok))
    assert dec.status() == gb.EDEVICE
    assert device_status_clear() == 0


def test_bad_prompt_token_sets_device_error():
    # the chunked prefill's projections gather the prompt rows themselves
    wl = synth.GQA.with_(name="gqa_r1", R=1, L=64)
    dec = decoder_for(wl, synth.make_params(wl))
    prompt = synth.make_prompt(wl)
    prompt[0, wl.L - 1] = -1  # the last token: read by both prefill projections
    dec.prefill(_i32(prompt))
    assert dec.status() == gb.EDEVICE
    assert device_status_clear() == 0


@pytest.mark.parametrize("wl", [
    synth.tiny_workload(d=16, H=2, V=20, T=3, W=(6, 8, 5), d_model=32, L=12, seed=21, R=3),
    synth.GQA.with_(name="gqa_r3", R=3, L=64),
], ids=["tiny_f32_r3", "gqa_bf16_r3"])
def test_per_request_reset_and_prefill(wl):
    # request 1 is released and prefilled with a new prompt while requests 0
    # and 2 keep their contexts; the next decode equals a fresh decode of the
    # prompts with row 1 replaced, bit for bit
    p = synth.make_params(wl)
    P1 = synth.make_prompt(wl)
    P2 = synth.make_prompt(wl.with_(seed=wl.seed + 100))
    dec = decoder_for(wl, p)
    dec.prefill(_i32(P1))
    dec.decode(wl.W)
    dec.reset([1])
    with pytest.raises(gb.GdnbeamError) as ei:
        dec.step(0, wl.W[0], None, _i32(np.zeros((wl.R, wl.W[0]))))
    assert ei.value.status == gb.ESTATE
    dec.prefill_requests([1], _i32(P2[1:2]))
    got = dec.decode(wl.W, keep_logits=True)
    assert dec.status() == 0
    P3 = P1.copy()
    P3[1] = P2[1]
    ref = decoder_for(wl, p)
    ref.prefill(_i32(P3))
    want = ref.decode(wl.W, keep_logits=True)
    assert ref.status() == 0
    np.testing.assert_array_equal(host(dec.read_sctx()), host(ref.read_sctx()))
    np.testing.assert_array_equal(host(dec.root_logits), host(ref.root_logits))
    for s in range(wl.T):
        for a, b in ((got.parents, want.parents), (got.tokens, want.tokens), (got.cum, want.cum)):
            np.testing.assert_array_equal(a[s].cpu().numpy(), b[s].cpu().numpy())
    for t in range(wl.T - 1):
        np.testing.assert_array_equal(host(got.logits[t]), host(want.logits[t]))
    np.testing.assert_array_equal(got.sid.cpu().numpy(), want.sid.cpu().numpy())
