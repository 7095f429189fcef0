"""Each CUDA stage against the oracle on identical stored inputs, through the
tensor-level C ABI. Shapes span several tiles and end in ragged tails."""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
import linear_attention_beam_gb300 as gb
from gpu_util import (DEV, TOL_BF16, TOL_F32, cfg_for, device_status_clear, host, maxrel,
                      store, tdt, to_dev)

pytestmark = pytest.mark.gpu

U = 2.0 ** -8  # bf16 unit roundoff (storage rounding of a stored output)


def _tol(wl):
    return TOL_BF16 if wl.dtype == "bf16" else TOL_F32


def _check_stored(g, o, wl, what):
    """Stored output: within tol of max|o| plus the storage rounding of o."""
    g = np.asarray(g, np.float64); o = np.asarray(o, np.float64)
    extra = U * np.abs(o) if wl.dtype == "bf16" else 0.0
    bound = _tol(wl) * np.abs(o).max() + extra
    bad = np.abs(g - o) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements out of bound, maxrel={maxrel(g, o):.3g}"


def _unit_rows(rng, shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


# ------------------------------------------------------------------ selection

def _select_case(rng, R, W_t, W_next, V, dtype, ties=True, bias=True):
    z = rng.standard_normal((R, W_t, V)).astype(np.float32) * 2.0
    if ties:
        z[:, :, ::5] = z[:, :, :1]
        if W_t > 1:
            z[:, 1] = z[:, 0]
    z = synth.to_storage(z, dtype)
    lse = np.stack([oracle.log_normalizer(z[r]) for r in range(R)]).astype(np.float32)
    cum = np.sort(rng.standard_normal((R, W_t)).astype(np.float32))[:, ::-1].copy()
    if W_t > 2:
        cum[:, 2] = cum[:, 1]
    b = rng.standard_normal((R, W_t)).astype(np.float32) * 2.0 if bias else None
    return z, lse, cum, b


@pytest.mark.parametrize("R,W_t,W_next,V,dtype", [
    (1, 1, 8, 16, "f32"), (3, 5, 7, 300, "bf16"), (2, 37, 64, 513, "bf16"),
    (4, 64, 200, 100, "f32"), (2, 9, 45, 5, "bf16"), (1, 3, 1, 2, "f32")])
def test_select_topw_bit_exact(R, W_t, W_next, V, dtype):
    rng = np.random.default_rng(R * 1000 + W_t + V)
    z, lse, cum, b = _select_case(rng, R, W_t, W_next, V, dtype)
    lib = gb.load()
    tz = to_dev(z.reshape(R * W_t, V), torch.bfloat16 if dtype == "bf16" else torch.float32)
    scratch = torch.empty(lib.gdnbeam_select_scratch_bytes(R, W_t, W_next, V), dtype=torch.uint8, device=DEV)
    for bias in (None, b):
        par = torch.empty(R, W_next, dtype=torch.int32, device=DEV)
        tok = torch.empty_like(par)
        cn = torch.empty(R, W_next, dtype=torch.float32, device=DEV)
        st = lib.gdnbeam_select_topw(R, W_t, W_next, V, gb.BF16 if dtype == "bf16" else gb.F32,
                                     gb.ptr(tz), gb.ptr(to_dev(lse)), gb.ptr(to_dev(cum)),
                                     gb.ptr(to_dev(bias) if bias is not None else None),
                                     gb.ptr(par), gb.ptr(tok), gb.ptr(cn), gb.ptr(scratch),
                                     scratch.numel(), None)
        assert st == 0
        assert device_status_clear() == 0
        for r in range(R):
            p, t, s = oracle.select_top(z[r], lse[r], cum[r], W_next, None if bias is None else bias[r])
            np.testing.assert_array_equal(par[r].cpu().numpy(), p)
            np.testing.assert_array_equal(tok[r].cpu().numpy(), t)
            np.testing.assert_array_equal(cn[r].cpu().numpy().view(np.uint32), s.view(np.uint32))


def test_select_topw_full_size_sampled():
    # 64 requests x 512 beams x 8192 codes: the batched workload's selection
    R, W, V = 64, 512, 8192
    rng = np.random.default_rng(77)
    z, lse, cum, _ = _select_case(rng, R, W, W, V, "bf16", bias=False)
    lib = gb.load()
    scratch = torch.empty(lib.gdnbeam_select_scratch_bytes(R, W, W, V), dtype=torch.uint8, device=DEV)
    par = torch.empty(R, W, dtype=torch.int32, device=DEV)
    tok = torch.empty_like(par)
    cn = torch.empty(R, W, dtype=torch.float32, device=DEV)
    assert lib.gdnbeam_select_topw(R, W, W, V, gb.BF16, gb.ptr(to_dev(z.reshape(R * W, V), torch.bfloat16)),
                                   gb.ptr(to_dev(lse)), gb.ptr(to_dev(cum)), None, gb.ptr(par),
                                   gb.ptr(tok), gb.ptr(cn), gb.ptr(scratch), scratch.numel(), None) == 0
    assert device_status_clear() == 0
    for r in (0, 29, 63):
        p, t, s = oracle.select_top(z[r], lse[r], cum[r], W)
        np.testing.assert_array_equal(par[r].cpu().numpy(), p)
        np.testing.assert_array_equal(tok[r].cpu().numpy(), t)
        np.testing.assert_array_equal(cn[r].cpu().numpy(), s)
    # properties on every request: sorted keys, valid indices
    c = cn.cpu().numpy()
    assert np.all(np.diff(c, axis=1) <= 0)
    assert par.min().item() >= 0 and par.max().item() < W and tok.max().item() < V


# ------------------------------------------------------------------ ancestry

def test_ancestry_op_matches_walk():
    rng = np.random.default_rng(5)
    T, R, V = 5, 3, 11
    W = [4, 6, 3, 7, 5]
    parents = [np.zeros((R, W[0]), np.int32)] + [rng.integers(0, W[s - 1], (R, W[s])).astype(np.int32) for s in range(1, T)]
    tokens = [rng.integers(0, V, (R, W[s])).astype(np.int32) for s in range(T)]
    lib = gb.load()
    Wm = max(W)
    anc = [torch.zeros(R * Wm, T, dtype=torch.int32, device=DEV) for _ in range(2)]
    sid = [torch.zeros(R * Wm, T, dtype=torch.int32, device=DEV) for _ in range(2)]
    for t in range(T):
        cur, prev = anc[t & 1], anc[(t & 1) ^ 1]
        st = lib.gdnbeam_ancestry(R, t, T, V, W[t - 1] if t else 1, W[t], gb.ptr(to_dev(parents[t], torch.int32)),
                                  gb.ptr(to_dev(tokens[t], torch.int32)), gb.ptr(prev), gb.ptr(sid[(t & 1) ^ 1]),
                                  gb.ptr(cur), gb.ptr(sid[t & 1]), None)
        assert st == 0
        for r in range(R):
            exp = oracle.ancestry_slots([p[r] for p in parents], t)
            got = cur[r * W[t]:(r + 1) * W[t], :t].cpu().numpy()
            np.testing.assert_array_equal(got, exp)
    for r in range(R):
        exp = oracle.token_paths([p[r] for p in parents], [x[r] for x in tokens])
        np.testing.assert_array_equal(sid[(T - 1) & 1][r * W[-1]:(r + 1) * W[-1]].cpu().numpy(), exp)
    assert device_status_clear() == 0


# ------------------------------------------------------------------ replay

@pytest.mark.parametrize("dtype,d,H,R,W_t,t,resid", [
    ("f32", 16, 1, 1, 8, 2, False), ("bf16", 128, 3, 2, 37, 2, False),
    ("bf16", 64, 2, 3, 20, 3, True), ("f32", 128, 2, 2, 19, 1, False),
    ("bf16", 128, 2, 2, 300, 0, False), ("bf16", 32, 1, 1, 5, 5, False),
    ("bf16", 128, 4, 3, 64, 3, False), ("bf16", 128, 1, 1, 1, 1, False),
    ("bf16", 128, 2, 1, 96, 5, False), ("bf16", 128, 2, 2, 40, 1, True),
    ("bf16", 128, 3, 2, 512, 2, False), ("bf16", 128, 2, 2, 70, 4, False),
    # 96 (request, head) pairs of 8 beam tiles on 152 SMs: each pair's tiles
    # go in two unequal blocks (6 + 2); ragged and residual variants
    ("bf16", 128, 16, 6, 256, 2, False), ("bf16", 128, 16, 6, 250, 3, False),
    ("bf16", 128, 16, 6, 250, 1, True)])
def test_replay_op(dtype, d, H, R, W_t, t, resid):
    _replay_op(dtype, d, H, R, W_t, t, resid, H)


@pytest.mark.parametrize("dtype,dk,dv,H,Hk,R,W_t,t", [
    ("bf16", 256, 256, 2, 1, 2, 70, 1), ("bf16", 128, 512, 2, 2, 1, 40, 2), ("bf16", 256, 128, 2, 1, 2, 33, 0),
    ("bf16", 256, 512, 2, 1, 1, 64, 2), ("f32", 256, 512, 2, 1, 1, 19, 2), ("f32", 32, 256, 3, 3, 2, 17, 1)])
def test_replay_op_wide_heads(dtype, dk, dv, H, Hk, R, W_t, t):
    # key widths up to 256 and value widths up to 512 (blocks of 128 value
    # rows)
    _replay_op(dtype, dk, H, R, W_t, t, False, Hk, dv=dv)


@pytest.mark.parametrize("dtype,d,H,Hk,R,W_t,t", [
    ("f32", 16, 4, 2, 2, 9, 2), ("f32", 32, 6, 3, 1, 20, 3), ("bf16", 128, 4, 1, 2, 70, 2),
    ("bf16", 128, 8, 4, 2, 96, 1)])
def test_replay_op_grouped_key_heads(dtype, d, H, Hk, R, W_t, t):
    # value head h reads query/key head h // (H // Hk) and that head's
    # ancestor keys; the tensor-core kernel and the CUDA-core one alike
    _replay_op(dtype, d, H, R, W_t, t, False, Hk)


def _replay_op(dtype, d, H, R, W_t, t, resid, Hk, dv=None):
    dk = d
    dv = dv or d
    wl = synth.tiny_workload(d=dk, d_v=dv, V=7, H=H, R=R, dtype=dtype, H_k=Hk)
    g = H // Hk
    rng = np.random.default_rng(d + H + W_t + t + 100 * Hk + dv)
    st_ = lambda a: store(a, wl)
    S_ctx = (rng.standard_normal((R, H, dv, dk)) * 0.05).astype(np.float32).astype(np.float64)
    Wj = [int(rng.integers(1, 40)) for _ in range(t)]
    rec_k = [st_(_unit_rows(rng, (R, Wj[j], Hk, dk))) for j in range(t)]
    rec_d = [st_(rng.standard_normal((R, Wj[j], H, dv)) * 0.5) for j in range(t)]
    rec_a = [rng.uniform(0.2, 1.0, (R, Wj[j], H)).astype(np.float32).astype(np.float64) for j in range(t)]
    q = st_(_unit_rows(rng, (R, W_t, Hk, dk)))
    k = st_(_unit_rows(rng, (R, W_t, Hk, dk)))
    v = st_(rng.standard_normal((R, W_t, H, dv)))
    al = rng.uniform(0.1, 1.0, (R, W_t, H)).astype(np.float32).astype(np.float64)
    be = rng.uniform(0.0, 1.0, (R, W_t, H)).astype(np.float32).astype(np.float64)
    anc = np.stack([rng.integers(0, Wj[j], (R, W_t)) for j in range(t)], -1).astype(np.int32) if t else np.zeros((R, W_t, 1), np.int32)
    x0 = rng.standard_normal((R, W_t, H * dv)) if resid else None

    td = tdt(wl)
    keep = []
    recs = (gb.Records * max(t, 1))()
    for j in range(t):
        tk, tdl, ta = to_dev(rec_k[j].reshape(-1), td), to_dev(rec_d[j].reshape(-1), td), to_dev(rec_a[j].reshape(-1))
        keep += [tk, tdl, ta]
        recs[j] = gb.Records(gb.ptr(tk), gb.ptr(tdl), gb.ptr(ta), Wj[j])
    n = R * W_t
    d_out = torch.empty(n, H * dv, dtype=td, device=DEV)
    o_out = torch.empty_like(d_out)
    d_dump = torch.zeros(n, H * dv, device=DEV)
    o_dump = torch.zeros_like(d_dump)
    x_dev = to_dev(x0.reshape(n, H * dv)) if resid else None
    dm = gb.dumps(delta=d_dump, o=o_dump)
    cfg = cfg_for(wl, R=R, H=H, d_k=dk, d_v=dv, d_model=H * dv, T=max(t + 1, 2), H_k=Hk)
    lib = gb.load()
    st = lib.gdnbeam_replay(C.byref(cfg), t, W_t, gb.ptr(to_dev(S_ctx.reshape(-1))), H * dv * dk,
                            gb.ptr(to_dev(q.reshape(-1), td)), gb.ptr(to_dev(k.reshape(-1), td)),
                            gb.ptr(to_dev(v.reshape(-1), td)), gb.ptr(to_dev(al.reshape(-1))),
                            gb.ptr(to_dev(be.reshape(-1))), recs,
                            gb.ptr(to_dev(anc.reshape(n, -1), torch.int32)), anc.shape[-1],
                            gb.ptr(d_out), gb.ptr(o_out), gb.ptr(x_dev), C.byref(dm), None)
    assert st == 0
    assert device_status_clear() == 0
    exp_d = np.zeros((R, W_t, H, dv)); exp_o = np.zeros_like(exp_d)
    for r in range(R):
        for b in range(W_t):
            for h in range(H):
                hk = h // g
                chain = [(rec_a[j][r, anc[r, b, j], h], rec_d[j][r, anc[r, b, j], h], rec_k[j][r, anc[r, b, j], hk]) for j in range(t)]
                exp_d[r, b, h], exp_o[r, b, h] = oracle.step_from_records(
                    S_ctx[r, h], chain, q[r, b, hk], k[r, b, hk], v[r, b, h], al[r, b, h], be[r, b, h])
    tol = _tol(wl)
    assert maxrel(host(d_dump).reshape(exp_d.shape), exp_d) <= tol
    assert maxrel(host(o_dump).reshape(exp_o.shape), exp_o) <= tol
    _check_stored(host(d_out).reshape(exp_d.shape), exp_d, wl, "delta")
    _check_stored(host(o_out).reshape(exp_o.shape), exp_o, wl, "o")
    if resid:
        assert maxrel(host(x_dev).reshape(R, W_t, H * dv), x0 + exp_o.reshape(R, W_t, H * dv)) <= tol


@pytest.mark.parametrize("dtype,d", [("f32", 16), ("bf16", 128)])
def test_replay_rejects_out_of_range_slot(dtype, d):
    wl = synth.tiny_workload(d=d, V=7, H=1, R=1, dtype=dtype)
    lib = gb.load()
    t, W_t = 1, 4
    td = tdt(wl)
    keep = []
    def z(*s, dt=torch.float32):
        x = torch.zeros(*s, device=DEV, dtype=dt)
        keep.append(x)
        return x
    k1, d1, a1 = z(3 * d, dt=td), z(3 * d, dt=td), z(3)
    recs = (gb.Records * 1)(gb.Records(gb.ptr(k1), gb.ptr(d1), gb.ptr(a1), 3))
    anc = torch.tensor([[0], [1], [7], [2]], dtype=torch.int32, device=DEV)  # 7 >= W_j = 3
    cfg = cfg_for(wl)
    st = lib.gdnbeam_replay(C.byref(cfg), t, W_t, gb.ptr(z(d * d)), d * d, gb.ptr(z(W_t * d, dt=td)),
                            gb.ptr(z(W_t * d, dt=td)), gb.ptr(z(W_t * d, dt=td)), gb.ptr(z(W_t)), gb.ptr(z(W_t)),
                            recs, gb.ptr(anc), 1, gb.ptr(z(W_t * d, dt=td)), gb.ptr(z(W_t * d, dt=td)), None,
                            None, None)
    assert st == 0
    assert device_status_clear() & gb.DERR["slot"]
    assert device_status_clear() == 0


# ------------------------------------------------------------------ projections

@pytest.mark.parametrize("dtype,d,H,d_model,n", [("f32", 16, 1, 16, 8), ("bf16", 32, 3, 96, 70),
                                                 ("bf16", 128, 2, 256, 130), ("f32", 64, 2, 64, 33)])
def test_project_op(dtype, d, H, d_model, n):
    wl = synth.tiny_workload(d=d, V=9, H=H, d_model=d_model, dtype=dtype, seed=d + n)
    p = synth.make_params(wl)
    rng = np.random.default_rng(n)
    u = store(rng.standard_normal((n, d_model)), wl)
    q, k, v, a, b = oracle.gdn_inputs(wl, p, 0, u)
    td = tdt(wl)
    Wp = to_dev(np.concatenate([p.Wq[0], p.Wk[0], p.Wv[0], p.w_alpha[0], p.w_beta[0]]), td)
    lib = gb.load()
    cfg = cfg_for(wl)
    outs = [torch.empty(n, H * d, dtype=td, device=DEV) for _ in range(3)]
    al, be = torch.empty(n, H, device=DEV), torch.empty(n, H, device=DEV)
    dq, dk, dv = (torch.zeros(n, H * d, device=DEV) for _ in range(3))
    dm = gb.dumps(q=dq, k=dk, v=dv)
    sb = lib.gdnbeam_project_scratch_bytes(C.byref(cfg), n)
    scratch = torch.empty(max(sb, 1), dtype=torch.uint8, device=DEV)
    st = lib.gdnbeam_project(C.byref(cfg), n, gb.ptr(to_dev(u, td)), gb.ptr(Wp), gb.ptr(outs[0]),
                             gb.ptr(outs[1]), gb.ptr(outs[2]), gb.ptr(al), gb.ptr(be), gb.ptr(scratch),
                             sb, C.byref(dm), None)
    assert st == 0
    tol = _tol(wl)
    for got, dump, exp, nm in ((outs[0], dq, q, "q"), (outs[1], dk, k, "k"), (outs[2], dv, v, "v")):
        assert maxrel(host(dump), exp.reshape(n, -1)) <= tol, nm
        _check_stored(host(got), exp.reshape(n, -1), wl, nm)
    assert maxrel(host(al), a) <= tol and maxrel(host(be), b) <= tol


# ------------------------------------------------------------------ logits

@pytest.mark.parametrize("dtype,F,V,n", [("f32", 16, 16, 8), ("bf16", 128, 300, 70), ("bf16", 256, 1000, 129)])
def test_logits_op(dtype, F, V, n):
    d = min(F, 128)
    wl = synth.tiny_workload(d=d, V=V, H=F // d, d_model=F, dtype=dtype, seed=F + V)
    p = synth.make_params(wl)
    rng = np.random.default_rng(V)
    feat = store(rng.standard_normal((n, F)), wl)
    z = oracle.codebook_logits(p, feat)
    lse = oracle.log_normalizer(z)
    td = tdt(wl)
    lib = gb.load()
    cfg = cfg_for(wl)
    zo = torch.empty(n, V, dtype=td, device=DEV)
    lo = torch.empty(n, device=DEV)
    zd = torch.zeros(n, V, device=DEV)
    dm = gb.dumps(logits=zd)
    sb = lib.gdnbeam_logits_scratch_bytes(C.byref(cfg), n)
    scratch = torch.empty(max(sb, 1), dtype=torch.uint8, device=DEV)
    assert lib.gdnbeam_logits(C.byref(cfg), n, gb.ptr(to_dev(feat, td)), gb.ptr(to_dev(p.Wo, td)),
                              gb.ptr(zo), gb.ptr(lo), gb.ptr(scratch), sb, C.byref(dm), None) == 0
    tol = _tol(wl)
    assert maxrel(host(zd), z) <= tol
    _check_stored(host(zo), z, wl, "z")
    assert np.abs(host(lo) - lse).max() <= tol * np.abs(z).max()


# ------------------------------------------------------------------ prefill

@pytest.mark.parametrize("dtype,d,H,R,L,resid", [("f32", 16, 1, 1, 32, False), ("bf16", 32, 2, 2, 33, True),
                                                 ("bf16", 128, 2, 2, 65, False)])
def test_prefill_scan_op(dtype, d, H, R, L, resid):
    _prefill_scan_op(dtype, d, d, H, H, R, L, resid)


@pytest.mark.parametrize("dtype,dk,dv,H,Hk,R,L", [
    ("bf16", 256, 512, 2, 1, 1, 70), ("f32", 256, 256, 2, 2, 1, 33), ("bf16", 128, 256, 4, 2, 2, 40),
    ("f32", 16, 32, 4, 2, 1, 50)])
def test_prefill_scan_op_wide_and_grouped(dtype, dk, dv, H, Hk, R, L):
    # key widths up to 256, value widths up to 512 (blocks of 128 value rows),
    # grouped key heads
    _prefill_scan_op(dtype, dk, dv, H, Hk, R, L, False)


@pytest.mark.parametrize("H,Hk,R,L,a_lo,a_hi", [
    (2, 2, 1, 1, 0.3, 1.0), (2, 2, 2, 63, 0.3, 1.0), (2, 1, 1, 128, 0.3, 1.0),
    (4, 2, 2, 129, 0.3, 1.0), (2, 2, 1, 300, 0.01, 0.3), (1, 1, 1, 1000, 0.9, 1.0),
    (2, 2, 3, 257, 0.5, 1.0)])
def test_prefill_chunked_tensor_cores(H, Hk, R, L, a_lo, a_hi):
    # bf16, d_k = d_v = 128 without a residual stream: the chunked tcgen05
    # prefill (64-token chunks, 128-token stages; lengths around both
    # boundaries, fast and slow decay, grouped key heads)
    _prefill_scan_op("bf16", 128, 128, H, Hk, R, L, False, a_lo, a_hi)


@pytest.mark.parametrize("H,Hk,R,L,a_lo,a_hi", [
    (2, 2, 1, 1, 0.3, 1.0), (2, 2, 2, 64, 0.3, 1.0), (2, 1, 1, 65, 0.3, 1.0),
    (4, 2, 2, 129, 0.3, 1.0), (2, 2, 1, 300, 0.01, 0.3), (1, 1, 1, 1000, 0.9, 1.0),
    (2, 2, 3, 257, 0.5, 1.0)])
def test_prefill_chunked_all_positions(H, Hk, R, L, a_lo, a_hi):
    # stacked layers: the chunked tcgen05 prefill also adds o of every prompt
    # position to the residual stream (chunk states and records from the
    # chain, all positions' outputs from the parallel kernel); checked
    # against the oracle's recurrence at every position
    _prefill_scan_op("bf16", 128, 128, H, Hk, R, L, True, a_lo, a_hi)


def _prefill_scan_op(dtype, dk, dv, H, Hk, R, L, resid, a_lo=0.3, a_hi=1.0):
    wl = synth.tiny_workload(d=dk, d_v=dv, V=5, H=H, R=R, dtype=dtype, H_k=Hk)
    rng = np.random.default_rng(L + dk + dv)
    q = store(_unit_rows(rng, (R, L, Hk, dk)), wl)
    k = store(_unit_rows(rng, (R, L, Hk, dk)), wl)
    v = store(rng.standard_normal((R, L, H, dv)), wl)
    a = rng.uniform(a_lo, a_hi, (R, L, H)).astype(np.float32).astype(np.float64)
    b = rng.uniform(0.0, 1.0, (R, L, H)).astype(np.float32).astype(np.float64)
    x0 = rng.standard_normal((R, L, H * dv)) if resid else None
    td = tdt(wl)
    lib = gb.load()
    cfg = cfg_for(wl, R=R, H=H, d_k=dk, d_v=dv, d_model=H * dv, H_k=Hk)
    sc = torch.empty(R, H, dv, dk, dtype=torch.float32, device=DEV)
    ol = torch.empty(R, H * dv, dtype=td, device=DEV)
    xd = to_dev(x0.reshape(R * L, H * dv)) if resid else None
    sb = lib.gdnbeam_prefill_scan_scratch_bytes(C.byref(cfg), L, int(resid))
    scr = torch.empty(max(sb, 1), dtype=torch.uint8, device=DEV)
    args = (C.byref(cfg), L, gb.ptr(to_dev(q.reshape(-1), td)), gb.ptr(to_dev(k.reshape(-1), td)),
            gb.ptr(to_dev(v.reshape(-1), td)), gb.ptr(to_dev(a.reshape(-1))),
            gb.ptr(to_dev(b.reshape(-1))), gb.ptr(sc), H * dv * dk, gb.ptr(ol), gb.ptr(xd))
    if sb:  # the chunked form with a residual stream needs its scratch
        assert lib.gdnbeam_prefill_scan(*args, gb.ptr(scr), sb - 1, None) == gb.EWORKSPACE
    st = lib.gdnbeam_prefill_scan(*args, gb.ptr(scr), sb, None)
    assert st == 0
    g = H // Hk
    for r in range(R):
        qe, ke = np.repeat(q[r], g, axis=1), np.repeat(k[r], g, axis=1)
        S, o = oracle.prefill_scan(qe, ke, v[r], a[r], b[r])
        assert maxrel(host(sc[r]), S) <= _tol(wl), "S_ctx"
        _check_stored(host(ol[r]).reshape(H, dv), o[-1], wl, "o_last")
        if resid:  # what was added to the stream is o of every position
            added = host(xd).reshape(R, L, H * dv)[r].astype(np.float64) - x0[r]
            assert maxrel(added, o.reshape(L, H * dv)) <= _tol(wl), "o at every position"


# ------------------------------------------------------------------ tensor-core GEMMs

@pytest.mark.parametrize("H,d_model,n", [(16, 2048, 300), (8, 1024, 129), (2, 256, 1), (16, 2048, 1024)])
def test_project_op_tensor_cores(H, d_model, n):
    # bf16, head width 128: the tcgen05 projection GEMM (ragged row tails,
    # the gate columns in a partly filled last tile)
    test_project_op("bf16", 128, H, d_model, n)


@pytest.mark.parametrize("F,V,n", [(2048, 8192, 300), (1024, 4096, 129), (256, 1000, 1), (2048, 8192, 512),
                                   (2048, 8232, 700), (1024, 520, 257)])
def test_logits_op_tensor_cores(F, V, n):
    # ragged row tails around the 256-row pair tiles; last column tiles of
    # full width, 232 columns, and 40 or 8 columns (narrowed MMAs)
    test_logits_op("bf16", F, V, n)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_select_massive_ties_take_the_exact_fallback(dtype):
    # every candidate ties: the bound keeps all of them, the buffer overflows
    # and the two-stage exact path must still give the lowest flat indices
    R, W_t, W_next, V = 2, 64, 5, 100
    z = np.zeros((R, W_t, V), np.float32)
    lse = np.zeros((R, W_t), np.float32)
    cum = np.zeros((R, W_t), np.float32)
    lib = gb.load()
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    scratch = torch.empty(lib.gdnbeam_select_scratch_bytes(R, W_t, W_next, V), dtype=torch.uint8, device=DEV)
    par = torch.empty(R, W_next, dtype=torch.int32, device=DEV)
    tok = torch.empty_like(par)
    cn = torch.empty(R, W_next, device=DEV)
    tz, tl, tc_ = to_dev(z.reshape(R * W_t, V), td), to_dev(lse), to_dev(cum)
    assert lib.gdnbeam_select_topw(R, W_t, W_next, V, gb.BF16 if dtype == "bf16" else gb.F32, gb.ptr(tz),
                                   gb.ptr(tl), gb.ptr(tc_), None, gb.ptr(par), gb.ptr(tok), gb.ptr(cn),
                                   gb.ptr(scratch), scratch.numel(), None) == 0
    assert device_status_clear() == 0
    for r in range(R):
        np.testing.assert_array_equal(par[r].cpu().numpy(), [0] * 5)
        np.testing.assert_array_equal(tok[r].cpu().numpy(), [0, 1, 2, 3, 4])


@pytest.mark.parametrize("R,W_t,W_next,V,dtype,z_std,b_std,spike", [
    (3, 300, 64, 2000, "bf16", 0.05, 3.0, None),    # ragged last tile, many stored-value ties
    (2, 77, 200, 513, "f32", 0.01, 2.0, None),      # nearly every tile listed
    (2, 1024, 1024, 8192, "bf16", 1.0, 2.0, None),  # the skewed workload's selection shape
    (2, 200, 64, 1000, "f32", 0.01, 0.01, 20.0),    # one far outlier: two narrowing rounds
    (2, 300, 64, 2000, "bf16", 0.01, 0.01, 20.0),
])
def test_select_parent_dominated_scores_narrow_the_bound(R, W_t, W_next, V, dtype, z_std, b_std, spike):
    # per-parent score offsets much wider than the logit spread: whole rows of
    # the best parents clear the tile-maximum bound, far more candidates than
    # the buffer holds, and the selection must narrow the bound and stay exact
    rng = np.random.default_rng(W_t + V)
    z = synth.to_storage(rng.standard_normal((R, W_t, V)).astype(np.float32) * z_std, dtype)
    if spike is not None:
        z[:, 0, 0] = spike  # the best score sits far above the crowd at the bound
    lse = np.stack([oracle.log_normalizer(z[r]) for r in range(R)]).astype(np.float32)
    cum = np.sort(rng.standard_normal((R, W_t)).astype(np.float32) * 0.5)[:, ::-1].copy()
    bias = (rng.standard_normal((R, W_t)) * b_std).astype(np.float32)
    lib = gb.load()
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    scratch = torch.empty(lib.gdnbeam_select_scratch_bytes(R, W_t, W_next, V), dtype=torch.uint8, device=DEV)
    par = torch.empty(R, W_next, dtype=torch.int32, device=DEV)
    tok = torch.empty_like(par)
    cn = torch.empty(R, W_next, device=DEV)
    assert lib.gdnbeam_select_topw(R, W_t, W_next, V, gb.BF16 if dtype == "bf16" else gb.F32,
                                   gb.ptr(to_dev(z.reshape(R * W_t, V), td)), gb.ptr(to_dev(lse)),
                                   gb.ptr(to_dev(cum)), gb.ptr(to_dev(bias)), gb.ptr(par), gb.ptr(tok),
                                   gb.ptr(cn), gb.ptr(scratch), scratch.numel(), None) == 0
    assert device_status_clear() == 0
    for r in range(R):
        p, t, s = oracle.select_top(z[r], lse[r], cum[r], W_next, bias[r])
        np.testing.assert_array_equal(par[r].cpu().numpy(), p)
        np.testing.assert_array_equal(tok[r].cpu().numpy(), t)
        np.testing.assert_array_equal(cn[r].cpu().numpy().view(np.uint32), s.view(np.uint32))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("bad", ["nan_logit", "inf_logit", "nan_lse"])
def test_select_flags_non_finite_inputs(dtype, bad):
    # a NaN or +inf logit (tile maxima computed by the selection itself) or a
    # non-finite lse sets GDNBEAM_DERR_NONFINITE; the call still returns
    R, W_t, W_next, V = 2, 16, 8, 300
    rng = np.random.default_rng(7)
    z = rng.standard_normal((R * W_t, V)).astype(np.float32)
    lse = np.log(np.exp(z.astype(np.float64)).sum(1)).astype(np.float32)
    cum = np.zeros(R * W_t, np.float32)
    if bad == "nan_logit":
        z[5, 17] = np.nan
    elif bad == "inf_logit":
        z[20, 299] = np.inf
    else:
        lse[3] = np.nan
    lib = gb.load()
    assert device_status_clear() == 0
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    scratch = torch.empty(lib.gdnbeam_select_scratch_bytes(R, W_t, W_next, V), dtype=torch.uint8, device=DEV)
    par = torch.empty(R, W_next, dtype=torch.int32, device=DEV)
    tok = torch.empty_like(par)
    cn = torch.empty(R, W_next, device=DEV)
    assert lib.gdnbeam_select_topw(R, W_t, W_next, V, gb.BF16 if dtype == "bf16" else gb.F32,
                                   gb.ptr(to_dev(z, td)), gb.ptr(to_dev(lse)), gb.ptr(to_dev(cum)), None,
                                   gb.ptr(par), gb.ptr(tok), gb.ptr(cn), gb.ptr(scratch), scratch.numel(),
                                   None) == 0
    assert device_status_clear() & gb.DERR_NONFINITE


# ------------------------------------------------------------------ baselines

@pytest.mark.parametrize("dtype,d,H,Hk,R,W_t,W_prev,t", [
    ("f32", 16, 2, 2, 2, 9, 5, 0), ("f32", 16, 2, 1, 2, 9, 5, 1), ("bf16", 128, 2, 1, 2, 40, 17, 1),
    ("bf16", 128, 3, 3, 1, 70, 33, 0), ("bf16", 64, 4, 2, 2, 33, 20, 3)])
def test_fullstate_step_op(dtype, d, H, Hk, R, W_t, W_prev, t):
    # the FullState baseline: each beam's own state from its parent's (S_ctx
    # at t = 0), one eq. 3 transition, the child's state stored
    wl = synth.tiny_workload(d=d, V=7, H=H, R=R, dtype=dtype, H_k=Hk)
    g = H // Hk
    rng = np.random.default_rng(d + 7 * H + W_t + t)
    st_ = lambda a: store(a, wl)
    S_ctx = st_(rng.standard_normal((R, H, d, d)) * 0.05)
    prev = st_(rng.standard_normal((R, W_prev, H, d, d)) * 0.05)
    par = rng.integers(0, W_prev, (R, W_t)).astype(np.int32)
    q = st_(_unit_rows(rng, (R, W_t, Hk, d)))
    k = st_(_unit_rows(rng, (R, W_t, Hk, d)))
    v = st_(rng.standard_normal((R, W_t, H, d)))
    al = rng.uniform(0.1, 1.0, (R, W_t, H)).astype(np.float32).astype(np.float64)
    be = rng.uniform(0.0, 1.0, (R, W_t, H)).astype(np.float32).astype(np.float64)
    td = tdt(wl)
    n = R * W_t
    cur = torch.zeros(n, H, d, d, dtype=td, device=DEV)
    d_out = torch.empty(n, H * d, dtype=td, device=DEV)
    o_out = torch.empty_like(d_out)
    cfg = cfg_for(wl, R=R, H=H, d_k=d, d_v=d, d_model=H * d, T=t + 2, H_k=Hk)
    st = gb.load().gdnbeam_fullstate_step(
        C.byref(cfg), t, W_t, W_prev, gb.ptr(to_dev(S_ctx.reshape(-1), td)), H * d * d,
        gb.ptr(to_dev(prev.reshape(-1), td)), gb.ptr(cur), gb.ptr(to_dev(par.reshape(-1), torch.int32)),
        gb.ptr(to_dev(q.reshape(-1), td)), gb.ptr(to_dev(k.reshape(-1), td)),
        gb.ptr(to_dev(v.reshape(-1), td)), gb.ptr(to_dev(al.reshape(-1))), gb.ptr(to_dev(be.reshape(-1))),
        gb.ptr(d_out), gb.ptr(o_out), None)
    assert st == 0
    assert device_status_clear() == 0
    exp_S = np.zeros((R, W_t, H, d, d)); exp_d = np.zeros((R, W_t, H, d)); exp_o = np.zeros_like(exp_d)
    for r in range(R):
        for b in range(W_t):
            for h in range(H):
                S_par = S_ctx[r, h] if t == 0 else prev[r, par[r, b], h]
                exp_S[r, b, h], exp_d[r, b, h], exp_o[r, b, h] = oracle.gdn_transition(
                    S_par, q[r, b, h // g], k[r, b, h // g], v[r, b, h], al[r, b, h], be[r, b, h])
    _check_stored(host(cur).reshape(exp_S.shape), exp_S, wl, "states")
    _check_stored(host(d_out).reshape(exp_d.shape), exp_d, wl, "delta")
    _check_stored(host(o_out).reshape(exp_o.shape), exp_o, wl, "o")


@pytest.mark.parametrize("dtype,d,H,Hk,R,W_t,t", [
    ("f32", 16, 2, 2, 2, 9, 2), ("bf16", 128, 2, 1, 2, 40, 1), ("bf16", 128, 3, 3, 1, 70, 3),
    ("bf16", 64, 4, 2, 2, 33, 0), ("f32", 32, 2, 2, 1, 17, 5)])
def test_replayssm_step_op(dtype, d, H, Hk, R, W_t, t):
    # the ReplaySSM baseline: each (beam, head) rebuilds its parent state
    # from S_ctx (storage precision) and its ancestors' records, then steps
    wl = synth.tiny_workload(d=d, V=7, H=H, R=R, dtype=dtype, H_k=Hk)
    g = H // Hk
    rng = np.random.default_rng(3 * d + H + W_t + 11 * t)
    st_ = lambda a: store(a, wl)
    S_ctx = st_(rng.standard_normal((R, H, d, d)) * 0.05)
    Wj = [int(rng.integers(1, 40)) for _ in range(t)]
    rec_k = [st_(_unit_rows(rng, (R, Wj[j], Hk, d))) for j in range(t)]
    rec_d = [st_(rng.standard_normal((R, Wj[j], H, d)) * 0.5) for j in range(t)]
    rec_a = [rng.uniform(0.2, 1.0, (R, Wj[j], H)).astype(np.float32).astype(np.float64) for j in range(t)]
    q = st_(_unit_rows(rng, (R, W_t, Hk, d)))
    k = st_(_unit_rows(rng, (R, W_t, Hk, d)))
    v = st_(rng.standard_normal((R, W_t, H, d)))
    al = rng.uniform(0.1, 1.0, (R, W_t, H)).astype(np.float32).astype(np.float64)
    be = rng.uniform(0.0, 1.0, (R, W_t, H)).astype(np.float32).astype(np.float64)
    anc = (np.stack([rng.integers(0, Wj[j], (R, W_t)) for j in range(t)], -1) if t
           else np.zeros((R, W_t, 1))).astype(np.int32)
    td = tdt(wl)
    recs = (gb.Records * max(t, 1))()
    for j in range(t):
        recs[j] = gb.Records(gb.ptr(to_dev(rec_k[j].reshape(-1), td)), gb.ptr(to_dev(rec_d[j].reshape(-1), td)),
                             gb.ptr(to_dev(rec_a[j].reshape(-1))), Wj[j])
    n = R * W_t
    d_out = torch.empty(n, H * d, dtype=td, device=DEV)
    o_out = torch.empty_like(d_out)
    cfg = cfg_for(wl, R=R, H=H, d_k=d, d_v=d, d_model=H * d, T=t + 2, H_k=Hk)
    st = gb.load().gdnbeam_replayssm_step(
        C.byref(cfg), t, W_t, gb.ptr(to_dev(S_ctx.reshape(-1), td)), H * d * d,
        gb.ptr(to_dev(q.reshape(-1), td)), gb.ptr(to_dev(k.reshape(-1), td)), gb.ptr(to_dev(v.reshape(-1), td)),
        gb.ptr(to_dev(al.reshape(-1))), gb.ptr(to_dev(be.reshape(-1))), recs,
        gb.ptr(to_dev(anc.reshape(n, -1), torch.int32)), anc.shape[-1], gb.ptr(d_out), gb.ptr(o_out), None)
    assert st == 0
    assert device_status_clear() == 0
    exp_d = np.zeros((R, W_t, H, d)); exp_o = np.zeros_like(exp_d)
    for r in range(R):
        for b in range(W_t):
            for h in range(H):
                chain = [(rec_a[j][r, anc[r, b, j], h], rec_d[j][r, anc[r, b, j], h],
                          rec_k[j][r, anc[r, b, j], h // g]) for j in range(t)]
                exp_d[r, b, h], exp_o[r, b, h] = oracle.step_from_records(
                    S_ctx[r, h], chain, q[r, b, h // g], k[r, b, h // g], v[r, b, h], al[r, b, h], be[r, b, h])
    _check_stored(host(d_out).reshape(exp_d.shape), exp_d, wl, "delta")
    _check_stored(host(o_out).reshape(exp_o.shape), exp_o, wl, "o")


def test_baseline_steps_reject_wide_heads():
    wl = synth.tiny_workload(d=16, V=7, H=1, R=1, dtype="bf16")
    cfg = cfg_for(wl, d_k=256, d_v=128, d_model=128)
    lib = gb.load()
    z = torch.zeros(16, device=DEV)
    assert lib.gdnbeam_fullstate_step(C.byref(cfg), 0, 1, 1, gb.ptr(z), 0, None, gb.ptr(z), None, gb.ptr(z),
                                      gb.ptr(z), gb.ptr(z), gb.ptr(z), gb.ptr(z), gb.ptr(z), gb.ptr(z),
                                      None) == gb.EUNSUPPORTED
    assert lib.gdnbeam_replayssm_step(C.byref(cfg), 0, 1, gb.ptr(z), 0, gb.ptr(z), gb.ptr(z), gb.ptr(z),
                                      gb.ptr(z), gb.ptr(z), None, None, 0, gb.ptr(z), gb.ptr(z),
                                      None) == gb.EUNSUPPORTED
