"""The fused replay operator over the operator-sweep geometries (OneLA §3,
operator experiments, and §4.2: nine recurrent geometries spanning H_K 4-32,
H_V 4-64, K 128-256, V 128-512, with T = 2..6 decode calls, so replay depths
0..5) against the oracle, through the tensor-level C ABI.

Every geometry runs at every depth on R = 4, W = 128; three geometries also
run at R = 16, W = 512 and depth 5, where the pipeline holds one stage. Each
case checks sampled beams (all of their heads) against the oracle's explicit
state rebuild, and checks that the instantiation without fp32 dumps stores
the same bits as the one with them."""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
import linear_attention_beam_gb300 as gb
from gpu_util import DEV, TOL_BF16, device_status_clear, host, maxrel, to_dev

pytestmark = pytest.mark.gpu

U = 2.0 ** -8  # bf16 unit roundoff


def _unit(x):
    return (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)


def _sweep_case(geom, R, W, t, seed, n_sample):
    Hk, H, dk, dv = geom
    grp = H // Hk
    rng = np.random.default_rng(seed)
    bf = synth.round_bf16
    n = R * W
    S_ctx = (rng.standard_normal((R, H, dv, dk), dtype=np.float32) * 0.05).astype(np.float32)
    rec_k = [bf(_unit(rng.standard_normal((n, Hk, dk), dtype=np.float32))) for _ in range(t)]
    rec_d = [bf(rng.standard_normal((n, H, dv), dtype=np.float32) * 0.5) for _ in range(t)]
    rec_a = [rng.uniform(0.2, 1.0, (n, H)).astype(np.float32) for _ in range(t)]
    q = bf(_unit(rng.standard_normal((n, Hk, dk), dtype=np.float32)))
    k = bf(_unit(rng.standard_normal((n, Hk, dk), dtype=np.float32)))
    v = bf(rng.standard_normal((n, H, dv), dtype=np.float32))
    al = rng.uniform(0.1, 1.0, (n, H)).astype(np.float32)
    be = rng.uniform(0.0, 1.0, (n, H)).astype(np.float32)
    anc = (rng.integers(0, W, (n, t)) if t else np.zeros((n, 1))).astype(np.int32)

    lib = gb.load()
    cfg = gb.Config(R=R, layers=1, H=H, d_k=dk, d_v=dv, d_model=H * dv, V=256, T=t + 2, W_max=W,
                    L_max=1, dtype=gb.BF16, residual=0, H_k=Hk)
    recs = (gb.Records * max(t, 1))()
    for j in range(t):
        recs[j] = gb.Records(gb.ptr(to_dev(rec_k[j], torch.bfloat16)),
                             gb.ptr(to_dev(rec_d[j], torch.bfloat16)), gb.ptr(to_dev(rec_a[j])), W)
    args = (gb.ptr(to_dev(S_ctx)), H * dv * dk, gb.ptr(to_dev(q, torch.bfloat16)),
            gb.ptr(to_dev(k, torch.bfloat16)), gb.ptr(to_dev(v, torch.bfloat16)), gb.ptr(to_dev(al)),
            gb.ptr(to_dev(be)), recs, gb.ptr(to_dev(anc, torch.int32)), anc.shape[1])
    outs = []
    d_dump = torch.zeros(n, H * dv, device=DEV)
    o_dump = torch.zeros_like(d_dump)
    for dumps in (gb.dumps(delta=d_dump, o=o_dump), None):
        d_out = torch.empty(n, H * dv, dtype=torch.bfloat16, device=DEV)
        o_out = torch.empty_like(d_out)
        st = lib.gdnbeam_replay(C.byref(cfg), t, W, *args, gb.ptr(d_out), gb.ptr(o_out), None,
                                C.byref(dumps) if dumps is not None else None, None)
        assert st == 0
        assert device_status_clear() == 0
        outs.append((d_out, o_out))
    # the fast instantiation (no dumps) stores exactly what the dumping one stores
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))

    beams = sorted(set([0, W - 1] + list(rng.integers(0, W, n_sample - 2))))
    rows = [r * W + b for r in range(R) for b in beams]
    exp_d = np.zeros((len(rows), H, dv)); exp_o = np.zeros_like(exp_d)
    for i, row in enumerate(rows):
        r = row // W
        for h in range(H):
            hk = h // grp
            slot = [r * W + anc[row, j] for j in range(t)]  # ancestor rows of this beam
            chain = [(rec_a[j][slot[j], h], rec_d[j][slot[j], h], rec_k[j][slot[j], hk])
                     for j in range(t)]
            exp_d[i, h], exp_o[i, h] = oracle.step_from_records(
                S_ctx[r, h].astype(np.float64), chain, q[row, hk], k[row, hk], v[row, h], al[row, h],
                be[row, h])
    idx = torch.tensor(rows, device=DEV)
    got_d = host(d_dump[idx]).reshape(exp_d.shape)
    got_o = host(o_dump[idx]).reshape(exp_o.shape)
    assert maxrel(got_d, exp_d) <= TOL_BF16
    assert maxrel(got_o, exp_o) <= TOL_BF16
    for got, exp in ((outs[0][0], exp_d), (outs[0][1], exp_o)):
        g = host(got[idx]).reshape(exp.shape)
        bound = TOL_BF16 * np.abs(exp).max() + U * np.abs(exp)
        assert not (np.abs(g - exp) > bound).any()
    err = float(np.abs(got_o - exp_o).max())
    print(f"sweep-parity H_K={Hk} H_V={H} K={dk} V={dv} R={R} W={W} t={t}: "
          f"max|o - oracle| = {err:.3g} (max|o| = {np.abs(exp_o).max():.3g})")


@pytest.mark.parametrize("t", range(6))
@pytest.mark.parametrize("geom", synth.SWEEP_GEOMETRIES,
                         ids=lambda g: "hk{}_hv{}_k{}_v{}".format(*g))
def test_sweep_geometry_depths(geom, t):
    _sweep_case(geom, 4, 128, t, seed=sum(geom) * 10 + t, n_sample=6)


@pytest.mark.parametrize("geom", [(16, 16, 128, 128), (8, 8, 256, 256), (8, 8, 128, 512)],
                         ids=lambda g: "hk{}_hv{}_k{}_v{}".format(*g))
def test_sweep_full_size_deepest(geom):
    # R = 16, W = 512 at depth 5: one pipeline stage per block
    _sweep_case(geom, 16, 512, 5, seed=sum(geom) + 5, n_sample=4)
