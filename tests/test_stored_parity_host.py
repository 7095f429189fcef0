"""The stored-input stage check (tests/stored_parity.py) on the CPU.

Fed the oracle's own decode as if it were the GPU's dumps, every stage must
agree to fp32 rounding; a planted mistake in what the helper is given (a
wrong ancestor slot, a wrong token, a dropped residual layer) must show.
This pins the helper before the GPU tests rely on it.
"""
import numpy as np
import pytest

import oracle
import synth
from stored_parity import FIELDS, ancestry, selection_matches, stage_errors


def _calls_from_oracle(wl, tr):
    calls = []
    for c in tr.calls:
        d = {f: np.stack(getattr(c, f)) for f in FIELDS}
        d["logits"] = c.z
        d["lse"] = c.lse
        d["tokens"] = c.tokens
        calls.append(d)
    return calls


WLS = {
    "tiny_f32": synth.TINY,
    "gqa_f32": synth.tiny_workload(d=16, d_v=32, H=4, H_k=2, V=24, T=4, W=(8, 12, 10, 6),
                                   d_model=64, L=40, seed=3),
    "residual_f32": synth.tiny_workload(d=8, H=2, layers=3, residual=True, V=11, T=4,
                                        W=(5, 7, 6, 4), L=9, seed=5),
}


@pytest.mark.parametrize("name", list(WLS))
def test_oracle_decode_passes_the_stage_check(name):
    wl = WLS[name]
    p = synth.make_params(wl)
    prompt = synth.make_prompt(wl)[0]
    tr = oracle.decode_request(wl, p, prompt)
    calls = _calls_from_oracle(wl, tr)
    for t in range(wl.T - 1):
        anc = ancestry(tr.parents, t)
        e = stage_errors(wl, p, tr.S_ctx, calls, anc, t, range(wl.W[t]), chunk=3)
        assert set(e) >= set(FIELDS) | {"logits", "lse"}
        assert max(e.values()) < 1e-6, (t, e)
        # the selection contract on the oracle's own stored logits
        zs = oracle.kept_scores_f32(calls[t]["logits"], wl.dtype)
        selection_matches(zs, calls[t]["lse"].astype(np.float32), tr.cum[t], wl.W[t + 1], None,
                          tr.parents[t + 1], tr.tokens[t + 1], tr.cum[t + 1])


def test_planted_mistakes_show():
    wl = WLS["residual_f32"]
    p = synth.make_params(wl)
    tr = oracle.decode_request(wl, p, synth.make_prompt(wl)[0])
    calls = _calls_from_oracle(wl, tr)
    t = 2
    anc = ancestry(tr.parents, t)
    ok = stage_errors(wl, p, tr.S_ctx, calls, anc, t, range(wl.W[t]))
    assert max(ok.values()) < 1e-6
    # a wrong ancestor slot at depth 0 changes the replayed state
    bad = anc.copy()
    bad[:, 0] = (bad[:, 0] + 1) % wl.W[0]
    e = stage_errors(wl, p, tr.S_ctx, calls, bad, t, range(wl.W[t]))
    assert e["delta"] > 1e-3 and e["o"] > 1e-3
    # a wrong input token changes every projection
    wrong = [dict(c) for c in calls]
    wrong[t]["tokens"] = (calls[t]["tokens"] + 1) % wl.V
    e = stage_errors(wl, p, tr.S_ctx, wrong, anc, t, range(wl.W[t]))
    assert e["q"] > 1e-3 and e["v"] > 1e-3
    # a dropped layer output in the residual stream changes the feature
    drop = [dict(c) for c in calls]
    drop[t]["o"] = calls[t]["o"].copy()
    drop[t]["o"][0] = 0.0
    e = stage_errors(wl, p, tr.S_ctx, drop, anc, t, range(wl.W[t]))
    assert e["o"] > 1e-3 and e["q"] > 1e-3


def test_selection_mismatch_shows():
    wl = synth.TINY
    p = synth.make_params(wl)
    tr = oracle.decode_request(wl, p, synth.make_prompt(wl)[0])
    zs = oracle.kept_scores_f32(tr.calls[0].z, wl.dtype)
    par = tr.parents[1].copy()
    par[[0, 1]] = par[[1, 0]] if par[0] != par[1] else par[[0, 1]] + 1
    with pytest.raises(AssertionError):
        selection_matches(zs, tr.calls[0].lse.astype(np.float32), tr.cum[0], wl.W[1], None,
                          par, tr.tokens[1], tr.cum[1])
