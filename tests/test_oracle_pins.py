"""Pins for the CPU oracle: checks against closed forms, invariants, special
cases and brute force, so that a plausible mistake anywhere in the oracle (a
dropped term, a wrong sign or index, a transposed operand) fails one of them.

Sources are named by page title:
  OneLA   "OneLA: Scaling Linear-Attention Decoding to Large Beams in
           Generative Recommendation" (review page)
  RecoGEM "RecoGEM: A Serving System for Production-Scale Generative
           Recommendation"
"""
import itertools
import math

import numpy as np
import pytest

import oracle
import synth

RNG = np.random.default_rng(1234)


def unit(v):
    return v / np.linalg.norm(v)


# ---------------------------------------------------------------- inputs

def test_l2_normalize_closed_form():
    y = RNG.standard_normal((5, 7))
    yh = oracle.l2_normalize(y)
    ss = (y * y).sum(-1)
    # squared norm is ss / (ss + eps) and the direction is y's
    np.testing.assert_allclose((yh * yh).sum(-1), ss / (ss + 1e-6), rtol=1e-13)
    np.testing.assert_allclose(yh / np.linalg.norm(yh, axis=-1, keepdims=True),
                               y / np.linalg.norm(y, axis=-1, keepdims=True), rtol=1e-13)


def test_rms_normalize_constant_row():
    x = np.full((2, 8), 3.0)
    np.testing.assert_allclose(oracle.rms_normalize(x), 3.0 / math.sqrt(9.0 + 1e-6), rtol=1e-15)


def test_gates_special_values_and_identity():
    assert oracle.decay_gate(np.array(0.0)) == pytest.approx(0.5, abs=1e-15)
    assert oracle.write_gate(np.array(0.0)) == pytest.approx(0.5, abs=1e-15)
    z = np.linspace(-30, 30, 121)
    # exp(-softplus(z)) is the logistic function at -z
    np.testing.assert_allclose(oracle.decay_gate(z), 1.0 / (1.0 + np.exp(z)), rtol=1e-12)
    np.testing.assert_allclose(oracle.write_gate(z), 1.0 / (1.0 + np.exp(-z)), rtol=1e-12)
    # stable at extremes, in (0, 1]
    big = oracle.decay_gate(np.array([-800.0, 800.0]))
    assert big[0] == 1.0 and 0.0 <= big[1] < 1e-300


def test_gdn_inputs_reads_columns_of_the_weights():
    wl = synth.tiny_workload(d=4, V=3, H=2, d_model=6)
    p = synth.make_params(wl)
    for j in range(wl.d_model):
        u = np.zeros((1, wl.d_model)); u[0, j] = 1.0
        q, k, v, a, b = oracle.gdn_inputs(wl, p, 0, u)
        for h in range(wl.H):
            col_q = p.Wq[0][h * wl.d_k:(h + 1) * wl.d_k, j].astype(float)
            np.testing.assert_allclose(q[0, h], col_q / math.sqrt((col_q ** 2).sum() + 1e-6), rtol=1e-12)
            col_k = p.Wk[0][h * wl.d_k:(h + 1) * wl.d_k, j].astype(float)
            np.testing.assert_allclose(k[0, h], col_k / math.sqrt((col_k ** 2).sum() + 1e-6), rtol=1e-12)
            np.testing.assert_allclose(v[0, h], p.Wv[0][h * wl.d_v:(h + 1) * wl.d_v, j], rtol=1e-12)
            assert a[0, h] == pytest.approx(1 / (1 + math.exp(p.w_alpha[0][h, j])), rel=1e-12)
            assert b[0, h] == pytest.approx(1 / (1 + math.exp(-p.w_beta[0][h, j])), rel=1e-12)


# ---------------------------------------------------------------- recurrence

def _rand_state(dv=5, dk=4):
    return RNG.standard_normal((dv, dk)), unit(RNG.standard_normal(dk)), unit(RNG.standard_normal(dk)), RNG.standard_normal(dv)


def test_delta_rule_invariant():
    # beta = 1 and |k| = 1: the new state maps k exactly onto v (OneLA §1.2 eq. 3)
    S, q, k, v = _rand_state()
    for alpha in (0.0, 0.37, 1.0):
        Sn, _, _ = oracle.gdn_transition(S, q, k, v, np.array(alpha), np.array(1.0))
        np.testing.assert_allclose(Sn @ k, v, atol=1e-13)


def test_noop_and_pure_decay():
    S, q, k, v = _rand_state()
    Sn, d, o = oracle.gdn_transition(S, q, k, v, np.array(1.0), np.array(0.0))
    np.testing.assert_array_equal(Sn, S)
    np.testing.assert_array_equal(d, np.zeros_like(v))
    np.testing.assert_allclose(o, S @ q, rtol=1e-14)
    Sn, _, o = oracle.gdn_transition(S, q, k, v, np.array(0.3), np.array(0.0))
    np.testing.assert_allclose(Sn, 0.3 * S, rtol=1e-15)


def test_first_token_from_zero_state():
    # S = 0: S_1 = beta v k^T (rows follow v, columns follow k), o = beta v (k.q)
    _, q, k, v = _rand_state(dv=3, dk=5)
    beta = 0.8
    Sn, d, o = oracle.gdn_transition(np.zeros((3, 5)), q, k, v, np.array(0.6), np.array(beta))
    for i in range(3):
        for j in range(5):
            assert Sn[i, j] == pytest.approx(beta * v[i] * k[j], rel=1e-14, abs=1e-15)
    np.testing.assert_allclose(o, beta * v * (k @ q), rtol=1e-13)
    np.testing.assert_allclose(d, beta * v, rtol=1e-15)


def test_recorded_delta_is_the_rank_one_rewrite():
    # OneLA §2.2 eq. 4: S_t = alpha S + delta k^T with delta = beta (v - alpha S k)
    S, q, k, v = _rand_state(dv=6, dk=6)
    k = RNG.standard_normal(6)            # not unit: the identity holds for any k
    Sn, d, _ = oracle.gdn_transition(S, q, k, v, np.array(0.7), np.array(0.45))
    np.testing.assert_allclose(Sn, 0.7 * S + np.outer(d, k), rtol=1e-12, atol=1e-14)
    # and delta is read off the parent state, not the child
    np.testing.assert_allclose(d, 0.45 * (v - 0.7 * (S @ k)), rtol=1e-12)


def test_two_orthogonal_tokens():
    # k1 _|_ k2 unit, beta2 = 1: S2 k2 = v2 and S2 k1 = alpha2 * beta1 * v1
    basis = np.linalg.qr(RNG.standard_normal((4, 4)))[0]
    k1, k2 = basis[:, 0], basis[:, 1]
    v1, v2 = RNG.standard_normal(3), RNG.standard_normal(3)
    q = unit(RNG.standard_normal(4))
    ks = np.stack([k1, k2])[:, None, :]
    vs = np.stack([v1, v2])[:, None, :]
    S, o = oracle.prefill_scan(np.repeat(q[None, None], 2, 0), ks, vs,
                               np.array([[0.9], [0.4]]), np.array([[0.7], [1.0]]))
    np.testing.assert_allclose(S[0] @ k2, v2, atol=1e-14)
    np.testing.assert_allclose(S[0] @ k1, 0.4 * 0.7 * v1, atol=1e-14)
    np.testing.assert_allclose(o[1, 0], S[0] @ q, rtol=1e-14)


def test_state_from_records_matches_transitions():
    S0, q, _, _ = _rand_state(dv=4, dk=4)
    S = S0.copy()
    recs = []
    for _ in range(3):
        k = unit(RNG.standard_normal(4)); v = RNG.standard_normal(4)
        a, b = RNG.uniform(0.1, 1.0), RNG.uniform(0.0, 1.0)
        S, d, _ = oracle.gdn_transition(S, q, k, v, np.array(a), np.array(b))
        recs.append((a, d, k))
    np.testing.assert_allclose(oracle.state_from_records(S0, recs), S, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- head

def test_logits_read_columns_of_Wo():
    wl = synth.tiny_workload(d=4, V=5, H=2, d_model=8)
    p = synth.make_params(wl)
    for j in range(wl.feat_dim):
        f = np.zeros((1, wl.feat_dim)); f[0, j] = 1.0
        np.testing.assert_allclose(oracle.codebook_logits(p, f)[0], p.Wo[:, j], rtol=1e-15)


def test_log_normalizer():
    z = RNG.standard_normal((4, 11)) * 5
    lse = oracle.log_normalizer(z)
    np.testing.assert_allclose(np.exp(z - lse[:, None]).sum(-1), 1.0, rtol=1e-12)
    np.testing.assert_allclose(oracle.log_normalizer(np.full((1, 7), 2.5)), 2.5 + math.log(7), rtol=1e-15)
    # shift invariance of the normalised scores, with huge logits
    np.testing.assert_allclose(oracle.log_normalizer(z + 1e4) - 1e4, lse, rtol=1e-9)


# ---------------------------------------------------------------- selection

def _brute_select(z32, lse32, cum32, W_next, bias32=None):
    n, V = z32.shape
    items = []
    for b in range(n):
        cp = np.float32(cum32[b]) if bias32 is None else np.float32(np.float32(cum32[b]) + np.float32(bias32[b]))
        for v in range(V):
            s = np.float32(cp + np.float32(np.float32(z32[b, v]) - np.float32(lse32[b])))
            items.append((-float(s), b * V + v, float(s)))
    items.sort()
    keep = items[:W_next]
    return ([f // V for _, f, _ in keep], [f % V for _, f, _ in keep], [s for _, _, s in keep])


@pytest.mark.parametrize("n,V,W", [(1, 7, 3), (4, 5, 20), (6, 9, 6), (3, 4, 12)])
def test_select_matches_brute_force(n, V, W):
    rng = np.random.default_rng(n * 100 + V)
    z = synth.round_bf16(rng.standard_normal((n, V)).astype(np.float32))
    z[:, ::3] = z[:, :1]          # duplicate values inside rows
    if n > 1:
        z[1] = z[0]               # and across rows
    lse = oracle.log_normalizer(z).astype(np.float32)
    cum = rng.standard_normal(n).astype(np.float32)
    cum[-1] = cum[0]
    bias = rng.standard_normal(n).astype(np.float32)
    for bs in (None, bias):
        p, t, s = oracle.select_top(z, lse, cum, W, bs)
        bp, bt, bsc = _brute_select(z, lse, cum, W, bs)
        np.testing.assert_array_equal(p, bp)
        np.testing.assert_array_equal(t, bt)
        np.testing.assert_array_equal(s, np.array(bsc, np.float32))


def test_select_tie_goes_to_lower_flat_index():
    # every candidate equal: the first W flat indices win, in order
    z = np.zeros((3, 4), np.float32)
    p, t, _ = oracle.select_top(z, np.zeros(3, np.float32), np.zeros(3, np.float32), 5)
    np.testing.assert_array_equal(p, [0, 0, 0, 0, 1])
    np.testing.assert_array_equal(t, [0, 1, 2, 3, 0])


def test_select_fp32_rounding_creates_ties():
    # cum' = 2^24: adding 0.25 or 0.5 - 1 ... rounds back to 2^24, so the
    # candidates tie in fp32 and the lower flat index wins
    z = np.array([[0.0, -0.25, 0.5, -0.5]], np.float32)
    lse = np.zeros(1, np.float32)
    cum = np.array([2.0 ** 24], np.float32)
    p, t, s = oracle.select_top(z, lse, cum, 4)
    assert list(s) == [2.0 ** 24] * 4
    np.testing.assert_array_equal(t, [0, 1, 2, 3])


def test_two_stage_precut_is_exact():
    # RecoGEM §4.3: keeping each row's local top-K, then selecting among the
    # survivors, gives the same K winners as one flat selection
    rng = np.random.default_rng(7)
    for trial in range(20):
        n, V = rng.integers(1, 8), rng.integers(2, 12)
        K = int(rng.integers(1, n * V + 1))
        z = synth.round_bf16(rng.standard_normal((n, V)).astype(np.float32))
        z[:, rng.integers(0, V)] = z[:, 0]
        lse = np.zeros(n, np.float32)
        cum = synth.round_bf16(rng.standard_normal(n).astype(np.float32))
        p, t, _ = oracle.select_top(z, lse, cum, K)
        s = oracle.scores_f32(z, lse, cum)
        cand = []
        for b in range(n):
            order = sorted(range(V), key=lambda v: (-s[b, v], v))[:min(K, V)]
            cand += [(-s[b, v], b * V + v) for v in order]
        cand.sort()
        flat = [f for _, f in cand[:K]]
        np.testing.assert_array_equal(p, [f // V for f in flat])
        np.testing.assert_array_equal(t, [f % V for f in flat])


def test_kept_scores_rounding():
    z = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -3.0], np.float64)
    np.testing.assert_array_equal(oracle.kept_scores_f32(z, "bf16"), np.array([1.0, 1.0 + 2 ** -6, -3.0], np.float32))
    np.testing.assert_array_equal(oracle.kept_scores_f32(z, "f32"), z.astype(np.float32))


# ---------------------------------------------------------------- ancestry

def _eq9_ancestry(parents, t):
    # OneLA §2.4 eq. 9, applied call by call
    h = np.zeros((len(parents[0]), 0), np.int32)
    for s in range(1, t + 1):
        pi = parents[s]
        h = np.concatenate([h[pi], pi[:, None].astype(np.int32)], axis=1)
    return h


def test_ancestry_walk_equals_eq9():
    rng = np.random.default_rng(3)
    W = [3, 5, 4, 6, 2]
    parents = [np.zeros(3, np.int32)] + [rng.integers(0, W[s - 1], W[s]).astype(np.int32) for s in range(1, 5)]
    for t in range(5):
        np.testing.assert_array_equal(oracle.ancestry_slots(parents, t), _eq9_ancestry(parents, t))


def test_token_paths_hand_tree():
    parents = [np.array([0, 0]), np.array([1, 0, 1]), np.array([2, 2, 0])]
    tokens = [np.array([7, 8]), np.array([1, 2, 3]), np.array([4, 5, 6])]
    sid = oracle.token_paths(parents, tokens)
    # beam 0: parent 2 (token 3, parent 1 -> token 8); beam 2: parent 0 (token 1, parent 1 -> 8)
    np.testing.assert_array_equal(sid, [[8, 3, 4], [8, 3, 5], [8, 1, 6]])


# ---------------------------------------------------------------- decoder

def test_exhaustive_beam_keeps_every_sequence():
    # V = 3, T = 3, W >= V^T: every sequence survives, and each final score is
    # the sum of per-step log-probabilities of an independent single-path decode
    wl = synth.tiny_workload(d=4, V=3, T=3, W=(3, 9, 27), L=6, seed=5)
    p = synth.make_params(wl)
    prompt = synth.make_prompt(wl)[0]
    tr = oracle.decode_request(wl, p, prompt)
    assert sorted(map(tuple, tr.sid.tolist())) == sorted(itertools.product(range(3), repeat=3))
    S_ctx, _ = oracle.prefill(wl, p, prompt)
    for b, seq in enumerate(tr.sid.tolist()):
        _, zs, lses = oracle.chain_decode(wl, p, S_ctx, seq[:-1])
        logp = tr.root_z[seq[0]] - tr.root_lse
        for t in range(2):
            logp += zs[t][seq[t + 1]] - lses[t]
        assert tr.cum[-1][b] == pytest.approx(logp, rel=2e-6, abs=2e-6)


def test_greedy_width_one():
    wl = synth.tiny_workload(d=4, V=5, T=4, W=(1, 1, 1, 1), L=4, seed=6)
    p = synth.make_params(wl)
    prompt = synth.make_prompt(wl)[0]
    tr = oracle.decode_request(wl, p, prompt)
    S_ctx, feat = oracle.prefill(wl, p, prompt)
    seq = [int(np.argmax(oracle.codebook_logits(p, feat[None])[0]))]
    for t in range(3):
        _, zs, _ = oracle.chain_decode(wl, p, S_ctx, seq)
        seq.append(int(np.argmax(zs[-1])))
    assert tr.sid[0].tolist() == seq


def _replay(S_ctx, recs, h, t, q, k, v, alpha, beta):
    """Projection replay, OneLA §2.3 eqs. 6-8, for one beam and head."""
    uq, uk = S_ctx @ q, S_ctx @ k
    for j in range(t):
        a_j, d_j, k_j = recs[j][h[j]]
        uq = a_j * uq + d_j * (k_j @ q)
        uk = a_j * uk + d_j * (k_j @ k)
    delta = beta * (v - alpha * uk)
    return delta, alpha * uq + delta * (k @ q)


@pytest.mark.parametrize("residual,layers,forced", [(False, 1, False), (False, 1, True), (True, 2, True)])
def test_projection_replay_equals_fullstate(residual, layers, forced):
    # The method's claim (OneLA §2.3): replaying the two projections along the
    # ancestry gives the FullState o and delta exactly (up to rounding).
    wl = synth.tiny_workload(d=6, V=3, T=5, W=(3, 4, 4, 3, 2), H=2, layers=layers,
                             residual=residual, d_model=12, L=7, seed=8)
    p = synth.make_params(wl)
    prompt = synth.make_prompt(wl)[0]
    lin = None
    if forced:
        par, tok = synth.random_lineage(wl, seed=1)
        lin = ([x[0] for x in par], [x[0] for x in tok])
    tr = oracle.decode_request(wl, p, prompt, forced=lin)
    for t, call in enumerate(tr.calls):
        h = oracle.ancestry_slots(tr.parents, t)
        for layer in range(layers):
            for b in range(wl.W[t]):
                for hd in range(wl.H):
                    recs = [[(tr.calls[j].alpha[layer][s, hd], tr.calls[j].delta[layer][s, hd],
                              tr.calls[j].k[layer][s, hd]) for s in range(wl.W[j])] for j in range(t)]
                    d, o = _replay(tr.S_ctx[layer, hd], recs, h[b], t, call.q[layer][b, hd],
                                   call.k[layer][b, hd], call.v[layer][b, hd],
                                   call.alpha[layer][b, hd], call.beta[layer][b, hd])
                    np.testing.assert_allclose(d, call.delta[layer][b, hd], rtol=1e-12, atol=1e-13)
                    np.testing.assert_allclose(o, call.o[layer][b, hd], rtol=1e-12, atol=1e-13)


def test_step_from_records_equals_decode():
    wl = synth.tiny_workload(d=5, V=3, T=4, W=(3, 5, 4, 4), H=2, d_model=10, L=5, seed=9)
    p = synth.make_params(wl)
    tr = oracle.decode_request(wl, p, synth.make_prompt(wl)[0])
    t = 2
    h = oracle.ancestry_slots(tr.parents, t)
    c = tr.calls[t]
    for b in range(wl.W[t]):
        recs = [(tr.calls[j].alpha[0][h[b, j]], tr.calls[j].delta[0][h[b, j]], tr.calls[j].k[0][h[b, j]])
                for j in range(t)]
        d, o = oracle.step_from_records(tr.S_ctx[0], recs, c.q[0][b], c.k[0][b], c.v[0][b], c.alpha[0][b], c.beta[0][b])
        np.testing.assert_allclose(d, c.delta[0][b], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(o, c.o[0][b], rtol=1e-12, atol=1e-13)


def test_forced_lineage_is_followed():
    wl = synth.tiny_workload(d=4, V=3, T=3, W=(2, 3, 3), L=4, seed=10)
    p = synth.make_params(wl)
    par, tok = synth.random_lineage(wl, seed=2)
    lin = ([x[0] for x in par], [x[0] for x in tok])
    tr = oracle.decode_request(wl, p, synth.make_prompt(wl)[0], forced=lin)
    for s in range(wl.T):
        np.testing.assert_array_equal(tr.parents[s], lin[0][s])
        np.testing.assert_array_equal(tr.tokens[s], lin[1][s])
    for t in range(wl.T - 1):
        np.testing.assert_array_equal(tr.calls[t].tokens, lin[1][t])


def test_bias_shifts_parent_scores():
    # a bias on a parent adds to every candidate of its row (RecoGEM-style
    # per-parent score adjustment read as cum' = cum + bias)
    wl = synth.tiny_workload(d=4, V=3, T=2, W=(3, 3), L=4, seed=12)
    p = synth.make_params(wl)
    prompt = synth.make_prompt(wl)[0]
    bias = np.zeros((1, 3), np.float32); bias[0, 2] = 100.0
    tr = oracle.decode_request(wl, p, prompt, bias=bias)
    assert set(tr.parents[1].tolist()) == {2}


# ---------------------------------------------------------------- stacked glue

def _deep(seed=21, layers=2):
    return synth.tiny_workload(d=4, V=3, T=3, W=(2, 4, 8), H=2, layers=layers,
                               residual=True, d_model=8, L=5, seed=seed)


def test_prelayer_rmsnorm_makes_first_layer_scale_invariant():
    # RMSNorm before the first layer: scaling the embedding table leaves the
    # first layer's outputs unchanged (up to the eps inside the norm)
    wl = _deep()
    p = synth.make_params(wl)
    prompt = synth.make_prompt(wl)[0]
    lin = tuple([x[0] for x in y] for y in synth.random_lineage(wl, seed=4))
    a = oracle.decode_request(wl, p, prompt, forced=lin)
    p.E = p.E * 7.0
    b = oracle.decode_request(wl, p, prompt, forced=lin)
    np.testing.assert_allclose(b.calls[0].o[0], a.calls[0].o[0], rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(b.S_ctx[0], a.S_ctx[0], rtol=1e-5, atol=1e-7)


def test_silenced_top_layer_reduces_to_shallower_stack():
    # W_v = 0 in the top layer: its state stays 0, it adds nothing to the
    # residual stream, so the 2-layer model equals the 1-layer one
    wl2 = _deep(layers=2)
    p2 = synth.make_params(wl2)
    p2.Wv[1] = np.zeros_like(p2.Wv[1])
    wl1 = wl2.with_(layers=1)
    p1 = synth.Params(p2.E, p2.Wq[:1], p2.Wk[:1], p2.Wv[:1], p2.w_alpha[:1], p2.w_beta[:1], p2.Wo)
    prompt = synth.make_prompt(wl2)[0]
    a = oracle.decode_request(wl2, p2, prompt)
    b = oracle.decode_request(wl1, p1, prompt)
    np.testing.assert_allclose(a.root_z, b.root_z, rtol=1e-12)
    np.testing.assert_array_equal(a.sid, b.sid)
    np.testing.assert_allclose(a.calls[-1].z, b.calls[-1].z, rtol=1e-12)
    assert np.all(a.calls[-1].o[1] == 0.0)


def test_stacked_beam_decode_equals_single_paths():
    wl = _deep(layers=2).with_(W=(3, 9, 27))
    p = synth.make_params(wl)
    prompt = synth.make_prompt(wl)[0]
    tr = oracle.decode_request(wl, p, prompt)
    assert len({tuple(s) for s in tr.sid.tolist()}) == 27
    for b, seq in enumerate(tr.sid.tolist()):
        feats, zs, lses = oracle.chain_decode(wl, p, tr.S_ctx, seq[:-1])
        logp = tr.root_z[seq[0]] - tr.root_lse + sum(zs[t][seq[t + 1]] - lses[t] for t in range(2))
        assert tr.cum[-1][b] == pytest.approx(logp, rel=2e-6, abs=2e-6)


# ---------------------------------------------------------------- page figures

def test_page_record_size_figures():
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "onela_record_sizes.json")))
    d_v, d_k = g["d_v"], g["d_k"]
    # a record is (alpha, delta, k): 1 + d_v + d_k elements; a state d_v x d_k
    assert 1 + d_v + d_k == g["gtr_elements"]
    assert d_v * d_k == g["fullstate_elements"]
    assert round(g["fullstate_elements"] / g["gtr_elements"], 1) == g["per_record_saving_reviewer"]
    W, T = 512, 2
    ratio = W * d_v * d_k / (d_v * d_k + W * T * (d_v + d_k + 1))
    assert abs(ratio - g["capacity_ratio_W512_T2_approx"]) < 1.0
    c = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "recogem_candidates.json")))
    assert round(c["C"] * c["W"] / 1e6, 1) == c["candidates_millions_approx"]
    assert c["C"] * c["W"] * 2 / 2 ** 20 == c["fp16_MiB"]


# ---------------------------------------------------------------- grouped key heads

@pytest.mark.parametrize("residual", [False, True])
def test_gqa_equals_mha_with_repeated_key_weights(residual):
    # Grouped query attention (Hk key heads shared by consecutive value heads)
    # is the multi-head model whose query/key weight rows are repeated per
    # group: the two decodes must agree to rounding.
    layers = 2 if residual else 1
    g = synth.tiny_workload(d=4, V=5, T=3, W=(4, 6, 5), H=4, H_k=2, d_v=3, layers=layers,
                            residual=residual, d_model=12, L=6, seed=21)
    m = g.with_(H_k=0)
    pg = synth.make_params(g)
    rep = lambda Ws: [np.repeat(Wl.reshape(g.Hk, g.d_k, -1), g.H // g.Hk, axis=0).reshape(g.H * g.d_k, -1)
                      for Wl in Ws]
    import dataclasses
    pm = dataclasses.replace(pg, Wq=rep(pg.Wq), Wk=rep(pg.Wk))
    prompt = synth.make_prompt(g)[0]
    tg = oracle.decode_request(g, pg, prompt)
    tm = oracle.decode_request(m, pm, prompt)
    np.testing.assert_allclose(tg.S_ctx, tm.S_ctx, rtol=1e-12, atol=1e-14)
    for cg, cm in zip(tg.calls, tm.calls):
        np.testing.assert_allclose(cg.z, cm.z, rtol=1e-12, atol=1e-14)
        for layer in range(layers):
            np.testing.assert_allclose(oracle.per_value_head(g, cg.k[layer]), cm.k[layer], rtol=1e-12)
            np.testing.assert_allclose(cg.delta[layer], cm.delta[layer], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(tg.sid, tm.sid)


def test_gqa_value_heads_share_their_group_key():
    # value heads 0,1 read key head 0 and heads 2,3 key head 1: a decode where
    # only key head 1's weights change leaves value heads 0 and 1 untouched
    import dataclasses
    wl = synth.tiny_workload(d=4, V=5, T=2, W=(3, 3), H=4, H_k=2, d_model=10, L=5, seed=5)
    p = synth.make_params(wl)
    Wk2 = [w.copy() for w in p.Wk]
    Wk2[0][wl.d_k:] *= -0.5
    p2 = dataclasses.replace(p, Wk=Wk2)
    prompt = synth.make_prompt(wl)[0]
    S1 = oracle.prefill(wl, p, prompt)[0]
    S2 = oracle.prefill(wl, p2, prompt)[0]
    np.testing.assert_array_equal(S1[:, :2], S2[:, :2])
    assert np.abs(S1[:, 2:] - S2[:, 2:]).max() > 1e-6


def test_layer_feature_is_the_normalised_stream_or_the_outputs():
    # the codebook head reads RMSNorm(x) of the residual stream on stacked
    # layers (unit root-mean-square, no gain, direction kept) and concat_h o
    # unchanged on a single layer
    rng = np.random.default_rng(21)
    # (row scales >= 1, where the norm's eps of 1e-6 moves the result < 1e-6)
    x = rng.standard_normal((4, 96)) * np.array([[1.0], [3.0], [7.0], [300.0]])
    f = oracle.layer_feature(synth.DEEP, x)
    rms = np.sqrt((f ** 2).mean(axis=-1))
    np.testing.assert_allclose(rms, 1.0, rtol=1e-6)
    ratio = f / x
    np.testing.assert_allclose(ratio, ratio[:, :1] * np.ones_like(ratio), rtol=1e-12)
    assert np.all(ratio > 0)
    np.testing.assert_array_equal(oracle.layer_feature(synth.SINGLE, x), x)
