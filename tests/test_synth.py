"""The seeded input module: determinism and bf16 rounding (checked against
torch's own float32 -> bfloat16 conversion, an independent implementation)."""
import numpy as np
import torch

import synth


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 100000),
                        np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 65504.0], np.float32)]).astype(np.float32)
    ours = synth.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_params_deterministic_and_rounded():
    wl = synth.tiny_workload(d=4, V=6, H=2, d_model=8, dtype="bf16")
    a, b = synth.make_params(wl), synth.make_params(wl)
    np.testing.assert_array_equal(a.E, b.E)
    np.testing.assert_array_equal(a.Wo, b.Wo)
    np.testing.assert_array_equal(synth.round_bf16(a.Wq[0]), a.Wq[0])
    np.testing.assert_array_equal(synth.make_prompt(wl), synth.make_prompt(wl))


def test_workload_schedules():
    assert synth.TINY.W == (8, 8, 8)
    assert synth.BATCHED.W == (512, 512, 512, 512)
    assert synth.BATCHED.beam_steps == 3 * 64 * 512
    assert synth.SKEWED.W == (256, 1024, 1024, 1024)
    assert synth.DEEP.feat_dim == 1024 and synth.SINGLE.feat_dim == 2048


def test_random_lineage_valid():
    wl = synth.SKEWED.with_(R=3)
    par, tok = synth.random_lineage(wl, seed=0)
    assert np.all(par[0] == 0)
    for s in range(1, wl.T):
        assert par[s].shape == (3, wl.W[s]) and par[s].max() < wl.W[s - 1] and par[s].min() >= 0
        assert tok[s].max() < wl.V
