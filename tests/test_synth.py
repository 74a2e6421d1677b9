"""The seeded input generator: determinism, ranges and the workload recipes (no GPU)."""

import numpy as np
import pytest
import torch

from speculative_decoding_verification_58_gb300 import synth


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100_000).astype(np.float32) * 50,
                        np.array([0.0, -0.0, 1.0, -3.5, 1e-30, 3e38], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(synth.bf16_bits(x), want)
    back = torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(synth.bf16_to_f32(want), back)


def test_uniforms_strictly_inside_unit_interval():
    u = synth.uniform_24bit(np.random.default_rng(1), (1_000_000,))
    assert u.dtype == np.float32 and u.min() >= 0.0 and u.max() < 1.0
    assert np.all(u * 2**24 == np.floor(u * 2**24))


@pytest.mark.parametrize("recipe", synth.RECIPES)
def test_same_inputs_for_any_thread_count(recipe):
    a = synth.make_inputs(recipe, 8, 5, 333, "bf16", seed=5, threads=1)
    b = synth.make_inputs(recipe, 8, 5, 333, "bf16", seed=5, threads=4)
    for f in ("target", "draft", "tokens", "lengths", "uniforms", "temperature"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))


def test_recipe_shapes_and_ranges():
    x = synth.make_inputs("zipf_mixed_temp", 40, 16, 500, "f32", seed=3)
    assert x.target.shape == (40, 17, 500) and x.draft.shape == (40, 16, 500)
    assert x.tokens.shape == (40, 16) and x.uniforms.shape == (40, 17)
    assert (x.temperature == 0).sum() == 10
    t = x.temperature[x.temperature > 0]
    assert t.min() >= 0.5 and t.max() <= 1.2
    assert x.lengths.min() >= 1 and x.lengths.max() <= 16
    assert x.tokens.min() >= 0 and x.tokens.max() < 500
    # greedy requests draft the argmax of their draft row
    g = np.nonzero(x.temperature == 0)[0]
    np.testing.assert_array_equal(x.tokens[g], np.argmax(x.draft[g], axis=2))
    y = synth.make_inputs("zipf_mixed_noise", 40, 16, 500, "bf16", seed=3)
    assert y.lengths.min() >= 4 and np.all(y.temperature == 1)
    assert y.target.dtype == np.uint16


def test_mixed_noise_halves_differ_in_acceptance():
    # The two noise halves should visibly differ: the draft stays closer to the
    # target for the low-noise half.
    x = synth.make_inputs("zipf_mixed_noise", 16, 4, 2000, "f32", seed=9)
    d = np.abs(x.draft[:, 0] - x.target[:, 0]).mean(axis=1)
    lo, hi = np.sort(d)[:8], np.sort(d)[8:]
    assert hi.min() > 3 * lo.max()


def test_workload_table():
    assert synth.HEADLINE in synth.WORKLOADS
    w = synth.WORKLOADS[synth.HEADLINE]
    assert (w["B"], w["k"], w["V"], w["dtype"]) == (128, 16, 151936, "bf16")
