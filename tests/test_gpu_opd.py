"""OPD supervision statistics on the GPU vs the fp64 oracle, through the C-ABI (needs a GB300).

AdaFlash Section 3.1: per verified position the target argmax (exact, lowest
index on ties), -log q(argmax), the reverse KL and its entry-wise clipped
form, and per request the alpha mixture loss.

Tolerance.  The kernel works in fp32: each term q log(q/p) carries a relative
error of a few 1e-7 (one ex2.approx, the float normalisers), per-thread sums
run over at most a few hundred terms in fp32 and everything above that is
added in float-float.  The error of a sum is therefore about
(terms per thread) * 2^-24 * sum |term| ~ 1e-5 * sum |term| at worst, and
sum |term| stays below a few units for these rows; the test allows
3e-5 + 3e-5 * |value|.
"""

import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import speculative_decoding_verification_58_gb300 as sv
from speculative_decoding_verification_58_gb300 import synth
from parity import compare, oracle_opd_threads

pytestmark = pytest.mark.gpu

ATOL = 3e-5
RTOL = 3e-5
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.lib()


def run(inp, delta=0.01, alpha=0.8):
    d = sv.to_device(inp)
    r = sv.spec_opd_stats(d["target_logits"], d["draft_logits"], d["lengths"], delta=delta,
                          alpha=alpha)
    torch.cuda.synchronize()
    return {k: getattr(r, k).cpu().numpy() for k in ("x_star", "hard", "rkl", "rkl_clip", "loss")}


def check(inp, label, delta=0.01, alpha=0.8):
    g = run(inp, delta, alpha)
    o = oracle.opd_stats(inp.target, inp.draft, inp.lengths, delta=delta, alpha=alpha)
    np.testing.assert_array_equal(g["x_star"], o.x_star, err_msg=label)
    for name in ("hard", "rkl", "rkl_clip"):
        want = getattr(o, name)
        np.testing.assert_allclose(g[name], want, rtol=RTOL, atol=ATOL, equal_nan=True,
                                   err_msg=f"{label}: {name}")
    np.testing.assert_allclose(g["loss"], o.loss, rtol=RTOL, atol=ATOL, equal_nan=True,
                               err_msg=f"{label}: loss")
    return g, o


@pytest.mark.parametrize("recipe,B,k,V,dtype", [
    ("gauss", 1, 4, 1024, "f32"),
    ("zipf_mixed_temp", 9, 16, 5000, "bf16"),
    ("zipf_mixed_temp", 5, 7, 4099, "f32"),         # rows not 16-byte aligned: plain loads
    ("zipf_mixed_noise", 8, 3, 257, "bf16"),
    ("zipf_adaptive", 3, 16, 151936, "bf16"),       # the pages' vocabulary: clusters of 8
    ("zipf_mixed_noise", 2, 5, 151936, "f32"),      # clusters of 16
    ("zipf_adaptive", 4, 16, 32000, "bf16"),        # clusters of 2
    ("gauss", 2, 3, 70001, "f32"),                  # clusters of 4, rows not aligned
    ("gauss", 3, 2, 7, "f32"),
    ("gauss", 2, 3, 1, "bf16"),
])
def test_opd_matches_oracle(recipe, B, k, V, dtype):
    inp = synth.make_inputs(recipe, B, k, V, dtype, seed=60 + B + V)
    check(inp, f"{recipe} B={B} k={k} V={V} {dtype}")


def test_opd_worked_example_of_the_notes():
    g = json.load(open(os.path.join(GOLDEN, "opd_worked_example.json")))
    t = np.zeros((1, 2, 4), np.float32)
    d = np.zeros((1, 1, 4), np.float32)
    t[0, 0] = np.log(np.array(g["p_target"]))
    d[0, 0] = np.log(np.array(g["q_draft"]))
    inp = synth.SpecInputs(t, d, np.zeros((1, 1), np.int32), np.ones(1, np.int32),
                           np.zeros((1, 2), np.float32), np.ones(1, np.float32), "f32")
    r, _ = check(inp, "worked example", delta=g["delta"], alpha=g["alpha"])
    tol = g["printed_tolerance"]
    assert r["x_star"][0, 0] == g["printed"]["x_star"]
    assert abs(r["hard"][0, 0] - g["printed"]["hard"]) < tol
    assert abs(r["rkl"][0, 0] - g["printed"]["rkl"]) < tol


def _opd_close(g, o, label, rows=slice(None)):
    np.testing.assert_array_equal(g["x_star"][rows], o.x_star, err_msg=label)
    for name in ("hard", "rkl", "rkl_clip"):
        np.testing.assert_allclose(g[name][rows], getattr(o, name), rtol=RTOL, atol=ATOL,
                                   equal_nan=True, err_msg=f"{label}: {name}")
    np.testing.assert_allclose(g["loss"][rows], o.loss, rtol=RTOL, atol=ATOL, equal_nan=True,
                               err_msg=f"{label}: loss")


def test_opd_headline_workload_every_request():
    """B=128, k=16, V=151936 bf16 as the benchmark runs it; all 128 requests
    against the oracle (over host threads)."""
    inp = synth.make_workload(synth.HEADLINE)
    g = run(inp)
    _opd_close(g, oracle_opd_threads(inp), "headline")
    # Every position past L_b is -1 / NaN; every verified one is finite.
    for b in range(inp.B):
        L = inp.lengths[b]
        assert np.all(g["x_star"][b, L:] == -1) and np.all(np.isnan(g["rkl"][b, L:]))
        assert np.all(np.isfinite(g["rkl_clip"][b, :L])) and np.all(g["rkl"][b, :L] >= -ATOL)


# ---------------------------------------------------------------------------
# Verification and statistics in one pass (spec_verify_opd)
# ---------------------------------------------------------------------------

def run_fused(inp, delta=0.01, alpha=0.8):
    d = sv.to_device(inp)
    ws = sv.alloc_workspace(inp.B, inp.k, inp.V)
    out, n, st = sv.spec_verify_opd(**d, delta=delta, alpha=alpha, workspace=ws)
    rep = sv.spec_verify_report(ws)
    g = {k: getattr(st, k).cpu().numpy() for k in ("x_star", "hard", "rkl", "rkl_clip", "loss")}
    return out.cpu().numpy(), n.cpu().numpy(), g, rep


def check_fused(inp, label, delta=0.01, alpha=0.8):
    out, n, g, rep = run_fused(inp, delta, alpha)
    o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                      inp.temperature)
    info = compare(out, n, o, inp.temperature, label)
    _opd_close(g, oracle.opd_stats(inp.target, inp.draft, inp.lengths, delta=delta, alpha=alpha),
               label)
    return info, rep


@pytest.mark.parametrize("recipe,B,k,V,dtype", [
    ("gauss", 1, 4, 1024, "f32"),
    ("zipf_mixed_noise", 24, 16, 5000, "bf16"),     # T = 1: one set of normalisers
    ("zipf_mixed_temp", 40, 8, 6000, "bf16"),       # greedy and T != 1: second sums
    ("zipf_adaptive", 16, 16, 70001, "f32"),        # clusters of 4, rows not aligned
    ("zipf_mixed_temp", 12, 5, 151936, "bf16"),     # the pages' vocabulary
    ("gauss", 3, 2, 7, "f32"),
])
def test_fused_verification_and_statistics_match_oracle(recipe, B, k, V, dtype):
    inp = synth.make_inputs(recipe, B, k, V, dtype, seed=80 + B + V)
    info, rep = check_fused(inp, f"fused {recipe} B={B} k={k} V={V} {dtype}")
    assert rep.status == sv.SPEC_OK, rep


def test_fused_headline_workload_every_request():
    inp = synth.make_workload(synth.HEADLINE)
    out, n, g, rep = run_fused(inp)
    o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                      inp.temperature)
    compare(out, n, o, inp.temperature, "fused headline")
    _opd_close(g, oracle_opd_threads(inp), "fused headline")
    assert rep.status == sv.SPEC_OK, rep


def test_fused_invalid_request_keeps_its_statistics():
    """A token out of range invalidates the verification of its request (-1),
    while its statistics, which do not use tokens, are still computed."""
    inp = synth.make_inputs("zipf_mixed_noise", 6, 4, 900, "bf16", seed=85)
    inp.tokens[2, 0] = 900
    out, n, g, rep = run_fused(inp)
    o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                      inp.temperature)
    assert n[2] == -1 and np.all(out[2] == -1) and o.num_accepted[2] == -1
    compare(out, n, o, inp.temperature, "fused, one invalid request")
    _opd_close(g, oracle.opd_stats(inp.target, inp.draft, inp.lengths), "fused, invalid request")
    assert rep.status == sv.SPEC_ERR_BAD_INPUT and rep.bad_requests == 1


def test_opd_special_cases():
    rng = np.random.default_rng(4)
    B, k, V = 6, 3, 3000
    t = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    d = (t[:, :k] + rng.standard_normal((B, k, V))).astype(np.float32)
    d[0] = t[0, :k]                      # p == q: no divergence
    d[1, 0, :100] = -np.inf              # q = 0 entries add nothing
    t[2, 1, 200:300] = -np.inf           # q > 0 where p = 0: rkl = +inf, clipped to delta
    t[3, 0, 5] = t[3, 0, 9] = t[3, 0].max() + 1  # argmax tie: lowest index
    d[4, 2, 7] = np.nan                  # a row without finite mass
    lens = np.array([3, 3, 3, 2, 3, 0], np.int32)  # request 5: invalid length
    inp = synth.SpecInputs(t, d, np.zeros((B, k), np.int32), lens,
                           np.zeros((B, k + 1), np.float32), np.ones(B, np.float32), "f32")
    g, o = check(inp, "special cases")
    assert np.all(np.abs(g["rkl"][0]) < ATOL) and np.all(np.abs(g["rkl_clip"][0]) < ATOL)
    assert g["rkl"][2, 1] == np.inf and np.isfinite(g["rkl_clip"][2, 1])
    assert g["x_star"][3, 0] == 5
    assert np.isnan(g["hard"][4, 2]) and g["x_star"][4, 2] == -1 and np.isnan(g["loss"][4])
    assert np.all(g["x_star"][5] == -1) and np.isnan(g["loss"][5])


@pytest.mark.parametrize("shift", [12.0, -9.0])
def test_opd_shifted_draft_logits(shift):
    """Logits are defined up to a constant per row: a draft row shifted by a
    large constant has the same q.  Every term q (dz - c) then holds the shift
    twice, in dz = z_d - z_t and in c = lse_d - lse_t, so this checks that the
    divergence, small here, is not lost to the large parts that cancel."""
    rng = np.random.default_rng(int(abs(shift)) + 30)
    B, k, V = 4, 4, 151936
    t = (rng.standard_normal((B, k + 1, V)) * 1.5).astype(np.float32)
    d = (t[:, :k] + rng.standard_normal((B, k, V)).astype(np.float32) * np.float32(0.05)
         + np.float32(shift)).astype(np.float32)
    inp = synth.SpecInputs(t, d, np.zeros((B, k), np.int32), np.array([4, 3, 2, 1], np.int32),
                           np.zeros((B, k + 1), np.float32), np.ones(B, np.float32), "f32")
    check(inp, f"draft shifted by {shift}")


def test_opd_sharply_peaked_rows():
    """Logits scaled so that p and q are nearly one-hot: where the two
    argmaxes differ the reverse KL and the hard-label term reach tens of nats
    and a few entries carry them; a row pair that differs only by a shift
    has no divergence."""
    rng = np.random.default_rng(77)
    B, k, V = 6, 4, 30000
    t = (rng.standard_normal((B, k + 1, V)) * 40).astype(np.float32)
    d = (t[:, :k] + rng.standard_normal((B, k, V)).astype(np.float32) * np.float32(8)).astype(
        np.float32)
    d[0] = t[0, :k] + np.float32(0.5)  # same argmaxes, shifted rows: divergence 0
    inp = synth.SpecInputs(t, d, np.zeros((B, k), np.int32), np.full(B, k, np.int32),
                           np.zeros((B, k + 1), np.float32), np.ones(B, np.float32), "f32")
    g, o = check(inp, "peaked rows")
    assert np.max(o.rkl) > 10 and np.max(o.hard) > 10


def test_opd_host_checks():
    d = sv.to_device(synth.make_inputs("gauss", 2, 3, 64, "f32", seed=1))
    for kw in (dict(delta=0.0), dict(delta=float("inf")), dict(alpha=1.5), dict(alpha=-0.1)):
        with pytest.raises(sv.SpecVerifyError):
            sv.spec_opd_stats(d["target_logits"], d["draft_logits"], d["lengths"], **kw)


def test_opd_many_requests():
    """More requests than a grid's y extent holds; every position in one launch."""
    rng = np.random.default_rng(8)
    B, k, V = 70000, 2, 16
    t = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    d = (t[:, :k] + rng.standard_normal((B, k, V))).astype(np.float32)
    L = rng.integers(1, k + 1, B).astype(np.int32)
    big = synth.SpecInputs(t, d, np.zeros((B, k), np.int32), L, np.zeros((B, k + 1), np.float32),
                           np.ones(B, np.float32), "f32")
    check(big, "B=70000")


def test_opd_largest_vocabulary():
    V = 1 << 21
    rng = np.random.default_rng(21)
    t = (rng.standard_normal((2, 3, V)) * 2).astype(np.float32)
    d = (t[:, :2] + rng.standard_normal((2, 2, V))).astype(np.float32)
    inp = synth.SpecInputs(t, d, np.zeros((2, 2), np.int32), np.array([2, 1], np.int32),
                           np.zeros((2, 3), np.float32), np.ones(2, np.float32), "f32")
    check(inp, "V=2^21")
