"""CUDA path vs the CPU oracle, through the C-ABI (needs a GB300).

out_tokens and num_accepted must match bit for bit, except for requests
whose outcome depends on a decision within 1e-6 of its threshold (counted,
at most 1e-5 of the logit rows evaluated); greedy requests match with no
exemption.  Per-row max and argmax are exact, log-sum-exp within 1e-5
relative.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import speculative_decoding_verification_58_gb300 as sv
from speculative_decoding_verification_58_gb300 import synth
from parity import compare

pytestmark = pytest.mark.gpu

LSE_RTOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.lib()


def run_gpu(inp, full_sweep=False, workspace=None):
    d = sv.to_device(inp)
    ws = workspace if workspace is not None else sv.alloc_workspace(inp.B, inp.k, inp.V)
    out, n = sv.spec_verify(**d, workspace=ws, full_sweep=full_sweep)
    rep = sv.spec_verify_report(ws)
    return out.cpu().numpy(), n.cpu().numpy(), rep


def check(inp, label, full_sweep=False):
    out, n, rep = run_gpu(inp, full_sweep=full_sweep)
    o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms, inp.temperature)
    info = compare(out, n, o, inp.temperature, label)
    assert rep.status == sv.SPEC_OK, rep
    assert rep.bad_requests == 0
    return info, rep, o


# ---------------------------------------------------------------------------
# Row statistics (the sweep alone)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 7, 1000, 4097, 151936])
def test_row_stats_match_oracle(dtype, V):
    rng = np.random.default_rng(V)
    rows = 24 if V > 100000 else 61
    z = (rng.standard_normal((rows, V)) * 2.5).astype(np.float32)
    if V > 3:
        z[0, V // 3] = z[0, V // 2] = z[0].max() + 2  # argmax tie
    buf = synth.bf16_bits(z) if dtype == "bf16" else z
    temp = rng.uniform(0.5, 1.5, rows).astype(np.float32)
    temp[::5] = 0.0
    mx_o, lse_o, arg_o = oracle.row_stats(buf, temp)
    t = torch.from_numpy(buf.view(np.int16)).view(torch.bfloat16) if dtype == "bf16" \
        else torch.from_numpy(buf)
    mx, lse, arg = sv.spec_row_stats(t.cuda(), torch.from_numpy(temp).cuda())
    mx, lse, arg = mx.cpu().numpy(), lse.cpu().numpy(), arg.cpu().numpy()
    np.testing.assert_array_equal(mx.astype(np.float64), mx_o)
    greedy = temp == 0
    np.testing.assert_array_equal(arg[greedy], arg_o[greedy])
    np.testing.assert_allclose(lse[~greedy], lse_o[~greedy], rtol=LSE_RTOL, atol=1e-6)


# ---------------------------------------------------------------------------
# Verification on reduced and full workloads
# ---------------------------------------------------------------------------

SMALL = [
    ("gauss", 1, 4, 1024, "f32"),
    ("zipf", 3, 16, 4096, "bf16"),
    ("zipf_adaptive", 32, 16, 8200, "bf16"),
    ("zipf_mixed_noise", 64, 16, 5000, "bf16"),
    ("zipf_mixed_temp", 64, 16, 6000, "f32"),
    ("zipf_mixed_temp", 40, 7, 1001, "bf16"),   # rows not 16-byte aligned
    ("zipf_mixed_noise", 17, 3, 333, "f32"),
    ("zipf_adaptive", 5, 1, 9, "bf16"),
    ("zipf_adaptive", 40, 31, 2000, "bf16"),   # SPEC_MAX_K: 31 positions, 32-bit masks
    ("zipf_mixed_temp", 24, 31, 1500, "f32"),
]


@pytest.mark.parametrize("recipe,B,k,V,dtype", SMALL)
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_verify_small_matches_oracle(recipe, B, k, V, dtype, seed):
    inp = synth.make_inputs(recipe, B, k, V, dtype, seed=seed)
    check(inp, f"{recipe} B={B} k={k} V={V} {dtype} seed={seed}")


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_verify_full_workloads_match_oracle(name):
    inp = synth.make_workload(name)
    info, rep, o = check(inp, name)
    # Every row the oracle needed was swept, and no more than the plan.
    assert rep.rows_planned == int(np.sum(np.where(inp.temperature == 0, 1, 2) * inp.lengths))
    assert rep.chunks_swept <= rep.rows_planned * rep.chunks_per_row


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
@pytest.mark.parametrize("extra", [1, 2, 3, 4])
def test_full_workloads_more_seeds_match_oracle(name, extra):
    """Four more seeded instances of every workload, each compared in full."""
    seed = synth.WORKLOADS[name]["seed"] + 1000 * extra
    inp = synth.make_workload(name, seed=seed)
    check(inp, f"{name} seed={seed}")


@pytest.mark.parametrize("name", ["b128_k16_v151936_bf16_zipf_mixed_noise"])
def test_full_sweep_flag_gives_same_outputs(name):
    inp = synth.make_workload(name, seed=777)
    a_out, a_n, a_rep = run_gpu(inp)
    b_out, b_n, b_rep = run_gpu(inp, full_sweep=True)
    np.testing.assert_array_equal(a_out, b_out)
    np.testing.assert_array_equal(a_n, b_n)
    assert b_rep.chunks_swept == b_rep.rows_planned * b_rep.chunks_per_row
    assert a_rep.chunks_swept <= b_rep.chunks_swept


def test_repeated_calls_are_deterministic_and_reuse_workspace():
    inp = synth.make_inputs("zipf_mixed_temp", 48, 16, 20000, "bf16", seed=5)
    small = synth.make_inputs("gauss", 2, 4, 300, "bf16", seed=6)
    ws = sv.alloc_workspace(48, 16, 20000)
    a = run_gpu(inp, workspace=ws)
    run_gpu(small, workspace=ws)  # a different, smaller call on the same workspace
    b = run_gpu(inp, workspace=ws)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ---------------------------------------------------------------------------
# Edge cases
# ---------------------------------------------------------------------------

def _inputs(B, k, V, dtype="f32", seed=0, T=1.0):
    rng = np.random.default_rng(seed)
    tl = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    dl = (tl[:, :k] + rng.standard_normal((B, k, V)) * 0.7).astype(np.float32)
    inp = synth.SpecInputs(tl, dl, rng.integers(0, V, (B, k)).astype(np.int32),
                           np.full(B, k, np.int32), synth.uniform_24bit(rng, (B, k + 1)),
                           np.full(B, T, np.float32), "f32")
    if dtype == "bf16":
        inp.target, inp.draft, inp.dtype = synth.bf16_bits(tl), synth.bf16_bits(dl), "bf16"
    return inp


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_p_equals_q_always_accepts(dtype):
    inp = _inputs(64, 8, 3000, dtype, seed=1)
    inp.draft = inp.target[:, :8].copy()
    inp.uniforms[:, :8] = np.float32(1.0 - 2.0**-24)
    inp.lengths = np.random.default_rng(2).integers(1, 9, 64).astype(np.int32)
    out, n, _ = run_gpu(inp)
    np.testing.assert_array_equal(n, inp.lengths)
    check(inp, "p == q")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [1e-3, 0.05, 0.2, 8.0, 100.0])
def test_extreme_temperatures_match_oracle(dtype, T):
    """Every request at one temperature far from 1: at T = 1e-3 both rows are
    nearly one-hot (scaled logits in the thousands of bits), at T = 100 both
    are nearly uniform and the residual max(0, p - q) is small.  Each draft
    token is drawn from q at the request's own temperature (Gumbel-max on
    the stored draft logits), as a drafter sampling at T would; one position
    per request carries the uniform 0.999 so that rejections, and with them
    the residual draw, happen at every temperature.  (A token the drafter
    gives almost no probability can leave a residual below what single or
    double precision resolves; such draws are decided by rounding on both
    sides and are not what this test compares.)"""
    B, k, V = 48, 6, 20000
    inp = synth.make_inputs("zipf_mixed_noise", B, k, V, dtype, seed=int(T * 1000) % 9973 + 7)
    inp.temperature[:] = np.float32(T)
    rng = np.random.default_rng(12)
    zd = (inp.draft.astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" else inp.draft
    g = rng.gumbel(size=zd.shape)
    inp.tokens[:] = np.argmax(zd.astype(np.float64) / np.float64(np.float32(T)) + g,
                              axis=2).astype(np.int32)
    forced = rng.integers(0, k, size=B)
    inp.uniforms[np.arange(B), forced] = np.float32(0.999)
    info, rep, o = check(inp, f"T={T} {dtype}")
    rejected = o.num_accepted < inp.lengths
    assert np.sum(rejected) >= 10, "too few rejections to exercise the residual"
    assert rep.residual_zero == 0, rep


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_logits_far_from_zero_match_oracle(dtype):
    """Softmax is shift-invariant, and the kernels subtract row maxima in
    scaled form: target rows shifted by +3000 and draft rows by -2000 must
    still give the oracle's outputs, at mixed temperatures and with greedy
    requests.  The shifted values are stored in the call's dtype (in bf16
    they lie 16 apart, so the rows become sharply peaked), and both sides
    read exactly those values."""
    inp = synth.make_inputs("zipf_mixed_temp", 40, 8, 30000, "f32", seed=314)
    t = (inp.target + np.float32(3000.0)).astype(np.float32)
    d = (inp.draft - np.float32(2000.0)).astype(np.float32)
    if dtype == "bf16":
        inp.target, inp.draft, inp.dtype = synth.bf16_bits(t), synth.bf16_bits(d), "bf16"
    else:
        inp.target, inp.draft = t, d
    info, rep, o = check(inp, f"shifted logits {dtype}")
    assert np.sum(o.num_accepted < inp.lengths) >= 5


def test_single_token_vocabulary():
    inp = _inputs(4, 3, 1)
    inp.tokens[:] = 0
    out, n, _ = run_gpu(inp)
    assert np.all(n == 3) and np.all(out == 0)


def test_greedy_ties_and_worked_example_structure():
    B, k, V = 3, 8, 64
    tl = np.zeros((B, k + 1, V), np.float32)
    tl[:, :, 10] = 1.0
    tl[:, :, 40] = 1.0                   # tie: argmax is 10
    tl[0, 4, 10] = 0.0                   # request 0: position 4 prefers 40
    dl = np.zeros((B, k, V), np.float32)
    tok = np.full((B, k), 10, np.int32)
    inp = synth.SpecInputs(tl, dl, tok, np.array([8, 8, 3], np.int32),
                           np.full((B, k + 1), np.nan, np.float32), np.zeros(B, np.float32), "f32")
    out, n, rep = run_gpu(inp)
    assert n.tolist() == [4, 8, 3]
    assert out[0].tolist() == [10, 10, 10, 10, 40, -1, -1, -1, -1]
    assert out[1].tolist() == [10] * 9
    assert out[2].tolist() == [10, 10, 10, 10, -1, -1, -1, -1, -1]
    assert rep.status == sv.SPEC_OK


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_rows_with_nan_and_inf_match_oracle(dtype):
    """Greedy rows are only argmaxed: a NaN entry is never the maximum, +inf is
    a maximum like any other (lowest index wins), and only a row with nothing
    above -inf makes the request invalid."""
    B, k, V = 24, 6, 2000
    rng = np.random.default_rng(71)
    tl = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    dl = rng.standard_normal((B, k, V)).astype(np.float32)
    for b in range(B):
        for i in range(k + 1):
            tl[b, i, rng.integers(0, V, 5)] = np.nan       # NaN entries anywhere
    for b in range(0, B, 3):
        i = b % (k + 1)
        tl[b, i, np.argmax(np.nan_to_num(tl[b, i], nan=-np.inf))] = np.nan  # NaN at the max
    for b in range(1, B, 4):
        i = (b + 2) % (k + 1)
        tl[b, i, [700, 300, 1500]] = np.inf               # +inf wins, lowest index (300)
    tl[5, 2] = -np.inf
    tl[5, 2, 17] = np.nan                                  # nothing above -inf: invalid
    # Draft tokens: the argmax where it exists (so rounds run on), with a
    # seeded wrong token now and then.
    best = np.nanargmax(np.where(np.isnan(tl[:, :k]), -np.inf, tl[:, :k]), axis=2).astype(np.int32)
    tok = best.copy()
    wrong = rng.random((B, k)) < 0.2
    tok[wrong] = rng.integers(0, V, wrong.sum())
    tok[5, :2] = best[5, :2]                               # request 5 reaches its bad row 2
    inp = synth.SpecInputs(tl, dl, tok, rng.integers(1, k + 1, B).astype(np.int32),
                           synth.uniform_24bit(rng, (B, k + 1)), np.zeros(B, np.float32), "f32")
    inp.lengths[5] = k
    if dtype == "bf16":
        inp.target, inp.draft, inp.dtype = synth.bf16_bits(tl), synth.bf16_bits(dl), "bf16"
    out, n, rep = run_gpu(inp)
    o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                      inp.temperature)
    np.testing.assert_array_equal(n, o.num_accepted)
    np.testing.assert_array_equal(out, o.out_tokens)
    assert o.num_accepted[5] == -1 and o.bad_requests == 1
    assert rep.status == sv.SPEC_ERR_BAD_INPUT and rep.bad_requests == 1
    # Some request was stopped by, or emitted, a +inf argmax at index 300.
    assert np.any(out == 300)


def test_disjoint_supports_and_masked_logits():
    inp = _inputs(50, 4, 512, "f32", seed=3)
    inp.target[:, :, 256:] = -np.inf
    inp.draft[:, :, :256] = -np.inf
    inp.tokens[:] = np.random.default_rng(4).integers(256, 512, inp.tokens.shape)
    out, n, _ = run_gpu(inp)
    assert np.all(n == 0)
    check(inp, "disjoint supports")


@pytest.mark.parametrize("field", ["length0", "length_big", "token", "uniform", "temp_neg",
                                   "temp_nan", "temp_subnormal", "nan_logit_reached"])
def test_invalid_inputs_flagged_on_device(field):
    inp = _inputs(6, 4, 700, "bf16", seed=7)
    if field == "length0":
        inp.lengths[2] = 0
    elif field == "length_big":
        inp.lengths[2] = 5
    elif field == "token":
        inp.tokens[2, 1] = 700
    elif field == "uniform":
        inp.uniforms[2, 4] = 1.0
    elif field == "temp_neg":
        inp.temperature[2] = -0.5
    elif field == "temp_nan":
        inp.temperature[2] = np.nan
    elif field == "temp_subnormal":
        inp.temperature[2] = 1e-40
    else:
        inp.target[2, 0, 5] = 0x7FC0  # bf16 NaN in a row every round reads
    out, n, rep = run_gpu(inp)
    o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms, inp.temperature)
    assert n[2] == -1 and np.all(out[2] == -1)
    assert o.num_accepted[2] == -1
    assert rep.status == sv.SPEC_ERR_BAD_INPUT and rep.bad_requests == 1
    assert rep.first_bad_request == 2
    keep = np.arange(6) != 2
    np.testing.assert_array_equal(n[keep], o.num_accepted[keep])


def test_host_argument_errors_launch_nothing():
    inp = _inputs(2, 3, 64)
    d = sv.to_device(inp)
    ws = sv.alloc_workspace(2, 3, 64)
    L = sv.lib()
    args = [d["target_logits"].data_ptr(), d["draft_logits"].data_ptr(), sv.SPEC_F32,
            d["draft_tokens"].data_ptr(), d["lengths"].data_ptr(), d["uniforms"].data_ptr(),
            d["temperature"].data_ptr(), 2, 3, 64, 0, 0, ws.data_ptr(), ws.numel(), 0]
    out = torch.empty((2, 4), dtype=torch.int32, device="cuda")
    n = torch.empty(2, dtype=torch.int32, device="cuda")
    args[10], args[11] = out.data_ptr(), n.data_ptr()
    assert L.spec_verify(*args) == sv.SPEC_OK
    bad = list(args); bad[13] = 16
    assert L.spec_verify(*bad) == sv.SPEC_ERR_WORKSPACE
    bad = list(args); bad[0] = 0
    assert L.spec_verify(*bad) == sv.SPEC_ERR_INVALID_ARG
    bad = list(args); bad[8] = 40
    assert L.spec_verify(*bad) == sv.SPEC_ERR_UNSUPPORTED
    bad = list(args); bad[0] += 1
    assert L.spec_verify(*bad) == sv.SPEC_ERR_INVALID_ARG
    # An empty batch, no draft positions or an empty vocabulary: nothing to do.
    for idx in (7, 8, 9):
        bad = list(args); bad[idx] = 0
        assert L.spec_verify(*bad) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_verify_workspace_bytes(0, 3, 64) == 0
    # Beyond the largest supported sizes: refused, not an argument error.
    for idx, big in ((7, (1 << 18) + 1), (9, (1 << 21) + 1)):
        bad = list(args); bad[idx] = big
        assert L.spec_verify(*bad) == sv.SPEC_ERR_UNSUPPORTED
    torch.cuda.synchronize()


def test_bound_call_matches_spec_verify_and_sees_new_contents():
    a = synth.make_inputs("zipf_mixed_temp", 32, 16, 9000, "bf16", seed=21)
    b = synth.make_inputs("zipf_mixed_temp", 32, 16, 9000, "bf16", seed=22)
    d = sv.to_device(a)
    call = sv.Verifier(**d)
    for inp in (a, b):
        # Same buffers, new contents: the bound call reads what is there now.
        for key, t in sv.to_device(inp).items():
            d[key].copy_(t)
        out, n = call()
        want_out, want_n = sv.spec_verify(**d)
        np.testing.assert_array_equal(out.cpu().numpy(), want_out.cpu().numpy())
        np.testing.assert_array_equal(n.cpu().numpy(), want_n.cpu().numpy())
        o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                          inp.temperature)
        compare(out.cpu().numpy(), n.cpu().numpy(), o, inp.temperature, "bound call")


def test_round_captured_in_a_cuda_graph_replays_with_new_contents():
    """A serving loop captures one round (three kernels, launch overlap kept) and replays it."""
    a = synth.make_inputs("zipf_mixed_temp", 32, 16, 9000, "bf16", seed=41)
    b = synth.make_inputs("zipf_mixed_temp", 32, 16, 9000, "bf16", seed=42)
    s = torch.cuda.Stream()
    d = sv.to_device(a)
    ws = sv.alloc_workspace(a.B, a.k, a.V)
    out = torch.empty((a.B, a.k + 1), dtype=torch.int32, device="cuda")
    nacc = torch.empty(a.B, dtype=torch.int32, device="cuda")
    call = sv.Verifier(**d, workspace=ws, out_tokens=out, num_accepted=nacc, stream=s)
    with torch.cuda.stream(s):
        call()  # first call on the device sets the kernels up, outside the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for inp in (a, b, a):
        for key, t in sv.to_device(inp).items():
            d[key].copy_(t)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                          inp.temperature)
        compare(out.cpu().numpy(), nacc.cpu().numpy(), o, inp.temperature, "graph replay")
        assert sv.spec_verify_report(ws).status == sv.SPEC_OK


@pytest.mark.parametrize("B,k,V,dtype", [
    (70000, 3, 24, "f32"),      # more requests than a grid's y extent holds
    (1 << 18, 1, 16, "bf16"),   # SPEC_MAX_B
])
def test_largest_batches(B, k, V, dtype):
    inp = _inputs(B, k, V, dtype, seed=B % 97)
    inp.lengths = np.random.default_rng(B).integers(1, k + 1, B).astype(np.int32)
    inp.temperature[::7] = 0.0
    info, rep, o = check(inp, f"B={B}")
    assert rep.rows_planned == int(np.sum(np.where(inp.temperature == 0, 1, 2) * inp.lengths))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_largest_vocabulary(dtype):
    """V = SPEC_MAX_V (2^21): the most segments the final pass holds in shared memory."""
    V = 1 << 21
    inp = _inputs(2, 3, V, dtype, seed=21)
    inp.lengths[:] = [3, 1]
    inp.temperature[1] = 0.0
    check(inp, f"V=2^21 {dtype}")


def test_timed_call_and_device_status():
    """spec_verify_timed gives the same outputs as spec_verify and records its
    four events in order; spec_verify_device_status reads the recorded status."""
    inp = synth.make_inputs("zipf_mixed_temp", 24, 16, 5000, "bf16", seed=61)
    d = sv.to_device(inp)
    ws = sv.alloc_workspace(inp.B, inp.k, inp.V)
    want_out, want_n = sv.spec_verify(**d, workspace=ws)
    want_out, want_n = want_out.cpu().numpy(), want_n.cpu().numpy()
    assert sv.spec_verify_device_status(ws) == sv.SPEC_OK
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    out, n = sv.spec_verify(**d, workspace=ws, events=evs)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), want_out)
    np.testing.assert_array_equal(n.cpu().numpy(), want_n)
    times = [evs[0].elapsed_time(e) for e in evs]
    assert all(b >= a for a, b in zip(times, times[1:])) and times[-1] > 0
    d["lengths"][3] = 0  # an invalid length: recorded on the device
    sv.spec_verify(**d, workspace=ws)
    assert sv.spec_verify_device_status(ws) == sv.SPEC_ERR_BAD_INPUT


def test_timed_out_slices_leave_minus_one_and_the_next_call_works():
    """A final-pass slice that gives up waiting still counts itself in, and the
    request then reports -1 (not stale outputs).  The testing flag makes every
    slice but the first of each request wait, bounded, for an event that never
    happens; the workspace records SPEC_ERR_TIMEOUT, and a normal call on the
    same workspace right after matches the oracle."""
    inp = synth.make_inputs("zipf_mixed_temp", 8, 6, 4096, "bf16", seed=61)
    d = sv.to_device(inp)
    ws = sv.alloc_workspace(inp.B, inp.k, inp.V)
    out = torch.full((inp.B, inp.k + 1), 123, dtype=torch.int32, device="cuda")
    n = torch.full((inp.B,), 123, dtype=torch.int32, device="cuda")
    sv.spec_verify(**d, workspace=ws, out_tokens=out, num_accepted=n,
                   flags=sv.SPEC_FLAG_TEST_LATE_SLICES)
    assert sv.spec_verify_device_status(ws) == sv.SPEC_ERR_TIMEOUT
    # 8 requests over 16 segments: every request has several slices.
    assert np.all(n.cpu().numpy() == -1)
    assert np.all(out.cpu().numpy() == -1)
    out2, n2 = sv.spec_verify(**d, workspace=ws, out_tokens=out, num_accepted=n)
    rep = sv.spec_verify_report(ws)
    assert rep.status == sv.SPEC_OK, rep
    o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                      inp.temperature)
    compare(out2.cpu().numpy(), n2.cpu().numpy(), o, inp.temperature, "after timeouts")


def test_one_slice_per_request_is_not_affected_by_the_late_flag():
    """With a single segment per row every request has exactly one slice (the
    first), so the testing flag changes nothing."""
    inp = synth.make_inputs("zipf_mixed_temp", 12, 5, 200, "f32", seed=62)
    d = sv.to_device(inp)
    ws = sv.alloc_workspace(inp.B, inp.k, inp.V)
    out, n = sv.spec_verify(**d, workspace=ws, flags=sv.SPEC_FLAG_TEST_LATE_SLICES)
    assert sv.spec_verify_device_status(ws) == sv.SPEC_OK
    o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                      inp.temperature)
    compare(out.cpu().numpy(), n.cpu().numpy(), o, inp.temperature, "one slice")
