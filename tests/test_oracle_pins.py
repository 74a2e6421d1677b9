"""Pins of the CPU oracle to facts the pages and mathematics fix (no GPU).

Each test checks the oracle against something other than itself:
  * losslessness by exact enumeration: the verification outcome, extended by
    plain sampling from the target, has exactly the target's joint
    distribution (AdaFlash Section 2.1: "the output distribution is identical
    to that of the target model"; DFlash notes Section 5.2 for drafters whose
    per-position distributions are marginals);
  * the mean number of emitted tokens E[tau] = (1 - Acc^(k+1)) / (1 - Acc)
    for i.i.d. positions (AdaFlash Section 2.1), by Monte Carlo;
  * p == q always accepts; disjoint supports always reject and resample p;
  * the residual mass equals the total-variation distance 1 - sum min(p, q);
  * per-row logsumexp against torch.logsumexp in float64, argmax against numpy;
  * the greedy worked example of the DFlash notes (Section 5.2, example #4).

The enumeration finds the oracle's decision thresholds by bisection on its
double-precision uniforms, so it never re-implements the rule it checks.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_58_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def softmax(z, T):
    z = np.asarray(z, np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


# --------------------------------------------------------------------------
# Exact enumeration of the output distribution on tiny vocabularies.
# --------------------------------------------------------------------------

def _bisect_sup(pred_batch, n_problems, iters=62):
    """For each problem, sup{t in [0,1) : pred(t)} for a predicate true on [0, a) only."""
    top = np.nextafter(1.0, 0.0)
    lo = np.zeros(n_problems)
    hi = np.ones(n_problems)
    for _ in range(iters):
        mid = np.minimum(0.5 * (lo + hi), top)  # (lo + hi) / 2 can round up to 1.0
        ok = pred_batch(mid)
        lo = np.where(ok, mid, lo)
        hi = np.where(ok, hi, mid)
    ok_top = pred_batch(np.full(n_problems, top))
    return np.where(ok_top, 1.0, lo)


class ToyModel:
    """Random target table p(.|prefix) for prefixes of length <= k, and a drafter.

    ``kind='marginal'``: q_i(.) depends only on the position (diffusion drafter).
    ``kind='ar'``: q(.|prefix) depends on the prefix (autoregressive drafter).
    """

    def __init__(self, V, k, kind, T, seed):
        rng = np.random.default_rng(seed)
        # The C-ABI takes temperatures as float32: define p at that value.
        self.V, self.k, self.kind, self.T = V, k, kind, float(np.float32(T))
        self.t_logits = {}
        for m in range(k + 1):
            for pre in itertools.product(range(V), repeat=m):
                self.t_logits[pre] = (rng.standard_normal(V) * 1.5).astype(np.float32)
        self.q_pos = [(rng.standard_normal(V) * 1.5).astype(np.float32) for _ in range(k)]
        self.q_pre = {}
        if kind == "ar":
            for m in range(k):
                for pre in itertools.product(range(V), repeat=m):
                    self.q_pre[pre] = (rng.standard_normal(V) * 1.5).astype(np.float32)

    def draft_logits(self, i, prefix):
        return self.q_pre[prefix] if self.kind == "ar" else self.q_pos[i]

    def p(self, prefix):
        return softmax(self.t_logits[prefix], self.T)

    def draft_weight(self, x):
        w = 1.0
        for i, xi in enumerate(x):
            w *= softmax(self.draft_logits(i, tuple(x[:i])), self.T)[xi]
        return w


def _enumerate_output_distribution(model, L):
    V, k = model.V, model.k
    xs = list(itertools.product(range(V), repeat=k))
    X = len(xs)
    tl = np.empty((X, k + 1, V), np.float32)
    dl = np.empty((X, k, V), np.float32)
    for s, x in enumerate(xs):
        for i in range(k + 1):
            tl[s, i] = model.t_logits[tuple(x[:i])]
        for i in range(k):
            dl[s, i] = model.draft_logits(i, tuple(x[:i]))
    tok = np.array(xs, np.int32).reshape(X, k)
    temp = np.full(X, model.T, np.float32)
    lens = np.full(X, L, np.int32)

    def run(u):
        return oracle.verify(tl, dl, tok, lens, u, temp)

    # Acceptance threshold a_i of every position, with all earlier positions
    # accepted (u = 0), found by bisection on u_i.
    acc = np.zeros((X, L))
    for i in range(L):
        def pred(t, i=i):
            u = np.full((X, k + 1), 0.5)
            u[:, :i] = 0.0
            u[:, i] = t
            return run(u).num_accepted > i
        acc[:, i] = _bisect_sup(pred, X)

    # For every outcome n (first rejection, or L), the final-token CDF as a
    # function of u_L, again by bisection.
    emitted = {}
    for n in range(L + 1):
        reach = np.prod(acc[:, :n], axis=1)
        if n < L:
            reach = reach * (1.0 - acc[:, n])
        live = np.nonzero(reach > 0)[0]
        if live.size == 0:
            continue
        base = np.full((X, k + 1), 0.5)
        base[:, :n] = 0.0
        if n < L:
            base[:, n] = np.minimum(0.5 * (acc[:, n] + 1.0), np.nextafter(1.0, 0.0))
        edges = np.zeros((X, V + 1))
        edges[:, V] = 1.0
        for j in range(V - 1):
            def pred(t, j=j):
                u = base.copy()
                u[:, L] = t
                r = run(u)
                assert np.all(r.num_accepted[live] == n)
                return r.out_tokens[:, n] <= j
            edges[:, j + 1] = _bisect_sup(pred, X)
        probs = np.diff(edges, axis=1)
        for s in live:
            x = xs[s]
            w = model.draft_weight(x) * reach[s]
            for y in range(V):
                if probs[s, y] > 0:
                    key = tuple(x[:n]) + (y,)
                    emitted[key] = emitted.get(key, 0.0) + w * probs[s, y]
    return emitted


@pytest.mark.parametrize("kind", ["marginal", "ar"])
@pytest.mark.parametrize("V,k,L,T", [(3, 1, 1, 1.0), (3, 2, 2, 1.0), (4, 2, 1, 0.7),
                                     (3, 3, 2, 1.3), (4, 3, 3, 1.0)])
def test_output_distribution_equals_target(kind, V, k, L, T):
    model = ToyModel(V, k, kind, T, seed=1000 + 31 * V + 7 * k + L)
    emitted = _enumerate_output_distribution(model, L)
    assert abs(sum(emitted.values()) - 1.0) < 1e-12
    # Continue every emitted prefix with plain sampling from the target up to
    # k+1 tokens; the result must be the target's own joint distribution.
    worst = 0.0
    for seq in itertools.product(range(V), repeat=k + 1):
        target = 1.0
        for j in range(k + 1):
            target *= model.p(seq[:j])[seq[j]] if j <= k else 1.0
        got = 0.0
        for m in range(1, L + 2):
            pre = seq[:m]
            if pre in emitted:
                tail = 1.0
                for j in range(m, k + 1):
                    tail *= model.p(seq[:j])[seq[j]]
                got += emitted[pre] * tail
        worst = max(worst, abs(got - target))
    assert worst < 1e-12, worst


def test_first_token_marginal_is_target_row0():
    model = ToyModel(4, 1, "marginal", 1.0, seed=7)
    emitted = _enumerate_output_distribution(model, 1)
    first = np.zeros(4)
    for key, w in emitted.items():
        first[key[0]] += w
    np.testing.assert_allclose(first, model.p(()), rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# Monte Carlo: mean emitted tokens per round.
# --------------------------------------------------------------------------

def _mc_rounds(p_logits_per_pos, q_logits_per_pos, target_bonus, N, seed):
    rng = np.random.default_rng(seed)
    L = len(q_logits_per_pos)
    V = len(target_bonus)
    tl = np.empty((N, L + 1, V), np.float32)
    dl = np.empty((N, L, V), np.float32)
    tok = np.empty((N, L), np.int32)
    for i in range(L):
        tl[:, i] = p_logits_per_pos[i]
        dl[:, i] = q_logits_per_pos[i]
        tok[:, i] = rng.choice(V, size=N, p=softmax(q_logits_per_pos[i], 1.0))
    tl[:, L] = target_bonus
    u = rng.random((N, L + 1))
    r = oracle.verify(tl, dl, tok, np.full(N, L, np.int32), u, np.ones(N, np.float32))
    assert r.bad_requests == 0
    return r.num_accepted.astype(np.float64) + 1.0


@pytest.mark.slow
def test_mean_emitted_tokens_iid_closed_form():
    V, k = 6, 4
    rng = np.random.default_rng(11)
    zp = (rng.standard_normal(V) * 1.2).astype(np.float32)
    zq = (zp + rng.standard_normal(V) * 0.9).astype(np.float32)
    acc = np.minimum(softmax(zp, 1.0), softmax(zq, 1.0)).sum()
    expected = (1 - acc ** (k + 1)) / (1 - acc)
    tau = _mc_rounds([zp] * k, [zq] * k, zp, 1_000_000, seed=12)
    se = tau.std() / math.sqrt(tau.size)
    assert abs(tau.mean() - expected) < 5 * se, (tau.mean(), expected, se)


@pytest.mark.slow
def test_mean_emitted_tokens_per_position_acceptance():
    # Independent positions with their own Acc_i: E[n+1] = 1 + sum_{i=1..L} prod_{j<i} Acc_j.
    V, L = 5, 3
    rng = np.random.default_rng(21)
    zps = [(rng.standard_normal(V) * 1.5).astype(np.float32) for _ in range(L)]
    zqs = [(z + rng.standard_normal(V) * s).astype(np.float32) for z, s in zip(zps, (0.3, 1.0, 2.0))]
    accs = [np.minimum(softmax(a, 1.0), softmax(b, 1.0)).sum() for a, b in zip(zps, zqs)]
    expected = 1.0 + sum(np.prod(accs[:i]) for i in range(1, L + 1))
    tau = _mc_rounds(zps, zqs, zps[0], 600_000, seed=22)
    se = tau.std() / math.sqrt(tau.size)
    assert abs(tau.mean() - expected) < 5 * se, (tau.mean(), expected, se)


# --------------------------------------------------------------------------
# Special cases.
# --------------------------------------------------------------------------

def test_p_equals_q_always_accepts():
    rng = np.random.default_rng(3)
    B, k, V = 64, 5, 97
    tl = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    dl = tl[:, :k].copy()
    tok = rng.integers(0, V, (B, k)).astype(np.int32)
    lens = rng.integers(1, k + 1, B).astype(np.int32)
    u = rng.random((B, k + 1)).astype(np.float32)
    u[:, 0] = np.float32(np.nextafter(np.float32(1), np.float32(0)))
    temp = rng.uniform(0.3, 2.0, B).astype(np.float32)
    r = oracle.verify(tl, dl, tok, lens, u, temp)
    np.testing.assert_array_equal(r.num_accepted, lens)
    for b in range(B):
        np.testing.assert_array_equal(r.out_tokens[b, :lens[b]], tok[b, :lens[b]])
        assert 0 <= r.out_tokens[b, lens[b]] < V
        assert np.all(r.out_tokens[b, lens[b] + 1:] == -1)


def test_residual_mass_is_total_variation():
    rng = np.random.default_rng(5)
    B, k, V = 40, 3, 50
    tl = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    dl = (tl[:, :k] + rng.standard_normal((B, k, V))).astype(np.float32)
    tok = np.zeros((B, k), np.int32)
    temp = rng.uniform(0.5, 1.5, B).astype(np.float32)
    for b in range(B):
        p = softmax(tl[b, 0], temp[b])
        q = softmax(dl[b, 0], temp[b])
        tok[b, 0] = int(np.argmax(q / p))  # p/q smallest: rejected for u close to 1
    u = np.full((B, k + 1), 0.999999, np.float32)
    u[:, k] = rng.random(B)
    r = oracle.verify(tl, dl, tok, np.full(B, k, np.int32), u, temp)
    assert np.all(r.num_accepted == 0)
    for b in range(B):
        tv = 1.0 - np.minimum(softmax(tl[b, 0], temp[b]), softmax(dl[b, 0], temp[b])).sum()
        assert abs(r.final_mass[b] - tv) < 1e-12


@pytest.mark.parametrize("T", [0.05, 0.2, 8.0, 100.0])
def test_residual_draw_matches_extended_precision(T):
    """The residual draw (AdaFlash Section 2.1: a token from
    normalize(max(0, p - q)) by inverse CDF with u_L) recomputed in 50-digit
    arithmetic from the same float32 logits and temperature: nearly one-hot
    rows at T = 0.05, nearly uniform ones at T = 100.  Position 0 is
    rejected by construction (the token with the smallest p/q, u = 0.999999);
    a draw whose u_L * TV lies within 1e-9 of a CDF edge is skipped."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(int(T * 100) + 3)
    B, k, V = 30, 2, 200
    tl = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    dl = (tl[:, :k] + rng.standard_normal((B, k, V)) * 0.5).astype(np.float32)
    Tf = np.float32(T)
    tok = np.zeros((B, k), np.int32)
    for b in range(B):
        p, q = softmax(tl[b, 0], Tf), softmax(dl[b, 0], Tf)
        tok[b, 0] = int(np.argmax(q / p))
    u = np.full((B, k + 1), 0.999999, np.float32)
    u[:, k] = rng.random(B).astype(np.float32)
    r = oracle.verify(tl, dl, tok, np.full(B, k, np.int32), u, np.full(B, Tf, np.float32))
    assert np.all(r.num_accepted == 0)
    checked = 0
    for b in range(B):
        Tm = mp.mpf(float(Tf))
        et = [mp.exp(mp.mpf(float(z)) / Tm) for z in tl[b, 0]]
        ed = [mp.exp(mp.mpf(float(z)) / Tm) for z in dl[b, 0]]
        st, sd = mp.fsum(et), mp.fsum(ed)
        res = [max(mp.mpf(0), a / st - c / sd) for a, c in zip(et, ed)]
        tv = mp.fsum(res)
        target = mp.mpf(float(u[b, k])) * tv
        acc, want, edge = mp.mpf(0), None, None
        for y, w in enumerate(res):
            if acc + w > target:
                want, edge = y, min(target - acc, acc + w - target)
                break
            acc += w
        if want is None or edge < mp.mpf("1e-9") * tv:
            continue
        assert r.out_tokens[b, 0] == want, (T, b)
        assert abs(r.final_mass[b] - float(tv)) <= 1e-12 * max(1.0, float(tv)) + 1e-300
        checked += 1
    assert checked >= B - 2


def test_disjoint_supports_reject_and_resample_target():
    rng = np.random.default_rng(9)
    B, k, V = 200, 2, 16
    tl = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    dl = rng.standard_normal((B, k, V)).astype(np.float32)
    tl[:, :, V // 2:] = -np.inf   # target lives on the lower half
    dl[:, :, : V // 2] = -np.inf  # draft lives on the upper half
    tok = rng.integers(V // 2, V, (B, k)).astype(np.int32)
    u = rng.random((B, k + 1)).astype(np.float32)
    r = oracle.verify(tl, dl, tok, np.full(B, k, np.int32), u, np.ones(B, np.float32))
    assert np.all(r.num_accepted == 0)
    for b in range(B):
        p = softmax(tl[b, 0, : V // 2], 1.0)
        c = np.cumsum(p)
        want = int(np.searchsorted(c, np.float64(u[b, k]) * c[-1], side="right"))
        assert r.out_tokens[b, 0] == want
        assert abs(r.final_mass[b] - 1.0) < 1e-12


# --------------------------------------------------------------------------
# Row statistics and greedy.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_row_stats_match_library_routines(dtype):
    from speculative_decoding_verification_58_gb300 import synth
    rng = np.random.default_rng(4)
    rows, V = 37, 1531
    z = (rng.standard_normal((rows, V)) * 3).astype(np.float32)
    z[5, 100] = z[5, 900] = z[5].max() + 1.0  # argmax tie: lowest index wins
    buf = synth.bf16_bits(z) if dtype == "bf16" else z
    zf = synth.bf16_to_f32(buf) if dtype == "bf16" else z
    temp = rng.uniform(0.2, 2.0, rows).astype(np.float32)
    temp[3] = 0.0
    mx, lse, arg = oracle.row_stats(buf, temp)
    np.testing.assert_array_equal(mx, zf.max(axis=1).astype(np.float64))
    np.testing.assert_array_equal(arg, np.argmax(zf, axis=1))
    assert arg[5] == 100
    ref = torch.logsumexp(torch.from_numpy(zf.astype(np.float64)) /
                          torch.from_numpy(temp.astype(np.float64))[:, None], dim=1).numpy()
    sampled = temp > 0
    np.testing.assert_allclose(lse[sampled], ref[sampled], rtol=1e-12, atol=0)
    assert np.isnan(lse[3])


def test_greedy_worked_example():
    with open(os.path.join(GOLDEN, "greedy_worked_example.json")) as f:
        ex = json.load(f)
    vocab = ex["vocab"]
    V, k = len(vocab), ex["k"]
    ids = {w: i for i, w in enumerate(vocab)}
    tl = np.zeros((1, k + 1, V), np.float32)
    for i, w in enumerate(ex["target_argmax"]):
        tl[0, i, ids[w]] = 5.0
    dl = np.zeros((1, k, V), np.float32)
    tok = np.array([[ids[w] for w in ex["draft"]]], np.int32)
    r = oracle.verify(tl, dl, tok, np.array([k], np.int32),
                      np.full((1, k + 1), np.nan, np.float32), np.zeros(1, np.float32))
    assert r.num_accepted[0] == ex["expected_num_accepted"]
    want = [ids[w] if w is not None else -1 for w in ex["expected_out"]]
    assert r.out_tokens[0].tolist() == want


def test_greedy_all_accepted_emits_argmax_of_row_L_and_ties_go_low():
    V, k = 10, 3
    tl = np.zeros((2, k + 1, V), np.float32)
    tl[:, :, 7] = 1.0
    tl[:, :, 2] = 1.0  # tie with index 7: argmax is 2
    dl = np.zeros((2, k, V), np.float32)
    tok = np.full((2, k), 2, np.int32)
    lens = np.array([k, 2], np.int32)
    r = oracle.verify(tl, dl, tok, lens, np.zeros((2, k + 1), np.float32), np.zeros(2, np.float32))
    assert r.num_accepted.tolist() == [3, 2]
    assert r.out_tokens[0].tolist() == [2, 2, 2, 2]
    assert r.out_tokens[1].tolist() == [2, 2, 2, -1]


def test_bf16_input_matches_widened_f32():
    from speculative_decoding_verification_58_gb300 import synth
    inp = synth.make_inputs("zipf_adaptive", 6, 5, 700, "bf16", seed=77, threads=1)
    a = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms, inp.temperature)
    b = oracle.verify(synth.bf16_to_f32(inp.target), synth.bf16_to_f32(inp.draft), inp.tokens,
                      inp.lengths, inp.uniforms, inp.temperature)
    np.testing.assert_array_equal(a.out_tokens, b.out_tokens)
    np.testing.assert_array_equal(a.num_accepted, b.num_accepted)


@pytest.mark.parametrize("field,value", [
    ("length", 0), ("length", 5), ("temperature", -1.0), ("temperature", float("nan")),
    ("temperature", float("inf")), ("token", 40), ("token", -1), ("uniform", 1.0),
    ("uniform", float("nan"))])
def test_invalid_inputs_are_reported(field, value):
    B, k, V = 3, 4, 40
    rng = np.random.default_rng(1)
    tl = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    dl = rng.standard_normal((B, k, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, k)).astype(np.int32)
    lens = np.full(B, 3, np.int32)
    u = rng.random((B, k + 1)).astype(np.float32)
    temp = np.ones(B, np.float32)
    if field == "length":
        lens[1] = value
    elif field == "temperature":
        temp[1] = value
    elif field == "token":
        tok[1, 2] = value
    else:
        u[1, 3] = value  # u_L with L = 3 is read
    r = oracle.verify(tl, dl, tok, lens, u, temp)
    assert r.bad_requests == 1
    assert r.num_accepted[1] == -1 and np.all(r.out_tokens[1] == -1)
    assert r.num_accepted[0] >= 0 and r.num_accepted[2] >= 0


def test_greedy_ignores_uniforms():
    V, k = 6, 2
    tl = np.zeros((1, k + 1, V), np.float32)
    tl[0, :, 1] = 1
    u = np.full((1, k + 1), np.nan, np.float32)
    r = oracle.verify(tl, np.zeros((1, k, V), np.float32), np.array([[1, 1]], np.int32),
                      np.array([2], np.int32), u, np.zeros(1, np.float32))
    assert r.bad_requests == 0 and r.num_accepted[0] == 2


def test_zero_mass_tokens_are_never_sampled():
    # A token of probability zero cannot be drawn, even at u = 0: the inverse
    # CDF picks the first index whose cumulative mass exceeds u * total.
    V, k = 9, 2
    z = np.linspace(0.0, 1.0, V, dtype=np.float32)
    tl = np.tile(z, (1, k + 1, 1))
    tl[0, k, :3] = -np.inf          # bonus row: the first three tokens have p = 0
    dl = tl[:, :k].copy()           # p == q: every draft is accepted
    r = oracle.verify(tl, dl, np.zeros((1, k), np.int32), np.array([k], np.int32),
                      np.zeros((1, k + 1), np.float32), np.ones(1, np.float32))
    assert r.num_accepted[0] == k
    assert r.out_tokens[0, k] == 3


def test_first_rejection_ends_the_round():
    # Position 0 is rejected for sure (p(x_0) = 0) and position 1 would be too:
    # the round must end at position 0 and resample there.
    V, k = 8, 3
    rng = np.random.default_rng(2)
    tl = rng.standard_normal((1, k + 1, V)).astype(np.float32)
    dl = rng.standard_normal((1, k, V)).astype(np.float32)
    tl[0, :, 0] = -np.inf
    tok = np.array([[0, 0, 0]], np.int32)
    r = oracle.verify(tl, dl, tok, np.array([k], np.int32), np.full((1, k + 1), 0.5, np.float32),
                      np.ones(1, np.float32))
    assert r.num_accepted[0] == 0
    assert r.out_tokens[0, 0] != 0 and np.all(r.out_tokens[0, 1:] == -1)


def test_token_impossible_under_both_is_rejected():
    # p(x) = q(x) = 0: the target never emits x, so the draft cannot be kept.
    V, k = 6, 1
    tl = np.zeros((1, k + 1, V), np.float32)
    dl = np.zeros((1, k, V), np.float32)
    tl[0, 0, 2] = dl[0, 0, 2] = -np.inf
    r = oracle.verify(tl, dl, np.array([[2]], np.int32), np.array([1], np.int32),
                      np.zeros((1, k + 1), np.float32), np.ones(1, np.float32))
    assert r.num_accepted[0] == 0 and r.out_tokens[0, 0] != 2


def test_unreadable_rows_invalidate_only_when_reached():
    V, k = 8, 3
    rng = np.random.default_rng(6)
    tl = rng.standard_normal((2, k + 1, V)).astype(np.float32)
    dl = rng.standard_normal((2, k, V)).astype(np.float32)
    tl[:, 0, 5] = -np.inf
    tok = np.full((2, k), 5, np.int32)  # p(x_0) = 0: position 0 always rejects
    tl[:, 2, 3] = np.nan                # row 2 is never reached
    dl[1, 0, 1] = np.nan                # ... but request 1's row 0 is
    r = oracle.verify(tl, dl, tok, np.full(2, k, np.int32), np.full((2, k + 1), 0.5, np.float32),
                      np.ones(2, np.float32))
    assert r.num_accepted.tolist() == [0, -1] and r.bad_requests == 1


def test_subnormal_temperature_is_invalid():
    V, k = 4, 1
    r = oracle.verify(np.zeros((1, k + 1, V), np.float32), np.zeros((1, k, V), np.float32),
                      np.zeros((1, k), np.int32), np.array([1], np.int32),
                      np.zeros((1, k + 1), np.float32), np.array([1e-39], np.float32))
    assert r.num_accepted[0] == -1


# ---------------------------------------------------------------------------
# OPD supervision statistics (AdaFlash Section 3.1)
# ---------------------------------------------------------------------------

def _opd_one(p, q, delta, alpha, dtype=np.float64):
    """One position whose softmaxes are p and q: logits log p, log q (float32)."""
    V = len(p)
    t = np.zeros((1, 2, V), np.float32)
    d = np.zeros((1, 1, V), np.float32)
    with np.errstate(divide="ignore"):
        t[0, 0] = np.log(np.asarray(p, dtype))
        d[0, 0] = np.log(np.asarray(q, dtype))
    return oracle.opd_stats(t, d, np.array([1], np.int32), delta=delta, alpha=alpha)


def test_opd_worked_example_of_the_notes():
    g = json.load(open(os.path.join(GOLDEN, "opd_worked_example.json")))
    tol = g["printed_tolerance"]
    r = _opd_one(g["p_target"], g["q_draft"], g["delta"], g["alpha"])
    assert r.x_star[0, 0] == g["printed"]["x_star"]
    assert abs(r.hard[0, 0] - g["printed"]["hard"]) < tol
    assert abs(r.rkl[0, 0] - g["printed"]["rkl"]) < tol
    entries = g["printed"]["rkl_entries"]
    # Clipped at delta = 0.01: the negative entry stays, the three others become delta.
    assert abs(r.rkl_clip[0, 0] - (entries[0] + 3 * g["delta"])) < tol
    unclipped = _opd_one(g["p_target"], g["q_draft"], 1e300, g["alpha"])
    assert abs(unclipped.loss[0] - g["printed"]["opd_unclipped"]) < tol
    assert abs(r.loss[0] - (g["alpha"] * r.hard[0, 0] + (1 - g["alpha"]) * r.rkl_clip[0, 0])) < 1e-12


def test_opd_reverse_kl_matches_scipy_entropy_and_gibbs():
    stats = pytest.importorskip("scipy.stats")
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    B, k, V = 3, 4, 333
    t = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    d = (t[:, :k] + rng.standard_normal((B, k, V))).astype(np.float32)
    lens = np.array([4, 1, 3], np.int32)
    r = oracle.opd_stats(t, d, lens, delta=0.05, alpha=0.3)
    for b in range(B):
        for i in range(k):
            if i >= lens[b]:
                assert r.x_star[b, i] == -1 and np.isnan(r.hard[b, i]) and np.isnan(r.rkl[b, i])
                continue
            p = special.softmax(t[b, i].astype(np.float64))
            q = special.softmax(d[b, i].astype(np.float64))
            assert abs(r.rkl[b, i] - stats.entropy(q, p)) < 1e-12 * max(1, stats.entropy(q, p))
            assert r.rkl[b, i] >= 0                               # Gibbs' inequality
            assert r.rkl_clip[b, i] <= r.rkl[b, i] + 1e-15        # clipping only lowers
            assert r.x_star[b, i] == int(np.argmax(t[b, i]))
            ce = special.logsumexp(d[b, i].astype(np.float64)) - float(d[b, i, r.x_star[b, i]])
            assert abs(r.hard[b, i] - ce) < 1e-12 * max(1, ce)
        L = lens[b]
        mix = 0.3 * r.hard[b, :L].mean() + 0.7 * r.rkl_clip[b, :L].mean()
        assert abs(r.loss[b] - mix) < 1e-12
    # A threshold above every entry clips nothing; alpha 1 and 0 pick one term.
    big = oracle.opd_stats(t, d, lens, delta=1e300, alpha=0.0)
    np.testing.assert_allclose(big.rkl_clip, big.rkl, rtol=0, atol=0)
    one = oracle.opd_stats(t, d, lens, delta=0.05, alpha=1.0)
    for b in range(B):
        assert abs(one.loss[b] - r.hard[b, :lens[b]].mean()) < 1e-12


def test_opd_special_cases():
    # p == q: no divergence anywhere; the hard term is the drafter's cross-entropy on its own mode.
    p = np.array([0.1, 0.6, 0.2, 0.1])
    r = _opd_one(p, p, 0.01, 0.8)
    assert abs(r.rkl[0, 0]) < 1e-12 and abs(r.rkl_clip[0, 0]) < 1e-12
    assert r.x_star[0, 0] == 1 and abs(r.hard[0, 0] + np.log(0.6)) < 1e-6
    # Argmax ties go to the lowest index.
    r = _opd_one([0.4, 0.1, 0.4, 0.1], [0.25] * 4, 0.01, 0.8)
    assert r.x_star[0, 0] == 0
    # q = 0 entries add nothing (0 log 0 = 0); q > 0 where p = 0 is an infinite entry, clipped to delta.
    r = _opd_one([0.5, 0.5, 0.0], [0.5, 0.5, 0.0], 0.01, 0.8)
    assert abs(r.rkl[0, 0]) < 1e-12
    r = _opd_one([0.5, 0.5, 0.0], [0.4, 0.4, 0.2], 0.01, 0.8)
    assert r.rkl[0, 0] == np.inf
    want = 2 * 0.4 * np.log(0.4 / 0.5) + 0.01
    assert abs(r.rkl_clip[0, 0] - want) < 1e-6
    # An invalid length makes the request NaN; a row without finite mass, its position.
    t = np.zeros((2, 3, 5), np.float32)
    d = np.zeros((2, 2, 5), np.float32)
    d[1, 0] = np.nan
    r = oracle.opd_stats(t, d, np.array([3, 2], np.int32))
    assert r.bad_requests == 1 and np.isnan(r.loss[0]) and np.all(r.x_star[0] == -1)
    assert np.isnan(r.hard[1, 0]) and np.isnan(r.loss[1]) and r.x_star[1, 1] == 0


# ---------------------------------------------------------------------------
# D3D branch selection (D3D paper, Methodology, asynchronous inference)
# ---------------------------------------------------------------------------

def test_d3d_budget_layout_of_the_paper():
    # Main D3D configuration: block size 16, coverage C = 12, fan-out F = 2;
    # packed budget N_async = B [(C - 1) F + 2] tokens.
    assert synth.d3d_branch_count(12, 2) * 16 == 16 * ((12 - 1) * 2 + 2) == 384
    br = synth.make_d3d_branches(np.array([16, 3], np.int32), 1000, C=12, F=2, blk=16, seed=1)
    assert br.pos.shape == (2, 24) and br.block.shape == (2, 24, 16)
    assert list(br.pos[0, :22]) == [j // 2 for j in range(22)] and list(br.pos[0, 22:]) == [16, 16]
    assert list(br.pos[1, :6]) == [0, 0, 1, 1, 2, 2] and np.all(br.pos[1, 6:22] == -1)


def _outcome(B, k, V, rng):
    """Made-up verification outcomes: n in [0, L], n + 1 tokens then -1."""
    L = rng.integers(1, k + 1, B).astype(np.int32)
    n = np.array([rng.integers(0, l + 1) for l in L], np.int32)
    out = np.full((B, k + 1), -1, np.int32)
    for b in range(B):
        out[b, :n[b] + 1] = rng.integers(0, V, n[b] + 1)
    return L, n, out


def test_d3d_select_finds_the_planted_branch_and_only_it():
    rng = np.random.default_rng(3)
    B, k, V, C, F, blk = 64, 16, 500, 12, 2, 16
    L, n, out = _outcome(B, k, V, rng)
    br = synth.make_d3d_branches(L, V, C, F, blk, seed=4)
    NB = br.pos.shape[1]
    want = np.full(B, -1, np.int32)
    for b in range(B):
        tok_n = out[b, n[b]]
        # No accidental matches: every branch assumes another token.
        br.tok[b][br.tok[b] == tok_n] = (tok_n + 1) % V
        if b % 4 != 3:  # plant the verified outcome in a random slot (3 in 4 requests)
            s = int(rng.integers(0, NB))
            br.pos[b, s], br.tok[b, s] = n[b], tok_n
            want[b] = s
    n[5] = -1  # an invalid request never hits
    want[5] = -1
    hit, nxt, hits = oracle.d3d_select(n, out, br.pos, br.tok, br.block)
    np.testing.assert_array_equal(hit, want)
    assert hits == int((want >= 0).sum())
    for b in range(B):
        if want[b] >= 0:
            np.testing.assert_array_equal(nxt[b], br.block[b, want[b]])
        else:
            assert np.all(nxt[b] == -1)


def test_d3d_select_tie_and_unused_slots():
    n = np.array([2, 0], np.int32)
    out = np.array([[7, 8, 9, -1], [4, -1, -1, -1]], np.int32)
    pos = np.array([[1, 2, 2, -1], [-1, 0, 0, 0]], np.int32)
    tok = np.array([[9, 9, 9, 9], [4, 5, 4, 4]], np.int32)
    blocks = np.arange(2 * 4 * 3, dtype=np.int32).reshape(2, 4, 3)
    hit, nxt, hits = oracle.d3d_select(n, out, pos, tok, blocks)
    # Request 0: slots 1 and 2 both match, the lowest wins; request 1: slot 0
    # is unused although its token matches, slot 2 is the first real match.
    assert list(hit) == [1, 2] and hits == 2
    np.testing.assert_array_equal(nxt, blocks[[0, 1], [1, 2]])
