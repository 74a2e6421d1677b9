"""Packed (ragged) batch layout on the CPU: the oracle's packed entry and the host checks.

AdaFlash Section 3.3 packs the verification batch to a total length of
sum_b k_b instead of B x k.  Packing only moves rows, so the oracle on a
packed batch must give exactly what it gives on the same rows padded; rows
that no request owns are filled with NaN there, which also pins that the rule
never reads past row L_b (target) or L_b - 1 (draft).
"""

import numpy as np
import pytest

import oracle
import speculative_decoding_verification_58_gb300 as sv
from speculative_decoding_verification_58_gb300 import synth


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("recipe", ["zipf_mixed_temp", "zipf_adaptive", "gauss"])
def test_packed_oracle_equals_padded_oracle(recipe, dtype):
    inp = synth.make_inputs(recipe, 24, 8, 700, dtype, seed=31)
    want = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                         inp.temperature)
    order = np.random.default_rng(5).permutation(inp.B)
    for pk in (synth.pack_rows(inp), synth.pack_rows(inp, order=order, gap=3)):
        assert pk.target_rows.shape[0] >= int(inp.lengths.sum()) + inp.B
        got = oracle.verify_packed(pk.target_rows, pk.draft_rows, pk.target_row_start,
                                   pk.draft_row_start, inp.tokens, inp.lengths, inp.uniforms,
                                   inp.temperature)
        np.testing.assert_array_equal(got.num_accepted, want.num_accepted)
        np.testing.assert_array_equal(got.out_tokens, want.out_tokens)
        np.testing.assert_array_equal(got.margin, want.margin)


def test_packed_oracle_flags_rows_outside_their_buffer():
    inp = synth.make_inputs("zipf_mixed_temp", 8, 4, 64, "f32", seed=2)
    inp.temperature[:] = 1.0
    pk = synth.pack_rows(inp)
    rows_t, rows_d = pk.target_rows.shape[0], pk.draft_rows.shape[0]
    t0, d0 = pk.target_row_start.copy(), pk.draft_row_start.copy()
    t0[1] = -1                                   # before the buffer
    t0[2] = rows_t - int(inp.lengths[2])         # one row short of L_b + 1
    d0[3] = rows_d - int(inp.lengths[3]) + 1     # draft rows run past the end
    got = oracle.verify_packed(pk.target_rows, pk.draft_rows, t0, d0, inp.tokens, inp.lengths,
                               inp.uniforms, inp.temperature)
    want = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                         inp.temperature)
    bad = np.zeros(8, bool)
    bad[[1, 2, 3]] = True
    assert np.all(got.num_accepted[bad] == -1) and np.all(got.out_tokens[bad] == -1)
    np.testing.assert_array_equal(got.num_accepted[~bad], want.num_accepted[~bad])
    np.testing.assert_array_equal(got.out_tokens[~bad], want.out_tokens[~bad])
    assert got.bad_requests == 3


def test_packed_oracle_greedy_requests_need_no_draft_rows():
    inp = synth.make_inputs("zipf_mixed_temp", 6, 4, 50, "bf16", seed=3)
    inp.temperature[:] = 0.0
    pk = synth.pack_rows(inp)
    empty = pk.draft_rows[:0]
    got = oracle.verify_packed(pk.target_rows, empty, pk.target_row_start,
                               np.full(6, 10**6, np.int32), inp.tokens, inp.lengths, inp.uniforms,
                               inp.temperature)
    want = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                         inp.temperature)
    np.testing.assert_array_equal(got.num_accepted, want.num_accepted)
    np.testing.assert_array_equal(got.out_tokens, want.out_tokens)


def test_packed_entry_host_checks_return_before_any_cuda_call():
    sv.build()
    f = sv.lib().spec_verify_packed
    ok = dict(t=16, rt=10, d=16, rd=10, dt=0, ts=16, ds=16, tok=16, L=16, u=16, T=16, B=2, k=3,
              V=64, out=16, n=16, ws=256, wsb=1 << 20, s=None, fl=0)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["t"], a["rt"], a["d"], a["rd"], a["dt"], a["ts"], a["ds"], a["tok"], a["L"],
                 a["u"], a["T"], a["B"], a["k"], a["V"], a["out"], a["n"], a["ws"], a["wsb"],
                 a["s"], a["fl"])

    assert call(ts=None) == sv.SPEC_ERR_INVALID_ARG
    assert call(ds=None) == sv.SPEC_ERR_INVALID_ARG
    assert call(ts=18) == sv.SPEC_ERR_INVALID_ARG          # misaligned row starts
    assert call(rt=0) == sv.SPEC_ERR_INVALID_ARG
    assert call(rd=-1) == sv.SPEC_ERR_INVALID_ARG
    assert call(rt=1 << 31) == sv.SPEC_ERR_INVALID_ARG
    assert call(d=None) == sv.SPEC_ERR_INVALID_ARG          # rows_d > 0 needs a buffer
    assert call(fl=8) == sv.SPEC_ERR_INVALID_ARG
    assert call(k=40) == sv.SPEC_ERR_UNSUPPORTED
    assert call(wsb=8) == sv.SPEC_ERR_WORKSPACE
