"""Packed (ragged) verification batches on the GPU, through the C-ABI (needs a GB300).

AdaFlash Section 3.3 packs the candidates of all requests into one
verification batch of total length sum_b k_b.  spec_verify_packed must give
what the oracle gives on the packed rows, and bit for bit what spec_verify
gives on the same rows laid out padded.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import speculative_decoding_verification_58_gb300 as sv
from speculative_decoding_verification_58_gb300 import synth
from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.lib()


def run_packed(inp, pk, full_sweep=False):
    d = sv.to_device(inp)
    rows = sv.to_device_packed(pk)
    ws = sv.alloc_workspace(inp.B, inp.k, inp.V)
    out, n = sv.spec_verify_packed(**rows, draft_tokens=d["draft_tokens"], lengths=d["lengths"],
                                   uniforms=d["uniforms"], temperature=d["temperature"],
                                   workspace=ws, full_sweep=full_sweep)
    rep = sv.spec_verify_report(ws)
    return out.cpu().numpy(), n.cpu().numpy(), rep


@pytest.mark.parametrize("recipe,B,k,V,dtype,gap", [
    ("gauss", 1, 4, 1024, "f32", 0),
    ("zipf_mixed_temp", 37, 16, 5000, "bf16", 2),
    ("zipf_mixed_temp", 19, 7, 4099, "f32", 1),       # rows not 16-byte aligned
    ("zipf_adaptive", 64, 16, 32000, "bf16", 0),
    ("zipf_mixed_noise", 8, 3, 257, "bf16", 5),
])
def test_packed_matches_oracle(recipe, B, k, V, dtype, gap):
    inp = synth.make_inputs(recipe, B, k, V, dtype, seed=40 + B)
    order = np.random.default_rng(B).permutation(B)
    pk = synth.pack_rows(inp, order=order, gap=gap)
    out, n, rep = run_packed(inp, pk)
    o = oracle.verify_packed(pk.target_rows, pk.draft_rows, pk.target_row_start,
                             pk.draft_row_start, inp.tokens, inp.lengths, inp.uniforms,
                             inp.temperature)
    compare(out, n, o, inp.temperature, f"packed {recipe} B={B}")
    assert rep.status == sv.SPEC_OK and rep.bad_requests == 0


def test_packed_equals_padded_at_full_size():
    """The benchmark's workload (B=128, k=16, V=151936 bf16), packed in shuffled order."""
    inp = synth.make_workload(synth.HEADLINE)
    d = sv.to_device(inp)
    ws = sv.alloc_workspace(inp.B, inp.k, inp.V)
    want_out, want_n = sv.spec_verify(**d, workspace=ws)
    want_out, want_n = want_out.cpu().numpy(), want_n.cpu().numpy()
    pk = synth.pack_rows(inp, order=np.random.default_rng(9).permutation(inp.B))
    for full in (False, True):
        out, n, rep = run_packed(inp, pk, full_sweep=full)
        np.testing.assert_array_equal(n, want_n)
        np.testing.assert_array_equal(out, want_out)
        assert rep.status == sv.SPEC_OK


def test_packed_rows_outside_their_buffer_are_flagged_on_device():
    inp = synth.make_inputs("zipf_mixed_temp", 12, 6, 3000, "bf16", seed=77)
    inp.temperature[:4] = 1.0  # requests 1..3 below sample, so their draft rows are checked
    pk = synth.pack_rows(inp)
    rows_t, rows_d = pk.target_rows.shape[0], pk.draft_rows.shape[0]
    pk.target_row_start[1] = -5
    pk.target_row_start[2] = rows_t - int(inp.lengths[2])
    pk.draft_row_start[3] = rows_d - int(inp.lengths[3]) + 1
    out, n, rep = run_packed(inp, pk)
    o = oracle.verify_packed(pk.target_rows, pk.draft_rows, pk.target_row_start,
                             pk.draft_row_start, inp.tokens, inp.lengths, inp.uniforms,
                             inp.temperature)
    assert list(np.nonzero(n < 0)[0]) == [1, 2, 3]
    assert np.all(out[[1, 2, 3]] == -1)
    compare(out, n, o, inp.temperature, "packed, bad placements")
    assert rep.status == sv.SPEC_ERR_BAD_INPUT and rep.bad_requests == 3
    assert rep.first_bad_request == 1


def test_packed_all_greedy_without_draft_rows():
    inp = synth.make_inputs("zipf_mixed_temp", 20, 16, 7000, "bf16", seed=13)
    inp.temperature[:] = 0.0
    pk = synth.pack_rows(inp)
    pk.draft_rows = pk.draft_rows[:0]
    pk.draft_row_start[:] = 123456  # never read, never checked at T = 0
    out, n, rep = run_packed(inp, pk)
    o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                      inp.temperature)
    np.testing.assert_array_equal(n, o.num_accepted)
    np.testing.assert_array_equal(out, o.out_tokens)
    assert rep.status == sv.SPEC_OK
