"""spec_verify_static: verification for callers that cannot allocate (needs a GPU).

Some callers get only their input and output buffers from the runtime they
run in and may not allocate device memory, so they cannot pass spec_verify
a workspace.  spec_verify_static serves them from a fixed scratch array
inside the library.  These tests call it through the C ABI and check that
it returns exactly what spec_verify (with a caller workspace) returns, and
what the oracle returns under the parity rule, for two different batches in
a row on the shared scratch; that a warmed-up call changes neither torch's
allocations nor the device's free memory; and that a batch too large for the
scratch is refused with every output left untouched.

This file sorts last so that a run stopping at the first failure has run
every other test first; it also passes on its own in a fresh process.
"""

import ctypes

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


def _static(d, inp, out, n):
    return sv.lib().spec_verify_static(
        d["target_logits"].data_ptr(), d["draft_logits"].data_ptr(),
        sv.SPEC_BF16 if inp.dtype == "bf16" else sv.SPEC_F32, d["draft_tokens"].data_ptr(),
        d["lengths"].data_ptr(), d["uniforms"].data_ptr(), d["temperature"].data_ptr(),
        inp.B, inp.k, inp.V, out.data_ptr(), n.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _both(inp):
    d = sv.to_device(inp)
    ref_out, ref_n = sv.spec_verify(**d)
    out = torch.full((inp.B, inp.k + 1), 7, dtype=torch.int32, device="cuda")
    n = torch.full((inp.B,), 7, dtype=torch.int32, device="cuda")
    code = _static(d, inp, out, n)
    assert code == sv.SPEC_OK, sv.status_string(code)
    torch.cuda.synchronize()
    return (ref_out.cpu().numpy(), ref_n.cpu().numpy()), (out.cpu().numpy(), n.cpu().numpy())


def test_static_scratch_matches_workspace_entry_two_calls_in_a_row():
    # Two different batches back to back on the shared scratch: the second
    # must not see anything the first left behind.
    first = synth.make_inputs("zipf_mixed_temp", 48, 16, 20000, "bf16", seed=31)
    second = synth.make_inputs("zipf_mixed_noise", 20, 8, 3001, "f32", seed=32)
    for inp in (first, second):
        assert sv.spec_verify_workspace_bytes(inp.B, inp.k, inp.V) <= sv.SPEC_STATIC_SCRATCH_BYTES
        (ref_out, ref_n), (out, n) = _both(inp)
        # Same kernels on the same inputs: identical tokens and counts.
        np.testing.assert_array_equal(out, ref_out)
        np.testing.assert_array_equal(n, ref_n)
        assert np.all(n >= 0)
        o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                          inp.temperature)
        compare(out, n, o, inp.temperature, "spec_verify_static")


def test_static_call_allocates_nothing():
    inp = synth.make_inputs("zipf_adaptive", 16, 8, 5000, "bf16", seed=33)
    d = sv.to_device(inp)
    out = torch.empty((inp.B, inp.k + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((inp.B,), dtype=torch.int32, device="cuda")
    assert _static(d, inp, out, n) == sv.SPEC_OK  # first call on the device: set-up
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        assert _static(d, inp, out, n) == sv.SPEC_OK
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch_before
    assert free_after == free_before


def test_static_scratch_refuses_batches_beyond_its_size():
    # Real buffers of the refused size (so that nothing could read out of
    # bounds even if the check were missing), outputs set to a sentinel.
    B, k, V = 1 << 14, 16, 64
    assert sv.spec_verify_workspace_bytes(B, k, V) > sv.SPEC_STATIC_SCRATCH_BYTES
    inp = synth.SpecInputs(np.zeros((B, k + 1, V), np.float32), np.zeros((B, k, V), np.float32),
                           np.zeros((B, k), np.int32), np.full(B, k, np.int32),
                           np.zeros((B, k + 1), np.float32), np.ones(B, np.float32), "f32")
    d = sv.to_device(inp)
    out = torch.full((B, k + 1), 5, dtype=torch.int32, device="cuda")
    n = torch.full((B,), 5, dtype=torch.int32, device="cuda")
    assert _static(d, inp, out, n) == sv.SPEC_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool(torch.all(out == 5)) and bool(torch.all(n == 5))
