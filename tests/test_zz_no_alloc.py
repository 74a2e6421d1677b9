"""spec_verify_static: verification for callers that cannot allocate (needs a GPU).

Some callers get only their input and output buffers from the runtime they
run in and may not allocate device memory, so they cannot pass spec_verify
a workspace.  spec_verify_static serves them from a fixed scratch array
inside the library.  These tests call it through the C ABI and check that
it returns exactly what spec_verify (with a caller workspace) returns, for
two different batches in a row on the shared scratch, and that a batch too
large for the scratch is refused without launching anything.

This file sorts last so that a run stopping at the first failure has run
every other test first; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_verification_58_gb300 as sv
from speculative_decoding_verification_58_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.lib()


def _both(inp):
    d = sv.to_device(inp)
    ref_out, ref_n = sv.spec_verify(**d)
    out = torch.full((inp.B, inp.k + 1), 7, dtype=torch.int32, device="cuda")
    n = torch.full((inp.B,), 7, dtype=torch.int32, device="cuda")
    L = sv.lib()
    code = L.spec_verify_static(
        d["target_logits"].data_ptr(), d["draft_logits"].data_ptr(),
        sv.SPEC_BF16 if inp.dtype == "bf16" else sv.SPEC_F32, d["draft_tokens"].data_ptr(),
        d["lengths"].data_ptr(), d["uniforms"].data_ptr(), d["temperature"].data_ptr(),
        inp.B, inp.k, inp.V, out.data_ptr(), n.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
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


def test_static_scratch_refuses_batches_beyond_its_size():
    B, k, V = 4096, 16, 151936
    assert sv.spec_verify_workspace_bytes(B, k, V) > sv.SPEC_STATIC_SCRATCH_BYTES
    code = sv.lib().spec_verify_static(16, 16, sv.SPEC_BF16, 16, 16, 16, 16, B, k, V, 16, 16, None)
    assert code == sv.SPEC_ERR_UNSUPPORTED
