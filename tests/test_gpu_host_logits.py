"""Logits in pinned host memory, read by the kernels over the CPU-GPU link (needs a GPU).

When both logits buffers are pinned host memory that the GPU maps, the
library reads them directly (plain loads, no bulk copies, no staging copy):
only the rows a round reads cross the link.  The results must be those of
the same call on device-resident logits, bit for bit, and the oracle's under
the parity rule; mixed placements are refused before anything is launched.
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


def _pinned(t):
    return t.cpu().pin_memory()


@pytest.mark.parametrize("recipe,B,k,V,dt", [
    ("zipf_mixed_temp", 24, 16, 20000, "bf16"),
    ("zipf_mixed_noise", 16, 8, 151936, "bf16"),
    ("gauss", 9, 5, 1001, "f32"),            # rows not 16-byte aligned
])
def test_host_logits_match_device_logits_and_oracle(recipe, B, k, V, dt):
    inp = synth.make_inputs(recipe, B, k, V, dt, seed=B + k)
    d = sv.to_device(inp)
    out_d, n_d = sv.spec_verify(**d)
    h = dict(d, target_logits=_pinned(d["target_logits"]), draft_logits=_pinned(d["draft_logits"]))
    ws = sv.alloc_workspace(B, k, V)
    out_h, n_h = sv.spec_verify(**h, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d) and torch.equal(n_h, n_d)
    assert sv.spec_verify_device_status(ws) == sv.SPEC_OK
    o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                      inp.temperature)
    compare(out_h.cpu().numpy(), n_h.cpu().numpy(), o, inp.temperature, f"host logits {recipe}")


def test_packed_host_rows_and_static_entry():
    inp = synth.make_inputs("zipf_mixed_noise", 20, 16, 30000, "bf16", seed=77)
    d = sv.to_device(inp)
    out_d, n_d = sv.spec_verify(**d)
    pk = synth.pack_rows(inp, order=np.arange(inp.B)[::-1], gap=1)
    rows = sv.to_device_packed(pk)
    rows_h = dict(rows, target_rows=_pinned(rows["target_rows"]),
                  draft_rows=_pinned(rows["draft_rows"]))
    small = {key: d[key] for key in ("draft_tokens", "lengths", "uniforms", "temperature")}
    out_p, n_p = sv.spec_verify_packed(**rows_h, **small)
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_d) and torch.equal(n_p, n_d)
    if sv.spec_verify_workspace_bytes(inp.B, inp.k, inp.V) <= sv.SPEC_STATIC_SCRATCH_BYTES:
        h = dict(d, target_logits=_pinned(d["target_logits"]),
                 draft_logits=_pinned(d["draft_logits"]))
        out_s, n_s = sv.spec_verify_static(**h)
        torch.cuda.synchronize()
        assert torch.equal(out_s, out_d) and torch.equal(n_s, n_d)


def test_mixed_or_pageable_placements_are_refused():
    inp = synth.make_inputs("gauss", 4, 4, 512, "f32", seed=3)
    d = sv.to_device(inp)
    out = torch.full((inp.B, inp.k + 1), 9, dtype=torch.int32, device="cuda")
    n = torch.full((inp.B,), 9, dtype=torch.int32, device="cuda")
    mixed = dict(d, target_logits=_pinned(d["target_logits"]))
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify(**mixed, out_tokens=out, num_accepted=n)
    assert e.value.code == sv.SPEC_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool(torch.all(out == 9)) and bool(torch.all(n == 9))
    pageable = dict(d, target_logits=d["target_logits"].cpu(), draft_logits=d["draft_logits"].cpu())
    with pytest.raises(ValueError):
        sv.spec_verify(**pageable)


def test_row_stats_read_host_logits_and_opd_refuses_them():
    inp = synth.make_inputs("zipf_mixed_temp", 8, 4, 4096, "bf16", seed=5)
    d = sv.to_device(inp)
    rows = d["target_logits"].reshape(-1, inp.V)
    temp = torch.from_numpy(np.tile(np.array([0.0, 0.7, 1.0, 1.3], np.float32),
                                    rows.shape[0] // 4 + 1)[:rows.shape[0]]).cuda()
    mx_d, lse_d, arg_d = sv.spec_row_stats(rows, temp)
    mx_h, lse_h, arg_h = sv.spec_row_stats(_pinned(rows), temp)
    torch.cuda.synchronize()
    greedy = temp == 0
    assert torch.equal(mx_h, mx_d) and torch.equal(arg_h, arg_d)
    assert torch.equal(lse_h[~greedy], lse_d[~greedy])  # NaN on greedy rows
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_opd_stats(_pinned(d["target_logits"]), _pinned(d["draft_logits"]), d["lengths"])
    assert e.value.code == sv.SPEC_ERR_INVALID_ARG
