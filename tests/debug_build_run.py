"""Every entry point once through the range-checking build (run in a child
process with SPEC_VERIFY_DEBUG=1 by test_gpu_debug_build.py).

Runs the smoke checks (padded and packed verification, OPD statistics, D3D
selection, each against the oracle), then the fused verification + OPD call,
the no-allocation entry, the row statistics and a 64-request verification
with early exit and every recipe's edge (greedy, mixed temperatures,
lengths), comparing with the oracle; finally prints the range checks that
failed on the device.
"""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import __graft_entry__ as g  # noqa: E402
import oracle  # noqa: E402
import speculative_decoding_verification_58_gb300 as sv  # noqa: E402
from speculative_decoding_verification_58_gb300 import synth  # noqa: E402
from parity import compare  # noqa: E402


def main() -> None:
    assert sv.DEBUG_BUILD and sv.spec_debug_build(), "the range-checking build is not loaded"
    sv.spec_debug_checks(reset=True)
    g.smoke()
    for recipe, B, k, V, dt, seed in (("zipf_mixed_temp", 64, 16, 20000, "bf16", 41),
                                      ("zipf_mixed_noise", 48, 8, 3001, "f32", 42),
                                      ("gauss", 8, 31, 777, "f32", 43)):
        inp = synth.make_inputs(recipe, B, k, V, dt, seed=seed)
        d = sv.to_device(inp)
        o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                          inp.temperature)
        out, n = sv.spec_verify(**d)
        compare(out.cpu().numpy(), n.cpu().numpy(), o, inp.temperature, f"debug {recipe}")
        out_f, n_f, st = sv.spec_verify_opd(**d)
        compare(out_f.cpu().numpy(), n_f.cpu().numpy(), o, inp.temperature, f"debug fused {recipe}")
        out_s = torch.full_like(out, 7)
        n_s = torch.full_like(n, 7)
        if sv.spec_verify_workspace_bytes(B, k, V) <= sv.SPEC_STATIC_SCRATCH_BYTES:
            sv.spec_verify_static(**d, out_tokens=out_s, num_accepted=n_s)
            compare(out_s.cpu().numpy(), n_s.cpu().numpy(), o, inp.temperature,
                    f"debug static {recipe}")
        # Row statistics: argmax on greedy rows (T = 0), max on every row.
        rows = d["target_logits"].reshape(-1, V)[:16]
        temp_h = np.tile(np.array([0.0, 1.0], np.float32), 8)
        mx, lse, arg = sv.spec_row_stats(rows, torch.from_numpy(temp_h).cuda())
        want_mx, _, want_arg = oracle.row_stats(inp.target.reshape(-1, V)[:16], temp_h)
        assert np.array_equal(mx.cpu().numpy().astype(np.float64), want_mx)
        assert np.array_equal(arg.cpu().numpy()[temp_h == 0], want_arg[temp_h == 0])
    torch.cuda.synchronize()
    failures, site = sv.spec_debug_checks()
    print(f"range checks failed: {failures} (first site {site})")
    assert failures == 0, (failures, site)
    print("debug build ok")


if __name__ == "__main__":
    main()
