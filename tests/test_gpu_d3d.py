"""D3D branch selection on the GPU vs the oracle, through the C-ABI (needs a GB300).

Integer work: the hit index, the copied block and the hit count must match
bit for bit.
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


def run(n, out, br):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    hit, nxt, hits = sv.spec_d3d_select(t(n), t(out), t(br.pos), t(br.tok), t(br.block))
    torch.cuda.synchronize()
    return hit.cpu().numpy(), nxt.cpu().numpy(), int(hits.item())


def planted(B, k, V, C, F, blk, seed):
    rng = np.random.default_rng(seed)
    L = rng.integers(1, k + 1, B).astype(np.int32)
    n = np.array([rng.integers(0, l + 1) for l in L], np.int32)
    out = np.full((B, k + 1), -1, np.int32)
    for b in range(B):
        out[b, :n[b] + 1] = rng.integers(0, V, n[b] + 1)
    br = synth.make_d3d_branches(L, V, C, F, blk, seed=seed + 1)
    NB = br.pos.shape[1]
    for b in range(B):
        if rng.random() < 0.6:
            s = int(rng.integers(0, NB))
            br.pos[b, s], br.tok[b, s] = n[b], out[b, n[b]]
            if rng.random() < 0.3:  # a second, later copy: the first one must win
                s2 = int(rng.integers(s, NB))
                br.pos[b, s2], br.tok[b, s2] = n[b], out[b, n[b]]
    n[rng.random(B) < 0.05] = -1
    return n, out, br


@pytest.mark.parametrize("B,k,V,C,F,blk", [
    (128, 16, 151936, 12, 2, 16),   # the paper's main configuration
    (1, 4, 10, 3, 1, 4),
    (300, 16, 50, 12, 6, 40),       # 68 branches (three ballot rounds), blocks of 40
    (7, 31, 1000, 32, 1, 1),
])
def test_d3d_matches_oracle(B, k, V, C, F, blk):
    n, out, br = planted(B, k, V, C, F, blk, seed=B + C)
    want = oracle.d3d_select(n, out, br.pos, br.tok, br.block)
    got = run(n, out, br)
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1], want[1])
    assert got[2] == want[2]


def test_d3d_after_verification_on_the_device():
    """spec_verify then spec_d3d_select on the same stream, tables planted from the oracle."""
    inp = synth.make_inputs("zipf_mixed_temp", 64, 16, 20000, "bf16", seed=91)
    o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                      inp.temperature)
    br = synth.make_d3d_branches(inp.lengths, inp.V, 12, 2, 16, seed=92)
    rng = np.random.default_rng(93)
    for b in range(inp.B):
        if o.num_accepted[b] >= 0 and rng.random() < 0.7:
            s = int(rng.integers(0, br.pos.shape[1]))
            br.pos[b, s], br.tok[b, s] = o.num_accepted[b], o.out_tokens[b, o.num_accepted[b]]
    d = sv.to_device(inp)
    out, nacc = sv.spec_verify(**d)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    hit, nxt, hits = sv.spec_d3d_select(nacc, out, t(br.pos), t(br.tok), t(br.block))
    torch.cuda.synchronize()
    want_hit, want_nxt, _ = oracle.d3d_select(o.num_accepted, o.out_tokens, br.pos, br.tok,
                                             br.block)
    gpu_out, gpu_n = out.cpu().numpy(), nacc.cpu().numpy()
    # Verification under the parity rule: differences only at near-ties.
    compare(gpu_out, gpu_n, o, inp.temperature, "verification before D3D selection")
    same = (gpu_n == o.num_accepted) & np.all(gpu_out == o.out_tokens, 1)
    np.testing.assert_array_equal(hit.cpu().numpy()[same], want_hit[same])
    np.testing.assert_array_equal(nxt.cpu().numpy()[same], want_nxt[same])
    assert int(hits.item()) == int((hit.cpu().numpy() >= 0).sum())


def test_d3d_many_requests():
    n, out, br = planted(70000, 4, 100, 3, 2, 8, seed=70)
    want = oracle.d3d_select(n, out, br.pos, br.tok, br.block)
    got = run(n, out, br)
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1], want[1])
    assert got[2] == want[2]
