"""The C-ABI library builds, loads and exports what include/spec_verify.h declares (no GPU).

Only host-side logic runs here: size queries, status strings, and argument
checks that return before any CUDA call.
"""

import ctypes
import os
import re

import pytest

import speculative_decoding_verification_58_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    sv.build()
    return sv.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert sorted(sv.EXPORTS) == declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_abi_version_and_status_strings(lib):
    assert lib.spec_abi_version() == 1
    for code in range(8):
        s = sv.status_string(code)
        assert s and "unknown" not in s
    assert "unknown" in sv.status_string(99)


def test_workspace_sizes(lib):
    a = sv.spec_verify_workspace_bytes(128, 16, 151936)
    b = sv.spec_verify_workspace_bytes(256, 16, 151936)
    assert 0 < a < b
    assert a % 256 == 0
    assert sv.spec_verify_workspace_bytes(0, 16, 100) == 0
    assert sv.spec_verify_workspace_bytes(4, 32, 100) == 0        # k > SPEC_MAX_K
    assert sv.spec_verify_workspace_bytes(4, 16, (1 << 21) + 1) == 0
    assert lib.spec_row_stats_workspace_bytes(10, 1000) > 0


def test_host_checks_return_before_any_cuda_call(lib):
    f = lib.spec_verify
    ws = ctypes.create_string_buffer(1 << 20)
    # Null pointers.
    assert f(None, None, 0, None, None, None, None, 2, 3, 64, None, None, None, 0, None) == \
        sv.SPEC_ERR_INVALID_ARG
    # Unsupported sizes.
    assert f(1, 1, 0, 1, 1, 1, 1, 2, 40, 64, 1, 1, None, 0, None) == sv.SPEC_ERR_UNSUPPORTED
    assert f(1, 1, 0, 1, 1, 1, 1, 0, 3, 64, 1, 1, None, 0, None) == sv.SPEC_ERR_INVALID_ARG
    # Bad dtype and flags.
    assert f(16, 16, 7, 16, 16, 16, 16, 2, 3, 64, 16, 16, 256, 1 << 20, None) == \
        sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_verify_ex(16, 16, 0, 16, 16, 16, 16, 2, 3, 64, 16, 16, 256, 1 << 20, None,
                              8) == sv.SPEC_ERR_INVALID_ARG
    # Misaligned logits, then a missing / small / misaligned workspace.
    assert f(18, 16, 0, 16, 16, 16, 16, 2, 3, 64, 16, 16, 256, 1 << 20, None) == \
        sv.SPEC_ERR_INVALID_ARG
    assert f(16, 16, 0, 16, 16, 16, 16, 2, 3, 64, 16, 16, None, 1 << 20, None) == \
        sv.SPEC_ERR_WORKSPACE
    assert f(16, 16, 0, 16, 16, 16, 16, 2, 3, 64, 16, 16, 256, 8, None) == sv.SPEC_ERR_WORKSPACE
    assert f(16, 16, 0, 16, 16, 16, 16, 2, 3, 64, 16, 16, 264, 1 << 20, None) == \
        sv.SPEC_ERR_WORKSPACE
    g = lib.spec_row_stats
    assert g(None, 0, 4, 10, None, None, None, None, None, 0, None) == sv.SPEC_ERR_INVALID_ARG
    assert g(16, 0, 4, 10, 16, 16, 16, 16, 256, 0, None) == sv.SPEC_ERR_WORKSPACE
    del ws


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(sv, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        sv.lib()


def test_bound_call_checks_buffers_once_at_construction():
    torch = pytest.importorskip("torch")
    B, k, V = 2, 3, 16
    t = torch.zeros(B, k + 1, V)
    good = dict(target_logits=t, draft_logits=torch.zeros(B, k, V),
                draft_tokens=torch.zeros(B, k, dtype=torch.int32),
                lengths=torch.ones(B, dtype=torch.int32), uniforms=torch.zeros(B, k + 1),
                temperature=torch.ones(B))
    for key, bad in (("draft_logits", torch.zeros(B, k + 1, V)),
                     ("draft_tokens", torch.zeros(B, k, dtype=torch.int64)),
                     ("uniforms", torch.zeros(B, k)),
                     ("temperature", torch.ones(B + 1)),
                     ("draft_logits", torch.zeros(B, k, V, dtype=torch.bfloat16))):
        with pytest.raises((TypeError, ValueError)):
            sv.Verifier(**{**good, key: bad})


def test_d3d_select_host_checks(lib):
    f = lib.spec_d3d_select
    ok = dict(n=16, out=16, pos=16, tok=16, blk_=16, B=2, k=3, NB=4, blk=5, hit=16, nxt=16, hits=None)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["n"], a["out"], a["pos"], a["tok"], a["blk_"], a["B"], a["k"], a["NB"], a["blk"],
                 a["hit"], a["nxt"], a["hits"], None)

    assert call(B=0) == sv.SPEC_ERR_INVALID_ARG
    assert call(NB=0) == sv.SPEC_ERR_INVALID_ARG
    assert call(blk=0) == sv.SPEC_ERR_INVALID_ARG
    assert call(k=40) == sv.SPEC_ERR_UNSUPPORTED
    assert call(pos=None) == sv.SPEC_ERR_INVALID_ARG
    assert call(nxt=18) == sv.SPEC_ERR_INVALID_ARG
    assert call(hits=18) == sv.SPEC_ERR_INVALID_ARG


def test_range_checking_build_exports_the_same_symbols(lib):
    # The -DSPEC_DEBUG build sits beside the release library: same entry
    # points, and it says which one it is.
    from speculative_decoding_verification_58_gb300 import make_lib
    dbg = ctypes.CDLL(make_lib.LIB_DEBUG)
    for name in declared_functions():
        assert hasattr(dbg, name), name
    assert dbg.spec_debug_build() == 1
    assert lib.spec_debug_build() == 0
    # A release build has no checks to report and touches no device for it.
    f, site = ctypes.c_int32(7), ctypes.c_int32(7)
    assert lib.spec_debug_checks(ctypes.addressof(f), ctypes.addressof(site), 1, None) == sv.SPEC_OK
    assert (f.value, site.value) == (0, 0)
