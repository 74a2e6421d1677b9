"""Host-side pieces of bench.py that need no GPU."""

import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_code_digest_ignores_comments_and_blank_lines_only():
    """A recorded ncu capture stays valid across comment edits, not code edits."""
    digest = _bench().code_digest
    base = digest([("sweep.cuh", "int x = 1;  // a count\n\nint y;\n")])
    assert base == digest([("sweep.cuh", "// header\nint x = 1;   // the count, reworded\nint y;")])
    assert base != digest([("sweep.cuh", "int x = 2;  // a count\n\nint y;\n")])
    assert base != digest([("plan.cuh", "int x = 1;  // a count\n\nint y;\n")])
    assert base != digest([("sweep.cuh", "int x = 1;\nint y;"), ("plan.cuh", "")])


def test_csrc_digest_covers_the_sweep_sources():
    bench = _bench()
    d = bench.csrc_digest()
    assert len(d) == 16 and int(d, 16) >= 0
