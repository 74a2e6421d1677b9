"""Plain fp64 CPU oracle for batched speculative-decoding verification.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package.  The product
library and its Python binding never import, load or call it.

The arithmetic lives in ``oracle.cpp`` (plain single-threaded C++17 in IEEE
double); this module only compiles it with g++ and marshals numpy arrays.
See ``oracle.h`` for the passages each step follows and the readings taken.

Functions whose result is not pinned by an independent check are marked
"parity unpinned" in their docstring; at present every exported function is
pinned by ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

F32 = 0
BF16 = 1

_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.cpp`` into ``liboracle.so`` beside it (g++, no FMA contraction)."""
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest_src:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    vp, i32p, f32p, f64p = (ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32),
                            ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double))
    common = [vp, vp, ctypes.c_int, i32p, i32p]
    tail = [f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, i32p, f64p, f64p, i32p]
    lib.oracle_verify.argtypes = common + [f32p] + tail
    lib.oracle_verify.restype = ctypes.c_int
    lib.oracle_verify_f64u.argtypes = common + [f64p] + tail
    lib.oracle_verify_f64u.restype = ctypes.c_int
    lib.oracle_row_stats.argtypes = [vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int, f32p,
                                     f64p, f64p, i32p]
    lib.oracle_row_stats.restype = None
    lib.oracle_opd_stats.argtypes = [vp, vp, ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_double, ctypes.c_double, i32p, f64p,
                                     f64p, f64p, f64p]
    lib.oracle_opd_stats.restype = ctypes.c_int
    lib.oracle_d3d_select.argtypes = [i32p, i32p, i32p, i32p, i32p, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, i32p, i32p]
    lib.oracle_d3d_select.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _logits(a: np.ndarray) -> tuple[np.ndarray, int]:
    """Accept float32 logits or bf16 logits given as their raw uint16 bits."""
    if a.dtype == np.float32:
        return np.ascontiguousarray(a), F32
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


@dataclass
class OracleResult:
    out_tokens: np.ndarray     # int32 [B, k+1]
    num_accepted: np.ndarray   # int32 [B], -1 for rejected inputs
    margin: np.ndarray         # float64 [B], distance of the outcome's decisions from their thresholds
    final_mass: np.ndarray     # float64 [B], unnormalised mass of the final sampling distribution
    residual_zero: np.ndarray  # int32 [B], 1 where the residual mass was exactly zero
    bad_requests: int


def verify(target_logits, draft_logits, draft_tokens, lengths, uniforms, temperature) -> OracleResult:
    """Run the oracle on host arrays shaped like the C-ABI's buffers.

    ``uniforms`` may be float32 (as the C-ABI takes them) or float64 (used by
    the exact-enumeration pins, which bisect on the uniforms).
    """
    tl, dt = _logits(target_logits)
    dl, dt2 = _logits(draft_logits)
    if dt != dt2:
        raise TypeError("target and draft logits must have the same dtype")
    B, k1, V = tl.shape
    k = k1 - 1
    if dl.shape != (B, k, V):
        raise ValueError(f"draft logits shape {dl.shape} != {(B, k, V)}")
    tok = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, k)
    lens = np.ascontiguousarray(lengths, dtype=np.int32).reshape(B)
    temp = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    out = np.empty((B, k + 1), np.int32)
    nacc = np.empty(B, np.int32)
    margin = np.empty(B, np.float64)
    fmass = np.empty(B, np.float64)
    rzero = np.empty(B, np.int32)
    lib = _load()
    if np.asarray(uniforms).dtype == np.float64:
        u = np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B, k + 1)
        fn, uptr = lib.oracle_verify_f64u, _ptr(u, ctypes.c_double)
    else:
        u = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, k + 1)
        fn, uptr = lib.oracle_verify, _ptr(u, ctypes.c_float)
    bad = fn(tl.ctypes.data, dl.ctypes.data, dt, _ptr(tok, ctypes.c_int32),
             _ptr(lens, ctypes.c_int32), uptr, _ptr(temp, ctypes.c_float), B, k, V,
             _ptr(out, ctypes.c_int32), _ptr(nacc, ctypes.c_int32), _ptr(margin, ctypes.c_double),
             _ptr(fmass, ctypes.c_double), _ptr(rzero, ctypes.c_int32))
    return OracleResult(out, nacc, margin, fmass, rzero, int(bad))


def row_stats(logits, temperature_per_row):
    """Per-row (max, natural-log logsumexp of z/T, lowest argmax) of a [rows, V] buffer."""
    a, dt = _logits(logits)
    V = a.shape[-1]
    rows = a.size // V
    temp = np.ascontiguousarray(np.broadcast_to(np.asarray(temperature_per_row, np.float32),
                                                (rows,)))
    mx = np.empty(rows, np.float64)
    lse = np.empty(rows, np.float64)
    arg = np.empty(rows, np.int32)
    _load().oracle_row_stats(a.ctypes.data, dt, rows, V, _ptr(temp, ctypes.c_float),
                             _ptr(mx, ctypes.c_double), _ptr(lse, ctypes.c_double),
                             _ptr(arg, ctypes.c_int32))
    return mx, lse, arg


def verify_packed(target_rows, draft_rows, target_row_start, draft_row_start, draft_tokens,
                  lengths, uniforms, temperature) -> OracleResult:
    """The oracle on a packed batch (AdaFlash Section 3.3: a verification batch of
    total length sum_b k_b instead of B x k).

    Request b's target rows are ``target_rows[target_row_start[b] + i]`` for
    i = 0..L_b and its draft rows ``draft_rows[draft_row_start[b] + i]`` for
    i < L_b.  A request whose rows fall outside a buffer is invalid (the draft
    rows of a greedy request are not used and not checked).  The rows are
    gathered into the padded layout, the positions no request owns filled with
    NaN (the rule never reads them), and ``verify`` runs on that.
    """
    tr, dt = _logits(target_rows)
    dr, dt2 = _logits(draft_rows) if np.asarray(draft_rows).size else (None, dt)
    if dt != dt2:
        raise TypeError("target and draft rows must have the same dtype")
    tok = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    B, k = tok.shape
    V = tr.shape[1]
    lens = np.asarray(lengths, np.int32).reshape(B)
    temp = np.asarray(temperature, np.float32).reshape(B)
    t0 = np.asarray(target_row_start, np.int64).reshape(B)
    d0 = np.asarray(draft_row_start, np.int64).reshape(B)
    rows_t, rows_d = tr.shape[0], (0 if dr is None else dr.shape[0])
    nan = np.float32(np.nan) if dt == F32 else np.uint16(0x7FC0)
    target = np.full((B, k + 1, V), nan, dtype=tr.dtype)
    draft = np.full((B, k, V), nan, dtype=tr.dtype)
    placed = np.zeros(B, bool)
    for b in range(B):
        L = int(lens[b])
        if not 1 <= L <= k:
            continue  # verify() rejects the length itself
        ok = 0 <= t0[b] and t0[b] + L + 1 <= rows_t
        if temp[b] != 0:
            ok = ok and 0 <= d0[b] and d0[b] + L <= rows_d
        if not ok:
            continue
        placed[b] = True
        target[b, :L + 1] = tr[t0[b]:t0[b] + L + 1]
        if temp[b] != 0:
            draft[b, :L] = dr[d0[b]:d0[b] + L]
    res = verify(target, draft, tok, lens, uniforms, temp)
    for b in range(B):
        if 1 <= lens[b] <= k and not placed[b] and res.num_accepted[b] >= 0:
            res.num_accepted[b] = -1
            res.out_tokens[b] = -1
            res.bad_requests += 1
    return res


@dataclass
class OpdResult:
    x_star: np.ndarray    # int32 [B, k]: argmax of p per position, -1 past L_b
    hard: np.ndarray      # float64 [B, k]: -log q(x_star)
    rkl: np.ndarray       # float64 [B, k]: sum_y q log(q/p)
    rkl_clip: np.ndarray  # float64 [B, k]: sum_y min(q log(q/p), delta)
    loss: np.ndarray      # float64 [B]: alpha * mean hard + (1 - alpha) * mean rkl_clip
    bad_requests: int


def opd_stats(target_logits, draft_logits, lengths, delta=0.01, alpha=0.8) -> OpdResult:
    """OPD supervision statistics per verified position (AdaFlash Section 3.1).

    Same buffers as ``verify``: target [B, k+1, V], draft [B, k, V]; positions
    i < lengths[b].  Defaults are the paper's delta = 0.01 and alpha = 0.8.
    """
    tl, dt = _logits(target_logits)
    dl, dt2 = _logits(draft_logits)
    if dt != dt2:
        raise TypeError("target and draft logits must have the same dtype")
    B, k1, V = tl.shape
    k = k1 - 1
    if dl.shape != (B, k, V):
        raise ValueError(f"draft logits shape {dl.shape} != {(B, k, V)}")
    lens = np.ascontiguousarray(lengths, dtype=np.int32).reshape(B)
    xs = np.empty((B, k), np.int32)
    hard = np.empty((B, k), np.float64)
    rkl = np.empty((B, k), np.float64)
    clip = np.empty((B, k), np.float64)
    loss = np.empty(B, np.float64)
    bad = _load().oracle_opd_stats(tl.ctypes.data, dl.ctypes.data, dt, _ptr(lens, ctypes.c_int32),
                                   B, k, V, float(delta), float(alpha), _ptr(xs, ctypes.c_int32),
                                   _ptr(hard, ctypes.c_double), _ptr(rkl, ctypes.c_double),
                                   _ptr(clip, ctypes.c_double), _ptr(loss, ctypes.c_double))
    return OpdResult(xs, hard, rkl, clip, loss, int(bad))


def d3d_select(num_accepted, out_tokens, branch_pos, branch_tok, branch_block):
    """D3D branch selection (D3D paper, Methodology, asynchronous inference).

    Returns (hit [B] int32: matching branch index or -1, next_block [B, blk]
    int32: that branch's block or -1s, hits: number of requests that hit).
    """
    n = np.ascontiguousarray(num_accepted, dtype=np.int32)
    out = np.ascontiguousarray(out_tokens, dtype=np.int32)
    pos = np.ascontiguousarray(branch_pos, dtype=np.int32)
    tok = np.ascontiguousarray(branch_tok, dtype=np.int32)
    blocks = np.ascontiguousarray(branch_block, dtype=np.int32)
    B, k1 = out.shape
    NB, blk = blocks.shape[1], blocks.shape[2]
    hit = np.empty(B, np.int32)
    nxt = np.empty((B, blk), np.int32)
    hits = _load().oracle_d3d_select(_ptr(n, ctypes.c_int32), _ptr(out, ctypes.c_int32),
                                     _ptr(pos, ctypes.c_int32), _ptr(tok, ctypes.c_int32),
                                     _ptr(blocks, ctypes.c_int32), B, k1 - 1, NB, blk,
                                     _ptr(hit, ctypes.c_int32), _ptr(nxt, ctypes.c_int32))
    return hit, nxt, int(hits)
