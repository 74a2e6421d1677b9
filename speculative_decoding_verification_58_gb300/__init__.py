"""GB300-native batched speculative-decoding verification.

A thin Python binding over the C ABI of ``libspecverify.so`` (declared in
``include/spec_verify.h``).  Every step of verification runs in the
library's CUDA kernels; this module only checks tensor shapes, passes raw
device pointers and the current CUDA stream, and turns status codes into
exceptions.  There is no CPU fallback: if the library has not been built,
every call raises.

The functions keep the C names:

``spec_verify(...)``                 batched verification (asynchronous)
``spec_verify_packed(...)``          the same over a packed (ragged) batch of rows
``Verifier(...)``                    spec_verify bound to fixed buffers (one C call per round)
``spec_verify_workspace_bytes(...)`` workspace size for (B, k, V)
``spec_verify_report(ws)``           what the device recorded for the last call
``spec_verify_device_status(ws)``    just the recorded status
``spec_row_stats(...)``              the row sweep alone: max, logsumexp, argmax
``spec_opd_stats(...)``              OPD supervision statistics (hard label, reverse KL, clipped)
``spec_verify_opd(...)``             verification and OPD statistics in one pass over the rows
``spec_d3d_select(...)``             D3D branch selection: reuse a prepared successor block
``spec_status_string(code)``
``spec_debug_build()``, ``spec_debug_checks()``  the range-checking build (SPEC_VERIFY_DEBUG=1)
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
# SPEC_VERIFY_DEBUG=1 in the environment loads the range-checking build
# (same entry points; see spec_debug_checks) instead of the release one.
DEBUG_BUILD = os.environ.get("SPEC_VERIFY_DEBUG", "") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "libspecverify_debug.so" if DEBUG_BUILD else "libspecverify.so")

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_UNSUPPORTED = 2
SPEC_ERR_WORKSPACE = 3
SPEC_ERR_CUDA = 4
SPEC_ERR_BAD_INPUT = 5
SPEC_ERR_TIMEOUT = 6
SPEC_ERR_INTERNAL = 7
SPEC_F32 = 0
SPEC_BF16 = 1
SPEC_FLAG_FULL_SWEEP = 1
SPEC_FLAG_TEST_LATE_SLICES = 2

# Every entry point include/spec_verify.h declares.
EXPORTS = ("spec_verify_workspace_bytes", "spec_verify", "spec_verify_ex", "spec_verify_timed",
           "spec_verify_packed", "spec_verify_report",
           "spec_verify_device_status", "spec_row_stats_workspace_bytes", "spec_row_stats",
           "spec_status_string", "spec_abi_version", "spec_verify_static", "spec_opd_stats",
           "spec_verify_opd", "spec_d3d_select", "spec_debug_build", "spec_debug_checks")
SPEC_STATIC_SCRATCH_BYTES = 8 << 20


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


class _Report(ctypes.Structure):
    _fields_ = [("status", ctypes.c_int32), ("bad_requests", ctypes.c_int32),
                ("first_bad_request", ctypes.c_int32), ("rows_planned", ctypes.c_int32),
                ("chunks_swept", ctypes.c_int64), ("chunks_per_row", ctypes.c_int32),
                ("chunk_elems", ctypes.c_int32), ("final_rows", ctypes.c_int64),
                ("residual_zero", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("sweep_bytes", ctypes.c_int64), ("final_bytes", ctypes.c_int64)]


@dataclass
class Report:
    status: int
    bad_requests: int
    first_bad_request: int
    rows_planned: int
    chunks_swept: int
    chunks_per_row: int
    chunk_elems: int
    final_rows: int
    residual_zero: int
    sweep_bytes: int
    final_bytes: int


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded ``libspecverify.so``; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32p, f32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    ci, csz = ctypes.c_int, ctypes.c_size_t
    L.spec_verify_workspace_bytes.argtypes = [ci, ci, ci]
    L.spec_verify_workspace_bytes.restype = csz
    L.spec_verify.argtypes = [vp, vp, ci, i32p, i32p, f32p, f32p, ci, ci, ci, i32p, i32p, vp, csz, vp]
    L.spec_verify.restype = ci
    L.spec_verify_ex.argtypes = L.spec_verify.argtypes + [ctypes.c_uint]
    L.spec_verify_ex.restype = ci
    L.spec_verify_timed.argtypes = L.spec_verify_ex.argtypes + [vp, vp, vp, vp]
    L.spec_verify_timed.restype = ci
    L.spec_verify_packed.argtypes = [vp, ctypes.c_longlong, vp, ctypes.c_longlong, ci, i32p, i32p,
                                     i32p, i32p, f32p, f32p, ci, ci, ci, i32p, i32p, vp, csz, vp,
                                     ctypes.c_uint]
    L.spec_verify_packed.restype = ci
    L.spec_verify_static.argtypes = [vp, vp, ci, i32p, i32p, f32p, f32p, ci, ci, ci, i32p, i32p, vp]
    L.spec_verify_static.restype = ci
    L.spec_verify_report.argtypes = [vp, vp, ctypes.POINTER(_Report)]
    L.spec_verify_report.restype = ci
    L.spec_verify_device_status.argtypes = [vp, vp]
    L.spec_verify_device_status.restype = ci
    L.spec_row_stats_workspace_bytes.argtypes = [ci, ci]
    L.spec_row_stats_workspace_bytes.restype = csz
    L.spec_row_stats.argtypes = [vp, ci, ci, ci, f32p, f32p, f32p, i32p, vp, csz, vp]
    L.spec_row_stats.restype = ci
    L.spec_opd_stats.argtypes = [vp, vp, ci, i32p, ci, ci, ci, ctypes.c_float, ctypes.c_float,
                                 i32p, f32p, f32p, f32p, f32p, vp]
    L.spec_opd_stats.restype = ci
    L.spec_verify_opd.argtypes = [vp, vp, ci, i32p, i32p, f32p, f32p, ci, ci, ci, ctypes.c_float,
                                  ctypes.c_float, i32p, i32p, i32p, f32p, f32p, f32p, f32p, vp, csz,
                                  vp]
    L.spec_verify_opd.restype = ci
    L.spec_d3d_select.argtypes = [i32p, i32p, i32p, i32p, i32p, ci, ci, ci, ci, i32p, i32p, i32p,
                                  vp]
    L.spec_d3d_select.restype = ci
    L.spec_status_string.argtypes = [ci]
    L.spec_status_string.restype = ctypes.c_char_p
    L.spec_abi_version.argtypes = []
    L.spec_abi_version.restype = ci
    L.spec_debug_build.argtypes = []
    L.spec_debug_build.restype = ci
    L.spec_debug_checks.argtypes = [vp, vp, ci, vp]
    L.spec_debug_checks.restype = ci
    _lib = L
    return L


def build(force: bool = False) -> str:
    """Compile the library and its range-checking build in-tree with nvcc
    for sm_103a; return the path of the one this process loads."""
    global _lib
    from . import make_lib
    make_lib.build_all(force=force)
    _lib = None
    return LIB_PATH


def spec_debug_build() -> bool:
    """Whether the loaded library is the range-checking build."""
    return bool(lib().spec_debug_build())


def spec_debug_checks(reset: bool = False, stream=None) -> tuple[int, int]:
    """(failed range checks on the current device since the last reset, site
    of the first); both 0 in a release build."""
    import torch
    f, site = ctypes.c_int32(0), ctypes.c_int32(0)
    st = torch.cuda.current_stream() if stream is None else stream
    code = lib().spec_debug_checks(ctypes.addressof(f), ctypes.addressof(site), int(reset),
                                   ctypes.c_void_p(st.cuda_stream))
    if code != SPEC_OK:
        raise SpecVerifyError(code, "spec_debug_checks")
    return f.value, site.value


def status_string(code: int) -> str:
    try:
        return lib().spec_status_string(code).decode()
    except RuntimeError:
        return f"status {code}"


spec_status_string = status_string


def _check(code: int, where: str) -> None:
    if code != SPEC_OK:
        raise SpecVerifyError(code, where)


def _torch():
    import torch
    return torch


def _stream_ptr(stream) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _need(t, name, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_logits(t, name, dtype, shape, device):
    """Logits on ``device``, or in pinned host memory, which the kernels then
    read themselves over the CPU-GPU link (no copy; early exit also spares
    the link the rows it skips)."""
    if t.device.type == "cpu":
        if not t.is_pinned():
            raise ValueError(f"{name} is in pageable host memory: pin it (pin_memory()) or move it "
                             f"to {device}")
        _need(t, name, dtype, shape, t.device)
    else:
        _need(t, name, dtype, shape, device)


def spec_verify_workspace_bytes(B: int, k: int, V: int) -> int:
    return int(lib().spec_verify_workspace_bytes(B, k, V))


def alloc_workspace(B: int, k: int, V: int, device=None):
    """A device workspace (torch uint8 tensor, 256-byte aligned by the caching allocator)."""
    torch = _torch()
    n = spec_verify_workspace_bytes(B, k, V)
    if n == 0:
        raise SpecVerifyError(SPEC_ERR_UNSUPPORTED, "spec_verify_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def spec_verify(target_logits, draft_logits, draft_tokens, lengths, uniforms, temperature, *,
                workspace=None, out_tokens=None, num_accepted=None, stream=None,
                full_sweep: bool = False, events=None, flags: int = 0):
    """Batched verification on the current (or given) CUDA stream.

    Shapes: target [B, k+1, V], draft [B, k, V] (float32 or bfloat16, same),
    draft_tokens int32 [B, k], lengths int32 [B], uniforms float32 [B, k+1],
    temperature float32 [B].  Returns (out_tokens int32 [B, k+1],
    num_accepted int32 [B]); results are ready when the stream reaches them.

    ``events``: optional four recorded ``torch.cuda.Event`` objects (or None
    entries) marking plan / sweep / final / end, for per-kernel timing
    (measurement only: it disables the kernels' launch overlap).
    ``flags``: further SPEC_FLAG_* bits passed through unchanged.
    """
    torch = _torch()
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = draft_tokens.device
    dt = _dtype_code(target_logits)
    _need_logits(target_logits, "target_logits", target_logits.dtype, (B, k + 1, V), dev)
    _need_logits(draft_logits, "draft_logits", target_logits.dtype, (B, k, V), dev)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k), dev)
    _need(lengths, "lengths", torch.int32, (B,), dev)
    _need(uniforms, "uniforms", torch.float32, (B, k + 1), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    if workspace is None:
        workspace = alloc_workspace(B, k, V, dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, k + 1), dev)
    _need(num_accepted, "num_accepted", torch.int32, (B,), dev)
    flags = int(flags) | (SPEC_FLAG_FULL_SWEEP if full_sweep else 0)
    args = (target_logits.data_ptr(), draft_logits.data_ptr(), dt, draft_tokens.data_ptr(),
            lengths.data_ptr(), uniforms.data_ptr(), temperature.data_ptr(), B, k, V,
            out_tokens.data_ptr(), num_accepted.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_ptr(stream), flags)
    if events is None:
        code = lib().spec_verify_ex(*args)
    else:
        handles = [None if e is None else (e.cuda_event or None) for e in events]
        code = lib().spec_verify_timed(*args, *handles)
    _check(code, "spec_verify")
    return out_tokens, num_accepted


def spec_verify_packed(target_rows, draft_rows, target_row_start, draft_row_start, draft_tokens,
                       lengths, uniforms, temperature, *, workspace=None, out_tokens=None,
                       num_accepted=None, stream=None, full_sweep: bool = False):
    """Verification over a packed batch (AdaFlash Section 3.3: total length sum_b k_b).

    ``target_rows`` [rows_t, V] and ``draft_rows`` [rows_d, V] (float32 or
    bfloat16, same); request b reads target rows ``target_row_start[b] + 0..L_b``
    and draft rows ``draft_row_start[b] + 0..L_b-1`` (int32 [B] each).
    ``draft_tokens`` int32 [B, k] fixes k.  Other arguments and the results are
    those of ``spec_verify``.
    """
    torch = _torch()
    rows_t, V = target_rows.shape
    B, k = draft_tokens.shape
    dev = draft_tokens.device
    dt = _dtype_code(target_rows)
    rows_d = draft_rows.shape[0]
    _need_logits(target_rows, "target_rows", target_rows.dtype, (rows_t, V), dev)
    _need_logits(draft_rows, "draft_rows", target_rows.dtype, (rows_d, V), dev)
    _need(target_row_start, "target_row_start", torch.int32, (B,), dev)
    _need(draft_row_start, "draft_row_start", torch.int32, (B,), dev)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k), dev)
    _need(lengths, "lengths", torch.int32, (B,), dev)
    _need(uniforms, "uniforms", torch.float32, (B, k + 1), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    if workspace is None:
        workspace = alloc_workspace(B, k, V, dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, k + 1), dev)
    _need(num_accepted, "num_accepted", torch.int32, (B,), dev)
    code = lib().spec_verify_packed(
        target_rows.data_ptr(), rows_t, draft_rows.data_ptr() if rows_d else None, rows_d, dt,
        target_row_start.data_ptr(), draft_row_start.data_ptr(), draft_tokens.data_ptr(),
        lengths.data_ptr(), uniforms.data_ptr(), temperature.data_ptr(), B, k, V,
        out_tokens.data_ptr(), num_accepted.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream),
        SPEC_FLAG_FULL_SWEEP if full_sweep else 0)
    _check(code, "spec_verify_packed")
    return out_tokens, num_accepted


class Verifier:
    """``spec_verify`` bound to one fixed set of device buffers.

    A serving loop verifies into the same buffers every round; this object
    checks their shapes, dtypes and devices once, at construction, and keeps
    the C call's argument tuple, so that each round costs the host one ctypes
    call (the Python checks of ``spec_verify`` cost more than a short round
    on the GPU).  The buffers' contents may change between calls; the
    tensors themselves must stay alive and keep their storage.
    """

    def __init__(self, target_logits, draft_logits, draft_tokens, lengths, uniforms, temperature,
                 *, workspace=None, out_tokens=None, num_accepted=None, stream=None,
                 full_sweep: bool = False):
        torch = _torch()
        B, k1, V = target_logits.shape
        k = k1 - 1
        dev = draft_tokens.device
        dt = _dtype_code(target_logits)
        _need_logits(target_logits, "target_logits", target_logits.dtype, (B, k + 1, V), dev)
        _need_logits(draft_logits, "draft_logits", target_logits.dtype, (B, k, V), dev)
        _need(draft_tokens, "draft_tokens", torch.int32, (B, k), dev)
        _need(lengths, "lengths", torch.int32, (B,), dev)
        _need(uniforms, "uniforms", torch.float32, (B, k + 1), dev)
        _need(temperature, "temperature", torch.float32, (B,), dev)
        if workspace is None:
            workspace = alloc_workspace(B, k, V, dev)
        if out_tokens is None:
            out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
        if num_accepted is None:
            num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
        _need(out_tokens, "out_tokens", torch.int32, (B, k + 1), dev)
        _need(num_accepted, "num_accepted", torch.int32, (B,), dev)
        # Keep every buffer referenced for as long as the bound call exists.
        self._keep = (target_logits, draft_logits, draft_tokens, lengths, uniforms, temperature,
                      workspace)
        self.workspace, self.out_tokens, self.num_accepted = workspace, out_tokens, num_accepted
        self._fn = lib().spec_verify_ex
        self._args = (target_logits.data_ptr(), draft_logits.data_ptr(), dt,
                      draft_tokens.data_ptr(), lengths.data_ptr(), uniforms.data_ptr(),
                      temperature.data_ptr(), B, k, V, out_tokens.data_ptr(),
                      num_accepted.data_ptr(), workspace.data_ptr(),
                      workspace.numel() * workspace.element_size(), _stream_ptr(stream),
                      SPEC_FLAG_FULL_SWEEP if full_sweep else 0)

    def __call__(self):
        """Enqueue one round on the bound stream; returns (out_tokens, num_accepted)."""
        code = self._fn(*self._args)
        if code != SPEC_OK:
            raise SpecVerifyError(code, "spec_verify")
        return self.out_tokens, self.num_accepted


def spec_verify_static(target_logits, draft_logits, draft_tokens, lengths, uniforms, temperature,
                       *, out_tokens=None, num_accepted=None, stream=None):
    """spec_verify for callers that cannot allocate: no workspace argument.

    The library uses its own fixed scratch array (SPEC_STATIC_SCRATCH_BYTES
    per GPU, held until exit) instead.  Calls that overlap on the GPU share it
    and race.  If ``out_tokens`` / ``num_accepted`` are given, this wrapper
    allocates nothing either.
    """
    torch = _torch()
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = draft_tokens.device
    dt = _dtype_code(target_logits)
    _need_logits(target_logits, "target_logits", target_logits.dtype, (B, k + 1, V), dev)
    _need_logits(draft_logits, "draft_logits", target_logits.dtype, (B, k, V), dev)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k), dev)
    _need(lengths, "lengths", torch.int32, (B,), dev)
    _need(uniforms, "uniforms", torch.float32, (B, k + 1), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, k + 1), dev)
    _need(num_accepted, "num_accepted", torch.int32, (B,), dev)
    code = lib().spec_verify_static(
        target_logits.data_ptr(), draft_logits.data_ptr(), dt, draft_tokens.data_ptr(),
        lengths.data_ptr(), uniforms.data_ptr(), temperature.data_ptr(), B, k, V,
        out_tokens.data_ptr(), num_accepted.data_ptr(), _stream_ptr(stream))
    _check(code, "spec_verify_static")
    return out_tokens, num_accepted


def spec_verify_report(workspace, stream=None) -> Report:
    """Synchronise the stream and read what the last call on ``workspace`` recorded."""
    r = _Report()
    _check(lib().spec_verify_report(workspace.data_ptr(), _stream_ptr(stream), ctypes.byref(r)),
           "spec_verify_report")
    return Report(r.status, r.bad_requests, r.first_bad_request, r.rows_planned, r.chunks_swept,
                  r.chunks_per_row, r.chunk_elems, r.final_rows, r.residual_zero, r.sweep_bytes,
                  r.final_bytes)


def spec_verify_device_status(workspace, stream=None) -> int:
    return int(lib().spec_verify_device_status(workspace.data_ptr(), _stream_ptr(stream)))


def spec_row_stats(logits, temperature, *, stream=None):
    """Row sweep alone over [rows, V] logits: (max, natural-log logsumexp of z/T, argmax).

    ``lse`` is NaN for T == 0 rows; ``argmax`` is -1 for T > 0 rows.
    """
    torch = _torch()
    rows, V = logits.shape
    dev = temperature.device
    dt = _dtype_code(logits)
    _need_logits(logits, "logits", logits.dtype, (rows, V), dev)
    _need(temperature, "temperature", torch.float32, (rows,), dev)
    n = int(lib().spec_row_stats_workspace_bytes(rows, V))
    if n == 0:
        raise SpecVerifyError(SPEC_ERR_UNSUPPORTED, "spec_row_stats_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    mx = torch.empty(rows, dtype=torch.float32, device=dev)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    arg = torch.empty(rows, dtype=torch.int32, device=dev)
    _check(lib().spec_row_stats(logits.data_ptr(), dt, rows, V, temperature.data_ptr(),
                                mx.data_ptr(), lse.data_ptr(), arg.data_ptr(), ws.data_ptr(), n,
                                _stream_ptr(stream)), "spec_row_stats")
    return mx, lse, arg


def _logits_to_device(a, device):
    torch = _torch()
    import numpy as np
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def to_device_packed(packed, device="cuda"):
    """Copy a ``synth.PackedRows`` layout to the device (the packed entry's row buffers)."""
    torch = _torch()
    return dict(target_rows=_logits_to_device(packed.target_rows, device),
                draft_rows=_logits_to_device(packed.draft_rows, device),
                target_row_start=torch.from_numpy(packed.target_row_start).to(device),
                draft_row_start=torch.from_numpy(packed.draft_row_start).to(device))


@dataclass
class OpdStats:
    x_star: object    # int32 [B, k]
    hard: object      # float32 [B, k]
    rkl: object       # float32 [B, k]
    rkl_clip: object  # float32 [B, k]
    loss: object      # float32 [B]


def spec_opd_stats(target_logits, draft_logits, lengths, *, delta: float = 0.01,
                   alpha: float = 0.8, out=None, stream=None) -> OpdStats:
    """OPD supervision statistics (AdaFlash Section 3.1) on the verification buffers.

    target [B, k+1, V], draft [B, k, V] (float32 or bfloat16), lengths int32 [B].
    Per verified position: target argmax, -log q(argmax), reverse KL and its
    entry-wise clipped form; per request the alpha mixture loss.  ``out`` may
    be an ``OpdStats`` of preallocated tensors.
    """
    torch = _torch()
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = lengths.device
    dt = _dtype_code(target_logits)
    # Host-resident logits reach the library, which refuses them.
    _need_logits(target_logits, "target_logits", target_logits.dtype, (B, k + 1, V), dev)
    _need_logits(draft_logits, "draft_logits", target_logits.dtype, (B, k, V), dev)
    _need(lengths, "lengths", torch.int32, (B,), dev)
    if out is None:
        f = dict(dtype=torch.float32, device=dev)
        out = OpdStats(torch.empty((B, k), dtype=torch.int32, device=dev), torch.empty((B, k), **f),
                       torch.empty((B, k), **f), torch.empty((B, k), **f), torch.empty(B, **f))
    _need(out.x_star, "x_star", torch.int32, (B, k), dev)
    for name in ("hard", "rkl", "rkl_clip"):
        _need(getattr(out, name), name, torch.float32, (B, k), dev)
    _need(out.loss, "loss", torch.float32, (B,), dev)
    _check(lib().spec_opd_stats(target_logits.data_ptr(), draft_logits.data_ptr(), dt,
                                lengths.data_ptr(), B, k, V, float(delta), float(alpha),
                                out.x_star.data_ptr(), out.hard.data_ptr(), out.rkl.data_ptr(),
                                out.rkl_clip.data_ptr(), out.loss.data_ptr(), _stream_ptr(stream)),
           "spec_opd_stats")
    return out


def spec_verify_opd(target_logits, draft_logits, draft_tokens, lengths, uniforms, temperature, *,
                    delta: float = 0.01, alpha: float = 0.8, workspace=None, out_tokens=None,
                    num_accepted=None, out=None, stream=None):
    """Verification and OPD statistics in one pass over the rows.

    Arguments as ``spec_verify`` plus ``delta`` and ``alpha`` as
    ``spec_opd_stats``; ``out`` may be an ``OpdStats`` of preallocated
    tensors.  Returns (out_tokens, num_accepted, OpdStats).
    """
    torch = _torch()
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    dt = _dtype_code(target_logits)
    _need(target_logits, "target_logits", target_logits.dtype, (B, k + 1, V), dev)
    _need(draft_logits, "draft_logits", target_logits.dtype, (B, k, V), dev)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k), dev)
    _need(lengths, "lengths", torch.int32, (B,), dev)
    _need(uniforms, "uniforms", torch.float32, (B, k + 1), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    if workspace is None:
        workspace = alloc_workspace(B, k, V, dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, k + 1), dev)
    _need(num_accepted, "num_accepted", torch.int32, (B,), dev)
    if out is None:
        f = dict(dtype=torch.float32, device=dev)
        out = OpdStats(torch.empty((B, k), dtype=torch.int32, device=dev), torch.empty((B, k), **f),
                       torch.empty((B, k), **f), torch.empty((B, k), **f), torch.empty(B, **f))
    _need(out.x_star, "x_star", torch.int32, (B, k), dev)
    for name in ("hard", "rkl", "rkl_clip"):
        _need(getattr(out, name), name, torch.float32, (B, k), dev)
    _need(out.loss, "loss", torch.float32, (B,), dev)
    _check(lib().spec_verify_opd(
        target_logits.data_ptr(), draft_logits.data_ptr(), dt, draft_tokens.data_ptr(),
        lengths.data_ptr(), uniforms.data_ptr(), temperature.data_ptr(), B, k, V, float(delta),
        float(alpha), out_tokens.data_ptr(), num_accepted.data_ptr(), out.x_star.data_ptr(),
        out.hard.data_ptr(), out.rkl.data_ptr(), out.rkl_clip.data_ptr(), out.loss.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
        "spec_verify_opd")
    return out_tokens, num_accepted, out


def spec_d3d_select(num_accepted, out_tokens, branch_pos, branch_tok, branch_block, *,
                    hit=None, next_block=None, hits=None, stream=None):
    """D3D branch selection (D3D paper, Methodology, asynchronous inference).

    num_accepted int32 [B], out_tokens int32 [B, k+1] (spec_verify's outputs);
    branch_pos, branch_tok int32 [B, NB]; branch_block int32 [B, NB, blk].
    Returns (hit [B], next_block [B, blk], hits [1]) device tensors.
    """
    torch = _torch()
    B, k1 = out_tokens.shape
    NB, blk = branch_block.shape[1], branch_block.shape[2]
    dev = out_tokens.device
    i32 = torch.int32
    _need(num_accepted, "num_accepted", i32, (B,), dev)
    _need(out_tokens, "out_tokens", i32, (B, k1), dev)
    _need(branch_pos, "branch_pos", i32, (B, NB), dev)
    _need(branch_tok, "branch_tok", i32, (B, NB), dev)
    _need(branch_block, "branch_block", i32, (B, NB, blk), dev)
    if hit is None:
        hit = torch.empty(B, dtype=i32, device=dev)
    if next_block is None:
        next_block = torch.empty((B, blk), dtype=i32, device=dev)
    if hits is None:
        hits = torch.empty(1, dtype=i32, device=dev)
    _need(hit, "hit", i32, (B,), dev)
    _need(next_block, "next_block", i32, (B, blk), dev)
    _need(hits, "hits", i32, (1,), dev)
    _check(lib().spec_d3d_select(num_accepted.data_ptr(), out_tokens.data_ptr(),
                                 branch_pos.data_ptr(), branch_tok.data_ptr(),
                                 branch_block.data_ptr(), B, k1 - 1, NB, blk, hit.data_ptr(),
                                 next_block.data_ptr(), hits.data_ptr(), _stream_ptr(stream)),
           "spec_d3d_select")
    return hit, next_block, hits


def to_device(inputs, device="cuda"):
    """Copy a ``synth.SpecInputs`` batch to the device as the C-ABI's buffers."""
    torch = _torch()
    import numpy as np
    if inputs.dtype == "bf16":
        t = torch.from_numpy(inputs.target.view(np.int16)).view(torch.bfloat16)
        d = torch.from_numpy(inputs.draft.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(inputs.target)
        d = torch.from_numpy(inputs.draft)
    return dict(
        target_logits=t.to(device), draft_logits=d.to(device),
        draft_tokens=torch.from_numpy(inputs.tokens).to(device),
        lengths=torch.from_numpy(inputs.lengths).to(device),
        uniforms=torch.from_numpy(inputs.uniforms).to(device),
        temperature=torch.from_numpy(inputs.temperature).to(device))
