"""Seeded synthetic verification inputs, shared by the tests, the benchmark and the smoke check.

This module only draws random numbers: it holds none of the verification
arithmetic (no softmax, no ratio, no residual).  Draft tokens stand for the
drafter's own samples and are drawn with the Gumbel-max trick,
``argmax(z_d + T * G)`` with ``G`` standard Gumbel, which samples
``softmax(z_d / T)`` without normalising anything; at ``T == 0`` the draft
token is ``argmax(z_d)``.

Workloads mimic the pages' serving setting: Qwen3-sized vocabularies
(V = 151936), blocks of k = 16 draft tokens (AdaFlash Appendix B.1), batch
concurrency 1-128 (AdaFlash Table 1), per-request verification lengths
1 <= L_b <= k (AdaFlash Section 3.2) and acceptance that decays with the
draft position (AdaFlash reading notes, Figure 2c discussion).  No dataset or
trained weight is involved.

Recipes (logits generated in fp32, rounded to nearest-even bf16 where the
workload is bf16):

``gauss``            target ~ N(0, 2^2) i.i.d.; draft = target + N(0, 0.5^2).
``zipf``             target = N(0, 1) - 1.1 * log(rank + 1), rank from one seeded
                     vocabulary permutation per request (shared by all of its
                     target and draft rows); draft = target + N(0, 1).
``zipf_adaptive``    ``zipf`` with L_b ~ U{1..k} and T_b ~ U[0.6, 1.0].
``zipf_mixed_noise`` ``zipf`` target; a seeded half of the requests draws draft
                     noise sigma_b = 0.3 and the other half 2.0, growing by 1.08x
                     per position (sigma_b * 1.08^i); L_b ~ U{min(4,k)..k}; T = 1.
``zipf_mixed_temp``  ``zipf_mixed_noise`` logits; a seeded quarter of the requests
                     is greedy (T = 0), the rest T_b ~ U[0.5, 1.2]; L_b ~ U{1..k}.

Uniforms are ``(uint32 >> 8) * 2^-24``, strictly inside [0, 1).

Every request draws from its own child of ``numpy.random.SeedSequence(seed)``,
so the result is the same for any thread count.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

RECIPES = ("gauss", "zipf", "zipf_adaptive", "zipf_mixed_noise", "zipf_mixed_temp")

# The five workloads the library is measured and checked on, named by what they are.
WORKLOADS = {
    "b1_k4_v1024_f32_gauss": dict(recipe="gauss", B=1, k=4, V=1024, dtype="f32", seed=20260001),
    "b1_k16_v151936_bf16_zipf": dict(recipe="zipf", B=1, k=16, V=151936, dtype="bf16",
                                     seed=20260002),
    "b32_k16_v151936_bf16_zipf_adaptive": dict(recipe="zipf_adaptive", B=32, k=16, V=151936,
                                               dtype="bf16", seed=20260003),
    "b128_k16_v151936_bf16_zipf_mixed_noise": dict(recipe="zipf_mixed_noise", B=128, k=16,
                                                   V=151936, dtype="bf16", seed=20260004),
    "b256_k16_v151936_f32_zipf_mixed_temp": dict(recipe="zipf_mixed_temp", B=256, k=16,
                                                 V=151936, dtype="f32", seed=20260005),
}

HEADLINE = "b128_k16_v151936_bf16_zipf_mixed_noise"


@dataclass
class SpecInputs:
    """Host arrays laid out exactly like the C-ABI's buffers."""

    target: np.ndarray       # [B, k+1, V] float32, or uint16 holding bf16 bits
    draft: np.ndarray        # [B, k, V]   same dtype as target
    tokens: np.ndarray       # [B, k]   int32
    lengths: np.ndarray      # [B]      int32
    uniforms: np.ndarray     # [B, k+1] float32 in [0, 1)
    temperature: np.ndarray  # [B]      float32, 0 = greedy
    dtype: str               # "f32" or "bf16"

    @property
    def B(self) -> int:
        return self.target.shape[0]

    @property
    def k(self) -> int:
        return self.draft.shape[1]

    @property
    def V(self) -> int:
        return self.target.shape[2]


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest bf16 (ties to even); return the raw bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bits to float32 (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniform_24bit(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniforms (uint32 >> 8) * 2^-24: 24-bit float32 values strictly inside [0, 1)."""
    bits = rng.integers(0, 2**32, size=shape, dtype=np.uint64).astype(np.uint32)
    return ((bits >> np.uint32(8)).astype(np.float32) * np.float32(2.0**-24)).astype(np.float32)


def _zipf_table(V: int) -> np.ndarray:
    return (-1.1 * np.log(np.arange(V, dtype=np.float64) + 1.0)).astype(np.float32)


def make_inputs(recipe: str, B: int, k: int, V: int, dtype: str, seed: int,
                threads: int | None = None) -> SpecInputs:
    """Generate one batch of verification inputs for ``recipe`` (see module docstring)."""
    if recipe not in RECIPES:
        raise ValueError(f"unknown recipe {recipe!r}")
    if dtype not in ("f32", "bf16"):
        raise ValueError("dtype must be 'f32' or 'bf16'")
    if B < 1 or k < 1 or V < 1:
        raise ValueError("B, k and V must be positive")

    ss = np.random.SeedSequence(seed)
    batch_seq, *req_seqs = ss.spawn(B + 1)
    brng = np.random.default_rng(batch_seq)

    # Per-request scalars: verification length, temperature, draft noise scale.
    if recipe in ("gauss", "zipf"):
        lengths = np.full(B, k, np.int32)
        temps = np.ones(B, np.float32)
    elif recipe == "zipf_adaptive":
        lengths = brng.integers(1, k + 1, size=B).astype(np.int32)
        temps = brng.uniform(0.6, 1.0, size=B).astype(np.float32)
    elif recipe == "zipf_mixed_noise":
        lengths = brng.integers(min(4, k), k + 1, size=B).astype(np.int32)
        temps = np.ones(B, np.float32)
    else:  # zipf_mixed_temp
        lengths = brng.integers(1, k + 1, size=B).astype(np.int32)
        temps = brng.uniform(0.5, 1.2, size=B).astype(np.float32)
        greedy = brng.permutation(B)[: B // 4]
        temps[greedy] = 0.0

    if recipe in ("zipf_mixed_noise", "zipf_mixed_temp"):
        sigma = np.full(B, 2.0)
        sigma[brng.permutation(B)[: B // 2]] = 0.3
        sigma_pos = sigma[:, None] * (1.08 ** np.arange(k))[None, :]
    elif recipe == "gauss":
        sigma_pos = np.full((B, k), 0.5)
    else:
        sigma_pos = np.full((B, k), 1.0)

    uniforms = uniform_24bit(brng, (B, k + 1))

    store = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty((B, k + 1, V), store)
    draft = np.empty((B, k, V), store)
    tokens = np.empty((B, k), np.int32)
    zipf = _zipf_table(V) if recipe != "gauss" else None

    def one_request(b: int) -> None:
        rng = np.random.default_rng(req_seqs[b])
        if recipe == "gauss":
            zt = rng.standard_normal((k + 1, V), dtype=np.float32) * np.float32(2.0)
        else:
            zt = rng.standard_normal((k + 1, V), dtype=np.float32)
            zt += rng.permutation(zipf)[None, :]
        zd = zt[:k] + rng.standard_normal((k, V), dtype=np.float32) * \
            sigma_pos[b].astype(np.float32)[:, None]
        if dtype == "bf16":
            target[b] = bf16_bits(zt)
            draft[b] = bf16_bits(zd)
            zd_stored = bf16_to_f32(draft[b])
        else:
            target[b] = zt
            draft[b] = zd
            zd_stored = zd
        T = float(temps[b])
        if T == 0.0:
            tokens[b] = np.argmax(zd_stored, axis=1)
        else:
            g = rng.gumbel(size=(k, V))
            tokens[b] = np.argmax(zd_stored.astype(np.float64) + T * g, axis=1)

    n_threads = threads or min(16, os.cpu_count() or 1, B)
    if n_threads <= 1:
        for b in range(B):
            one_request(b)
    else:
        with ThreadPoolExecutor(n_threads) as pool:
            list(pool.map(one_request, range(B)))

    return SpecInputs(target, draft, tokens, lengths, uniforms, temps, dtype)


LOW_TV_FORCED_U = np.float32(0.999)


def make_low_tv_inputs(B: int, k: int, V: int, dtype: str, sigma: float, seed: int,
                       threads: int | None = None) -> SpecInputs:
    """A batch whose draft rows are close to the target rows, with forced rejections.

    Target rows as the ``zipf`` recipe; draft = target + N(0, sigma^2) element
    by element (in fp32, before any bf16 rounding), so p and q differ by a
    small total variation and the residual max(0, p - q) carries little mass.
    Every request verifies all k positions at T = 1.  At one seeded position
    j_b < k the uniform is ``LOW_TV_FORCED_U`` (0.999), so the request is
    rejected there whenever p(x)/q(x) < 0.999 (about half the time when the
    earlier positions were accepted) instead of almost never; every other
    uniform is a 24-bit draw.  0.999 keeps the forced decision 1e-3 away from
    the ratio cap 1, so an accepting request is not a near-tie.  Only random
    numbers are drawn here.
    """
    if dtype not in ("f32", "bf16"):
        raise ValueError("dtype must be 'f32' or 'bf16'")
    ss = np.random.SeedSequence(seed)
    batch_seq, *req_seqs = ss.spawn(B + 1)
    brng = np.random.default_rng(batch_seq)
    lengths = np.full(B, k, np.int32)
    temps = np.ones(B, np.float32)
    uniforms = uniform_24bit(brng, (B, k + 1))
    forced = brng.integers(0, k, size=B)
    uniforms[np.arange(B), forced] = LOW_TV_FORCED_U
    store = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty((B, k + 1, V), store)
    draft = np.empty((B, k, V), store)
    tokens = np.empty((B, k), np.int32)
    zipf = _zipf_table(V)

    def one_request(b: int) -> None:
        rng = np.random.default_rng(req_seqs[b])
        zt = rng.standard_normal((k + 1, V), dtype=np.float32)
        zt += rng.permutation(zipf)[None, :]
        zd = zt[:k] + rng.standard_normal((k, V), dtype=np.float32) * np.float32(sigma)
        if dtype == "bf16":
            target[b] = bf16_bits(zt)
            draft[b] = bf16_bits(zd)
            zd_stored = bf16_to_f32(draft[b])
        else:
            target[b] = zt
            draft[b] = zd
            zd_stored = zd
        g = rng.gumbel(size=(k, V))
        tokens[b] = np.argmax(zd_stored.astype(np.float64) + g, axis=1)

    n_threads = threads or min(16, os.cpu_count() or 1, B)
    if n_threads <= 1:
        for b in range(B):
            one_request(b)
    else:
        with ThreadPoolExecutor(n_threads) as pool:
            list(pool.map(one_request, range(B)))
    return SpecInputs(target, draft, tokens, lengths, uniforms, temps, dtype)


def make_workload(name: str, seed: int | None = None, threads: int | None = None,
                  **overrides) -> SpecInputs:
    """Inputs of one named workload; ``overrides`` may shrink B, k or V for fast checks."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    if seed is not None:
        cfg["seed"] = seed
    return make_inputs(cfg["recipe"], cfg["B"], cfg["k"], cfg["V"], cfg["dtype"], cfg["seed"],
                       threads=threads)


@dataclass
class PackedRows:
    """A batch laid out as the packed C-ABI entry takes it (row buffers + first rows)."""

    target_rows: np.ndarray       # [rows_t, V] same dtype as SpecInputs.target
    draft_rows: np.ndarray        # [rows_d, V]
    target_row_start: np.ndarray  # [B] int32
    draft_row_start: np.ndarray   # [B] int32


def pack_rows(inp: SpecInputs, order=None, gap: int = 0) -> PackedRows:
    """Copy each request's rows into flat buffers, requests in ``order``.

    Request b contributes its target rows 0..L_b and draft rows 0..L_b-1 (a
    verification batch of total length sum_b L_b, AdaFlash Section 3.3).
    ``gap`` rows of filler (copies of row 0 of the batch) go after every request, so
    that placements need not be contiguous.  Only copies rows: no arithmetic.
    """
    B = inp.B
    order = np.arange(B) if order is None else np.asarray(order)
    t_start = np.zeros(B, np.int32)
    d_start = np.zeros(B, np.int32)
    trows, drows = [], []
    nt = nd = 0
    for b in order:
        L = int(inp.lengths[b])
        t_start[b], d_start[b] = nt, nd
        trows.append(inp.target[b, :L + 1])
        drows.append(inp.draft[b, :L])
        nt += L + 1
        nd += L
        if gap:
            trows.append(np.repeat(inp.target[0, :1], gap, axis=0))
            drows.append(np.repeat(inp.target[0, :1], gap, axis=0))
            nt += gap
            nd += gap
    return PackedRows(np.ascontiguousarray(np.concatenate(trows)),
                      np.ascontiguousarray(np.concatenate(drows)), t_start, d_start)


@dataclass
class D3DBranches:
    """Successor blocks prepared during verification (D3D asynchronous inference)."""

    pos: np.ndarray    # [B, NB] int32: first-rejection position each branch assumes (-1: unused)
    tok: np.ndarray    # [B, NB] int32: token the branch assumes is emitted there
    block: np.ndarray  # [B, NB, blk] int32: the successor block drafted for it


def d3d_branch_count(C: int, F: int) -> int:
    """Branches per request for position coverage C and token fan-out F: (C - 1) F + 2."""
    return (C - 1) * F + 2


def make_d3d_branches(lengths: np.ndarray, V: int, C: int = 12, F: int = 2, blk: int = 16,
                      seed: int = 0) -> D3DBranches:
    """Seeded branch tables laid out like the D3D packed budget B [(C - 1) F + 2].

    F candidate tokens for each of the C - 1 earliest rejection positions
    (slots past a request's length stay unused), then two for full acceptance
    (position L_b).  Tokens and blocks are uniform draws: a stand-in for the
    drafter's guesses, with no verification arithmetic.
    """
    B = len(lengths)
    NB = d3d_branch_count(C, F)
    rng = np.random.default_rng(seed)
    pos = np.full((B, NB), -1, np.int32)
    for b in range(B):
        L = int(lengths[b])
        for j in range((C - 1) * F):
            if j // F < L:
                pos[b, j] = j // F
        pos[b, NB - 2:] = L
    tok = rng.integers(0, V, (B, NB)).astype(np.int32)
    block = rng.integers(0, V, (B, NB, blk)).astype(np.int32)
    return D3DBranches(pos, tok, block)
