// Row sweep: one streaming pass over every logit row verification needs.
//
// For a sampling row (T > 0) it computes the row's online max and sum of
// 2^((z - max) * log2(e) / T) (p and q must be normalised over the whole
// vocabulary: AdaFlash Section 2.1); for a greedy row (T == 0) the max and
// its lowest index (DFlash notes, section 5.2, worked example #4).
//
// Persistent, warp-specialised CTAs:
//   - lane 0 of the producer warp claims work units (one vocabulary chunk of
//     one row) from a global counter and streams each chunk into a ring of
//     shared-memory stages with 1-D bulk async copies (cp.async.bulk,
//     completion counted on an mbarrier, L2 evict_first: each byte is read
//     once);
//   - eight consumer warps copy their share of a stage into registers, free
//     the stage, take one packed max over it, rescale at most once, and then
//     do independent FMA / ex2 / adds (or an argmax) on it;
//   - at the end of a unit the consumer warps leave their warp-reduced
//     accumulators in shared memory for the bookkeeping warp, which merges
//     them, stores the unit's partial and, in verification mode, does the
//     global counting and the accept decision, off the consumers' path.
//
// Verification mode: the CTA that completes the last chunk of (request b,
// position i) combines the partials, gathers p(x_i) and q(x_i), and applies
// the accept test u_i < min(1, p(x_i)/q(x_i)) (or argmax == x_i at T == 0)
// with float-float log-probabilities.  A rejection is published in first_reject[b]; the
// producer skips chunks of positions behind a known rejection, since only
// tokens before the first rejection are kept (AdaFlash Section 2.1).
#pragma once

#include "common.cuh"

namespace specv {

struct SweepParams {
  const void* target;        // verify: [B, k+1, V]; stats: [rows, V]
  const void* draft;         // verify: [B, k, V]
  const int32_t* tokens;     // [B, k]
  const float* uniforms;     // [B, k+1]
  int B, k, V, nch, chunk_elems;
  int early_exit;
  int direct;                // rows in pinned host memory: no bulk copies (kFlagDirect)
  long long rows_t, rows_d;  // rows of the target and draft buffers (range checks)
  long long parts_total;     // partial slots in the workspace (range checks)
  unsigned char* ws;
  WsLayout lay;
};

// kFlagDiscard closes a unit whose request was rejected at an earlier
// position while it streamed: its partial is neither stored nor counted.
// kFlagDirect: the stage was not copied; the consumers load its bytes from the
// row itself (logits in pinned host memory, read over the CPU-GPU link).
constexpr int kFlagFirst = 1, kFlagLast = 2, kFlagGreedy = 4, kFlagEnd = 8, kFlagDiscard = 16,
              kFlagDirect = 32;

struct StageInfo {
  const void* row;  // row base (element 0)
  int part;         // Partial index: slot * nch + chunk
  int flags;
  int elem0;        // element index of the stage buffer's first byte
  int nbytes;       // bulk bytes in the stage (multiple of 16, may be 0)
  int head0, headn; // elements before the 16-byte aligned range (first stage)
  int tail0, tailn; // elements after it (last stage)
  float sc;         // log2(e) / T
  int slot;         // row slot ((b*k+i)<<1 | tensor) or row index
};

// What the bookkeeping warp needs to know about a finished unit.
struct UnitMeta {
  int part;
  int slot;
  int flags;
  float sc;
};

constexpr int kNC = kSweepConsumerWarps;
constexpr int kNCT = kNC * 32;
// The bookkeeping and producer warps come first: a warp scheduler that
// favours older warps then does not starve them behind the consumers, which
// are ready to issue most of the time.
constexpr int kBookWarp = 0;
constexpr int kProducerWarp = 1;
constexpr int kFirstConsumerWarp = 2;
constexpr int kVecPerThread = kStageBytes / 16 / kNCT;  // 16-byte vectors per consumer thread
static_assert(kSweepThreads == (kNC + 2) * 32, "kNC consumer warps + producer + bookkeeping");
static_assert(kStageBytes % (16 * kNCT) == 0, "a stage splits evenly over the consumer threads");
static_assert((kVecPerThread & (kVecPerThread - 1)) == 0, "batch_max reduces a power-of-two batch");
static_assert(kNC <= 32, "unit-end merge gives one lane of the bookkeeping warp per consumer warp");

struct SweepSmem {
  alignas(128) unsigned char stage[kStages][kStageBytes];
  uint64_t full[kStages];        // 1 arrival + bulk bytes: stage loaded
  uint64_t empty[kStages];       // kNC arrivals: stage copied into registers
  uint64_t red_bar[kRedDepth];   // kNC arrivals: unit accumulators posted
  uint64_t red_free[kRedDepth];  // 1 arrival: bookkeeping warp has read the slot
  StageInfo info[kStages];
  UnitMeta meta[kRedDepth];
  float4 red[kRedDepth][kNC];
  int abort_flag;
};

__device__ __forceinline__ void sweep_abort(WsHeader* h, SweepSmem& sm) {
  record_status(h, SPEC_ERR_TIMEOUT);
  *(volatile int*)&sm.abort_flag = 1;
}

// ---------------------------------------------------------------------------
// Producer: one warp.  The warp claims a few consecutive units per atomic,
// resolves their descriptors and skip checks with one lane per unit, and
// claims the next batch before lane 0 issues this batch's bulk copies, so the
// claim's round trip overlaps the copy issue.  Near the end of the work list
// it claims single units so that the CTAs finish together.
// ---------------------------------------------------------------------------
constexpr int kClaim = 4;

// The descriptor of a CTA's first unit (unit blockIdx.x), loaded before the
// unit count is known so that the two loads travel together: the grid has
// at most one CTA per unit slot, so the index lies inside the descriptor
// array; the caller uses the descriptor only if the unit exists.
__device__ __forceinline__ int4 first_descriptor(const SweepParams& p, const int4* rowdesc) {
  return __ldcg(&rowdesc[SPEC_CHECKED((int)blockIdx.x / p.nch, p.parts_total / p.nch,
                                      kSiteSweepRowdesc)]);
}

template <typename TIn, bool kVerify>
__device__ void sweep_producer(const SweepParams& p, SweepSmem& sm, WsHeader* h) {
  using Tr = ElemTraits<TIn>;
  const int lane = threadIdx.x & 31;
  const int4* rowdesc = reinterpret_cast<const int4*>(p.ws + p.lay.rowdesc);
  const int32_t* first_reject = reinterpret_cast<const int32_t*>(p.ws + p.lay.first_reject);
  // The first unit's descriptor goes out with the unit count (see
  // first_descriptor).
  const int4 rd_first = first_descriptor(p, rowdesc);
  const int units_total = __ldcg(&h->units_total);
  const int small_after = units_total - 4 * kClaim * (int)gridDim.x;
  volatile int* abort_flag = &sm.abort_flag;
  int it = 0;  // stages issued (lane 0)
  bool ok = true;
  unsigned long long my_chunks = 0, my_bytes = 0;

  auto acquire = [&](int& s) -> bool {
    s = it % kStages;
    const int round = it / kStages;
    if (round > 0 && !mbar_wait_bounded(&sm.empty[s], (round - 1) & 1, abort_flag)) {
      sweep_abort(h, sm);
      return false;
    }
    return true;
  };

  // Batches move through a three-deep pipeline: claimed (atomic in flight),
  // described (row descriptors loaded, one lane per unit), checked (skip
  // flag loaded), then issued.  Each step consumes values loaded one loop
  // iteration earlier, so no global round trip stands in front of a copy.
  // Units 0 .. gridDim.x-1 are the CTAs' first units, one each, taken
  // without a claim so that the first copy waits for no round trip; the
  // counter hands out the units after them.
  auto want_at = [&](int base) { return base < small_after ? kClaim : 1; };
  auto claim = [&](int want) {
    int v = 0;
    if (lane == 0) v = (int)gridDim.x + atomicAdd(&h->work_next, want);
    return v;  // lane 0 only; broadcast when needed
  };
  auto describe = [&](int base, int want) {
    int4 rd = make_int4(-1, 0, 0, 0);
    if (lane < want && base + lane < units_total)
      rd = __ldcg(&rowdesc[SPEC_CHECKED((base + lane) / p.nch, units_total / p.nch,
                                        kSiteSweepRowdesc)]);
    return rd;
  };
  auto check = [&](int4 rd) {  // first known rejection of the unit's request, or k
    int fr = INT32_MAX;
    if (kVerify && p.early_exit && rd.x >= 0) {
      const int b = (rd.x >> 1) / p.k;
      fr = *(volatile const int32_t*)&first_reject[b];
    }
    return fr;
  };

  int wantC = 1;
  int baseC = (int)blockIdx.x;
  int4 rdC = (lane == 0 && baseC < units_total) ? rd_first : make_int4(-1, 0, 0, 0);
  // No decision can precede a CTA's first unit by much; the check before
  // each stage still applies to it.
  int frC = INT32_MAX;
  int wantB = want_at(baseC + wantC);
  int baseB = __shfl_sync(0xffffffffu, claim(wantB), 0);
  int4 rdB = describe(baseB, wantB);
  int wantA = want_at(baseB + wantB);
  int atomA = claim(wantA);

  while (baseC < units_total) {
    // Advance the look-ahead: skip flag for B, descriptors for A, a new claim.
    const int frB = check(rdB);
    const int baseA = __shfl_sync(0xffffffffu, atomA, 0);
    const int4 rdA = describe(baseA, wantA);
    const int wantN = want_at(baseA + wantA);
    const int atomN = claim(wantN);

    // Issue batch C: units not behind a known rejection of their request.
    bool live = rdC.x >= 0;
    if (kVerify && live && p.early_exit) {
      const int bi = rdC.x >> 1;
      if (frC < bi - (bi / p.k) * p.k) live = false;
    }
    unsigned mask = __ballot_sync(0xffffffffu, live);
    while (mask) {
      const int l = __ffs(mask) - 1;
      mask &= mask - 1;
      const int uu = baseC + l;
      const int slot = __shfl_sync(0xffffffffu, rdC.x, l);
      const float sc = __int_as_float(__shfl_sync(0xffffffffu, rdC.y, l));
      const int lrow = __shfl_sync(0xffffffffu, rdC.z, l);
      if (lane == 0) {
        const int chunk = uu - (uu / p.nch) * p.nch;
        // The descriptor's row is absolute within its buffer (target or draft).
        const bool drow = kVerify && (slot & 1);
        const TIn* rowp =
            static_cast<const TIn*>(drow ? p.draft : p.target) +
            (size_t)SPEC_CHECKED(lrow, drow ? p.rows_d : p.rows_t, kSiteSweepRow) * (size_t)p.V;
        const bool greedy = (sc == 0.0f);
        // Element range of the chunk and its 16-byte aligned core.
        const int e0 = chunk * p.chunk_elems;
        const int e1 = min(p.V, e0 + p.chunk_elems);
        const uintptr_t addr0 = reinterpret_cast<uintptr_t>(rowp + e0);
        int a0 = e0 + (int)(((16u - (unsigned)(addr0 & 15u)) & 15u) / Tr::kSize);
        if (a0 > e1) a0 = e1;
        const int core_bytes = (((e1 - a0) * Tr::kSize) & ~15);
        const int a1 = a0 + core_bytes / Tr::kSize;
        const int nstage = core_bytes > 0 ? (core_bytes + kStageBytes - 1) / kStageBytes : 1;
        const char* src0 = reinterpret_cast<const char*>(rowp + a0);
        // Position and request of the unit, for the per-stage skip check.
        const int ub = kVerify ? (slot >> 1) / p.k : 0;
        const int ui = kVerify ? (slot >> 1) - ub * p.k : 0;
        const bool recheck = kVerify && p.early_exit;
        for (int j = 0; j < nstage; ++j) {
          // Look again for a rejection at an earlier position of the request
          // before each stage; the load is issued before the ring wait, which
          // hides its latency.
          const int frj = recheck ? *(volatile const int32_t*)&first_reject[ub] : INT32_MAX;
          int s;
          if (!acquire(s)) {
            ok = false;
            break;
          }
          const bool drop = frj < ui;
          if (drop && j == 0) break;  // nothing issued yet: skip the unit
          const int off = j * kStageBytes;
          const int nb = (core_bytes > 0 && !drop) ? min(kStageBytes, core_bytes - off) : 0;
          StageInfo& I = sm.info[s];
          I.row = rowp;
          I.part = slot * p.nch + chunk;
          I.flags = (j == 0 ? kFlagFirst : 0) | (j == nstage - 1 || drop ? kFlagLast : 0) |
                    (drop ? kFlagDiscard : 0) | (greedy ? kFlagGreedy : 0);
          I.elem0 = a0 + off / Tr::kSize;
          I.nbytes = nb;
          I.head0 = e0;
          I.headn = a0 - e0;
          I.tail0 = a1;
          I.tailn = drop ? 0 : e1 - a1;
          I.sc = sc;
          I.slot = slot;
          if (p.direct) I.flags |= kFlagDirect;
          if (nb > 0 && !p.direct) {
            mbar_arrive_expect_tx(&sm.full[s], (uint32_t)nb);
            bulk_g2s_hint(sm.stage[s], src0 + off, (uint32_t)nb, &sm.full[s],
                      l2_policy_evict_first());
          } else {
            mbar_arrive(&sm.full[s]);
          }
          ++it;
          if (j == 0) {
            my_chunks += 1;
            my_bytes += (unsigned long long)(a0 - e0) * Tr::kSize;
          }
          my_bytes += (unsigned long long)nb;
          if (j == nstage - 1) my_bytes += (unsigned long long)(e1 - a1) * Tr::kSize;
          if (drop) break;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
    }
    if (!ok) break;

    // Rotate the pipeline.
    baseC = baseB;
    wantC = wantB;
    rdC = rdB;
    frC = frB;
    baseB = baseA;
    wantB = wantA;
    rdB = rdA;
    wantA = wantN;
    atomA = atomN;
  }

  if (lane != 0) return;
  atomicAdd(&h->chunks_swept, my_chunks);
  atomicAdd(&h->sweep_bytes, my_bytes);
  if (ok) {
    int s;
    if (acquire(s)) {
      sm.info[s].flags = kFlagEnd;
      mbar_arrive(&sm.full[s]);
      ++it;
      return;
    }
  }
  // Aborted: wait (bounded) for the copies still in flight into this CTA's
  // shared memory before the CTA may exit.
  for (int back = 1; back <= kStages && back <= it; ++back) {
    const int jt = it - back;
    int dummy = 0;
    mbar_wait_bounded(&sm.full[jt % kStages], (jt / kStages) & 1, (volatile int*)&dummy);
  }
}

// ---------------------------------------------------------------------------
// Producer for units of two stages or more (lane 0 of the producer warp).
// It claims one unit at a time, kLookStages stages before the current unit
// runs out: the claim goes out at that stage, the unit's descriptor load one
// stage later, so both round trips overlap copies already in flight and the
// units are streamed in the order they were claimed -- the position-major
// order of the work list, which makes a rejection known before the rows
// behind it are read.  Whether a unit is behind a known rejection is looked
// up before each of its stages (the load goes out before the ring wait).
// ---------------------------------------------------------------------------
constexpr int kLookStages = 3;

template <typename TIn, bool kVerify>
__device__ void sweep_producer_big(const SweepParams& p, SweepSmem& sm, WsHeader* h) {
  using Tr = ElemTraits<TIn>;
  if ((threadIdx.x & 31) != 0) return;
  const int4* rowdesc = reinterpret_cast<const int4*>(p.ws + p.lay.rowdesc);
  const int32_t* first_reject = reinterpret_cast<const int32_t*>(p.ws + p.lay.first_reject);
  const int4 rd_first = first_descriptor(p, rowdesc);
  const int units_total = __ldcg(&h->units_total);
  volatile int* abort_flag = &sm.abort_flag;
  const bool recheck = kVerify && p.early_exit;
  int it = 0;  // stages issued
  bool ok = true;
  unsigned long long my_chunks = 0, my_bytes = 0;

  auto acquire = [&](int& s) -> bool {
    s = it % kStages;
    const int round = it / kStages;
    if (round > 0 && !mbar_wait_bounded(&sm.empty[s], (round - 1) & 1, abort_flag)) {
      sweep_abort(h, sm);
      return false;
    }
    return true;
  };
  auto describe = [&](int u) {
    return u < units_total
               ? __ldcg(&rowdesc[SPEC_CHECKED(u / p.nch, units_total / p.nch, kSiteSweepRowdesc)])
               : make_int4(-1, 0, 0, 0);
  };

  // The CTA's first unit is unit blockIdx.x, taken without a claim so that
  // the first copy waits for no round trip; the counter hands out the units
  // after the grid's first ones.
  int nxt = (int)blockIdx.x;
  int4 nrd = nxt < units_total ? rd_first : make_int4(-1, 0, 0, 0);
  bool first_unit = true;
  while (nxt < units_total) {
    const int uu = nxt;
    const int4 rd = nrd;
    nxt = -1;
    bool described = false;
    const int slot = rd.x;
    const float sc = __int_as_float(rd.y);
    const int chunk = uu - (uu / p.nch) * p.nch;
    int ub = 0, ui = 0;
    if (kVerify) {
      const int bi = slot >> 1;
      ub = bi / p.k;
      ui = bi - ub * p.k;
    }
    // The descriptor's row is absolute within its buffer (target or draft).
    const bool drow = kVerify && (slot & 1);
    const TIn* rowp =
        static_cast<const TIn*>(drow ? p.draft : p.target) +
        (size_t)SPEC_CHECKED(rd.z, drow ? p.rows_d : p.rows_t, kSiteSweepRow) * (size_t)p.V;
    const bool greedy = (sc == 0.0f);
    // Element range of the chunk and its 16-byte aligned core.
    const int e0 = chunk * p.chunk_elems;
    const int e1 = min(p.V, e0 + p.chunk_elems);
    const uintptr_t addr0 = reinterpret_cast<uintptr_t>(rowp + e0);
    int a0 = e0 + (int)(((16u - (unsigned)(addr0 & 15u)) & 15u) / Tr::kSize);
    if (a0 > e1) a0 = e1;
    const int core_bytes = (((e1 - a0) * Tr::kSize) & ~15);
    const int a1 = a0 + core_bytes / Tr::kSize;
    const int nstage = core_bytes > 0 ? (core_bytes + kStageBytes - 1) / kStageBytes : 1;
    const char* src0 = reinterpret_cast<const char*>(rowp + a0);
    const int look = nstage > kLookStages ? nstage - kLookStages : 0;
    for (int j = 0; j < nstage; ++j) {
      // The CTA's first stage goes out without the look: no decision can
      // precede it by much, and its load would stand before the first copy.
      const int frj = (recheck && !(first_unit && j == 0))
                          ? *(volatile const int32_t*)&first_reject[ub]
                          : INT32_MAX;
      if (j == look) nxt = (int)gridDim.x + atomicAdd(&h->work_next, 1);
      if (j == look + 1) {
        nrd = describe(nxt);
        described = true;
      }
      int s;
      if (!acquire(s)) {
        ok = false;
        break;
      }
      const bool drop = frj < ui;
      if (drop && j == 0) break;  // nothing issued yet: skip the unit
      const int off = j * kStageBytes;
      const int nb = (core_bytes > 0 && !drop) ? min(kStageBytes, core_bytes - off) : 0;
      StageInfo& I = sm.info[s];
      I.row = rowp;
      I.part = slot * p.nch + chunk;
      I.flags = (j == 0 ? kFlagFirst : 0) | (j == nstage - 1 || drop ? kFlagLast : 0) |
                (drop ? kFlagDiscard : 0) | (greedy ? kFlagGreedy : 0);
      I.elem0 = a0 + off / Tr::kSize;
      I.nbytes = nb;
      I.head0 = e0;
      I.headn = a0 - e0;
      I.tail0 = a1;
      I.tailn = drop ? 0 : e1 - a1;
      I.sc = sc;
      I.slot = slot;
      if (p.direct) I.flags |= kFlagDirect;
      if (nb > 0 && !p.direct) {
        mbar_arrive_expect_tx(&sm.full[s], (uint32_t)nb);
        bulk_g2s_hint(sm.stage[s], src0 + off, (uint32_t)nb, &sm.full[s],
                      l2_policy_evict_first());
      } else {
        mbar_arrive(&sm.full[s]);
      }
      ++it;
      if (j == 0) {
        my_chunks += 1;
        my_bytes += (unsigned long long)(a0 - e0) * Tr::kSize;
      }
      my_bytes += (unsigned long long)nb;
      if (j == nstage - 1) my_bytes += (unsigned long long)(e1 - a1) * Tr::kSize;
      if (drop) break;
    }
    if (!ok) break;
    first_unit = false;
    // A unit that ended before its look-ahead point claims its successor now.
    if (nxt < 0) nxt = (int)gridDim.x + atomicAdd(&h->work_next, 1);
    if (!described) nrd = describe(nxt);
  }

  atomicAdd(&h->chunks_swept, my_chunks);
  atomicAdd(&h->sweep_bytes, my_bytes);
  if (ok) {
    int s;
    if (acquire(s)) {
      sm.info[s].flags = kFlagEnd;
      mbar_arrive(&sm.full[s]);
      ++it;
      return;
    }
  }
  // Aborted: wait (bounded) for the copies still in flight into this CTA's
  // shared memory before the CTA may exit.
  for (int back = 1; back <= kStages && back <= it; ++back) {
    const int jt = it - back;
    int dummy = 0;
    mbar_wait_bounded(&sm.full[jt % kStages], (jt / kStages) & 1, (volatile int*)&dummy);
  }
}

// ---------------------------------------------------------------------------
// Decision for (b, i) once all of its chunks are in (warp-cooperative).
// ---------------------------------------------------------------------------
// x, u and rb (token x_i, uniform u_i and the request's first target and
// draft rows) were loaded one unit earlier, when the chunk count was taken.  With dry set, the partials come from the
// workspace's made-up position and nothing is recorded: the call only brings
// this code into the instruction cache while memory is still quiet (its first
// real use comes when the sweep has HBM saturated, where every instruction
// fetch would wait in the queues).  Kept out of line so that both calls run
// the same code.
template <typename TIn>
__device__ __noinline__ void decide_position(const SweepParams& p, int bi, bool greedy, float sc,
                                             int x, float u_i, int2 rb, bool dry) {
  const int lane = threadIdx.x & 31;
  if (!dry) bi = (int)SPEC_CHECKED(bi, (long long)p.B * p.k, kSiteDecide);
  const int b = bi / p.k;
  const int i = bi - b * p.k;
  const Partial* parts = reinterpret_cast<const Partial*>(p.ws + p.lay.partials);
  const Partial* pt =
      dry ? reinterpret_cast<const Partial*>(p.ws + p.lay.warm) : parts + (size_t)(bi << 1) * p.nch;
  float4* pos_c = reinterpret_cast<float4*>(p.ws + p.lay.pos_c);
  int32_t* pos_arg = reinterpret_cast<int32_t*>(p.ws + p.lay.pos_arg);
  uint32_t* bad_bits = reinterpret_cast<uint32_t*>(p.ws + p.lay.bad_bits);
  unsigned long long* state = reinterpret_cast<unsigned long long*>(p.ws + p.lay.state);
  int32_t* first_reject = reinterpret_cast<int32_t*>(p.ws + p.lay.first_reject);

  bool accept, row_ok, late;
  if (greedy) {
    float v;
    int g;
    row_argmax_from_parts(pt, p.nch, &v, &g, &late);
    row_ok = (g != INT32_MAX);
    accept = (g == x);
    if (lane == 0 && !dry) __stcg(&pos_arg[bi], g);
  } else {
    // The gathers of z_t[x] and z_d[x] go out first and overlap the partial
    // loads.  Target chunks then draft chunks: the two slots are adjacent.
    // The dry run gathers from the workspace instead, which always exists.
    const TIn* trow =
        dry ? reinterpret_cast<const TIn*>(p.ws + p.lay.warm)
            : static_cast<const TIn*>(p.target) +
                  (size_t)SPEC_CHECKED((long long)rb.x + i, p.rows_t, kSiteSweepRow) * (size_t)p.V;
    const TIn* drow =
        dry ? reinterpret_cast<const TIn*>(p.ws + p.lay.warm)
            : static_cast<const TIn*>(p.draft) +
                  (size_t)SPEC_CHECKED((long long)rb.y + i, p.rows_d, kSiteSweepRow) * (size_t)p.V;
    // A token out of range (the final pass turns its request into -1) reads
    // element 0 instead and counts as a row without mass.
    const bool x_ok = (unsigned)x < (unsigned)p.V;
    const float zt = ElemTraits<TIn>::load(trow, x_ok ? x : 0);
    const float zd = ElemTraits<TIn>::load(drow, x_ok ? x : 0);
    FF ct, cd;
    bool okt, okd;
    pair_log2_normalisers(pt, p.nch, sc, &ct, &cd, &okt, &okd, &late);
    row_ok = okt && okd && x_ok;
    // A token the target gives probability zero is never accepted; a token
    // the drafter gives probability zero (and the target not) always is.
    // Otherwise d = log2 p(x) - log2 q(x) = (zt*sc - ct) - (zd*sc - cd) in
    // float-float (the products exact), and the ratio 2^d in single
    // precision: near any threshold u its absolute error is below 1e-7.
    float ratio;
    if (zt == -INFINITY) {
      ratio = 0.0f;
    } else if (zd == -INFINITY) {
      ratio = 1.0f;
    } else {
      const FF d = ff_sub(ff_sub(two_prod(zt, sc), ct), ff_sub(two_prod(zd, sc), cd));
      const float df = ff_to_float(d);
      ratio = df >= 0.0f ? 1.0f : exp2f(df);
    }
    accept = u_i < ratio;
    if (lane == 0 && !dry) __stcg(&pos_c[bi], make_float4(ct.hi, ct.lo, cd.hi, cd.lo));
  }
  // A row without finite mass makes the request invalid if the round reaches
  // it; it also ends the round there so no later row is read for nothing.
  if (!row_ok) accept = false;
  if (lane == 0 && !dry) {
    if (late) record_status(reinterpret_cast<WsHeader*>(p.ws + p.lay.header), SPEC_ERR_TIMEOUT);
    if (!row_ok) atomicOr(&bad_bits[b], 1u << i);
    // The early-exit hint first, so that producers see it as soon as possible.
    if (!accept) atomicMin(&first_reject[b], i);
    // An accept only sets its bits.  A rejection (or a row without mass)
    // releases with them: a final-pass CTA that sees the bit also sees this
    // position's normalisers, argmax and bad-row bit, written above.
    if (accept) atomicOr(&state[b], decision_bits(i, true));
    else atom_or_release_u64(&state[b], decision_bits(i, false));
  }
}

// ---------------------------------------------------------------------------
// Consumers: warps kFirstConsumerWarp .. kFirstConsumerWarp + kNC - 1.
// ---------------------------------------------------------------------------

// Post this warp's accumulator for the unit (or the end marker) in reduction
// slot `units % kRedDepth`, once the bookkeeping warp has released it.
__device__ __forceinline__ bool post_unit(SweepSmem& sm, WsHeader* h, int units, const float4& acc,
                                          const UnitMeta& meta) {
  const int warp = (threadIdx.x >> 5) - kFirstConsumerWarp, lane = threadIdx.x & 31;
  const int rs = units % kRedDepth;
  if (units >= kRedDepth &&
      !mbar_wait_bounded(&sm.red_free[rs], ((units / kRedDepth) - 1) & 1, &sm.abort_flag)) {
    sweep_abort(h, sm);
    return false;
  }
  if (lane == 0) {
    sm.red[rs][warp] = acc;
    if (warp == 0) sm.meta[rs] = meta;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&sm.red_bar[rs]);
  return true;
}

template <typename TIn>
__device__ void sweep_consumers(SweepSmem& sm, WsHeader* h) {
  using Tr = ElemTraits<TIn>;
  constexpr int EPV = Tr::kPerVec;
  const int warp = (threadIdx.x >> 5) - kFirstConsumerWarp;  // consumer warp 0 .. kNC-1
  const int lane = threadIdx.x & 31;
  const int ctid = threadIdx.x - kFirstConsumerWarp * 32;
  volatile int* abort_flag = &sm.abort_flag;

  SoftAcc sa;
  ArgAcc aa;
  soft_init(sa);
  arg_init(aa);
  int it = 0, units = 0;
  for (;;) {
    const int s = it % kStages;
    if (!mbar_wait_bounded(&sm.full[s], (it / kStages) & 1, abort_flag)) {
      sweep_abort(h, sm);
      return;
    }
    const StageInfo I = sm.info[s];
    if (I.flags & kFlagEnd) {
      UnitMeta end = {0, 0, kFlagEnd, 0.0f};
      post_unit(sm, h, units, make_float4(0.f, 0.f, 0.f, 0.f), end);
      return;
    }
    const bool greedy = (I.flags & kFlagGreedy) != 0;
    const TIn* row = static_cast<const TIn*>(I.row);
    if (I.flags & kFlagFirst) {
      soft_init(sa);
      arg_init(aa);
      if (warp == 0 && lane < I.headn) {
        const float x = Tr::load(row, I.head0 + lane);
        if (greedy) arg_add(aa, x, I.head0 + lane);
        else soft_add1(sa, x, I.sc);
      }
    }
    // Copy this thread's vectors out of the stage, then hand the stage back.
    const int nvec = I.nbytes >> 4;
    uint4 v[kVecPerThread];
    if (I.flags & kFlagDirect) {
      // Not copied: the same 16-byte aligned range, loaded from the row.
      const uint4* src = reinterpret_cast<const uint4*>(row + I.elem0);
#pragma unroll
      for (int t = 0; t < kVecPerThread; ++t) {
        const int j = ctid + t * kNCT;
        v[t] = j < nvec ? __ldg(src + j) : neg_inf_vec<TIn>();
      }
    } else {
      const uint4* buf = reinterpret_cast<const uint4*>(sm.stage[s]);
#pragma unroll
      for (int t = 0; t < kVecPerThread; ++t) {
        const int j = ctid + t * kNCT;
        v[t] = j < nvec ? buf[j] : neg_inf_vec<TIn>();
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
    ++it;

    if (greedy) arg_stage<TIn>(aa, v, I.elem0 + ctid * EPV, kNCT * EPV);
    else soft_stage<TIn>(sa, v, I.sc);
    if ((I.flags & kFlagLast) && warp == 0 && lane < I.tailn) {
      const float x = Tr::load(row, I.tail0 + lane);
      if (greedy) arg_add(aa, x, I.tail0 + lane);
      else soft_add1(sa, x, I.sc);
    }
    if (!(I.flags & kFlagLast)) continue;

    // ---- end of a unit: warp-reduce and post for the bookkeeping warp ----
    float4 acc;
    if (greedy) {
      arg_warp_reduce(aa);
      acc = make_float4(aa.v, __int_as_float(aa.i), 0.f, 0.f);
    } else {
      soft_warp_reduce(sa);
      acc = make_float4(sa.m, sa.ms, sa.s, 0.f);
    }
    const UnitMeta meta = {I.part, I.slot, I.flags, I.sc};
    if (!post_unit(sm, h, units, acc, meta)) return;
    ++units;
  }
}

// ---------------------------------------------------------------------------
// Bookkeeping warp: merges the consumer warps' accumulators of each unit,
// stores the unit's partial and, in verification mode, counts the chunks of
// (b, i) and decides when the last one is in.
// ---------------------------------------------------------------------------
template <typename TIn, bool kVerify>
__device__ void sweep_bookkeeper(const SweepParams& p, SweepSmem& sm, WsHeader* h) {
  const int lane = threadIdx.x & 31;
  Partial* parts = reinterpret_cast<Partial*>(p.ws + p.lay.partials);
  int32_t* done = reinterpret_cast<int32_t*>(p.ws + p.lay.done);
  // The chunk count of a unit is looked at one unit later, so that the
  // atomic's round trip overlaps the next unit's merge and store.  No fence
  // orders a partial before its count: the deciding CTA instead waits for
  // each partial slot of (b, i) to leave the empty marker, which it does
  // because every counted unit has already issued its store.
  int pend_bi = -1, pend_old = 0, pend_need = 0, pend_x = 0;
  bool pend_greedy = false;
  float pend_sc = 0.0f, pend_u = 0.0f;
  int2 pend_rb = make_int2(0, 0);
  if (kVerify) {
    // Run the decision paths the round's rows need once, without effect,
    // while the first units are still streaming in (see decide_position).
    const int kinds = __ldcg(&h->row_kinds);
    if (kinds & 2) decide_position<TIn>(p, 0, false, 1.0f, 0, 0.5f, make_int2(0, 0), true);
    if (kinds & 1) decide_position<TIn>(p, 0, true, 0.0f, 0, 0.5f, make_int2(0, 0), true);
  }
  auto resolve_pending = [&]() {
    if (!kVerify || pend_bi < 0) return;
    const int old = __shfl_sync(0xffffffffu, pend_old, 0);
    if (old == pend_need - 1)
      decide_position<TIn>(p, pend_bi, pend_greedy, pend_sc, pend_x, pend_u, pend_rb, false);
    pend_bi = -1;
  };
  for (int u = 0;; ++u) {
    const int rs = u % kRedDepth;
    const uint32_t par = (u / kRedDepth) & 1;
    // Nothing to merge yet: settle the previous unit's count while waiting.
    const bool ready = mbar_test_wait(&sm.red_bar[rs], par);
    if (!__all_sync(0xffffffffu, ready)) resolve_pending();
    if (!mbar_wait_bounded(&sm.red_bar[rs], par, &sm.abort_flag)) {
      sweep_abort(h, sm);
      return;
    }
    const UnitMeta meta = sm.meta[rs];
    const float4 r = lane < kNC ? sm.red[rs][lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.red_free[rs]);
    if (meta.flags & kFlagEnd) {
      resolve_pending();
      return;
    }
    if (meta.flags & kFlagDiscard) continue;

    const bool greedy = (meta.flags & kFlagGreedy) != 0;
    float out_m;
    uint32_t out_aux;
    if (greedy) {
      ArgAcc a;
      arg_init(a);
      if (lane < kNC) {
        a.v = r.x;
        a.i = __float_as_int(r.y);
      }
      arg_warp_reduce(a);
      out_m = a.v;
      out_aux = (uint32_t)a.i;
    } else {
      SoftAcc a;
      soft_init(a);
      if (lane < kNC) {
        a.m = r.x;
        a.ms = r.y;
        a.s = r.z;
      }
      soft_warp_reduce(a);
      out_m = a.m;
      out_aux = __float_as_uint(a.s);
    }
    if (lane == 0)
      store_partial(&parts[SPEC_CHECKED(meta.part, p.parts_total, kSiteSweepPartial)], out_m,
                    out_aux);

    if (kVerify) {
      // Count this chunk of (b, i); the CTA that brings the count to its
      // total decides.
      int old = 0;
      if (lane == 0)
        old = atomicAdd(&done[SPEC_CHECKED(meta.slot >> 1, (long long)p.B * p.k, kSiteSweepCount)],
                        1);
      resolve_pending();
      pend_bi = meta.slot >> 1;
      pend_old = old;
      pend_need = greedy ? p.nch : 2 * p.nch;
      pend_greedy = greedy;
      pend_sc = meta.sc;
      // What a decision would need, loaded now so that it is in registers
      // if this chunk turns out to be the last of (b, i).
      const int pb = pend_bi / p.k;
      const int pi = pend_bi - pb * p.k;
      pend_x = __ldg(&p.tokens[(size_t)pb * p.k + pi]);
      pend_u = __ldg(&p.uniforms[(size_t)pb * (p.k + 1) + pi]);
      pend_rb = __ldcg(reinterpret_cast<const int2*>(p.ws + p.lay.rowbase) + pb);
    }
  }
}

template <typename TIn, bool kVerify>
__global__ void __launch_bounds__(kSweepThreads, kSweepMinBlocks) sweep_kernel(SweepParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SweepSmem& sm = *reinterpret_cast<SweepSmem*>(smem_raw);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kNC);
    }
    for (int r = 0; r < kRedDepth; ++r) {
      mbar_init(&sm.red_bar[r], kNC);
      mbar_init(&sm.red_free[r], 1);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Everything below reads what the plan kernel wrote.
  pdl_wait();
  // The final pass may launch now: its CTAs take the SMs this grid leaves
  // during its tail and each waits for its own request's decisions.
  if (kVerify) pdl_launch_dependents();
  WsHeader* h = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
  // Warp 0 keeps the books, warp 1 produces, warps 2..kNC+1 consume; the
  // mbarrier counts and reduction slots are sized for exactly this split.
  const int warp = threadIdx.x >> 5;
  if (warp >= kFirstConsumerWarp) {
    sweep_consumers<TIn>(sm, h);
  } else if (warp == kProducerWarp) {
    // Units of two stages or more get the one-unit look-ahead producer;
    // smaller ones the batched one, which keeps enough bytes in flight.
    if (p.chunk_elems * (int)sizeof(TIn) >= 2 * kStageBytes)
      sweep_producer_big<TIn, kVerify>(p, sm, h);
    else
      sweep_producer<TIn, kVerify>(p, sm, h);
  } else if (warp == kBookWarp) {
    sweep_bookkeeper<TIn, kVerify>(p, sm, h);
  }
  // Count the CTA out once all its work is done, so that the final pass can
  // hold its own completion until every sweep CTA has finished.
  __syncthreads();
  if (kVerify && threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&h->sweep_exited, 1);
  }
}

}  // namespace specv
