// C ABI of the verification library: argument checks, workspace sizing and
// the launch sequence plan -> sweep -> final on the caller's stream.  The
// sweep and final kernels use programmatic dependent launch so that their
// prologues overlap the previous kernel's tail; each waits for its
// predecessor's results with griddepcontrol.wait before reading them.

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "d3d.cuh"
#include "final.cuh"
#include "opd.cuh"
#include "plan.cuh"
#include "sweep.cuh"

namespace specv {

// A named NVTX range for the lifetime of the object (host side: what an
// entry point enqueues, and each launch within it, shows as a labelled range
// in a timeline profiler; without one attached it costs a pointer check).
class NvtxRange {
 public:
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// ---------------------------------------------------------------------------
// Row-statistics kernels (spec_row_stats).
// ---------------------------------------------------------------------------

WsLayout stats_layout(int rows, int C) {
  WsLayout l = {};
  l.header = 0;
  l.rowdesc = align256(sizeof(WsHeader));
  l.partials = l.rowdesc + align256((size_t)rows * sizeof(int4));
  l.total = l.partials + align256((size_t)rows * C * sizeof(Partial));
  return l;
}

// Row descriptors {row, bits of log2(e)/T, row, 0} for the sweep, and the header.
__global__ void stats_plan_kernel(unsigned char* ws, WsLayout lay, int rows, int nch,
                                  int chunk_elems, const float* temperature) {
  pdl_launch_dependents();
  int4* rowdesc = reinterpret_cast<int4*>(ws + lay.rowdesc);
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) {
    const float T = temperature[r];
    rowdesc[r] = make_int4(r, __float_as_int(T == 0.0f ? 0.0f : softmax_scale(T)), r, 0);
  }
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  WsHeader* h = reinterpret_cast<WsHeader*>(ws + lay.header);
  h->status = SPEC_OK;
  h->bad_requests = 0;
  h->first_bad = INT32_MAX;
  h->work_next = 0;
  h->rows_planned = rows;
  h->units_total = rows * nch;
  h->chunks_per_row = nch;
  h->chunk_elems = chunk_elems;
  h->chunks_swept = 0;
  h->final_rows = 0;
  h->residual_zero = 0;
  h->sweep_bytes = 0;
  h->final_bytes = 0;
}

// One warp per row: combine the chunk partials into max, natural-log
// logsumexp of z/T (sampling rows) and argmax (greedy rows).
__global__ void stats_finalize_kernel(const unsigned char* ws, WsLayout lay, int rows, int nch,
                                      const float* temperature, float* row_max, float* row_lse,
                                      int32_t* row_arg) {
  pdl_wait();
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int lane = threadIdx.x & 31;
  const Partial* parts = reinterpret_cast<const Partial*>(ws + lay.partials) + (size_t)r * nch;
  const float T = temperature[r];
  if (T == 0.0f) {
    float v;
    int g;
    bool late;
    row_argmax_from_parts(parts, nch, &v, &g, &late);
    if (lane == 0) {
      row_max[r] = v;
      row_lse[r] = __int_as_float(0x7fc00000);
      row_arg[r] = (g == INT32_MAX) ? -1 : g;
    }
  } else {
    const float sc = softmax_scale(T);
    FF c;
    float m;
    bool late;
    const bool ok = row_log2_normaliser(parts, nch, sc, &c, &m, &late);
    if (lane == 0) {
      row_max[r] = m;
      row_lse[r] = ok ? ff_to_float(ff_mul_f(c, kLn2f)) : __int_as_float(0x7fc00000);
      row_arg[r] = -1;
    }
  }
}

// ---------------------------------------------------------------------------
// Per-device launch facts.
// ---------------------------------------------------------------------------

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int sweep_blocks_per_sm[2][2] = {{0, 0}, {0, 0}};  // [dtype][verify]
  size_t final_smem_optin = 0;
  bool opd_ready = false;
  int opd_clusters[2][4] = {};  // [dtype][cluster size - 1]: co-resident OPD clusters
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

template <typename TIn, bool kVerify>
cudaError_t sweep_blocks(int* out) {
  cudaError_t e = cudaFuncSetAttribute(sweep_kernel<TIn, kVerify>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(SweepSmem));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, sweep_kernel<TIn, kVerify>,
                                                       kSweepThreads, sizeof(SweepSmem));
}

cudaError_t device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    int optin = 0;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
        cudaSuccess)
      return e;
    d.final_smem_optin = (size_t)optin;
    if ((e = sweep_blocks<float, true>(&d.sweep_blocks_per_sm[0][1])) != cudaSuccess) return e;
    if ((e = sweep_blocks<uint16_t, true>(&d.sweep_blocks_per_sm[1][1])) != cudaSuccess) return e;
    if ((e = sweep_blocks<float, false>(&d.sweep_blocks_per_sm[0][0])) != cudaSuccess) return e;
    if ((e = sweep_blocks<uint16_t, false>(&d.sweep_blocks_per_sm[1][0])) != cudaSuccess) return e;
    const int fsm = (int)std::max(kMaxSegs * sizeof(float2), (size_t)kFinalStages * kFinalStageBytes);
    if ((e = cudaFuncSetAttribute(final_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  fsm)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(final_kernel<uint16_t>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, fsm)) != cudaSuccess)
      return e;
    d.ready = true;
  }
  *out = &d;
  return cudaSuccess;
}

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t record(void* const* ev, int j, cudaStream_t stream) {
  if (ev == nullptr || ev[j] == nullptr) return cudaSuccess;
  return cudaEventRecord(static_cast<cudaEvent_t>(ev[j]), stream);
}

bool sizes_ok(int B, int k, int V) {
  if (B < 1 || k < 1 || V < 1) return false;
  if (B > SPEC_MAX_B || k > SPEC_MAX_K || V > SPEC_MAX_V) return false;
  // Row slots (b*k + i) * 2 + tensor and work units must fit in int32.
  const long long slots = 2LL * B * k;
  if (slots * (long long)chunks_per_row(slots, V) >= (1LL << 31)) return false;
  return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// For the duration of one entry point, make the device that owns `p` current
// on this thread (the caller's framework may keep its own notion of the
// current device), and give the caller's current device back on return.
// Host or unregistered pointers leave the current device alone.
class DeviceOf {
 public:
  explicit DeviceOf(const void* p) {
    cudaPointerAttributes a;
    err_ = cudaPointerGetAttributes(&a, p);
    if (err_ != cudaSuccess) return;
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return;
    if ((err_ = cudaGetDevice(&prev_)) != cudaSuccess) return;
    if (a.device >= 0 && a.device != prev_) {
      err_ = cudaSetDevice(a.device);
      switched_ = (err_ == cudaSuccess);
    }
  }
  ~DeviceOf() {
    if (switched_) cudaSetDevice(prev_);
  }
  bool ok() const { return err_ == cudaSuccess; }

 private:
  cudaError_t err_ = cudaSuccess;
  int prev_ = -1;
  bool switched_ = false;
};

// Launch the plan kernel (padded layout: t_start == nullptr).
cudaError_t launch_plan(const int32_t* draft_tokens, const int32_t* lengths, const float* uniforms,
                        const float* temperature, int B, int k, int V, int C, int ce, int nch,
                        unsigned char* ws, const WsLayout& lay, cudaStream_t stream, bool pdl,
                        const int32_t* t_start, const int32_t* d_start, long long rows_t,
                        long long rows_d, bool skip_t01 = false) {
  NvtxRange r("plan_kernel");
  PlanParams pp;
  pp.skip_t01 = skip_t01 ? 1 : 0;
  pp.tokens = draft_tokens;
  pp.lengths = lengths;
  pp.uniforms = uniforms;
  pp.temperature = temperature;
  pp.t_start = t_start;
  pp.d_start = d_start;
  pp.rows_t = rows_t;
  pp.rows_d = rows_d;
  pp.B = B;
  pp.k = k;
  pp.V = V;
  pp.C = C;
  pp.chunk_elems = ce;
  pp.nch = nch;
  pp.ws = ws;
  pp.lay = lay;
  return launch(plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, pdl, pp);
}

// Launch the final pass behind a grid of `decider_grid` CTAs that publish the
// decisions (the row sweep, or the OPD kernel in verification mode).
template <typename TIn>
cudaError_t launch_final(const DeviceInfo* d, const void* target_logits, const void* draft_logits,
                         const int32_t* draft_tokens, const int32_t* lengths, const float* uniforms,
                         const float* temperature, int B, int k, int V, int32_t* out_tokens,
                         int32_t* num_accepted, unsigned char* ws, const WsLayout& lay,
                         int decider_grid, unsigned flags, cudaStream_t stream, bool pdl,
                         long long rows_t, long long rows_d, bool direct = false) {
  NvtxRange r("final_kernel");
  FinalParams fp;
  fp.target = target_logits;
  fp.draft = draft_logits;
  fp.tokens = draft_tokens;
  fp.lengths = lengths;
  fp.uniforms = uniforms;
  fp.temperature = temperature;
  fp.B = B;
  fp.k = k;
  fp.V = V;
  fp.out_tokens = out_tokens;
  fp.num_accepted = num_accepted;
  fp.ws = ws;
  fp.lay = lay;
  fp.sweep_grid = decider_grid;
  fp.test_late = (flags & SPEC_FLAG_TEST_LATE_SLICES) ? 1 : 0;
  fp.rows_t = rows_t;
  fp.rows_d = rows_d;
  fp.direct = direct ? 1 : 0;
  const int nseg = segments_of(V);
  // Slices per request: one wave of three CTAs per SM over the batch, but at
  // least two (a request's residual pair is 1.2 MB in fp32, too much for one
  // CTA at the end of a round), each slice at least one segment.
  int P = std::max(2, (3 * d->sms) / B);
  if (P > kMaxSlices) P = kMaxSlices;
  if (P > nseg) P = nseg;
  if (P < 1) P = 1;
  fp.P = P;
  // Dynamic shared memory: the slice ring, later reused for the combine's
  // segment records.
  const size_t fsm = std::max((size_t)nseg * sizeof(float2), (size_t)kFinalStages * kFinalStageBytes);
  return launch(final_kernel<TIn>, dim3((unsigned)(P * B)), dim3(kFinalThreads), fsm, stream, pdl,
                fp);
}

// Sweep CTAs for rows in host memory: the SM count divided by this.
constexpr int kDirectSweepDivisor = 4;

// Launch the verification sweep (persistent, a multiple of the SM count);
// *grid_out: its CTAs.
template <typename TIn>
cudaError_t launch_sweep(const DeviceInfo* d, const void* target_logits, const void* draft_logits,
                         const int32_t* draft_tokens, const float* uniforms, int B, int k, int V,
                         int nch, int ce, unsigned char* ws, const WsLayout& lay, bool early_exit,
                         int dtype_index, cudaStream_t stream, bool pdl, int* grid_out,
                         long long rows_t, long long rows_d, bool direct = false) {
  NvtxRange r("sweep_kernel");
  SweepParams sp;
  sp.target = target_logits;
  sp.draft = draft_logits;
  sp.tokens = draft_tokens;
  sp.uniforms = uniforms;
  sp.B = B;
  sp.k = k;
  sp.V = V;
  sp.nch = nch;
  sp.chunk_elems = ce;
  sp.early_exit = early_exit ? 1 : 0;
  sp.ws = ws;
  sp.lay = lay;
  sp.rows_t = rows_t;
  sp.rows_d = rows_d;
  sp.direct = direct ? 1 : 0;
  sp.parts_total = 2LL * B * k * nch;
  const long long max_units = 2LL * B * k * nch;
  // Rows in host memory arrive at the link's rate, which a fraction of the
  // SMs saturates with their loads: fewer CTAs keep fewer units in flight,
  // so the claim front runs less far past the decisions and fewer rows
  // behind a rejection cross the link.
  long long grid = direct ? (long long)d->sms / kDirectSweepDivisor
                          : (long long)d->sms * d->sweep_blocks_per_sm[dtype_index][1];
  // A work list much longer than one wave of CTAs (mid-size batches: 32
  // requests are 16 positions of 128 units for 456 CTAs) is claimed nearly
  // whole at once, far ahead of the decisions; at most two positions' units
  // in flight (but every SM busy) keep the claim front near the decisions,
  // so fewer rows behind a rejection are read (32 requests: 112 MB a round
  // instead of 149, 49.4 µs instead of 51.4).  Small batches keep every unit
  // in flight: their rounds are latency chains.
  if (!direct && max_units > 2 * grid) {
    const long long per_position = 2LL * B * nch;
    grid = std::min(grid, std::max((long long)d->sms, 2 * per_position));
  }
  if (grid > max_units) grid = max_units;
  if (grid < 1) grid = 1;
  *grid_out = (int)grid;
  return launch(sweep_kernel<TIn, true>, dim3((unsigned)grid), dim3(kSweepThreads),
                sizeof(SweepSmem), stream, pdl, sp);
}

template <typename TIn>
spec_status_t verify_typed(const void* target_logits, const void* draft_logits,
                           const int32_t* draft_tokens, const int32_t* lengths,
                           const float* uniforms, const float* temperature, int B, int k, int V,
                           int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                           cudaStream_t stream, unsigned flags, int dtype_index,
                           void* const* ev, const int32_t* t_start = nullptr,
                           const int32_t* d_start = nullptr, long long rows_t = 0,
                           long long rows_d = 0, bool direct = false) {
  NvtxRange r(t_start != nullptr ? "spec_verify_packed" : "spec_verify");
  DeviceInfo* d = nullptr;
  if (device_info(&d) != cudaSuccess) return SPEC_ERR_CUDA;
  const long long slots = 2LL * B * k;
  const int C = chunks_per_row(slots, V);
  const int ce = chunk_elems_for(V, C);
  const int nch = (V + ce - 1) / ce;
  const WsLayout lay = ws_layout(B, k, C, V);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  // With timing events between the kernels there is nothing to overlap.
  const bool pdl = (ev == nullptr);
  if (record(ev, 0, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  if (launch_plan(draft_tokens, lengths, uniforms, temperature, B, k, V, C, ce, nch, ws, lay,
                  stream, pdl, t_start, d_start, rows_t, rows_d) != cudaSuccess)
    return SPEC_ERR_CUDA;

  int grid = 0;
  if (record(ev, 1, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  // Rows of the two buffers: the padded layout's, or the caller's for packed rows.
  const long long nrt = t_start != nullptr ? rows_t : (long long)B * (k + 1);
  const long long nrd = t_start != nullptr ? rows_d : (long long)B * k;
  if (launch_sweep<TIn>(d, target_logits, draft_logits, draft_tokens, uniforms, B, k, V, nch, ce,
                        ws, lay, (flags & SPEC_FLAG_FULL_SWEEP) == 0, dtype_index, stream, pdl,
                        &grid, nrt, nrd, direct) != cudaSuccess)
    return SPEC_ERR_CUDA;

  if (record(ev, 2, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  if (launch_final<TIn>(d, target_logits, draft_logits, draft_tokens, lengths, uniforms,
                        temperature, B, k, V, out_tokens, num_accepted, ws, lay, grid, flags,
                        stream, pdl, nrt, nrd, direct) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (record(ev, 3, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

template <typename TIn>
spec_status_t row_stats_typed(const void* logits, int rows, int V, const float* temperature,
                              float* row_max, float* row_lse, int32_t* row_arg, void* workspace,
                              cudaStream_t stream, int dtype_index, bool direct = false) {
  DeviceInfo* d = nullptr;
  if (device_info(&d) != cudaSuccess) return SPEC_ERR_CUDA;
  const int C = chunks_per_row(rows, V);
  const int ce = chunk_elems_for(V, C);
  const int nch = (V + ce - 1) / ce;
  // Stats mode: header, one descriptor per row, partials at row * nch + chunk.
  const WsLayout lay = stats_layout(rows, C);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  if (launch(stats_plan_kernel, dim3((rows + 255) / 256), dim3(256), 0, stream, false, ws, lay,
             rows, nch, ce, temperature) != cudaSuccess)
    return SPEC_ERR_CUDA;
  SweepParams sp = {};
  sp.target = logits;
  sp.B = rows;
  sp.k = 1;
  sp.V = V;
  sp.nch = nch;
  sp.chunk_elems = ce;
  sp.early_exit = 0;
  sp.ws = ws;
  sp.lay = lay;
  sp.rows_t = rows;
  sp.rows_d = rows;
  sp.direct = direct ? 1 : 0;
  sp.parts_total = (long long)rows * nch;
  long long grid = (long long)d->sms * d->sweep_blocks_per_sm[dtype_index][0];
  if (grid > (long long)rows * nch) grid = (long long)rows * nch;
  if (launch(sweep_kernel<TIn, false>, dim3((unsigned)grid), dim3(kSweepThreads),
             sizeof(SweepSmem), stream, true, sp) != cudaSuccess)
    return SPEC_ERR_CUDA;
  const int wpb = 8;
  if (launch(stats_finalize_kernel, dim3((rows + wpb - 1) / wpb), dim3(wpb * 32), 0, stream, true,
             (const unsigned char*)ws, lay, rows, nch, temperature, row_max, row_lse,
             row_arg) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

size_t row_stats_ws_bytes(int rows, int V) { return stats_layout(rows, chunks_per_row(rows, V)).total; }

// ---------------------------------------------------------------------------
// OPD statistics: cluster shape and launch.
// ---------------------------------------------------------------------------
// Clusters of four CTAs (each a quarter of the vocabulary) for large rows,
// two for medium ones, single CTAs for small vocabularies.
int opd_cluster_size(int V) { return V >= 65536 ? 4 : (V > 16384 ? 2 : 1); }

template <typename TIn>
cudaError_t opd_prepare() {
  cudaError_t e = cudaFuncSetAttribute(opd_kernel<TIn, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(OpdSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(opd_kernel<TIn, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sizeof(OpdSmem));
}

template <typename TIn>
cudaError_t opd_max_clusters(int cs, int* out) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs * 64);
  cfg.blockDim = dim3(kOpdThreads);
  cfg.dynamicSmemBytes = sizeof(OpdSmem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Both instances have the same shape and launch bounds; the statistics
  // instance stands for both.
  return cudaOccupancyMaxActiveClusters(out, opd_kernel<TIn, false>, &cfg);
}

// Verification fields of an OPD launch (spec_verify_opd); null tokens means
// statistics only (spec_opd_stats).
struct OpdVerify {
  const int32_t* tokens = nullptr;
  const float* uniforms = nullptr;
  const float* temperature = nullptr;
  int32_t* out_tokens = nullptr;
  int32_t* num_accepted = nullptr;
  unsigned char* ws = nullptr;
};

template <typename TIn>
spec_status_t opd_typed(const void* target, const void* draft, const int32_t* lengths, int B,
                        int k, int V, float delta, float alpha, int32_t* x_star, float* hard,
                        float* rkl, float* rkl_clip, float* loss, cudaStream_t stream,
                        int dtype_index, bool vec_ok, const OpdVerify& vf = OpdVerify()) {
  NvtxRange r(vf.tokens != nullptr ? "spec_verify_opd" : "spec_opd_stats");
  DeviceInfo* d = nullptr;
  if (device_info(&d) != cudaSuccess) return SPEC_ERR_CUDA;
  const int cs = opd_cluster_size(V);
  int* slot = &d->opd_clusters[dtype_index][cs - 1];
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!d->opd_ready) {
      if (opd_prepare<float>() != cudaSuccess || opd_prepare<uint16_t>() != cudaSuccess)
        return SPEC_ERR_CUDA;
      d->opd_ready = true;
    }
    if (*slot == 0) {
      int n = 0;
      if (opd_max_clusters<TIn>(cs, &n) != cudaSuccess || n < 1) return SPEC_ERR_CUDA;
      *slot = n;
    }
  }
  const bool verify = vf.tokens != nullptr;
  const long long clusters = std::min<long long>((long long)B * k, *slot);
  OpdParams op = {};
  op.target = target;
  op.draft = draft;
  op.lengths = lengths;
  op.B = B;
  op.k = k;
  op.V = V;
  op.slice = (((V + cs - 1) / cs) + 7) & ~7;
  op.vec_ok = vec_ok ? 1 : 0;
  op.delta = delta;
  op.x_star = x_star;
  op.hard = hard;
  op.rkl = rkl;
  op.rkl_clip = rkl_clip;
  int C = 0, ce = 0, nch = 0;
  WsLayout lay = {};
  if (verify) {
    // The plan kernel checks the inputs and resets the workspace state the
    // decisions and the final pass use (its row list is not needed here).
    C = chunks_per_row(2LL * B * k, V);
    ce = chunk_elems_for(V, C);
    nch = (V + ce - 1) / ce;
    lay = ws_layout(B, k, C, V);
    if (launch_plan(vf.tokens, lengths, vf.uniforms, vf.temperature, B, k, V, C, ce, nch, vf.ws,
                    lay, stream, true, nullptr, nullptr, 0, 0, /*skip_t01=*/true) != cudaSuccess)
      return SPEC_ERR_CUDA;
    op.verify = 1;
    op.tokens = vf.tokens;
    op.uniforms = vf.uniforms;
    op.temperature = vf.temperature;
    op.ws = vf.ws;
    op.lay = lay;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * cs));
  cfg.blockDim = dim3(kOpdThreads);
  cfg.dynamicSmemBytes = sizeof(OpdSmem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = verify ? 2 : 1;
  {
    NvtxRange ro("opd_kernel");
    if ((verify ? cudaLaunchKernelEx(&cfg, opd_kernel<TIn, true>, op)
                : cudaLaunchKernelEx(&cfg, opd_kernel<TIn, false>, op)) != cudaSuccess)
      return SPEC_ERR_CUDA;
  }
  if (verify) {
    // Requests at other temperatures: the row sweep, over the rows the plan
    // listed (none when every request is at T = 0 or 1).
    int sweep_grid = 0;
    if (launch_sweep<TIn>(d, target, draft, vf.tokens, vf.uniforms, B, k, V, nch, ce, vf.ws, lay,
                          true, dtype_index, stream, true, &sweep_grid, (long long)B * (k + 1),
                          (long long)B * k) != cudaSuccess)
      return SPEC_ERR_CUDA;
    if (launch_final<TIn>(d, target, draft, vf.tokens, lengths, vf.uniforms, vf.temperature, B, k,
                          V, vf.out_tokens, vf.num_accepted, vf.ws, lay,
                          (int)(clusters * cs) + sweep_grid, 0u, stream, true,
                          (long long)B * (k + 1), (long long)B * k) != cudaSuccess)
      return SPEC_ERR_CUDA;
  }
  const int wpb = 8;
  if (launch(opd_loss_kernel, dim3((B + wpb - 1) / wpb), dim3(wpb * 32), 0, stream, true, lengths,
             (const float*)hard, (const float*)rkl_clip, B, k, alpha, loss) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

}  // namespace specv

using namespace specv;

extern "C" {

int spec_abi_version(void) { return SPEC_VERIFY_ABI_VERSION; }

int spec_debug_build(void) {
#ifdef SPEC_DEBUG
  return 1;
#else
  return 0;
#endif
}

spec_status_t spec_debug_checks(int32_t* failures, int32_t* first_site, int reset, void* stream) {
  int32_t f = 0, site = 0;
#ifdef SPEC_DEBUG
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyFromSymbolAsync(&f, g_debug_failures, sizeof f, 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&site, g_debug_site, sizeof site, 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (reset) {
    const int32_t zero = 0;
    if (cudaMemcpyToSymbolAsync(g_debug_failures, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                                s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_debug_site, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return SPEC_ERR_CUDA;
  }
#else
  (void)reset;
  (void)stream;
#endif
  if (failures) *failures = f;
  if (first_site) *first_site = site;
  return SPEC_OK;
}

const char* spec_status_string(spec_status_t s) {
  switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument (size, null or misaligned pointer)";
    case SPEC_ERR_UNSUPPORTED: return "unsupported size";
    case SPEC_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
    case SPEC_ERR_BAD_INPUT: return "invalid value in device inputs (see num_accepted == -1)";
    case SPEC_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    case SPEC_ERR_INTERNAL: return "internal consistency check failed";
  }
  return "unknown status";
}

size_t spec_verify_workspace_bytes(int B, int k, int V) {
  if (!sizes_ok(B, k, V)) return 0;
  const long long slots = 2LL * B * k;
  return ws_layout(B, k, chunks_per_row(slots, V), V).total;
}

// Where the two logits buffers live.  Pinned host memory that the GPU maps
// (cudaHostAlloc, cudaHostRegister, torch's pin_memory) is read by the
// kernels themselves over the CPU-GPU link, with plain loads and no bulk
// copies ("direct"); *t and *d become the device-side addresses.  Anything
// else is taken as device memory, as before.  Returns false if one buffer is
// host memory and the other is not, or a host buffer is not mapped.
static bool resolve_logits(const void** t, const void** d, bool* direct) {
  auto host_of = [](const void* p, const void** dev) -> int {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
      (void)cudaGetLastError();
      return 0;
    }
    if (a.type != cudaMemoryTypeHost) return 0;
    if (a.devicePointer == nullptr) return -1;
    *dev = a.devicePointer;
    return 1;
  };
  const void* td = *t;
  const void* dd = *d;
  const int ht = host_of(*t, &td), hd = host_of(*d, &dd);
  if (ht < 0 || hd < 0 || ht != hd) return false;
  *direct = (ht == 1);
  *t = td;
  *d = dd;
  return true;
}

// Padded layout: t_start == nullptr.  Packed layout: t_start / d_start give
// each request's first row in buffers of rows_t / rows_d rows; a draft buffer
// of zero rows may be null (then only greedy requests are valid).
static spec_status_t verify_entry(const void* target_logits, const void* draft_logits,
                             spec_dtype_t dtype, const int32_t* draft_tokens,
                             const int32_t* lengths, const float* uniforms,
                             const float* temperature, int B, int k, int V, int32_t* out_tokens,
                             int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                             void* stream, unsigned flags, void* const* ev,
                             const int32_t* t_start = nullptr, const int32_t* d_start = nullptr,
                             long long rows_t = 0, long long rows_d = 0) {
  if (B < 1 || k < 1 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (!sizes_ok(B, k, V)) return SPEC_ERR_UNSUPPORTED;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if ((flags & ~(SPEC_FLAG_FULL_SWEEP | SPEC_FLAG_TEST_LATE_SLICES)) != 0)
    return SPEC_ERR_INVALID_ARG;
  const bool packed = (t_start != nullptr);
  if (packed) {
    if (!d_start || !aligned(t_start, 4) || !aligned(d_start, 4)) return SPEC_ERR_INVALID_ARG;
    if (rows_t < 1 || rows_t > INT32_MAX || rows_d < 0 || rows_d > INT32_MAX)
      return SPEC_ERR_INVALID_ARG;
    if (rows_d == 0 && !draft_logits) draft_logits = target_logits;  // never read
  }
  if (!target_logits || !draft_logits || !draft_tokens || !lengths || !uniforms || !temperature ||
      !out_tokens || !num_accepted)
    return SPEC_ERR_INVALID_ARG;
  const size_t esize = dtype == SPEC_F32 ? 4 : 2;
  if (!aligned(target_logits, esize) || !aligned(draft_logits, esize) || !aligned(draft_tokens, 4) ||
      !aligned(lengths, 4) || !aligned(uniforms, 4) || !aligned(temperature, 4) ||
      !aligned(out_tokens, 4) || !aligned(num_accepted, 4))
    return SPEC_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) ||
      workspace_bytes < spec_verify_workspace_bytes(B, k, V))
    return SPEC_ERR_WORKSPACE;
  DeviceOf on_device(workspace);
  if (!on_device.ok()) return SPEC_ERR_CUDA;
  bool direct = false;
  if (!resolve_logits(&target_logits, &draft_logits, &direct)) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SPEC_F32)
    return verify_typed<float>(target_logits, draft_logits, draft_tokens, lengths, uniforms,
                               temperature, B, k, V, out_tokens, num_accepted, workspace, s, flags, 0,
                               ev, t_start, d_start, rows_t, rows_d, direct);
  return verify_typed<uint16_t>(target_logits, draft_logits, draft_tokens, lengths, uniforms,
                                temperature, B, k, V, out_tokens, num_accepted, workspace, s, flags,
                                1, ev, t_start, d_start, rows_t, rows_d, direct);
}

spec_status_t spec_verify_packed(const void* target_rows, long long rows_t, const void* draft_rows,
                                 long long rows_d, spec_dtype_t dtype,
                                 const int32_t* target_row_start, const int32_t* draft_row_start,
                                 const int32_t* draft_tokens, const int32_t* lengths,
                                 const float* uniforms, const float* temperature, int B, int k,
                                 int V, int32_t* out_tokens, int32_t* num_accepted,
                                 void* workspace, size_t workspace_bytes, void* stream,
                                 unsigned flags) {
  if (!target_row_start || !draft_row_start) return SPEC_ERR_INVALID_ARG;
  return verify_entry(target_rows, draft_rows, dtype, draft_tokens, lengths, uniforms,
                      temperature, B, k, V, out_tokens, num_accepted, workspace, workspace_bytes,
                      stream, flags, nullptr, target_row_start, draft_row_start, rows_t, rows_d);
}

spec_status_t spec_verify_ex(const void* target_logits, const void* draft_logits,
                             spec_dtype_t dtype, const int32_t* draft_tokens,
                             const int32_t* lengths, const float* uniforms,
                             const float* temperature, int B, int k, int V, int32_t* out_tokens,
                             int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                             void* stream, unsigned flags) {
  return verify_entry(target_logits, draft_logits, dtype, draft_tokens, lengths, uniforms,
                      temperature, B, k, V, out_tokens, num_accepted, workspace, workspace_bytes,
                      stream, flags, nullptr);
}

spec_status_t spec_verify_timed(const void* target_logits, const void* draft_logits,
                                spec_dtype_t dtype, const int32_t* draft_tokens,
                                const int32_t* lengths, const float* uniforms,
                                const float* temperature, int B, int k, int V,
                                int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                                size_t workspace_bytes, void* stream, unsigned flags,
                                void* ev_plan, void* ev_sweep, void* ev_final, void* ev_end) {
  void* const ev[4] = {ev_plan, ev_sweep, ev_final, ev_end};
  return verify_entry(target_logits, draft_logits, dtype, draft_tokens, lengths, uniforms,
                      temperature, B, k, V, out_tokens, num_accepted, workspace, workspace_bytes,
                      stream, flags, ev);
}

spec_status_t spec_verify(const void* target_logits, const void* draft_logits, spec_dtype_t dtype,
                          const int32_t* draft_tokens, const int32_t* lengths,
                          const float* uniforms, const float* temperature, int B, int k, int V,
                          int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return spec_verify_ex(target_logits, draft_logits, dtype, draft_tokens, lengths, uniforms,
                        temperature, B, k, V, out_tokens, num_accepted, workspace, workspace_bytes,
                        stream, 0u);
}

spec_status_t spec_verify_report(const void* workspace, void* stream, spec_verify_report_t* report) {
  if (!workspace || !report) return SPEC_ERR_INVALID_ARG;
  WsHeader h;
  DeviceOf on_device(workspace);
  if (!on_device.ok()) return SPEC_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&h, workspace, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_CUDA;
  report->status = h.status;
  report->bad_requests = h.bad_requests;
  report->first_bad_request = h.first_bad == INT32_MAX ? -1 : h.first_bad;
  report->rows_planned = h.rows_planned;
  report->chunks_swept = (int64_t)h.chunks_swept;
  report->chunks_per_row = h.chunks_per_row;
  report->chunk_elems = h.chunk_elems;
  report->final_rows = (int64_t)h.final_rows;
  report->residual_zero = h.residual_zero;
  report->reserved = 0;
  report->sweep_bytes = (int64_t)h.sweep_bytes;
  report->final_bytes = (int64_t)h.final_bytes;
  return SPEC_OK;
}

spec_status_t spec_verify_device_status(const void* workspace, void* stream) {
  spec_verify_report_t r;
  spec_status_t st = spec_verify_report(workspace, stream, &r);
  if (st != SPEC_OK) return st;
  return (spec_status_t)r.status;
}

spec_status_t spec_opd_stats(const void* target_logits, const void* draft_logits,
                             spec_dtype_t dtype, const int32_t* lengths, int B, int k, int V,
                             float delta, float alpha, int32_t* x_star, float* hard, float* rkl,
                             float* rkl_clip, float* loss, void* stream) {
  if (B < 1 || k < 1 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (!sizes_ok(B, k, V)) return SPEC_ERR_UNSUPPORTED;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (!(delta > 0.0f && delta <= FLT_MAX) || !(alpha >= 0.0f && alpha <= 1.0f))
    return SPEC_ERR_INVALID_ARG;
  if (!target_logits || !draft_logits || !lengths || !x_star || !hard || !rkl || !rkl_clip ||
      !loss)
    return SPEC_ERR_INVALID_ARG;
  const size_t esize = dtype == SPEC_F32 ? 4 : 2;
  if (!aligned(target_logits, esize) || !aligned(draft_logits, esize) || !aligned(lengths, 4) ||
      !aligned(x_star, 4) || !aligned(hard, 4) || !aligned(rkl, 4) || !aligned(rkl_clip, 4) ||
      !aligned(loss, 4))
    return SPEC_ERR_INVALID_ARG;
  const bool vec_ok = aligned(target_logits, 16) && aligned(draft_logits, 16) &&
                      ((size_t)V * esize) % 16 == 0;
  // The statistics stream every row twice through bulk copies: device memory only.
  {
    bool direct = false;
    const void* t = target_logits;
    const void* d = draft_logits;
    if (!resolve_logits(&t, &d, &direct) || direct) return SPEC_ERR_INVALID_ARG;
  }
  DeviceOf on_device(target_logits);
  if (!on_device.ok()) return SPEC_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SPEC_F32)
    return opd_typed<float>(target_logits, draft_logits, lengths, B, k, V, delta, alpha, x_star,
                            hard, rkl, rkl_clip, loss, s, 0, vec_ok);
  return opd_typed<uint16_t>(target_logits, draft_logits, lengths, B, k, V, delta, alpha, x_star,
                             hard, rkl, rkl_clip, loss, s, 1, vec_ok);
}

spec_status_t spec_verify_opd(const void* target_logits, const void* draft_logits,
                              spec_dtype_t dtype, const int32_t* draft_tokens,
                              const int32_t* lengths, const float* uniforms,
                              const float* temperature, int B, int k, int V, float delta,
                              float alpha, int32_t* out_tokens, int32_t* num_accepted,
                              int32_t* x_star, float* hard, float* rkl, float* rkl_clip,
                              float* loss, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 1 || k < 1 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (!sizes_ok(B, k, V)) return SPEC_ERR_UNSUPPORTED;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (!(delta > 0.0f && delta <= FLT_MAX) || !(alpha >= 0.0f && alpha <= 1.0f))
    return SPEC_ERR_INVALID_ARG;
  if (!target_logits || !draft_logits || !draft_tokens || !lengths || !uniforms || !temperature ||
      !out_tokens || !num_accepted || !x_star || !hard || !rkl || !rkl_clip || !loss)
    return SPEC_ERR_INVALID_ARG;
  const size_t esize = dtype == SPEC_F32 ? 4 : 2;
  if (!aligned(target_logits, esize) || !aligned(draft_logits, esize) || !aligned(draft_tokens, 4) ||
      !aligned(lengths, 4) || !aligned(uniforms, 4) || !aligned(temperature, 4) ||
      !aligned(out_tokens, 4) || !aligned(num_accepted, 4) || !aligned(x_star, 4) ||
      !aligned(hard, 4) || !aligned(rkl, 4) || !aligned(rkl_clip, 4) || !aligned(loss, 4))
    return SPEC_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) ||
      workspace_bytes < spec_verify_workspace_bytes(B, k, V))
    return SPEC_ERR_WORKSPACE;
  const bool vec_ok = aligned(target_logits, 16) && aligned(draft_logits, 16) &&
                      ((size_t)V * esize) % 16 == 0;
  // The statistics stream every row twice through bulk copies: device memory only.
  {
    bool direct = false;
    const void* t = target_logits;
    const void* d = draft_logits;
    if (!resolve_logits(&t, &d, &direct) || direct) return SPEC_ERR_INVALID_ARG;
  }
  DeviceOf on_device(target_logits);
  if (!on_device.ok()) return SPEC_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  OpdVerify vf;
  vf.tokens = draft_tokens;
  vf.uniforms = uniforms;
  vf.temperature = temperature;
  vf.out_tokens = out_tokens;
  vf.num_accepted = num_accepted;
  vf.ws = static_cast<unsigned char*>(workspace);
  if (dtype == SPEC_F32)
    return opd_typed<float>(target_logits, draft_logits, lengths, B, k, V, delta, alpha, x_star,
                            hard, rkl, rkl_clip, loss, s, 0, vec_ok, vf);
  return opd_typed<uint16_t>(target_logits, draft_logits, lengths, B, k, V, delta, alpha, x_star,
                             hard, rkl, rkl_clip, loss, s, 1, vec_ok, vf);
}

spec_status_t spec_d3d_select(const int32_t* num_accepted, const int32_t* out_tokens,
                              const int32_t* branch_pos, const int32_t* branch_tok,
                              const int32_t* branch_block, int B, int k, int NB, int blk,
                              int32_t* hit, int32_t* next_block, int32_t* hits, void* stream) {
  if (B < 1 || k < 1 || NB < 1 || blk < 1) return SPEC_ERR_INVALID_ARG;
  if (B > SPEC_MAX_B || k > SPEC_MAX_K) return SPEC_ERR_UNSUPPORTED;
  if ((long long)B * NB * blk >= (1LL << 40)) return SPEC_ERR_UNSUPPORTED;
  if (!num_accepted || !out_tokens || !branch_pos || !branch_tok || !branch_block || !hit ||
      !next_block)
    return SPEC_ERR_INVALID_ARG;
  if (!aligned(num_accepted, 4) || !aligned(out_tokens, 4) || !aligned(branch_pos, 4) ||
      !aligned(branch_tok, 4) || !aligned(branch_block, 4) || !aligned(hit, 4) ||
      !aligned(next_block, 4) || (hits && !aligned(hits, 4)))
    return SPEC_ERR_INVALID_ARG;
  DeviceOf on_device(num_accepted);
  if (!on_device.ok()) return SPEC_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch(d3d_select_kernel, dim3((B + kD3dWarps - 1) / kD3dWarps), dim3(kD3dWarps * 32), 0, s,
             true, num_accepted, out_tokens, branch_pos, branch_tok, branch_block, B, k, NB, blk,
             hit, next_block) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (hits && launch(d3d_count_kernel, dim3(1), dim3(kD3dCountThreads), 0, s, true,
                     (const int32_t*)hit, B, hits) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

size_t spec_row_stats_workspace_bytes(int rows, int V) {
  if (rows < 1 || V < 1 || V > SPEC_MAX_V) return 0;
  if ((long long)rows * chunks_per_row(rows, V) >= (1LL << 31)) return 0;
  return row_stats_ws_bytes(rows, V);
}

spec_status_t spec_row_stats(const void* logits, spec_dtype_t dtype, int rows, int V,
                             const float* temperature, float* row_max, float* row_lse,
                             int32_t* row_arg, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (rows < 1 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (V > SPEC_MAX_V || spec_row_stats_workspace_bytes(rows, V) == 0) return SPEC_ERR_UNSUPPORTED;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (!logits || !temperature || !row_max || !row_lse || !row_arg) return SPEC_ERR_INVALID_ARG;
  const size_t esize = dtype == SPEC_F32 ? 4 : 2;
  if (!aligned(logits, esize) || !aligned(temperature, 4) || !aligned(row_max, 4) ||
      !aligned(row_lse, 4) || !aligned(row_arg, 4))
    return SPEC_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) ||
      workspace_bytes < spec_row_stats_workspace_bytes(rows, V))
    return SPEC_ERR_WORKSPACE;
  DeviceOf on_device(workspace);
  if (!on_device.ok()) return SPEC_ERR_CUDA;
  bool direct = false;
  const void* unused = logits;
  if (!resolve_logits(&logits, &unused, &direct)) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SPEC_F32)
    return row_stats_typed<float>(logits, rows, V, temperature, row_max, row_lse, row_arg, workspace,
                                  s, 0, direct);
  return row_stats_typed<uint16_t>(logits, rows, V, temperature, row_max, row_lse, row_arg,
                                   workspace, s, 1, direct);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// spec_verify_static: verification that uses the library's own fixed scratch
// instead of a caller-provided workspace, for callers that cannot allocate
// device memory.  Nothing here allocates.
// ---------------------------------------------------------------------------

namespace specv {
namespace {

// The scratch: one fixed array on every GPU that loads this library, held
// until the process exits.  All spec_verify_static calls on a GPU share it.
static __device__ __align__(256) unsigned char g_static_scratch[SPEC_STATIC_SCRATCH_BYTES];

void* g_static_ptr[kMaxDevices];
std::mutex g_static_mu;

// Device address of the current GPU's scratch array.  The array's name is
// only a host-side stand-in in host code, so the address is looked up once
// per device, with that device current, and cached.
cudaError_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace specv

extern "C" spec_status_t spec_verify_static(const void* target_logits, const void* draft_logits,
                                            spec_dtype_t dtype, const int32_t* draft_tokens,
                                            const int32_t* lengths, const float* uniforms,
                                            const float* temperature, int B, int k, int V,
                                            int32_t* out_tokens, int32_t* num_accepted,
                                            void* stream) {
  using namespace specv;
  if (B < 1 || k < 1 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (!sizes_ok(B, k, V)) return SPEC_ERR_UNSUPPORTED;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (!target_logits || !draft_logits || !draft_tokens || !lengths || !uniforms || !temperature ||
      !out_tokens || !num_accepted)
    return SPEC_ERR_INVALID_ARG;
  const size_t esize = dtype == SPEC_F32 ? 4 : 2;
  if (!aligned(target_logits, esize) || !aligned(draft_logits, esize) || !aligned(draft_tokens, 4) ||
      !aligned(lengths, 4) || !aligned(uniforms, 4) || !aligned(temperature, 4) ||
      !aligned(out_tokens, 4) || !aligned(num_accepted, 4))
    return SPEC_ERR_INVALID_ARG;
  // The batch must fit the fixed scratch.
  const size_t need = spec_verify_workspace_bytes(B, k, V);
  if (need == 0 || need > SPEC_STATIC_SCRATCH_BYTES) return SPEC_ERR_UNSUPPORTED;
  DeviceOf on_device(num_accepted);
  if (!on_device.ok()) return SPEC_ERR_CUDA;
  bool direct = false;
  if (!resolve_logits(&target_logits, &draft_logits, &direct)) return SPEC_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) return SPEC_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SPEC_F32)
    return verify_typed<float>(target_logits, draft_logits, draft_tokens, lengths, uniforms,
                               temperature, B, k, V, out_tokens, num_accepted, scratch, s, 0u, 0,
                               nullptr, nullptr, nullptr, 0, 0, direct);
  return verify_typed<uint16_t>(target_logits, draft_logits, draft_tokens, lengths, uniforms,
                                temperature, B, k, V, out_tokens, num_accepted, scratch, s, 0u, 1,
                                nullptr, nullptr, nullptr, 0, 0, direct);
}
