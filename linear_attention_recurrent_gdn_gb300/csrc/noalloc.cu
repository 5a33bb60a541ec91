// dl_step_noalloc: one DeltaLog decode step that allocates no device memory.
//
// Who needs this.  Some callers cannot let a library call cudaMalloc while
// they run.  Typical cases:
//   * a serving engine that reserves almost all of the GPU's memory for its own
//     pools (states, caches, activations) when it starts: an allocation made
//     later by a library can fail, or can take memory the engine has budgeted;
//   * code that runs under a custom allocator, which must own every device
//     buffer so that it can account for, reuse and free them itself;
//   * latency-sensitive loops, because cudaMalloc can synchronise the device.
// Such callers allocate everything themselves: the dense bases, the logs, the
// device slot table, the per-token inputs and outputs.  They pass all of it
// here.  The only other memory the step needs is the ReplayPrep coefficient
// scratch (and a status word).  This file keeps them in file-scope __device__
// arrays, which are part of the library image and are set up when the library
// is loaded on a device, so this entry point calls no allocator.
//
// Rules for users:
//   * The scratch holds at most DL_NOALLOC_SCRATCH_FLOATS floats.  A step needs
//     n * num_heads * CB floats, where CB is the coefficient block size for
//     (op, M, d_k).  Larger steps are refused with DL_EINVAL and a message
//     naming the limit.
//   * Every call shares the one scratch array; it keeps the last call's
//     contents.  Within a call, ReplayPrep writes every coefficient that
//     AppendDecode then uses, so nothing left from an earlier call is used;
//     the status word must start at zero and is cleared at the start of
//     each call.  Calls that overlap on the GPU (on
//     different streams, without ordering between them) race on the scratch;
//     order them on one stream.
//   * The first call on a device does a one-time set-up with that device
//     current: it resolves the device address of the scratch
//     (cudaGetSymbolAddress) and sets the kernels' shared-memory limits.  Make
//     this first call before any stream capture.
// The path is the same two kernels dl_step launches (ReplayPrep, then
// AppendDecode with the merge fused), with the same arguments except for the
// location of the scratch.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/deltalog.h"
#include "dl_device.cuh"
#include "launch.h"
#include "layout.h"

namespace {

constexpr int MAX_DEVICES = 64;

struct DeviceSetup {
  bool ready = false;
  float* coef = nullptr;       // device address of g_noalloc_coef
  int32_t* status = nullptr;   // device address of g_noalloc_status
  int num_sms = 0;
  int smem_optin = 0;
  int smem_per_sm = 0;
  int l2_bytes = 0;
  size_t smem_configured[3][2] = {{0, 0}, {0, 0}, {0, 0}};   // per (op, d_k 64/128)
};

DeviceSetup g_dev[MAX_DEVICES];
std::mutex g_setup_mutex;
thread_local dl::StepArgs t_args;   // launch arguments (12 KiB), reused: no per-call allocation

}  // namespace

static __device__ __align__(256) float g_noalloc_coef[DL_NOALLOC_SCRATCH_FLOATS];
static __device__ __align__(256) int32_t g_noalloc_status[4];

namespace {

struct ErrOut {
  char* buf;
  int32_t len;
  dl_status operator()(dl_status s, const char* fmt, ...) const {
    if (buf && len > 0) {
      va_list ap;
      va_start(ap, fmt);
      vsnprintf(buf, (size_t)len, fmt, ap);
      va_end(ap);
    }
    return s;
  }
};

}  // namespace

extern "C" dl_status dl_step_noalloc(const dl_config* cfg, const dl_state_view* st,
                                     const int32_t* plan, int32_t n, const void* q,
                                     const void* k, const void* v, const float* g,
                                     const float* beta, void* o, void* stream, char* errbuf,
                                     int32_t errlen) {
  const ErrOut fail{errbuf, errlen};
  if (errbuf && errlen > 0) errbuf[0] = 0;
  if (!cfg || !st || n < 0 || (n > 0 && !plan)) return fail(DL_EINVAL, "NULL argument");
  const dl_config f = *cfg;
  if (f.op < DL_GDN || f.op > DL_RWKV6 || f.num_heads < 1 || f.num_slots < 1 ||
      f.merge_interval < 1 || f.merge_interval > 32 || (f.d_k != 64 && f.d_k != 128) ||
      f.d_v != f.d_k || (f.out_bf16 != 0 && f.out_bf16 != 1))
    return fail(DL_EUNSUPPORTED, "configuration not supported");
  if (n == 0) return DL_OK;
  if (n > dl::MAX_ROWS) return fail(DL_EINVAL, "at most 1024 slots per call");
  if (!st->Sbar || !st->alog || !st->klog || !st->Llog || !st->n_log || !st->base_of ||
      !q || !k || !v || !g || !o || (f.op != DL_RWKV6 && !beta) || (f.op == DL_RWKV6 && !st->bonus))
    return fail(DL_EINVAL, "NULL tensor pointer");
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!a16(q) || !a16(k) || !a16(v) || !a16(st->Sbar) || !a16(st->alog) || !a16(st->klog) ||
      (f.op != DL_GDN && !a16(g)))
    return fail(DL_EINVAL, "q, k, v, the state and log arrays (and per-key g) need 16-byte alignment");
  const dl::Layout L = dl::make_layout(f.op, f.merge_interval, f.d_k, f.d_v);
  const size_t need = (size_t)n * f.num_heads * L.CB;
  if (need > (size_t)DL_NOALLOC_SCRATCH_FLOATS)
    return fail(DL_EINVAL,
                "step needs %zu scratch floats (n=%d x H=%d x %d), the static scratch holds %d "
                "(DL_NOALLOC_SCRATCH_FLOATS); split the slots over several calls",
                need, n, f.num_heads, L.CB, DL_NOALLOC_SCRATCH_FLOATS);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t* p = plan + 4 * (size_t)i;
    if (p[0] < 0 || p[0] >= f.num_slots || p[1] < 0 || p[1] >= f.num_slots || p[2] < 0 ||
        p[2] >= f.merge_interval)
      return fail(DL_EINVAL, "plan entry out of range");
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
    return fail(DL_ECUDA, "cudaGetDevice failed");
  DeviceSetup& d = g_dev[dev];
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!d.ready) {
      // one-time set-up on this device (it is current here)
      if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.coef), g_noalloc_coef) != cudaSuccess ||
          cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_noalloc_status) != cudaSuccess)
        return fail(DL_ECUDA, "cudaGetSymbolAddress of the static scratch failed");
      if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
              cudaSuccess ||
          cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
              cudaSuccess ||
          cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
        return fail(DL_ECUDA, "device query failed");
      d.ready = true;
    }
  }

  dl::StepArgs& a = t_args;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.g = g;
  a.beta = beta;
  a.o = o;
  a.Sbar = st->Sbar;
  a.alog = st->alog;
  a.klog = st->klog;
  a.Llog = st->Llog;
  a.coef = d.coef;
  a.bonus = st->bonus;
  a.nlog = st->n_log;
  a.base_of = st->base_of;
  a.status = d.status;
  a.rows = n;
  a.H = f.num_heads;
  a.M = f.merge_interval;
  a.Mcap = L.Mcap;
  a.Mcap4 = L.Mcap4;
  a.CB = L.CB;
  a.P0 = L.P0;
  a.out_bf16 = f.out_bf16;
  a.scale = f.scale;
  a.aux_bytes = L.aux_bytes;
  for (int32_t i = 0; i < n; ++i)
    a.items[i] = dl::StepItem{plan[4 * (size_t)i], plan[4 * (size_t)i + 1], plan[4 * (size_t)i + 2]};
  const int nvt = f.d_v / dl::BV;
  const long n_sh = (long)n * f.num_heads;
  if (n_sh >= 2L * d.num_sms) {
    a.G = nvt;
    a.NG = 1;
  } else {
    a.G = 1;
    a.NG = nvt;
  }
  const dl::PipePlan sh = dl::plan_pipeline(f.d_k, L.aux_bytes, a.G, d.smem_optin, d.smem_per_sm);
  if (sh.ns == 0) return fail(DL_EUNSUPPORTED, "pipeline does not fit in shared memory");
  a.ns = sh.ns;
  a.na = sh.na;
  a.ncw = sh.ncw;
  a.npw = sh.npw;
  a.tps = dl::tiles_per_stage(f.d_k, a.G);
  a.l2_stream = (double)n * f.num_heads * f.d_v * f.d_k * 4 > 0.75 * d.l2_bytes ? 1 : 0;
  a.pdl_prefetch = 0;
  a.plan_dev = nullptr;
  a.rows_dev = nullptr;
  const long units = n_sh * a.NG;
  const long slots_gpu = (long)sh.cps * d.num_sms;
  const int grid = (int)(units < slots_gpu ? units : slots_gpu);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  const int di = f.d_k == 64 ? 0 : 1;
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (d.smem_configured[f.op][di] < (size_t)sh.smem) {
      e = dl::configure_append_decode(f.op, f.d_k, sh.smem);
      if (e == cudaSuccess) d.smem_configured[f.op][di] = sh.smem;
    }
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(d.status, 0, sizeof(int32_t), s);   // starts at zero
  if (e == cudaSuccess) e = dl::launch_replay_prep(f.op, f.d_k, a, s);
  if (e == cudaSuccess) e = dl::launch_append_decode(f.op, f.d_k, a, grid, sh.smem, true, s);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();   // reported here, not left to the caller's next CUDA call
    return fail(DL_ECUDA, "launch failed: %s", cudaGetErrorString(e));
  }
  return DL_OK;
}
