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
//     AppendDecode then uses, so nothing left from an earlier call is used.
//     Calls that overlap on the GPU (on different streams, without ordering
//     between them) race on the scratch; order them on one stream.
//   * The status word starts at zero (static initialisation).  A kernel whose
//     bounded wait gives up records a code in it; the code stays until
//     dl_noalloc_sync reads it, reports DL_EDEVICE and clears it.  Outputs and
//     state of the calls since the last dl_noalloc_sync are then not to be
//     trusted.
//   * The first call on a device does a one-time set-up with that device
//     current: it resolves the device addresses of the scratch and the status
//     word (cudaGetSymbolAddress), reads the device's limits and the kernels'
//     register counts, and sets the kernels' shared-memory limits.  Make this
//     first call before any stream capture.
// The path is the two kernels dl_step launches in its two-kernel form
// (ReplayPrep, then AppendDecode with the merge fused), planned the same way,
// with the same arguments except for the location of the scratch.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
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
  int regs[3][2] = {{0, 0}, {0, 0}, {0, 0}};   // AppendDecode registers per (op, d_k 64/128)
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
  // The same rules as dl_step, plus the caller-owned state: what bulk copies
  // and 16-byte vector loads move needs 16-byte alignment, what is accessed
  // per element its element size.
  auto al = [](const void* p, uintptr_t b) { return (reinterpret_cast<uintptr_t>(p) & (b - 1)) == 0; };
  const bool perkey = f.op != DL_GDN;
  if (!al(q, 16) || !al(k, 16) || !al(v, 16) || !al(g, perkey ? 16 : 4) ||
      (beta && !al(beta, 4)) || !al(o, f.out_bf16 ? 2 : 4))
    return fail(DL_EINVAL, "misaligned tensor: q, k, v%s need 16-byte alignment, beta%s and o "
                "their element size", perkey ? ", g" : "", perkey ? "" : ", g");
  if (!al(st->Sbar, 16) || !al(st->alog, 16) || !al(st->klog, 16) ||
      !al(st->Llog, perkey ? 16 : 4) || !al(st->n_log, 4) || !al(st->base_of, 4) ||
      (st->bonus && !al(st->bonus, 16)))
    return fail(DL_EINVAL, "misaligned state: Sbar, alog, klog%s and bonus need 16-byte "
                "alignment, the slot table 4 bytes", perkey ? ", Llog" : "");
  const dl::Layout L = dl::make_layout(f.op, f.merge_interval, f.d_k, f.d_v);
  const size_t need = (size_t)n * f.num_heads * L.CB;
  if (need > (size_t)DL_NOALLOC_SCRATCH_FLOATS)
    return fail(DL_EINVAL,
                "step needs %zu scratch floats (n=%d x H=%d x %d), the static scratch holds %d "
                "(DL_NOALLOC_SCRATCH_FLOATS); split the slots over several calls",
                need, n, f.num_heads, L.CB, DL_NOALLOC_SCRATCH_FLOATS);
  // The plan must be what dl_table_step returned.  Check what the kernels rely
  // on: ids and log lengths in range, the merge flag consistent with the log
  // length, no slot twice (two units would update one base and log at once),
  // and no row reading the base of a slot that merges in this call (the merge
  // rewrites that base while the row reads it; dl_table_step never plans
  // either, because a fork source is frozen until its branches have merged).
  int32_t merging[dl::MAX_ROWS], sorted[dl::MAX_ROWS];
  int32_t nm = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t* p = plan + 4 * (size_t)i;
    if (p[0] < 0 || p[0] >= f.num_slots || p[1] < 0 || p[1] >= f.num_slots || p[2] < 0 ||
        p[2] >= f.merge_interval || p[3] != (p[2] + 1 == f.merge_interval ? 1 : 0))
      return fail(DL_EINVAL, "plan row %d out of range or inconsistent", i);
    sorted[i] = p[0];
    if (p[3]) merging[nm++] = p[0];
  }
  std::sort(sorted, sorted + n);
  for (int32_t i = 1; i < n; ++i)
    if (sorted[i] == sorted[i - 1]) return fail(DL_EINVAL, "slot %d appears twice in the plan", sorted[i]);
  std::sort(merging, merging + nm);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t* p = plan + 4 * (size_t)i;
    if (p[1] != p[0] && std::binary_search(merging, merging + nm, p[1]))
      return fail(DL_EINVAL, "slot %d reads the base of slot %d, which merges in the same call",
                  p[0], p[1]);
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
      for (int op = 0; op < 3; ++op)
        for (int di = 0; di < 2; ++di) d.regs[op][di] = dl::append_decode_regs(op, di ? 128 : 64, false, 1);
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
  a.arows = 0;   // aux slots sized for M log rows
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
  // as dl_step plans its two-kernel form: no tuning override, no prep warps,
  // the kernel's register count for residency
  const int di = f.d_k == 64 ? 0 : 1;
  const dl::PipePlan sh = dl::plan_pipeline(f.d_k, L.aux_bytes, a.G, d.smem_optin, d.smem_per_sm,
                                            nullptr, -1, d.regs[f.op][di], false);
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
  a.wait_ns = dl::WAIT_LIMIT_NS;
  a.test_stall = 0;
  // Test only: a shorter wait limit and the stall that makes one wait run out
  // (see dl_noalloc_sync); read on every call, unset in normal use.
  if (const char* e = getenv("DL_TEST_WAIT_MS")) {
    const long ms = atol(e);
    if (ms > 0 && ms < 2000) a.wait_ns = (unsigned long long)ms * 1000000ull;
  }
  if (const char* e = getenv("DL_TEST_STALL")) a.test_stall = atoi(e) == 1 ? 1 : 0;
  const long units = n_sh * a.NG;
  const long slots_gpu = (long)sh.cps * d.num_sms;
  const int grid = (int)(units < slots_gpu ? units : slots_gpu);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (d.smem_configured[f.op][di] < (size_t)sh.smem) {
      e = dl::configure_append_decode(f.op, f.d_k, sh.smem);
      if (e == cudaSuccess) d.smem_configured[f.op][di] = sh.smem;
    }
  }
  if (e == cudaSuccess) e = dl::launch_replay_prep(f.op, f.d_k, a, s);
  if (e == cudaSuccess) e = dl::launch_append_decode(f.op, f.d_k, a, grid, sh.smem, true, s);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();   // reported here, not left to the caller's next CUDA call
    return fail(DL_ECUDA, "launch failed: %s", cudaGetErrorString(e));
  }
  return DL_OK;
}

extern "C" dl_status dl_noalloc_sync(void* stream, int32_t* device_code, char* errbuf,
                                     int32_t errlen) {
  const ErrOut fail{errbuf, errlen};
  if (errbuf && errlen > 0) errbuf[0] = 0;
  if (device_code) *device_code = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(DL_ECUDA, "stream synchronisation failed: %s", cudaGetErrorString(e));
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
    return fail(DL_ECUDA, "cudaGetDevice failed");
  int32_t* status = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_dev[dev].ready) return DL_OK;   // no step ran on this device
    status = g_dev[dev].status;
  }
  int32_t code = 0;
  e = cudaMemcpy(&code, status, sizeof code, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(DL_ECUDA, "status read failed: %s", cudaGetErrorString(e));
  }
  if (code == 0) return DL_OK;
  if (device_code) *device_code = code;
  e = cudaMemset(status, 0, sizeof code);   // reported once; the next calls start clean
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(DL_ECUDA, "status reset failed: %s", cudaGetErrorString(e));
  }
  return fail(DL_EDEVICE, "kernel reported device status %d (%s)", code,
              dl::device_status_str(code));
}
