// C ABI of libdeltalog (declared and documented in include/deltalog.h).
//
// The context owns the dense bases S̄, the bounded logs, the device copy of the
// slot table, the ReplayPrep coefficient scratch and a device status word.  The
// host slot table (slot_table.cpp) validates every call and yields the per-row
// step plan (slot, base read, log length) that is passed to the kernels as a
// launch parameter, so that no host-device synchronisation is needed per step.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <new>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/deltalog.h"
#include "dl_device.cuh"
#include "launch.h"
#include "layout.h"

extern "C" dl_status dl_table_set_n(dl_table* t, const int32_t* slots, int32_t n,
                                   const int32_t* len);

namespace {

constexpr int NKIND = 4;   // timing kinds: ReplayPrep, AppendDecode, EagerStep, Merge/ReadState

struct TimedPair {
  cudaEvent_t a, b;
};

}  // namespace

// Staging sets of dl_decode_host.  A set is reused only after the download of
// the group before it, so with two sets the upload of group j + 2 waited on the
// download of group j and the chain download -> upload -> compute set the pace
// whenever the two copies together took longer than a group's compute.
// Measured on GB300 (GDN, 256 slots x 32 heads, one token a group, copies at
// 81 GB/s up and 27 GB/s down): two sets gave 59.1 M tokens·heads/s end to end,
// four give 83.7 M, against 87.1 M on the device.
constexpr int PIPE_SETS = 4;

struct dl_ctx {
  dl_config cfg{};
  cudaStream_t stream = nullptr;
  int device = 0, num_sms = 0, smem_optin = 0, smem_per_sm = 0, l2_bytes = 0;
  int regs[3] = {0, 0, 0};   // registers per thread: AppendDecode, fused AppendDecode, EagerStep
  // Set while a decode window is captured, from its second step on: the step
  // launches as a programmatic dependent of the previous step (both ours) and
  // may stream dense-base tiles of rows with a non-empty log before it waits.
  int pdl_chain = 0;
  // Set while a ragged window is captured: the step reads its rows and their
  // count from these device buffers (see dl_window_create_ragged).
  const dl::StepItem* dev_plan = nullptr;
  const int32_t* dev_rows = nullptr;
  dl_table* table = nullptr;
  dl::Layout L{};
  float* Sbar = nullptr;
  void* alog = nullptr;
  uint16_t* klog = nullptr;
  float* Llog = nullptr;
  int32_t* nlog = nullptr;
  int32_t* base_of = nullptr;
  float* coef = nullptr;
  float* bonus = nullptr;
  int32_t* status = nullptr;
  int32_t coef_rows = 0;
  void* stage = nullptr;        // device staging for dl_step_host
  size_t stage_bytes = 0;
  // dl_decode_host: PIPE_SETS device staging sets (token group j uses set
  // j % PIPE_SETS), an upload and a download stream, and the events that
  // order them
  void* pipe_stage = nullptr;
  size_t pipe_set_bytes = 0;
  int pipe_group = 1;          // tokens per staging set
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t ev_in[PIPE_SETS] = {}, ev_done[PIPE_SETS] = {}, ev_out[PIPE_SETS] = {};
  // dl_decode_host over whole decode windows: PIPE_SETS staging sets of M
  // tokens for the batch `wslots`, each with a decode window (CUDA graph)
  // captured on its buffers
  void* wstage = nullptr;
  size_t wset_bytes = 0;
  std::vector<int32_t> wslots;
  dl_window* wwin[PIPE_SETS] = {};
  std::vector<int32_t> plan;
  std::unique_ptr<dl::StepArgs> step_args;
  std::unique_ptr<dl::SlotListArgs> list_args;
  std::unique_ptr<dl::CkptArgs> ckpt_args;
  std::string err = "no error";
  dl_status sticky = DL_OK;
  // Bounded waits give up after wait_ns.  Tests may shorten it
  // (DL_TEST_WAIT_MS at dl_create) and set test_stall (DL_TEST_STALL=1), which
  // makes one consumer warp of each launch wait on a barrier nothing arrives
  // on, so that the device-side error path runs without any fault.
  unsigned long long wait_ns = dl::WAIT_LIMIT_NS;
  int test_stall = 0;
  bool timing = false;
  std::vector<TimedPair> timed[NKIND];
  double timed_ms[NKIND] = {0, 0, 0, 0};
  int64_t timed_n[NKIND] = {0, 0, 0, 0};
};

namespace {

dl_status set_err(dl_ctx* c, dl_status s, const char* fmt, ...) {
  if (c) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    c->err = buf;
    if (s == DL_ECUDA || s == DL_EDEVICE) c->sticky = s;
  }
  return s;
}

dl_status cuda_err(dl_ctx* c, cudaError_t e, const char* what) {
  (void)cudaGetLastError();   // the error is reported here; do not leave it to the caller's next call
  return set_err(c, DL_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define DL_CUDA(call, what)                   \
  do {                                        \
    cudaError_t e_ = (call);                  \
    if (e_ != cudaSuccess) return cuda_err(c, e_, what); \
  } while (0)

// Allocation with an optional countdown failure for tests (DL_TEST_FAIL_ALLOC=k
// makes the k-th device allocation of dl_create fail).
int g_fail_countdown = -1;

cudaError_t dev_alloc(void** p, size_t bytes) {
  if (g_fail_countdown > 0 && --g_fail_countdown == 0) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc(p, bytes < 16 ? 16 : bytes);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void free_windows(dl_ctx* c) {
  for (int b = 0; b < PIPE_SETS; ++b) {
    if (c->wwin[b]) dl_window_destroy(c->wwin[b]);
    c->wwin[b] = nullptr;
  }
  if (c->wstage) cudaFree(c->wstage);
  c->wstage = nullptr;
  c->wset_bytes = 0;
  c->wslots.clear();
}

void free_all(dl_ctx* c) {
  free_windows(c);
  void* ptrs[] = {c->Sbar, c->alog, c->klog, c->Llog, c->nlog, c->base_of,
                  c->coef, c->bonus, c->status, c->stage, c->pipe_stage};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  c->pipe_stage = nullptr;
  for (cudaEvent_t* ev : {c->ev_in, c->ev_done, c->ev_out})
    for (int b = 0; b < PIPE_SETS; ++b)
      if (ev[b]) {
        cudaEventDestroy(ev[b]);
        ev[b] = nullptr;
      }
  if (c->up) cudaStreamDestroy(c->up);
  if (c->down) cudaStreamDestroy(c->down);
  c->up = c->down = nullptr;
  c->Sbar = nullptr;
  c->alog = nullptr;
  c->klog = nullptr;
  c->Llog = nullptr;
  c->nlog = nullptr;
  c->base_of = nullptr;
  c->coef = nullptr;
  c->bonus = nullptr;
  c->status = nullptr;
  c->stage = nullptr;
  for (auto& v : c->timed)
    for (auto& p : v) {
      cudaEventDestroy(p.a);
      cudaEventDestroy(p.b);
    }
  if (c->table) dl_table_destroy(c->table);
  c->table = nullptr;
}

// DL_PIPE_SHAPE="cps,ncw,R" overrides the shape choice (a tuning knob for
// measurements; shapes that do not fit are ignored).
// Tuning override of the pipeline shape: DL_PIPE_SHAPE="cps,ncw,R[,npw[,max_na]]".
const int* shape_override() {
  static thread_local int v[5];
  const char* e = getenv("DL_PIPE_SHAPE");
  v[3] = -1;
  v[4] = 0;
  if (!e || sscanf(e, "%d,%d,%d,%d,%d", &v[0], &v[1], &v[2], &v[3], &v[4]) < 3) return nullptr;
  return v;
}

// Prep warps of the fused form.  A unit that is a single stage is handled by
// one consumer warp, which computes the unit's coefficients itself (0 prep
// warps: no hand-off between warps).  Units spread over several consumer
// warps share one prep warp's work.  GDN's scalar decays need one.  The
// per-key ops' coefficients (an exponential per key channel and log entry)
// need two to keep pace with the value-tile consumers once the log holds more
// than 16 entries; up to 16 one is as fast (measured on GB300 for KDA: M=32
// 38.0 against 31.0 M tokens·heads/s with one; M=16 78.4 against 77.9).
int prep_warps(int op, int dk, int G, int M) {
  if (G / dl::tiles_per_stage(dk, G) == 1) return 0;
  if (op == DL_GDN) return 1;
  return M <= 16 ? 1 : 2;
}

enum class Kern { Append, Fused, Eager };

// `L`: the launch's layout (its aux slots' size); `merge_launch`: every row of
// the launch merges (rows known on the host).
dl::PipePlan pipe_shape(const dl_ctx* c, const dl::Layout& L, int G, Kern k,
                        bool merge_launch = false) {
  const int aux = k == Kern::Append ? L.aux_bytes : k == Kern::Fused ? L.f_bytes : L.e_bytes;
  return dl::plan_pipeline(c->cfg.d_k, aux, G, c->smem_optin, c->smem_per_sm, shape_override(),
                           k == Kern::Fused ? prep_warps(c->cfg.op, c->cfg.d_k, G, c->cfg.merge_interval) : -1,
                           c->regs[(int)k], merge_launch && k == Kern::Fused);
}

bool record(dl_ctx* c, int kind, cudaEvent_t* ev) {
  if (!c->timing) return false;
  cudaEventCreate(ev);
  cudaEventRecord(*ev, c->stream);
  (void)kind;
  return true;
}

void record_end(dl_ctx* c, int kind, cudaEvent_t start) {
  cudaEvent_t stop;
  cudaEventCreate(&stop);
  cudaEventRecord(stop, c->stream);
  c->timed[kind].push_back(TimedPair{start, stop});
}

dl_status check_ctx(dl_ctx* c) {
  if (!c) return DL_EINVAL;
  if (c->sticky != DL_OK) return c->sticky;
  return DL_OK;
}

dl_status check_step_ptrs(dl_ctx* c, int32_t n, const void* q, const void* k, const void* v,
                          const float* g, const float* beta, const void* o) {
  if (n == 0) return DL_OK;
  if (!q || !k || !v || !g || !o || (c->cfg.op != DL_RWKV6 && !beta))
    return set_err(c, DL_EINVAL, "NULL tensor pointer");
  // q, k, v (and the per-key g rows) are moved by bulk copies / vector loads:
  // 16-byte alignment; the per-head g (GDN), beta and o are accessed per element.
  const bool perkey = c->cfg.op != DL_GDN;
  const uintptr_t osz = c->cfg.out_bf16 ? 2 : 4;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) ||
      (perkey ? !aligned16(g) : (reinterpret_cast<uintptr_t>(g) & 3u) != 0) ||
      (beta && (reinterpret_cast<uintptr_t>(beta) & 3u) != 0) ||
      (reinterpret_cast<uintptr_t>(o) & (osz - 1)) != 0)
    return set_err(c, DL_EINVAL, "misaligned tensor: q, k, v%s need 16-byte alignment, "
                   "other tensors their element size", perkey ? ", g" : "");
  if (c->cfg.op == DL_RWKV6 && !c->bonus)
    return set_err(c, DL_EINVAL, "RWKV6 needs dl_set_bonus before stepping");
  return DL_OK;
}

void fill_step_args(dl_ctx* c, dl::StepArgs& a, int32_t row0, int32_t rows, const void* q,
                    const void* k, const void* v, const float* g, const float* beta, void* o) {
  const dl_config& f = c->cfg;
  const size_t H = f.num_heads;
  const size_t gw = (f.op == DL_GDN) ? 1 : f.d_k;
  a.q = static_cast<const uint16_t*>(q) + (size_t)row0 * H * f.d_k;
  a.k = static_cast<const uint16_t*>(k) + (size_t)row0 * H * f.d_k;
  a.v = static_cast<const uint16_t*>(v) + (size_t)row0 * H * f.d_v;
  a.g = g + (size_t)row0 * H * gw;
  a.beta = beta ? beta + (size_t)row0 * H : nullptr;
  const size_t osz = f.out_bf16 ? 2 : 4;
  a.o = static_cast<unsigned char*>(o) + (size_t)row0 * H * f.d_v * osz;
  a.Sbar = c->Sbar;
  a.alog = c->alog;
  a.klog = c->klog;
  a.Llog = c->Llog;
  a.coef = c->coef;
  a.bonus = c->bonus;
  a.nlog = c->nlog;
  a.base_of = c->base_of;
  a.status = c->status;
  a.rows = rows;
  a.H = f.num_heads;
  a.M = f.merge_interval;
  a.Mcap = c->L.Mcap;
  a.Mcap4 = c->L.Mcap4;
  a.CB = c->L.CB;
  a.P0 = c->L.P0;
  a.out_bf16 = f.out_bf16;
  a.scale = f.scale;
  a.aux_bytes = c->L.aux_bytes;
  a.wait_ns = c->wait_ns;
  a.test_stall = c->test_stall;
  a.plan_dev = c->dev_plan ? c->dev_plan + row0 : nullptr;   // ragged windows only
  a.rows_dev = c->dev_rows;
  for (int32_t i = 0; i < rows; ++i) {
    const int32_t* p = &c->plan[4 * (size_t)(row0 + i)];
    a.items[i].slot = p[0];
    a.items[i].base = p[1];
    a.items[i].n = p[2];
  }
}

// Choose G (value tiles per work unit) for `rows` slot rows.
void unit_shape(const dl_ctx* c, dl::StepArgs& a) {
  const int nvt = c->cfg.d_v / dl::BV;
  const long n_sh = (long)a.rows * a.H;
  if (n_sh >= 2L * c->num_sms) {
    a.G = nvt;
    a.NG = 1;
  } else {
    a.G = 1;
    a.NG = nvt;
  }
}

dl_status run_step(dl_ctx* c, const int32_t* slots, int32_t n, const void* q, const void* k,
                   const void* v, const float* g, const float* beta, void* o, bool eager_call) {
  (void)slots;
  const dl_config& f = c->cfg;
  dl::StepArgs& a = *c->step_args;
  for (int32_t row0 = 0; row0 < n; row0 += dl::MAX_ROWS) {
    const int32_t rows = (n - row0) < dl::MAX_ROWS ? (n - row0) : dl::MAX_ROWS;
    fill_step_args(c, a, row0, rows, q, k, v, g, beta, o);
    unit_shape(c, a);
    // M = 1: every step is a merge of an empty log, which is the eager update.
    // When every row reads its own base (rows known on the host), the dedicated
    // EagerStep kernel runs it: measured on GB300 it streams the state faster
    // than the fused kernel's merge path (GDN 47.7 against 41.2, KDA 45.6
    // against 34.4, RWKV6 159.9 against 67.5 M tokens·heads/s).  A branch that
    // still reads a fork source's base takes the fused path, which writes its
    // private base.
    bool eager = eager_call;
    if (!eager && f.merge_interval == 1 && a.plan_dev == nullptr) {
      bool own = true;
      for (int32_t i = 0; i < rows && own; ++i) own = a.items[i].base == a.items[i].slot;
      if (own) eager = true;
    }
    const bool fused = !eager && f.staging == DL_STAGE_FUSED;
    // a launch where every row merges a window of M >= 8 gets the merge shape
    // (shorter rank-M updates are cheap enough that the append shape wins)
    bool all_merge = fused && a.plan_dev == nullptr && f.merge_interval >= 8;
    for (int32_t i = 0; i < rows && all_merge; ++i)
      all_merge = a.items[i].n + 1 == f.merge_interval;
    // Aux slots hold the launch's longest log when every row's log length is
    // known on the host, plus the current token's row where a step uses it:
    // RWKV6's v_t, and a merge step's u_t and k_t (delta-rule appends write
    // u_t straight to the log in HBM).  A ragged window's rows are only known
    // on the device, so its slots hold M rows.
    a.arows = 0;
    if (a.plan_dev == nullptr) {
      int32_t nmax = 0;
      bool any_merge = false;
      for (int32_t i = 0; i < rows; ++i) {
        nmax = a.items[i].n > nmax ? a.items[i].n : nmax;
        any_merge = any_merge || a.items[i].n + 1 == f.merge_interval;
      }
      const bool row_n = f.op == DL_RWKV6 || any_merge;
      a.arows = row_n ? nmax + 1 : (nmax > 0 ? nmax : 1);
    }
    const dl::Layout Ll = dl::make_layout(f.op, f.merge_interval, f.d_k, f.d_v, a.arows);
    a.aux_bytes = Ll.aux_bytes;
    const dl::PipePlan ps = pipe_shape(c, Ll, a.G, eager ? Kern::Eager : fused ? Kern::Fused : Kern::Append,
                                       all_merge);
    if (ps.ns == 0) return set_err(c, DL_EUNSUPPORTED, "pipeline does not fit in shared memory");
    a.ns = ps.ns;
    a.na = ps.na;
    a.ncw = ps.ncw;
    a.npw = ps.npw;
    a.tps = dl::tiles_per_stage(f.d_k, a.G);
    // stream the state through L2 unless the whole batch's state fits in 3/4 of it
    a.l2_stream = (double)n * f.num_heads * f.d_v * f.d_k * 4 > 0.75 * c->l2_bytes ? 1 : 0;
    const long units = (long)a.rows * a.H * a.NG;
    const long slots_gpu = (long)ps.cps * c->num_sms;
    const int grid = (int)(units < slots_gpu ? units : slots_gpu);
    cudaEvent_t e0;
    if (eager) {
      const bool t = record(c, 2, &e0);
      DL_CUDA(dl::launch_eager_step(f.op, f.d_k, a, grid, ps.smem, c->stream), "EagerStep launch");
      if (t) record_end(c, 2, e0);
    } else if (fused) {
      const bool t = record(c, 1, &e0);
      a.pdl_prefetch = c->pdl_chain;
      DL_CUDA(dl::launch_append_decode_fused(f.op, f.d_k, a, grid, ps.smem, c->pdl_chain != 0,
                                             c->stream),
              "AppendDecode launch");
      if (t) record_end(c, 1, e0);
    } else {
      bool t = record(c, 0, &e0);
      DL_CUDA(dl::launch_replay_prep(f.op, f.d_k, a, c->stream), "ReplayPrep launch");
      if (t) record_end(c, 0, e0);
      t = record(c, 1, &e0);
      DL_CUDA(dl::launch_append_decode(f.op, f.d_k, a, grid, ps.smem, !c->timing, c->stream),
              "AppendDecode launch");
      if (t) record_end(c, 1, e0);
    }
  }
  return DL_OK;
}

}  // namespace

extern "C" {

int32_t dl_abi_version(void) { return DL_ABI_VERSION; }

const char* dl_status_str(dl_status s) {
  switch (s) {
    case DL_OK: return "DL_OK";
    case DL_EINVAL: return "DL_EINVAL";
    case DL_ENOMEM: return "DL_ENOMEM";
    case DL_ECUDA: return "DL_ECUDA";
    case DL_EBUSY: return "DL_EBUSY";
    case DL_EDEVICE: return "DL_EDEVICE";
    case DL_EUNSUPPORTED: return "DL_EUNSUPPORTED";
  }
  return "DL_?";
}

const char* dl_last_error(const dl_ctx* c) { return c ? c->err.c_str() : "NULL context"; }

dl_status dl_create(const dl_config* cfg, void* stream, dl_ctx** out) {
  if (!out) return DL_EINVAL;
  *out = nullptr;
  if (!cfg) return DL_EINVAL;
  const dl_config f = *cfg;
  if (f.op < DL_GDN || f.op > DL_RWKV6 || f.num_slots < 1 || f.num_heads < 1 ||
      f.merge_interval < 1 || (f.out_bf16 != 0 && f.out_bf16 != 1) ||
      (f.staging != DL_STAGE_FUSED && f.staging != DL_STAGE_KERNELS))
    return DL_EINVAL;
  if (f.merge_interval > 32) return DL_EUNSUPPORTED;
  if ((f.d_k != 64 && f.d_k != 128) || f.d_v != f.d_k) return DL_EUNSUPPORTED;

  dl_ctx* c = new (std::nothrow) dl_ctx;
  if (!c) return DL_ENOMEM;
  c->cfg = f;
  c->stream = static_cast<cudaStream_t>(stream);
  c->L = dl::make_layout(f.op, f.merge_interval, f.d_k, f.d_v);
  c->plan.resize(4 * (size_t)f.num_slots);
  c->step_args.reset(new (std::nothrow) dl::StepArgs());
  c->list_args.reset(new (std::nothrow) dl::SlotListArgs());
  c->ckpt_args.reset(new (std::nothrow) dl::CkptArgs());
  if (const char* s = getenv("DL_TEST_FAIL_ALLOC")) g_fail_countdown = atoi(s);
  if (const char* s = getenv("DL_TEST_WAIT_MS")) {
    const long ms = atol(s);
    if (ms > 0 && ms < 2000) c->wait_ns = (unsigned long long)ms * 1000000ull;
  }
  if (const char* s = getenv("DL_TEST_STALL")) c->test_stall = atoi(s) == 1 ? 1 : 0;
  dl_status rc = DL_OK;
  do {
    if (!c->step_args || !c->list_args || !c->ckpt_args) { rc = DL_ENOMEM; break; }
    if (dl_table_create(f.num_slots, f.merge_interval, &c->table) != DL_OK) { rc = DL_ENOMEM; break; }
    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&c->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&c->smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, c->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->l2_bytes, cudaDevAttrL2CacheSize, c->device);
    if (e != cudaSuccess) { rc = cuda_err(c, e, "device query"); break; }
    const size_t S = f.num_slots, H = f.num_heads, dk = f.d_k, dv = f.d_v, Mcap = c->L.Mcap;
    const size_t esa = (f.op == DL_RWKV6) ? 2 : 4;
    const size_t lw = (f.op == DL_GDN) ? 1 : dk;
    c->coef_rows = f.num_slots < dl::MAX_ROWS ? f.num_slots : dl::MAX_ROWS;
    struct { void** p; size_t bytes; } al[] = {
        {reinterpret_cast<void**>(&c->Sbar), S * H * dv * dk * 4},
        {&c->alog, S * H * Mcap * dv * esa},
        {reinterpret_cast<void**>(&c->klog), S * H * Mcap * dk * 2},
        {reinterpret_cast<void**>(&c->Llog), S * H * Mcap * lw * 4},
        {reinterpret_cast<void**>(&c->nlog), S * 4},
        {reinterpret_cast<void**>(&c->base_of), S * 4},
        {reinterpret_cast<void**>(&c->coef), (size_t)c->coef_rows * H * c->L.CB * 4},
        {reinterpret_cast<void**>(&c->status), 16},
    };
    for (auto& x : al) {
      e = dev_alloc(x.p, x.bytes);
      if (e != cudaSuccess) break;
    }
    if (e != cudaSuccess) { rc = set_err(c, DL_ENOMEM, "device allocation failed"); break; }
    e = cudaMemsetAsync(c->Sbar, 0, S * H * dv * dk * 4, c->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->alog, 0, S * H * Mcap * dv * esa, c->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->klog, 0, S * H * Mcap * dk * 2, c->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->Llog, 0, S * H * Mcap * lw * 4, c->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->nlog, 0, S * 4, c->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->status, 0, 16, c->stream);
    if (e == cudaSuccess) {
      std::vector<int32_t> iota(S);
      for (size_t s = 0; s < S; ++s) iota[s] = (int32_t)s;
      e = cudaMemcpyAsync(c->base_of, iota.data(), S * 4, cudaMemcpyHostToDevice, c->stream);
      if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    }
    if (e != cudaSuccess) { rc = cuda_err(c, e, "context initialisation"); break; }
    // allow any shape the planner may pick (its budget never exceeds the opt-in limit)
    const size_t smem = (size_t)c->smem_optin;
    e = dl::configure_append_decode(f.op, f.d_k, smem);
    if (e == cudaSuccess) e = dl::configure_eager_step(f.op, f.d_k, smem);
    if (e != cudaSuccess) { rc = cuda_err(c, e, "kernel attribute"); break; }
    c->regs[(int)Kern::Append] = dl::append_decode_regs(f.op, f.d_k, false, f.merge_interval);
    c->regs[(int)Kern::Fused] = dl::append_decode_regs(f.op, f.d_k, true, f.merge_interval);
    c->regs[(int)Kern::Eager] = dl::eager_step_regs(f.op, f.d_k);
  } while (0);
  g_fail_countdown = -1;
  if (rc != DL_OK) {
    free_all(c);
    delete c;
    return rc;
  }
  *out = c;
  return DL_OK;
}

dl_status dl_destroy(dl_ctx* c) {
  if (!c) return DL_OK;
  cudaStreamSynchronize(c->stream);
  free_all(c);
  delete c;
  return DL_OK;
}

dl_status dl_set_stream(dl_ctx* c, void* stream) {
  if (!c) return DL_EINVAL;
  c->stream = static_cast<cudaStream_t>(stream);
  return DL_OK;
}

dl_status dl_set_state(dl_ctx* c, const int32_t* slots, int32_t n, const float* S) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 0 || (n > 0 && (!S || !aligned16(S)))) return set_err(c, DL_EINVAL, "bad state pointer");
  rc = dl_table_reset(c->table, slots, n);
  if (rc != DL_OK) return set_err(c, rc, "dl_set_state: invalid or frozen slot list");
  dl::SlotListArgs& a = *c->list_args;
  const size_t per = (size_t)c->cfg.num_heads * c->cfg.d_v * c->cfg.d_k;
  for (int32_t r0 = 0; r0 < n; r0 += dl::MAX_ROWS) {
    const int32_t rows = (n - r0) < dl::MAX_ROWS ? (n - r0) : dl::MAX_ROWS;
    a = dl::SlotListArgs{};
    a.Sbar = c->Sbar;
    a.nlog = c->nlog;
    a.base_of = c->base_of;
    a.S_in = S + (size_t)r0 * per;
    a.rows = rows;
    a.H = c->cfg.num_heads;
    a.Mcap = c->L.Mcap;
    for (int32_t i = 0; i < rows; ++i) a.items[i] = dl::StepItem{slots[r0 + i], slots[r0 + i], 0};
    DL_CUDA(dl::launch_set_state(c->cfg.d_k, c->cfg.d_v, a, c->stream), "SetState launch");
  }
  return DL_OK;
}

dl_status dl_set_bonus(dl_ctx* c, const float* bonus) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (c->cfg.op != DL_RWKV6) return set_err(c, DL_EINVAL, "bonus applies to RWKV6 only");
  if (!bonus) return set_err(c, DL_EINVAL, "NULL bonus");
  const size_t bytes = (size_t)c->cfg.num_heads * c->cfg.d_k * 4;
  if (!c->bonus) {
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&c->bonus), bytes);
    if (e != cudaSuccess) return set_err(c, DL_ENOMEM, "bonus allocation failed");
  }
  DL_CUDA(cudaMemcpyAsync(c->bonus, bonus, bytes, cudaMemcpyDeviceToDevice, c->stream), "bonus copy");
  return DL_OK;
}

dl_status dl_fork(dl_ctx* c, int32_t src, const int32_t* dsts, int32_t n) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 0) return set_err(c, DL_EINVAL, "negative count");
  int32_t src_base = 0, src_n = 0;
  if (src >= 0 && src < c->cfg.num_slots) {
    std::vector<int32_t> nl(c->cfg.num_slots), bo(c->cfg.num_slots);
    dl_table_get(c->table, nl.data(), bo.data(), nullptr);
    src_base = bo[src];
    src_n = nl[src];
  }
  rc = dl_table_fork(c->table, src, dsts, n);
  if (rc != DL_OK) return set_err(c, rc, "dl_fork: invalid or frozen slots");
  dl::SlotListArgs& a = *c->list_args;
  for (int32_t r0 = 0; r0 < n; r0 += dl::MAX_ROWS) {
    const int32_t rows = (n - r0) < dl::MAX_ROWS ? (n - r0) : dl::MAX_ROWS;
    a = dl::SlotListArgs{};
    a.alog = c->alog;
    a.klog = c->klog;
    a.Llog = c->Llog;
    a.nlog = c->nlog;
    a.base_of = c->base_of;
    a.rows = rows;
    a.H = c->cfg.num_heads;
    a.Mcap = c->L.Mcap;
    a.src_slot = src;
    a.src_n = src_n;
    a.src_base = src_base;
    for (int32_t i = 0; i < rows; ++i) a.items[i] = dl::StepItem{dsts[r0 + i], src_base, src_n};
    DL_CUDA(dl::launch_fork(c->cfg.op, c->cfg.d_k, a, c->stream), "Fork launch");
  }
  return DL_OK;
}

dl_status dl_step(dl_ctx* c, const int32_t* slots, int32_t n, const void* q, const void* k,
                  const void* v, const float* g, const float* beta, void* o) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 0) return set_err(c, DL_EINVAL, "negative count");
  rc = check_step_ptrs(c, n, q, k, v, g, beta, o);
  if (rc != DL_OK) return rc;
  rc = dl_table_step(c->table, slots, n, c->plan.data());
  if (rc != DL_OK) return set_err(c, rc, "dl_step: invalid or frozen slot list");
  return run_step(c, slots, n, q, k, v, g, beta, o, false);
}

dl_status dl_step_eager(dl_ctx* c, const int32_t* slots, int32_t n, const void* q, const void* k,
                        const void* v, const float* g, const float* beta, void* o) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 0) return set_err(c, DL_EINVAL, "negative count");
  rc = check_step_ptrs(c, n, q, k, v, g, beta, o);
  if (rc != DL_OK) return rc;
  rc = dl_table_step_eager(c->table, slots, n);
  if (rc != DL_OK)
    return set_err(c, rc, "dl_step_eager: slots must own their base and have an empty log");
  for (int32_t i = 0; i < n; ++i) {
    c->plan[4 * (size_t)i + 0] = slots[i];
    c->plan[4 * (size_t)i + 1] = slots[i];
    c->plan[4 * (size_t)i + 2] = 0;
    c->plan[4 * (size_t)i + 3] = 1;
  }
  return run_step(c, slots, n, q, k, v, g, beta, o, true);
}

dl_status dl_step_host(dl_ctx* c, const int32_t* slots, int32_t n, const void* q, const void* k,
                       const void* v, const float* g, const float* beta, void* o) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 0) return set_err(c, DL_EINVAL, "negative count");
  if (n == 0) return DL_OK;
  if (!q || !k || !v || !g || !o || (c->cfg.op != DL_RWKV6 && !beta))
    return set_err(c, DL_EINVAL, "NULL tensor pointer");
  const dl_config& f = c->cfg;
  const size_t H = f.num_heads;
  const size_t bq = (size_t)n * H * f.d_k * 2, bv = (size_t)n * H * f.d_v * 2;
  const size_t bg = (size_t)n * H * (f.op == DL_GDN ? 1 : f.d_k) * 4;
  const size_t bb = (size_t)n * H * 4, bo = (size_t)n * H * f.d_v * (f.out_bf16 ? 2 : 4);
  auto r16 = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t need = 2 * r16(bq) + r16(bv) + r16(bg) + r16(bb) + r16(bo);
  if (need > c->stage_bytes) {
    if (c->stage) cudaFree(c->stage);
    c->stage = nullptr;
    c->stage_bytes = 0;
    // size for the largest batch the context can take, so that later calls do not reallocate
    const size_t Sn = f.num_slots;
    const size_t full = 2 * r16(Sn * H * f.d_k * 2) + r16(Sn * H * f.d_v * 2) +
                        r16(Sn * H * (f.op == DL_GDN ? 1 : f.d_k) * 4) + r16(Sn * H * 4) +
                        r16(Sn * H * f.d_v * 4);
    if (cudaMalloc(&c->stage, full) != cudaSuccess) return set_err(c, DL_ENOMEM, "staging allocation");
    c->stage_bytes = full;
  }
  unsigned char* p = static_cast<unsigned char*>(c->stage);
  void* dq = p; p += r16(bq);
  void* dk = p; p += r16(bq);
  void* dv = p; p += r16(bv);
  float* dg = reinterpret_cast<float*>(p); p += r16(bg);
  float* db = reinterpret_cast<float*>(p); p += r16(bb);
  void* dout = p;
  // validate before any copy so that an error leaves nothing enqueued
  rc = dl_table_check(c->table, slots, n);
  if (rc != DL_OK) return set_err(c, rc, "dl_step_host: invalid slot list");
  DL_CUDA(cudaMemcpyAsync(dq, q, bq, cudaMemcpyHostToDevice, c->stream), "H2D q");
  DL_CUDA(cudaMemcpyAsync(dk, k, bq, cudaMemcpyHostToDevice, c->stream), "H2D k");
  DL_CUDA(cudaMemcpyAsync(dv, v, bv, cudaMemcpyHostToDevice, c->stream), "H2D v");
  DL_CUDA(cudaMemcpyAsync(dg, g, bg, cudaMemcpyHostToDevice, c->stream), "H2D g");
  if (f.op != DL_RWKV6)
    DL_CUDA(cudaMemcpyAsync(db, beta, bb, cudaMemcpyHostToDevice, c->stream), "H2D beta");
  rc = dl_step(c, slots, n, dq, dk, dv, dg, f.op != DL_RWKV6 ? db : nullptr, dout);
  if (rc != DL_OK) return rc;
  DL_CUDA(cudaMemcpyAsync(o, dout, bo, cudaMemcpyDeviceToHost, c->stream), "D2H o");
  DL_CUDA(cudaStreamSynchronize(c->stream), "stream sync");
  return DL_OK;
}

// The upload and download streams of dl_decode_host and the events that order
// them (made once per context).
static cudaError_t copy_streams(dl_ctx* c) {
  cudaError_t e = cudaSuccess;
  if (!c->up) e = cudaStreamCreateWithFlags(&c->up, cudaStreamNonBlocking);
  if (e == cudaSuccess && !c->down) e = cudaStreamCreateWithFlags(&c->down, cudaStreamNonBlocking);
  for (int b = 0; b < PIPE_SETS && e == cudaSuccess; ++b) {
    if (!c->ev_in[b]) e = cudaEventCreateWithFlags(&c->ev_in[b], cudaEventDisableTiming);
    if (e == cudaSuccess && !c->ev_done[b]) e = cudaEventCreateWithFlags(&c->ev_done[b], cudaEventDisableTiming);
    if (e == cudaSuccess && !c->ev_out[b]) e = cudaEventCreateWithFlags(&c->ev_out[b], cudaEventDisableTiming);
  }
  return e;
}

// Staging of window mode: at most this much device memory for the sets.
constexpr size_t WINDOW_STAGE_CAP = (size_t)2 << 30;

// dl_decode_host in whole decode windows (every slot owns its base and starts
// with an empty log, T a multiple of M): each staging set holds M tokens and
// runs as one decode window captured on its buffers (dl_window_create), so the
// host enqueues one graph per M tokens instead of M steps, and the steps inside
// a window chain as programmatic dependents.  The windows are captured once per
// batch (slot list) and kept.  Returns DL_EUNSUPPORTED, having enqueued
// nothing, when the staging would exceed WINDOW_STAGE_CAP.
static dl_status decode_host_windows(dl_ctx* c, const int32_t* slots, int32_t n, int32_t T,
                                     const unsigned char* hq, const unsigned char* hk,
                                     const unsigned char* hv, const unsigned char* hg,
                                     const unsigned char* hb, unsigned char* ho) {
  const dl_config& f = c->cfg;
  const int M = f.merge_interval;
  const size_t H = f.num_heads;
  const size_t bq = (size_t)n * H * f.d_k * 2, bv = (size_t)n * H * f.d_v * 2;
  const size_t bg = (size_t)n * H * (f.op == DL_GDN ? 1 : f.d_k) * 4;
  const size_t bb = (size_t)n * H * 4, bo = (size_t)n * H * f.d_v * (f.out_bf16 ? 2 : 4);
  auto r256 = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t Mz = (size_t)M;
  const size_t set = 2 * r256(Mz * bq) + r256(Mz * bv) + r256(Mz * bg) + r256(Mz * bb) + r256(Mz * bo);
  if (set * PIPE_SETS > WINDOW_STAGE_CAP) return DL_EUNSUPPORTED;
  auto region = [&](int b, unsigned char** dq, unsigned char** dk, unsigned char** dv,
                    unsigned char** dg, unsigned char** db, unsigned char** dout) {
    unsigned char* p = static_cast<unsigned char*>(c->wstage) + (size_t)b * c->wset_bytes;
    *dq = p; p += r256(Mz * bq);
    *dk = p; p += r256(Mz * bq);
    *dv = p; p += r256(Mz * bv);
    *dg = p; p += r256(Mz * bg);
    *db = p; p += r256(Mz * bb);
    *dout = p;
  };
  const bool same = c->wstage && c->wset_bytes == set && c->wslots.size() == (size_t)n &&
                    std::equal(c->wslots.begin(), c->wslots.end(), slots);
  if (!same) {
    cudaStreamSynchronize(c->stream);   // earlier windows may still run
    free_windows(c);
    if (dev_alloc(&c->wstage, PIPE_SETS * set) != cudaSuccess) {
      c->wstage = nullptr;
      return set_err(c, DL_ENOMEM, "window staging allocation");
    }
    c->wset_bytes = set;
    for (int b = 0; b < PIPE_SETS; ++b) {
      unsigned char *dq, *dk, *dv, *dg, *db, *dout;
      region(b, &dq, &dk, &dv, &dg, &db, &dout);
      dl_status rc = dl_window_create(c, slots, n, dq, dk, dv, reinterpret_cast<const float*>(dg),
                                      f.op != DL_RWKV6 ? reinterpret_cast<const float*>(db) : nullptr,
                                      dout, &c->wwin[b]);
      if (rc != DL_OK) {
        free_windows(c);
        return rc;
      }
    }
    c->wslots.assign(slots, slots + n);
  }
  const cudaError_t es = copy_streams(c);
  if (es != cudaSuccess) return cuda_err(c, es, "dl_decode_host set-up");
  dl_status rc = DL_OK;
  cudaError_t e = cudaSuccess;
  const int W = T / M;
  for (int w = 0; w < W && rc == DL_OK && e == cudaSuccess; ++w) {
    const int b = w % PIPE_SETS;
    unsigned char *dq, *dk, *dv, *dg, *db, *dout;
    region(b, &dq, &dk, &dv, &dg, &db, &dout);
    const size_t t0 = (size_t)w * Mz;
    // set b is free once window w - PIPE_SETS's outputs are back
    if (w >= PIPE_SETS) e = cudaStreamWaitEvent(c->up, c->ev_out[b], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dq, hq + t0 * bq, Mz * bq, cudaMemcpyHostToDevice, c->up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dk, hk + t0 * bq, Mz * bq, cudaMemcpyHostToDevice, c->up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dv, hv + t0 * bv, Mz * bv, cudaMemcpyHostToDevice, c->up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dg, hg + t0 * bg, Mz * bg, cudaMemcpyHostToDevice, c->up);
    if (e == cudaSuccess && f.op != DL_RWKV6)
      e = cudaMemcpyAsync(db, hb + t0 * bb, Mz * bb, cudaMemcpyHostToDevice, c->up);
    if (e == cudaSuccess) e = cudaEventRecord(c->ev_in[b], c->up);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->stream, c->ev_in[b], 0);
    if (e != cudaSuccess) break;
    rc = dl_window_launch(c->wwin[b]);
    if (rc != DL_OK) break;
    e = cudaEventRecord(c->ev_done[b], c->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->down, c->ev_done[b], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ho + t0 * bo, dout, Mz * bo, cudaMemcpyDeviceToHost, c->down);
    if (e == cudaSuccess) e = cudaEventRecord(c->ev_out[b], c->down);
  }
  const cudaError_t e1 = cudaStreamSynchronize(c->up);
  const cudaError_t e2 = cudaStreamSynchronize(c->stream);
  const cudaError_t e3 = cudaStreamSynchronize(c->down);
  if (rc != DL_OK) return rc;
  if (e != cudaSuccess) return cuda_err(c, e, "dl_decode_host copies");
  if (e1 != cudaSuccess) return cuda_err(c, e1, "dl_decode_host upload");
  if (e2 != cudaSuccess) return cuda_err(c, e2, "dl_decode_host compute");
  if (e3 != cudaSuccess) return cuda_err(c, e3, "dl_decode_host download");
  return DL_OK;
}

dl_status dl_decode_host(dl_ctx* c, const int32_t* slots, int32_t n, int32_t T, const void* q,
                         const void* k, const void* v, const float* g, const float* beta,
                         void* o) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 0 || T < 0) return set_err(c, DL_EINVAL, "negative count");
  if (n == 0 || T == 0) return DL_OK;
  if (!q || !k || !v || !g || !o || (c->cfg.op != DL_RWKV6 && !beta))
    return set_err(c, DL_EINVAL, "NULL tensor pointer");
  rc = dl_table_check(c->table, slots, n);
  if (rc != DL_OK) return set_err(c, rc, "dl_decode_host: invalid slot list");
  const dl_config& f = c->cfg;
  // whole windows when every slot starts a window on its own base
  if (f.merge_interval >= 2 && T % f.merge_interval == 0 && n <= dl::MAX_ROWS &&
      dl_table_step_eager(c->table, slots, n) == DL_OK) {
    rc = decode_host_windows(c, slots, n, T, static_cast<const unsigned char*>(q),
                             static_cast<const unsigned char*>(k), static_cast<const unsigned char*>(v),
                             reinterpret_cast<const unsigned char*>(g),
                             reinterpret_cast<const unsigned char*>(beta), static_cast<unsigned char*>(o));
    if (rc != DL_EUNSUPPORTED) return rc;
  }
  const size_t H = f.num_heads;
  const size_t bq = (size_t)n * H * f.d_k * 2, bv = (size_t)n * H * f.d_v * 2;
  const size_t bg = (size_t)n * H * (f.op == DL_GDN ? 1 : f.d_k) * 4;
  const size_t bb = (size_t)n * H * 4, bo = (size_t)n * H * f.d_v * (f.out_bf16 ? 2 : 4);
  auto r256 = [](size_t x) { return (x + 255) & ~(size_t)255; };
  if (!c->pipe_stage) {
    // PIPE_SETS staging sets, each for a group of tokens of the largest batch
    // the context can take: a group's inputs travel in one copy per tensor
    // and its outputs in one copy back.  Each copy has a fixed cost, so small
    // per-token tensors are grouped until a key tensor's copy reaches 2 MiB
    // (at most 8 tokens and 64 MiB a set); large ones go token by token,
    // which keeps the pipeline fine-grained.
    const size_t Sn = f.num_slots;
    const size_t per_tok = 2 * Sn * H * f.d_k * 2 + Sn * H * f.d_v * 2 +
                           Sn * H * (f.op == DL_GDN ? 1 : f.d_k) * 4 + Sn * H * 4 +
                           Sn * H * f.d_v * 4;
    const size_t key_bytes = Sn * H * f.d_k * 2;
    size_t tgz = (((size_t)2 << 20) + key_bytes - 1) / (key_bytes > 0 ? key_bytes : 1);
    const size_t cap = ((size_t)64 << 20) / (per_tok > 0 ? per_tok : 1);
    if (tgz > cap) tgz = cap;
    const int tg = tgz < 1 ? 1 : (tgz > 8 ? 8 : (int)tgz);
    const size_t set = 2 * r256(tg * Sn * H * f.d_k * 2) + r256(tg * Sn * H * f.d_v * 2) +
                       r256(tg * Sn * H * (f.op == DL_GDN ? 1 : f.d_k) * 4) +
                       r256(tg * Sn * H * 4) + r256(tg * Sn * H * f.d_v * 4);
    if (cudaMalloc(&c->pipe_stage, PIPE_SETS * set) != cudaSuccess) {
      c->pipe_stage = nullptr;
      return set_err(c, DL_ENOMEM, "staging allocation");
    }
    c->pipe_set_bytes = set;
    c->pipe_group = tg;
    const cudaError_t e = copy_streams(c);
    if (e != cudaSuccess) return cuda_err(c, e, "dl_decode_host set-up");
  }
  const unsigned char* hq = static_cast<const unsigned char*>(q);
  const unsigned char* hk = static_cast<const unsigned char*>(k);
  const unsigned char* hv = static_cast<const unsigned char*>(v);
  const unsigned char* hg = reinterpret_cast<const unsigned char*>(g);
  const unsigned char* hb = reinterpret_cast<const unsigned char*>(beta);
  unsigned char* ho = static_cast<unsigned char*>(o);
  const int TG = c->pipe_group;
  cudaError_t e = cudaSuccess;
  int grp = 0;
  for (int32_t t0 = 0; t0 < T && rc == DL_OK && e == cudaSuccess; t0 += TG, ++grp) {
    const int b = grp % PIPE_SETS;
    const int tn = (T - t0) < TG ? (T - t0) : TG;   // tokens in this group
    // the set's regions, each holding the group's tokens contiguously
    unsigned char* p = static_cast<unsigned char*>(c->pipe_stage) + (size_t)b * c->pipe_set_bytes;
    unsigned char* dq = p; p += r256((size_t)TG * bq);
    unsigned char* dk = p; p += r256((size_t)TG * bq);
    unsigned char* dv = p; p += r256((size_t)TG * bv);
    unsigned char* dg = p; p += r256((size_t)TG * bg);
    unsigned char* db = p; p += r256((size_t)TG * bb);
    unsigned char* dout = p;
    // set b is free once group grp - PIPE_SETS's outputs have been downloaded
    // (which also follows its kernels, the last readers of its inputs)
    if (grp >= PIPE_SETS) e = cudaStreamWaitEvent(c->up, c->ev_out[b], 0);
    const size_t t0s = (size_t)t0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(dq, hq + t0s * bq, tn * bq, cudaMemcpyHostToDevice, c->up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dk, hk + t0s * bq, tn * bq, cudaMemcpyHostToDevice, c->up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dv, hv + t0s * bv, tn * bv, cudaMemcpyHostToDevice, c->up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dg, hg + t0s * bg, tn * bg, cudaMemcpyHostToDevice, c->up);
    if (e == cudaSuccess && f.op != DL_RWKV6)
      e = cudaMemcpyAsync(db, hb + t0s * bb, tn * bb, cudaMemcpyHostToDevice, c->up);
    if (e == cudaSuccess) e = cudaEventRecord(c->ev_in[b], c->up);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->stream, c->ev_in[b], 0);
    if (e != cudaSuccess) break;
    for (int j = 0; j < tn && rc == DL_OK; ++j)
      rc = dl_step(c, slots, n, dq + j * bq, dk + j * bq, dv + j * bv,
                   reinterpret_cast<const float*>(dg + j * bg),
                   f.op != DL_RWKV6 ? reinterpret_cast<const float*>(db + j * bb) : nullptr,
                   dout + j * bo);
    if (rc != DL_OK) break;
    e = cudaEventRecord(c->ev_done[b], c->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->down, c->ev_done[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ho + t0s * bo, dout, tn * bo, cudaMemcpyDeviceToHost, c->down);
    if (e == cudaSuccess) e = cudaEventRecord(c->ev_out[b], c->down);
  }
  // nothing may still write the caller's buffers when the call returns
  const cudaError_t e1 = cudaStreamSynchronize(c->up);
  const cudaError_t e2 = cudaStreamSynchronize(c->stream);
  const cudaError_t e3 = cudaStreamSynchronize(c->down);
  if (rc != DL_OK) return rc;
  if (e != cudaSuccess) return cuda_err(c, e, "dl_decode_host copies");
  if (e1 != cudaSuccess) return cuda_err(c, e1, "dl_decode_host upload");
  if (e2 != cudaSuccess) return cuda_err(c, e2, "dl_decode_host compute");
  if (e3 != cudaSuccess) return cuda_err(c, e3, "dl_decode_host download");
  return DL_OK;
}

static dl_status merge_or_read(dl_ctx* c, const int32_t* slots, int32_t n, float* S_out) {
  std::vector<int32_t> nl(c->cfg.num_slots), bo(c->cfg.num_slots);
  dl_table_get(c->table, nl.data(), bo.data(), nullptr);
  std::vector<dl::StepItem> items(n);
  for (int32_t i = 0; i < n; ++i) items[i] = dl::StepItem{slots[i], bo[slots[i]], nl[slots[i]]};
  if (!S_out) {
    dl_status rc = dl_table_reset(c->table, slots, n);
    if (rc != DL_OK) return set_err(c, rc, "dl_merge: invalid or frozen slot list");
  }
  dl::SlotListArgs& a = *c->list_args;
  const size_t per = (size_t)c->cfg.num_heads * c->cfg.d_v * c->cfg.d_k;
  for (int32_t r0 = 0; r0 < n; r0 += dl::MAX_ROWS) {
    const int32_t rows = (n - r0) < dl::MAX_ROWS ? (n - r0) : dl::MAX_ROWS;
    a = dl::SlotListArgs{};
    a.Sbar = c->Sbar;
    a.alog = c->alog;
    a.klog = c->klog;
    a.Llog = c->Llog;
    a.nlog = c->nlog;
    a.base_of = c->base_of;
    a.S_out = S_out ? S_out + (size_t)r0 * per : nullptr;
    a.rows = rows;
    a.H = c->cfg.num_heads;
    a.Mcap = c->L.Mcap;
    for (int32_t i = 0; i < rows; ++i) a.items[i] = items[r0 + i];
    cudaEvent_t e0;
    const bool t = record(c, 3, &e0);
    DL_CUDA(dl::launch_merge(c->cfg.op, c->cfg.d_k, a, c->stream), "Merge launch");
    if (t) record_end(c, 3, e0);
  }
  return DL_OK;
}

dl_status dl_merge(dl_ctx* c, const int32_t* slots, int32_t n) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 0) return set_err(c, DL_EINVAL, "negative count");
  rc = dl_table_check(c->table, slots, n);
  if (rc != DL_OK) return set_err(c, rc, "dl_merge: invalid slot list");
  return merge_or_read(c, slots, n, nullptr);
}

dl_status dl_read_state(dl_ctx* c, const int32_t* slots, int32_t n, float* S_out) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 0) return set_err(c, DL_EINVAL, "negative count");
  if (n > 0 && (!S_out || !aligned16(S_out))) return set_err(c, DL_EINVAL, "bad output pointer");
  rc = dl_table_check(c->table, slots, n);
  if (rc != DL_OK) return set_err(c, rc, "dl_read_state: invalid slot list");
  return merge_or_read(c, slots, n, S_out);
}

dl_status dl_prefill(dl_ctx* c, const int32_t* slots, int32_t n, int32_t T, const void* q,
                     const void* k, const void* v, const float* g, const float* beta, void* o) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 0 || T < 0) return set_err(c, DL_EINVAL, "negative count");
  if (n == 0 || T == 0) return DL_OK;
  const bool delta = c->cfg.op != DL_RWKV6;
  if (!q || !k || !v || !g || (delta && !beta)) return set_err(c, DL_EINVAL, "NULL tensor pointer");
  if (!delta && !c->bonus) return set_err(c, DL_EINVAL, "RWKV6 needs dl_set_bonus before prefill");
  // q, k, v and the per-key g rows are read as 16-byte vectors
  const bool perkey = c->cfg.op != DL_GDN;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) ||
      (perkey ? !aligned16(g) : (reinterpret_cast<uintptr_t>(g) & 3u) != 0) ||
      (delta && (reinterpret_cast<uintptr_t>(beta) & 3u)) ||
      (o && (reinterpret_cast<uintptr_t>(o) & (c->cfg.out_bf16 ? 1u : 3u))))
    return set_err(c, DL_EINVAL, "misaligned tensor: q, k, v%s need 16-byte alignment, "
                   "other tensors their element size", perkey ? ", g" : "");
  if (n > dl::MAX_ROWS) return set_err(c, DL_EINVAL, "dl_prefill takes at most %d slots per call", dl::MAX_ROWS);
  rc = dl_table_step_eager(c->table, slots, n);
  if (rc != DL_OK)
    return set_err(c, rc, "dl_prefill: slots must own their base and have an empty log");
  dl::SlotListArgs& a = *c->list_args;
  a = dl::SlotListArgs{};
  a.Sbar = c->Sbar;
  a.nlog = c->nlog;
  a.base_of = c->base_of;
  a.rows = n;
  a.H = c->cfg.num_heads;
  a.Mcap = c->L.Mcap;
  for (int32_t i = 0; i < n; ++i) a.items[i] = dl::StepItem{slots[i], slots[i], 0};
  DL_CUDA(dl::launch_prefill(c->cfg.op, c->cfg.d_k, a, q, k, v, g, delta ? beta : nullptr,
                             c->bonus, o, T, c->cfg.out_bf16, c->cfg.scale, c->status,
                             c->stream),
          "Prefill launch");
  return DL_OK;
}

struct CkptLayout {
  size_t S, A, K, L, N, total;
};

static CkptLayout ckpt_layout(const dl_ctx* c) {
  const dl_config& f = c->cfg;
  const size_t H = f.num_heads, Mcap = c->L.Mcap;
  auto r16 = [](size_t x) { return (x + 15) & ~(size_t)15; };
  CkptLayout k;
  k.S = 0;
  k.A = k.S + r16(H * f.d_v * f.d_k * 4);
  k.K = k.A + r16(H * Mcap * f.d_v * (f.op == DL_RWKV6 ? 2 : 4));
  k.L = k.K + r16(H * Mcap * f.d_k * 2);
  k.N = k.L + r16(H * Mcap * (f.op == DL_GDN ? 1 : f.d_k) * 4);
  k.total = k.N + 16;
  return k;
}

int64_t dl_checkpoint_bytes(const dl_ctx* c) { return c ? (int64_t)ckpt_layout(c).total : -1; }

// One launch per MAX_ROWS slots moves the records (checkpoint_kernel).
static dl_status checkpoint_copy(dl_ctx* c, const int32_t* slots, int32_t n, unsigned char* buf,
                                 const int32_t* bases, int save) {
  const CkptLayout k = ckpt_layout(c);
  const dl_config& f = c->cfg;
  for (int32_t r0 = 0; r0 < n; r0 += dl::MAX_ROWS) {
    const int32_t rows = (n - r0) < dl::MAX_ROWS ? (n - r0) : dl::MAX_ROWS;
    dl::CkptArgs& a = *c->ckpt_args;
    a.Sbar = c->Sbar;
    a.alog = c->alog;
    a.klog = c->klog;
    a.Llog = c->Llog;
    a.nlog = c->nlog;
    a.base_of = c->base_of;
    a.buf = buf + (size_t)r0 * k.total;
    a.total = k.total;
    a.offS = k.S;
    a.offA = k.A;
    a.offK = k.K;
    a.offL = k.L;
    a.offN = k.N;
    a.rows = rows;
    a.H = f.num_heads;
    a.Mcap = c->L.Mcap;
    a.save = save;
    for (int32_t i = 0; i < rows; ++i)
      a.items[i] = dl::StepItem{slots[r0 + i], bases ? bases[r0 + i] : slots[r0 + i], 0};
    DL_CUDA(dl::launch_checkpoint(f.op, f.d_k, a, c->stream), save ? "checkpoint save" : "checkpoint restore");
  }
  return DL_OK;
}

dl_status dl_checkpoint_save(dl_ctx* c, const int32_t* slots, int32_t n, void* buf) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 0 || (n > 0 && (!buf || !aligned16(buf)))) return set_err(c, DL_EINVAL, "bad buffer");
  rc = dl_table_check(c->table, slots, n);
  if (rc != DL_OK) return set_err(c, rc, "dl_checkpoint_save: invalid slot list");
  if (n == 0) return DL_OK;
  std::vector<int32_t> nl(c->cfg.num_slots), bo(c->cfg.num_slots), bases(n);
  dl_table_get(c->table, nl.data(), bo.data(), nullptr);
  for (int32_t i = 0; i < n; ++i) bases[i] = bo[slots[i]];
  return checkpoint_copy(c, slots, n, static_cast<unsigned char*>(buf), bases.data(), 1);
}

dl_status dl_checkpoint_load(dl_ctx* c, const int32_t* slots, int32_t n, const void* buf) {
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 0 || (n > 0 && (!buf || !aligned16(buf)))) return set_err(c, DL_EINVAL, "bad buffer");
  rc = dl_table_check(c->table, slots, n);
  if (rc != DL_OK) return set_err(c, rc, "dl_checkpoint_load: invalid slot list");
  if (n == 0) return DL_OK;
  const CkptLayout k = ckpt_layout(c);
  // the saved log lengths, one strided copy, validated before anything changes
  std::vector<int32_t> ns(n);
  DL_CUDA(cudaMemcpy2DAsync(ns.data(), 4, static_cast<const unsigned char*>(buf) + k.N, k.total, 4,
                            n, cudaMemcpyDeviceToHost, c->stream),
          "checkpoint read");
  DL_CUDA(cudaStreamSynchronize(c->stream), "stream sync");
  for (int32_t i = 0; i < n; ++i)
    if (ns[i] < 0 || ns[i] >= c->cfg.merge_interval)
      return set_err(c, DL_EINVAL, "checkpoint %d holds log length %d, not valid for M=%d", i, ns[i],
                     c->cfg.merge_interval);
  rc = dl_table_reset(c->table, slots, n);     // validates frozen slots, owns base, n = 0
  if (rc != DL_OK) return set_err(c, rc, "dl_checkpoint_load: frozen slot");
  rc = checkpoint_copy(c, slots, n,
                       const_cast<unsigned char*>(static_cast<const unsigned char*>(buf)), nullptr, 0);
  if (rc != DL_OK) return rc;
  dl_table_set_n(c->table, slots, n, ns.data());
  return DL_OK;
}

}  // extern "C"

struct dl_window {
  dl_ctx* ctx = nullptr;
  std::vector<int32_t> slots;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  // ragged windows: per-token plans and counts, written on the host at each
  // launch and copied to the device by the graph's first node
  bool ragged = false;
  int32_t n_max = 0;
  void* plan_host = nullptr;   // pinned: [M][n_max] StepItem, then [M] int32 counts
  void* plan_dev = nullptr;
  size_t plan_bytes = 0;
  cudaEvent_t done = nullptr;  // end of the last launch (the host plan is free again)
  bool launched = false;
  std::vector<int32_t> scratch;   // one token's plan rows (4 ints each)
};

static void window_free(dl_window* w) {
  if (w->exec) cudaGraphExecDestroy(w->exec);
  if (w->graph) cudaGraphDestroy(w->graph);
  if (w->done) cudaEventDestroy(w->done);
  if (w->plan_host) cudaFreeHost(w->plan_host);
  if (w->plan_dev) cudaFree(w->plan_dev);
  w->exec = nullptr;
  w->graph = nullptr;
  w->done = nullptr;
  w->plan_host = w->plan_dev = nullptr;
}

extern "C" {

dl_status dl_window_create(dl_ctx* c, const int32_t* slots, int32_t n, const void* q,
                           const void* k, const void* v, const float* g, const float* beta,
                           void* o, dl_window** out) {
  if (!out) return DL_EINVAL;
  *out = nullptr;
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (n < 1 || n > dl::MAX_ROWS) return set_err(c, DL_EINVAL, "window batch must be 1..%d", dl::MAX_ROWS);
  rc = check_step_ptrs(c, n, q, k, v, g, beta, o);
  if (rc != DL_OK) return rc;
  rc = dl_table_step_eager(c->table, slots, n);   // own base, empty log, not frozen
  if (rc != DL_OK) return set_err(c, rc, "dl_window_create: slots must own their base and have an empty log");
  const dl_config& f = c->cfg;
  const int M = f.merge_interval;
  const size_t H = f.num_heads;
  const size_t sq = (size_t)n * H * f.d_k * 2, sv = (size_t)n * H * f.d_v * 2;
  const size_t sg = (size_t)n * H * (f.op == DL_GDN ? 1 : f.d_k) * 4, sb = (size_t)n * H * 4;
  const size_t so = (size_t)n * H * f.d_v * (f.out_bf16 ? 2 : 4);
  // every per-token slice must keep the alignment dl_step needs (q, k, v and
  // per-key g rows are always 16-byte multiples; the others are element-sized)
  (void)sb;
  std::unique_ptr<dl_window> w(new (std::nothrow) dl_window);
  if (!w) return set_err(c, DL_ENOMEM, "window allocation");
  w->ctx = c;
  w->slots.assign(slots, slots + n);
  cudaStream_t cap = nullptr;
  DL_CUDA(cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking), "capture stream");
  cudaStream_t saved = c->stream;
  const bool saved_timing = c->timing;
  c->stream = cap;
  c->timing = false;
  cudaError_t e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
  dl_status st = DL_OK;
  if (e == cudaSuccess) {
    for (int j = 0; j < M && st == DL_OK; ++j) {
      c->pdl_chain = (j > 0 && f.staging == DL_STAGE_FUSED) ? 1 : 0;
      for (int32_t i = 0; i < n; ++i) {
        c->plan[4 * (size_t)i + 0] = slots[i];
        c->plan[4 * (size_t)i + 1] = slots[i];
        c->plan[4 * (size_t)i + 2] = j;
        c->plan[4 * (size_t)i + 3] = (j + 1 == M);
      }
      st = run_step(c, slots, n, static_cast<const unsigned char*>(q) + j * sq,
                    static_cast<const unsigned char*>(k) + j * sq,
                    static_cast<const unsigned char*>(v) + j * sv,
                    reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(g) + j * sg),
                    beta ? reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(beta) + j * sb)
                         : nullptr,
                    static_cast<unsigned char*>(o) + j * so, false);
    }
    cudaError_t e2 = cudaStreamEndCapture(cap, &w->graph);
    if (e == cudaSuccess) e = e2;
  }
  c->stream = saved;
  c->timing = saved_timing;
  c->pdl_chain = 0;
  cudaStreamDestroy(cap);
  if (st != DL_OK) {
    if (w->graph) cudaGraphDestroy(w->graph);
    c->sticky = DL_OK;   // a failed capture leaves the context usable
    return set_err(c, DL_ECUDA, "window capture failed: %s", c->err.c_str());
  }
  if (e != cudaSuccess) {
    if (w->graph) cudaGraphDestroy(w->graph);
    return set_err(c, DL_ECUDA, "window capture: %s", cudaGetErrorString(e));
  }
  e = cudaGraphInstantiate(&w->exec, w->graph, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(w->graph);
    return set_err(c, DL_ECUDA, "graph instantiate: %s", cudaGetErrorString(e));
  }
  *out = w.release();
  return DL_OK;
}

dl_status dl_window_launch(dl_window* w) {
  if (!w) return DL_EINVAL;
  dl_ctx* c = w->ctx;
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (w->ragged) return set_err(c, DL_EINVAL, "a ragged window launches with dl_window_launch_ragged");
  const int32_t n = (int32_t)w->slots.size();
  rc = dl_table_step_eager(c->table, w->slots.data(), n);
  if (rc != DL_OK)
    return set_err(c, rc, "dl_window_launch: slots must own their base and have an empty log");
  DL_CUDA(cudaGraphLaunch(w->exec, c->stream), "graph launch");
  for (int j = 0; j < c->cfg.merge_interval; ++j) dl_table_step(c->table, w->slots.data(), n, nullptr);
  return DL_OK;
}

dl_status dl_window_destroy(dl_window* w) {
  if (!w) return DL_OK;
  if (w->done) cudaEventSynchronize(w->done);   // the graph may still read the plan buffers
  window_free(w);
  delete w;
  return DL_OK;
}

dl_status dl_window_create_ragged(dl_ctx* c, int32_t n_max, const void* q, const void* k,
                                  const void* v, const float* g, const float* beta, void* o,
                                  dl_window** out) {
  if (!out) return DL_EINVAL;
  *out = nullptr;
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  const dl_config& f = c->cfg;
  if (n_max < 1 || n_max > dl::MAX_ROWS || n_max > f.num_slots)
    return set_err(c, DL_EINVAL, "ragged window capacity must be 1..min(%d, num_slots)",
                   dl::MAX_ROWS);
  rc = check_step_ptrs(c, n_max, q, k, v, g, beta, o);
  if (rc != DL_OK) return rc;
  if (f.op == DL_RWKV6 && !c->bonus)
    return set_err(c, DL_EINVAL, "RWKV6 needs dl_set_bonus before a window is captured");
  const int M = f.merge_interval;
  const size_t H = f.num_heads;
  const size_t sq = (size_t)n_max * H * f.d_k * 2, sv = (size_t)n_max * H * f.d_v * 2;
  const size_t sg = (size_t)n_max * H * (f.op == DL_GDN ? 1 : f.d_k) * 4, sb = (size_t)n_max * H * 4;
  const size_t so = (size_t)n_max * H * f.d_v * (f.out_bf16 ? 2 : 4);
  std::unique_ptr<dl_window> w(new (std::nothrow) dl_window);
  if (!w) return set_err(c, DL_ENOMEM, "window allocation");
  w->ctx = c;
  w->ragged = true;
  w->n_max = n_max;
  w->plan_bytes = (size_t)M * n_max * sizeof(dl::StepItem) + (size_t)M * sizeof(int32_t);
  w->scratch.resize(4 * (size_t)n_max);
  if (cudaHostAlloc(&w->plan_host, w->plan_bytes, cudaHostAllocDefault) != cudaSuccess ||
      cudaMalloc(&w->plan_dev, w->plan_bytes) != cudaSuccess) {
    window_free(w.get());
    return set_err(c, DL_ENOMEM, "ragged window plan buffers");
  }
  memset(w->plan_host, 0, w->plan_bytes);
  DL_CUDA(cudaEventCreateWithFlags(&w->done, cudaEventDisableTiming), "window event");
  const dl::StepItem* items_dev = static_cast<const dl::StepItem*>(w->plan_dev);
  const int32_t* counts_dev =
      reinterpret_cast<const int32_t*>(static_cast<const unsigned char*>(w->plan_dev) +
                                       (size_t)M * n_max * sizeof(dl::StepItem));
  cudaStream_t cap = nullptr;
  DL_CUDA(cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking), "capture stream");
  cudaStream_t saved = c->stream;
  const bool saved_timing = c->timing;
  c->stream = cap;
  c->timing = false;
  cudaError_t e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
  dl_status st = DL_OK;
  if (e == cudaSuccess) {
    e = cudaMemcpyAsync(w->plan_dev, w->plan_host, w->plan_bytes, cudaMemcpyHostToDevice, cap);
    for (int j = 0; j < M && st == DL_OK && e == cudaSuccess; ++j) {
      c->pdl_chain = (j > 0 && f.staging == DL_STAGE_FUSED) ? 1 : 0;
      c->dev_plan = items_dev + (size_t)j * n_max;
      c->dev_rows = counts_dev + j;
      st = run_step(c, nullptr, n_max, static_cast<const unsigned char*>(q) + j * sq,
                    static_cast<const unsigned char*>(k) + j * sq,
                    static_cast<const unsigned char*>(v) + j * sv,
                    reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(g) + j * sg),
                    beta ? reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(beta) + j * sb)
                         : nullptr,
                    static_cast<unsigned char*>(o) + j * so, false);
    }
    cudaError_t e2 = cudaStreamEndCapture(cap, &w->graph);
    if (e == cudaSuccess) e = e2;
  }
  c->stream = saved;
  c->timing = saved_timing;
  c->pdl_chain = 0;
  c->dev_plan = nullptr;
  c->dev_rows = nullptr;
  cudaStreamDestroy(cap);
  if (st != DL_OK) {
    window_free(w.get());
    c->sticky = DL_OK;   // a failed capture leaves the context usable
    return set_err(c, DL_ECUDA, "window capture failed: %s", c->err.c_str());
  }
  if (e != cudaSuccess) {
    window_free(w.get());
    return set_err(c, DL_ECUDA, "window capture: %s", cudaGetErrorString(e));
  }
  e = cudaGraphInstantiate(&w->exec, w->graph, 0);
  if (e != cudaSuccess) {
    window_free(w.get());
    return set_err(c, DL_ECUDA, "graph instantiate: %s", cudaGetErrorString(e));
  }
  *out = w.release();
  return DL_OK;
}

dl_status dl_window_launch_ragged(dl_window* w, const int32_t* slots, const int32_t* counts) {
  if (!w) return DL_EINVAL;
  dl_ctx* c = w->ctx;
  dl_status rc = check_ctx(c);
  if (rc != DL_OK) return rc;
  if (!w->ragged) return set_err(c, DL_EINVAL, "not a ragged window");
  if (!counts || !slots) return set_err(c, DL_EINVAL, "NULL slot list");
  const int M = c->cfg.merge_interval;
  const int32_t n_max = w->n_max;
  // validate every token before any is applied: ids, duplicates, fork sources
  std::vector<int32_t> refs(c->cfg.num_slots);
  dl_table_get(c->table, nullptr, nullptr, refs.data());
  for (int j = 0; j < M; ++j) {
    const int32_t cnt = counts[j];
    if (cnt < 0 || cnt > n_max) return set_err(c, DL_EINVAL, "token %d: count out of range", j);
    const int32_t* sl = slots + (size_t)j * n_max;
    rc = dl_table_check(c->table, sl, cnt);
    if (rc != DL_OK) return set_err(c, rc, "token %d: invalid slot list", j);
    for (int32_t i = 0; i < cnt; ++i)
      if (refs[sl[i]] > 0) return set_err(c, DL_EBUSY, "token %d: slot %d is a fork source", j, sl[i]);
  }
  // the previous launch's graph has copied the plan only once it has run
  if (w->launched) DL_CUDA(cudaEventSynchronize(w->done), "window wait");
  dl::StepItem* items = static_cast<dl::StepItem*>(w->plan_host);
  int32_t* cnt_host = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(w->plan_host) +
                                                 (size_t)M * n_max * sizeof(dl::StepItem));
  for (int j = 0; j < M; ++j) {
    const int32_t cnt = counts[j];
    rc = dl_table_step(c->table, slots + (size_t)j * n_max, cnt, w->scratch.data());
    if (rc != DL_OK) return set_err(c, rc, "token %d: slot table refused the step", j);
    for (int32_t i = 0; i < cnt; ++i)
      items[(size_t)j * n_max + i] =
          dl::StepItem{w->scratch[4 * i], w->scratch[4 * i + 1], w->scratch[4 * i + 2]};
    cnt_host[j] = cnt;
  }
  DL_CUDA(cudaGraphLaunch(w->exec, c->stream), "graph launch");
  DL_CUDA(cudaEventRecord(w->done, c->stream), "window event");
  w->launched = true;
  return DL_OK;
}

dl_status dl_sync(dl_ctx* c) {
  if (!c) return DL_EINVAL;
  if (c->sticky != DL_OK) return c->sticky;
  DL_CUDA(cudaStreamSynchronize(c->stream), "stream sync");
  DL_CUDA(cudaGetLastError(), "pending CUDA error");
  int32_t st = 0;
  DL_CUDA(cudaMemcpy(&st, c->status, 4, cudaMemcpyDeviceToHost), "status read");
  if (st != 0)
    return set_err(c, DL_EDEVICE, "kernel reported device status %d (%s)", st, dl::device_status_str(st));
  return DL_OK;
}

dl_status dl_get_meta(dl_ctx* c, int32_t* n_log, int32_t* base_of) {
  dl_status rc = dl_sync(c);
  if (rc != DL_OK) return rc;
  const size_t S = c->cfg.num_slots;
  std::vector<int32_t> dn(S), db(S), hn(S), hb(S);
  DL_CUDA(cudaMemcpy(dn.data(), c->nlog, S * 4, cudaMemcpyDeviceToHost), "meta read");
  DL_CUDA(cudaMemcpy(db.data(), c->base_of, S * 4, cudaMemcpyDeviceToHost), "meta read");
  dl_table_get(c->table, hn.data(), hb.data(), nullptr);
  if (n_log) memcpy(n_log, dn.data(), S * 4);
  if (base_of) memcpy(base_of, db.data(), S * 4);
  if (dn != hn || db != hb) return set_err(c, DL_EDEVICE, "device slot table disagrees with host table");
  return DL_OK;
}

dl_status dl_set_timing(dl_ctx* c, int32_t enable) {
  if (!c) return DL_EINVAL;
  c->timing = enable != 0;
  for (int k = 0; k < NKIND; ++k) {
    c->timed_ms[k] = 0;
    c->timed_n[k] = 0;
  }
  return DL_OK;
}

dl_status dl_get_timing(dl_ctx* c, double* ms, int64_t* launches) {
  if (!c) return DL_EINVAL;
  DL_CUDA(cudaStreamSynchronize(c->stream), "stream sync");
  for (int k = 0; k < NKIND; ++k) {
    for (auto& p : c->timed[k]) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, p.a, p.b) == cudaSuccess) c->timed_ms[k] += t;
      c->timed_n[k] += 1;
      cudaEventDestroy(p.a);
      cudaEventDestroy(p.b);
    }
    c->timed[k].clear();
    if (ms) ms[k] = c->timed_ms[k];
    if (launches) launches[k] = c->timed_n[k];
  }
  return DL_OK;
}

}  // extern "C"
