// fnorm_api.cu -- the libfnorm C ABI: argument validation, choice of kernel
// and launch shape, stream-ordered launches, status codes and the device
// error word. Declarations and contracts are in include/fnorm.h.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "../../include/fnorm.h"
#include "fnorm_internal.h"

namespace fnorm {

// Device error word: kernels OR failure codes into it (bounded waits that
// expired); fnorm_get_last_error reads and clears it. One instance per device.
__device__ unsigned int g_fnorm_err_word;

namespace {

std::mutex g_mutex;
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_info_valid[kMaxDevices];
unsigned* g_err_ptr[kMaxDevices];
std::map<std::string, int> g_occupancy;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return d;
}

// Device address of this device's error word (looked up once per device with
// that device current).
unsigned* err_word() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mutex);
  if (!g_err_ptr[d]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fnorm_err_word) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_err_ptr[d] = static_cast<unsigned*>(ptr);
  }
  return g_err_ptr[d];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// [a, a+na) and [b, b+nb) share a byte (empty ranges never overlap).
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  return !__builtin_mul_overflow(a, b, out) && *out <= (int64_t(1) << 56);
}

bool finite_nonneg(float v) { return std::isfinite(v) && v >= 0.f; }

// Tuning and test switches (FNORM_* environment variables) are read once per
// process, on the first call that needs one, and again only when
// fnorm_tuning_reload() is called. With none of them set, env() returns at
// the first branch.
struct Knob {
  const char* name;
  std::string value;
  bool set;
};
Knob g_knobs[] = {
    {"FNORM_FORCE_PATH", {}, false},      {"FNORM_SPLIT_SHAPE", {}, false},
    {"FNORM_RESIDENT_THREADS", {}, false}, {"FNORM_FORCE_SCALAR", {}, false},
    {"FNORM_STREAM_UNROLL", {}, false},   {"FNORM_NO_PACK", {}, false},
    {"FNORM_EPI_CLUSTER", {}, false},     {"FNORM_EPI_KEEP", {}, false},
    {"FNORM_EPI_STREAM", {}, false},      {"FNORM_EPI_TWOPASS", {}, false},
    {"FNORM_BN_SPLIT", {}, false},        {"FNORM_BN_RESIDENT", {}, false},
    {"FNORM_BN_NO_COLUMNS", {}, false},   {"FNORM_DEBUG_PLAN", {}, false},
};
std::mutex g_knob_mutex;
std::atomic<int> g_knobs_state{0};   // 0: not read, 1: read, none set, 2: read, some set

void load_knobs() {
  std::lock_guard<std::mutex> lk(g_knob_mutex);
  bool any = false;
  for (Knob& k : g_knobs) {
    const char* v = std::getenv(k.name);
    k.set = v && *v;
    k.value = k.set ? v : "";
    any = any || k.set;
  }
  g_knobs_state.store(any ? 2 : 1, std::memory_order_release);
}

const char* env(const char* name) {
  int st = g_knobs_state.load(std::memory_order_acquire);
  if (st == 0) {
    static std::once_flag once;
    std::call_once(once, [] {
      if (g_knobs_state.load(std::memory_order_acquire) == 0) load_knobs();
    });
    st = g_knobs_state.load(std::memory_order_acquire);
  }
  if (st == 1) return nullptr;
  for (const Knob& k : g_knobs)
    if (std::strcmp(k.name, name) == 0) return k.set ? k.value.c_str() : nullptr;
  return nullptr;
}

// Test hook (fnorm_debug_force_timeout): one CTA of each launch waits on a
// barrier that nothing completes, so that its bounded wait expires.
std::atomic<int> g_force_timeout{0};
int force_timeout() { return g_force_timeout.load(std::memory_order_relaxed) ? 1 : 0; }

// Test hook (fnorm_debug_fail_launches): the next n calls that pass their
// argument checks return FNORM_ERR_CUDA instead of launching, as a failed
// launch would. Each call consumes one.
std::atomic<int> g_fail_launches{0};
bool injected_launch_failure() {
  int n = g_fail_launches.load(std::memory_order_relaxed);
  while (n > 0) {
    if (g_fail_launches.compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) return true;
  }
  return false;
}

// An NVTX range named after the entry point around the planning and launches
// of one call (visible to profilers that collect NVTX; nearly free otherwise).
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

int occupancy_cached(const std::string& key, int (*query)(const void*), const void* arg) {
  const int d = current_device();
  const std::string k = std::to_string(d) + "|" + key;
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    auto it = g_occupancy.find(k);
    if (it != g_occupancy.end()) return it->second;
  }
  const int v = query(arg);
  std::lock_guard<std::mutex> lk(g_mutex);
  g_occupancy[k] = v;
  return v;
}

fnorm_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FNORM_OK;
  cudaGetLastError();
  return FNORM_ERR_CUDA;
}

// ------------------------------------------------------------ InstanceNorm
struct InCall {
  int tin, tout;   // 0 = f32, 1 = bf16
  InPlan plan;
};

cudaError_t in_launch_dispatch(int tin, int tout, const InParams& p, const InPlan& plan,
                               cudaStream_t s) {
  if (tin == 0 && tout == 0) return in_launch_t<float, float>(p, plan, s);
  if (tin == 0 && tout == 1) return in_launch_t<float, __nv_bfloat16>(p, plan, s);
  if (tin == 1 && tout == 1) return in_launch_t<__nv_bfloat16, __nv_bfloat16>(p, plan, s);
  return in_launch_t<__nv_bfloat16, float>(p, plan, s);
}

struct InQuery {
  int tin, tout;
  InPlan plan;
};

int in_query(const void* arg) {
  const InQuery& q = *static_cast<const InQuery*>(arg);
  if (q.tin == 0 && q.tout == 0) return in_max_active_clusters_t<float, float>(q.plan);
  if (q.tin == 0 && q.tout == 1) return in_max_active_clusters_t<float, __nv_bfloat16>(q.plan);
  if (q.tin == 1 && q.tout == 1)
    return in_max_active_clusters_t<__nv_bfloat16, __nv_bfloat16>(q.plan);
  return in_max_active_clusters_t<__nv_bfloat16, float>(q.plan);
}

int in_capacity(int tin, int tout, const InPlan& plan) {
  char key[128];
  std::snprintf(key, sizeof key, "in|%d|%d|%d|%d|%d|%d|%d|%d|%d|%d", tin, tout,
                static_cast<int>(plan.path), plan.vec ? 1 : 0, plan.threads, plan.nv, plan.ns,
                plan.group, plan.cluster, plan.packed ? 1 : 0);
  InQuery q{tin, tout, plan};
  return occupancy_cached(key, in_query, &q);
}

// Parses FNORM_FORCE_PATH (test and tuning hook):
//   group:G:NV | resident:THREADS:NV:CLUSTER | split:THREADS:NR:NS:CLUSTER | stream:CLUSTER
bool in_forced_plan(InPlan* plan) {
  const char* f = env("FNORM_FORCE_PATH");
  if (!f) return false;
  int a = 0, b = 0, c = 0;
  if (std::sscanf(f, "group:%d:%d", &a, &b) == 2) {
    plan->path = InPath::kGroup;
    plan->group = a;
    plan->nv = b;
    plan->threads = 256;
    plan->cluster = 1;
    return true;
  }
  if (std::sscanf(f, "resident:%d:%d:%d", &a, &b, &c) == 3) {
    plan->path = InPath::kResident;
    plan->threads = a;
    plan->nv = b;
    plan->cluster = c;
    return true;
  }
  int d = 0;
  if (std::sscanf(f, "split:%d:%d:%d:%d", &a, &b, &c, &d) == 4) {
    plan->path = InPath::kSplit;
    plan->threads = a;
    plan->nv = b;
    plan->ns = c;
    plan->cluster = d;
    return plan->vec;   // the split kernel has no element-wise form
  }
  if (std::sscanf(f, "stream:%d", &a) == 1) {
    plan->path = InPath::kStream;
    plan->threads = kStreamThreads;
    plan->nv = kStreamUnroll;
    if (const char* u = env("FNORM_STREAM_UNROLL"))
      plan->nv = std::atoi(u) == kStreamUnrollFew ? kStreamUnrollFew : kStreamUnroll;
    plan->cluster = a;
    return true;
  }
  return false;
}

// Chooses the kernel and launch shape for an InstanceNorm call.
fnorm_status in_make_plan(int tin, int tout, const void* x, const void* y, int64_t NC, int64_t S,
                          InPlan* out) {
  const int es_in = tin == 0 ? 4 : 2, es_out = tout == 0 ? 4 : 2;
  const int W = 16 / es_in;
  const size_t out_vec_bytes = static_cast<size_t>(W) * es_out;
  InPlan plan{};
  plan.vec = aligned(x, 16) && aligned(y, out_vec_bytes < 16 ? out_vec_bytes : 16) && S % W == 0 &&
             !env("FNORM_FORCE_SCALAR");
  const int64_t slots = (S + W - 1) / W;

  if (env("FNORM_FORCE_PATH")) {
    if (!in_forced_plan(&plan)) return FNORM_ERR_UNSUPPORTED;
    int64_t cap = 0;
    if (plan.path == InPath::kGroup) cap = int64_t(plan.group) * plan.nv;
    if (plan.path == InPath::kResident) cap = int64_t(plan.threads) * plan.nv * plan.cluster;
    if (plan.path == InPath::kSplit)
      cap = int64_t(plan.threads) * (plan.nv + plan.ns) * plan.cluster;
    if (plan.path == InPath::kStream) cap = slots;
    if (cap < slots || plan.cluster < 1 || plan.cluster > kMaxCluster) return FNORM_ERR_UNSUPPORTED;
  } else if (slots <= 256) {
    plan.path = InPath::kGroup;
    plan.threads = 256;
    plan.cluster = 1;
    for (const auto& g : kGroupShapes) {
      if (int64_t(g[0]) * g[1] >= slots) {
        plan.group = g[0];
        plan.nv = g[1];
        break;
      }
    }
  } else if (plan.vec && slots <= int64_t(kMaxCluster) * 8192) {
    // Split-resident. Up to 4096 slots (64 KiB of input) a CTA of 64..512
    // threads holds the slice in registers (8 slots per thread); up to 8192
    // slots a 512-thread CTA holds 8 slots per thread in registers and 8 in
    // TMA-staged shared memory (two CTAs per SM); up to 65536 slots clusters
    // of up to 16 such 256-thread CTAs (four per SM), beyond that clusters of
    // 512-thread CTAs. FNORM_SPLIT_SHAPE=threads:nr:ns overrides the CTA shape.
    plan.path = InPath::kSplit;
    plan.nv = 8;
    plan.ns = 0;
    plan.cluster = 1;
    if (slots <= 512) plan.threads = 64;
    else if (slots <= 1024) plan.threads = 128;
    else if (slots <= 2048) plan.threads = 256;
    else if (slots <= 4096) plan.threads = 512;
    else if (slots <= 8192) {
      plan.threads = 512;
      plan.ns = 8;
    } else if (slots <= 16 * 4096) {
      // 256-thread CTAs of 64 KiB in clusters of up to 16 (four CTAs per SM):
      // 2-4 % faster than 512-thread CTAs of 128 KiB in half the clusters
      plan.threads = 256;
      plan.ns = 8;
      plan.cluster = static_cast<int>((slots + 4095) / 4096);
    } else {
      plan.threads = 512;
      plan.ns = 8;
      plan.cluster = static_cast<int>((slots + 8191) / 8192);
    }
    int t = 0, nr = 0, ns = 0;
    const char* shape = env("FNORM_SPLIT_SHAPE");
    if (shape && std::sscanf(shape, "%d:%d:%d", &t, &nr, &ns) == 3) {
      plan.threads = t;
      plan.nv = nr;
      plan.ns = ns;
      const int64_t per = int64_t(t) * (nr + ns);
      plan.cluster = static_cast<int>((slots + per - 1) / per);
      if (plan.cluster > kMaxCluster) return FNORM_ERR_UNSUPPORTED;
    }
  } else if (slots <= int64_t(kMaxCluster) * 8192) {
    plan.path = InPath::kResident;
    if (slots <= 8192) {
      plan.cluster = 1;
      for (const auto& r : kResidentShapes) {
        if (int64_t(r[0]) * r[1] >= slots) {
          plan.threads = r[0];
          plan.nv = r[1];
          break;
        }
      }
    } else {
      // Wide slices: CTA shape (threads x 8 slots) and cluster size. The CTA
      // shape is tunable through FNORM_RESIDENT_THREADS (512 or 1024).
      const char* t = env("FNORM_RESIDENT_THREADS");
      plan.threads = (t && std::atoi(t) == 512) ? 512 : 1024;
      plan.nv = 8;
      const int64_t per = int64_t(plan.threads) * plan.nv;
      plan.cluster = static_cast<int>((slots + per - 1) / per);
      if (plan.cluster > kMaxCluster) {
        plan.threads = 1024;
        plan.cluster = static_cast<int>((slots + 8191) / 8192);
      }
    }
  } else {
    plan.path = InPath::kStream;
    plan.threads = kStreamThreads;
    // few slices: 16 CTAs per slice (non-portable clusters) when 8 would leave
    // most SMs idle, and more loads in flight per thread
    const bool few = NC * 8 < device_info().sm_count;
    // 8 loads of 16 bytes per thread for fp32 input or few slices; 4 for bf16
    // input with many slices (measured: the same ~32 values per thread)
    plan.nv = (few || tin == 0) ? kStreamUnrollFew : kStreamUnroll;
    plan.cluster = few ? 16 : 8;
    if (const char* u = env("FNORM_STREAM_UNROLL"))
      plan.nv = std::atoi(u) == kStreamUnrollFew ? kStreamUnrollFew : kStreamUnroll;
  }

  // bf16 slices spread over clusters of more than 8 CTAs (shapes with 8
  // register and 8 staged slots) and slices held by one 64-thread CTA (8
  // register slots) take the packed pair arithmetic; FNORM_NO_PACK=1 keeps the
  // scalar loops
  auto set_packed = [&] {
    const bool clustered = plan.cluster > 8 && plan.ns == 8 &&
                           (plan.threads == 256 || plan.threads == 512 || plan.threads == 1024);
    const bool small = plan.cluster == 1 && plan.ns == 0 && plan.threads == 64;
    plan.packed = plan.path == InPath::kSplit && tin == 1 && plan.nv == 8 && (clustered || small) &&
                  !env("FNORM_NO_PACK");
  };
  set_packed();
  int cap = in_capacity(tin, tout, plan);
  if (cap <= 0 && plan.path == InPath::kSplit && plan.cluster > 8 && !env("FNORM_FORCE_PATH") &&
      !env("FNORM_SPLIT_SHAPE")) {
    // 16-CTA clusters not available: twice the chunk per CTA, half the CTAs
    plan.threads *= 2;
    plan.cluster = static_cast<int>((slots + plan.threads * 16 - 1) / (plan.threads * 16));
    set_packed();
    cap = in_capacity(tin, tout, plan);
  }
  if (cap <= 0 && plan.path != InPath::kGroup && plan.cluster > 8 && !env("FNORM_FORCE_PATH")) {
    // 16-CTA clusters not available: stream the slice with a portable cluster.
    plan.path = InPath::kStream;
    plan.threads = kStreamThreads;
    plan.nv = kStreamUnroll;
    plan.cluster = 8;
    set_packed();
    cap = in_capacity(tin, tout, plan);
  }
  if (cap <= 0) return FNORM_ERR_UNSUPPORTED;

  if (plan.path == InPath::kGroup) {
    const int64_t per_block = int64_t(8) * (32 / plan.group);
    const int64_t need = (NC + per_block - 1) / per_block;
    plan.grid = static_cast<int>(need < cap ? need : cap);
  } else {
    const int64_t clusters = NC < cap ? NC : cap;
    plan.grid = static_cast<int>(clusters * plan.cluster);
  }
  if (env("FNORM_DEBUG_PLAN"))
    std::fprintf(stderr,
                 "fnorm_instancenorm plan: path=%d vec=%d threads=%d nv=%d ns=%d group=%d "
                 "cluster=%d packed=%d grid=%d capacity=%d NC=%lld S=%lld\n",
                 static_cast<int>(plan.path), plan.vec ? 1 : 0, plan.threads, plan.nv, plan.ns,
                 plan.group,
                 plan.cluster, plan.packed ? 1 : 0, plan.grid, cap, static_cast<long long>(NC),
                 static_cast<long long>(S));
  *out = plan;
  return FNORM_OK;
}

// ------------------------------------------------------------ Epilogue
struct EpiQuery {
  EpiPlan plan;
};
int epi_query(const void* arg) { return epi_max_active_clusters(static_cast<const EpiQuery*>(arg)->plan); }

int epi_capacity(const EpiPlan& plan) {
  char key[128];
  std::snprintf(key, sizeof key, "epi|%d|%d|%d|%d|%zu|%d|%d", static_cast<int>(plan.path),
                plan.threads, plan.cluster, plan.want_arg ? 1 : 0, plan.smem,
                plan.keep == kEpiKeepMax ? 1 : 0, plan.onepass ? 1 : 0);
  EpiQuery q{plan};
  return occupancy_cached(key, epi_query, &q);
}

// Range plans: a cluster of CTAs per sample, each CTA owning a range of
// positions of all C channels (the L2 form: statistics from HBM, outputs
// re-read from L2), 4-CTA clusters unless FNORM_EPI_CLUSTER forces a size;
// FNORM_EPI_STREAM forces the element-wise fallback.
fnorm_status epi_make_plan(const float* x, const float* y, const int64_t* argmax, int64_t N,
                           int64_t C, int64_t S, EpiPlan* out) {
  const DeviceInfo& di = device_info();
  const bool vec = aligned(x, 16) && aligned(y, 16) && (!argmax || aligned(argmax, 16)) &&
                   S % 4 == 0 && !env("FNORM_EPI_STREAM");
  const char* force_cl = env("FNORM_EPI_CLUSTER");
  EpiPlan plan{};
  plan.threads = kEpiThreads;
  bool have = false;
  if (vec && C <= 1024) {
    // The range decomposition: statistics from HBM, outputs re-read from L2
    // (4-CTA clusters keep every sample of the page's shape resident at once).
    const int cl = force_cl ? std::atoi(force_cl) : 4;
    const int64_t nv4 = S / 4;
    const int64_t per = (nv4 + cl - 1) / cl;
    const int cl_eff = static_cast<int>((nv4 + per - 1) / per);
    const int64_t fixed = static_cast<int64_t>(epi_range_l2_smem(C, cl_eff, 0));
    int keep = fixed < kEpiSmemBudget ? static_cast<int>((kEpiSmemBudget - fixed) / (C * 16)) : 0;
    if (keep > kEpiKeepMax) keep = kEpiKeepMax;
    if (keep > per) keep = static_cast<int>(per);
    if (const char* k = env("FNORM_EPI_KEEP")) keep = std::atoi(k) < keep ? std::atoi(k) : keep;
    if (keep < 0) keep = 0;
    EpiPlan cand{EpiPath::kRangeL2, kEpiThreads, cl_eff, per, argmax != nullptr,
                 epi_range_l2_smem(C, cl_eff, keep), 0, keep,
                 per <= kEpiOnePassMaxPer && !env("FNORM_EPI_TWOPASS")};
    if (cl >= 1 && cl <= kMaxCluster && epi_capacity(cand) > 0) {
      plan = cand;
      have = true;
    }
  }
  if (!have) {
    plan.path = EpiPath::kStream;
    plan.cluster = kEpiStreamCluster;
    plan.per = 0;
    plan.smem = epi_stream_smem(C, plan.cluster);
    if (plan.smem > static_cast<size_t>(di.max_smem_optin)) return FNORM_ERR_UNSUPPORTED;
  }
  const int cap = epi_capacity(plan);
  if (cap <= 0) return FNORM_ERR_UNSUPPORTED;
  const int64_t clusters = N < cap ? N : cap;
  plan.grid = static_cast<int>(clusters * plan.cluster);
  if (env("FNORM_DEBUG_PLAN"))
    std::fprintf(stderr,
                 "fnorm_instancenorm_epilogue plan: path=%d threads=%d cluster=%d per=%lld "
                 "keep=%d onepass=%d smem=%zu grid=%d capacity=%d\n",
                 static_cast<int>(plan.path), plan.threads, plan.cluster,
                 static_cast<long long>(plan.per), plan.keep, plan.onepass ? 1 : 0, plan.smem,
                 plan.grid, cap);
  *out = plan;
  return FNORM_OK;
}

// ------------------------------------------------------------ BatchNorm
struct BnLayout {
  int64_t chunk, chunks, P;
  size_t part_bytes;   // [C][P] float4 partials
  size_t col_part_bytes = 0;   // short runs: [C*S][row blocks] partials (coefficients follow)
  size_t ws_bytes;     // the larger layout + 256 bytes holding the resident kernel's barrier counter
};

size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

BnLayout bn_layout(int64_t N, int64_t C, int64_t S) {
  BnLayout l{};
  l.chunk = kBnChunk;
  l.chunks = S > 0 ? (S + l.chunk - 1) / l.chunk : 0;
  l.P = N * l.chunks;
  l.part_bytes = round256(static_cast<size_t>(C) * l.P * 16);
  l.ws_bytes = l.part_bytes + 256;
  if (S > 0 && S <= kBnColMaxS) {
    // column form: [C*S][row blocks] partials, then [C] coefficients
    const int64_t nrb = (N + kBnColRows - 1) / kBnColRows;
    l.col_part_bytes = round256(static_cast<size_t>(C) * S * nrb * 16);
    const size_t col_bytes = l.col_part_bytes + round256(static_cast<size_t>(C) * 16);
    if (col_bytes + 256 > l.ws_bytes) l.ws_bytes = col_bytes + 256;
  }
  return l;
}

}  // namespace

const DeviceInfo& device_info() {
  static DeviceInfo fallback{1, 48 * 1024, 0};
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return fallback;
  std::lock_guard<std::mutex> lk(g_mutex);
  if (!g_info_valid[d]) {
    DeviceInfo di{};
    cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, d);
    cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    cudaDeviceGetAttribute(&di.cluster_launch, cudaDevAttrClusterLaunch, d);
    cudaGetLastError();
    g_info[d] = di;
    g_info_valid[d] = true;
  }
  return g_info[d];
}

}  // namespace fnorm

namespace fnorm {
namespace {

// Shared validation of the BatchNorm entry points. `need_stats` >= 2: the
// count N*S must allow the unbiased estimate (single-process training).
fnorm_status bn_check(const float* x, const float* y, const float* gamma, const float* beta,
                      float scale, const float* running_mean, const float* running_var,
                      float momentum, float eps, const float* save_mean, const float* save_rstd,
                      int64_t N, int64_t C, int64_t S, int64_t* total) {
  if (N < 0 || C < 0 || S < 0) return FNORM_ERR_INVALID_ARG;
  if (!finite_nonneg(eps) || !std::isfinite(scale) || !std::isfinite(momentum))
    return FNORM_ERR_INVALID_ARG;
  if ((running_mean == nullptr) != (running_var == nullptr)) return FNORM_ERR_INVALID_ARG;
  int64_t NC = 0, NS = 0;
  if (!mul_ok(N, C, &NC) || !mul_ok(NC, S, total) || !mul_ok(N, S, &NS))
    return FNORM_ERR_INVALID_ARG;
  if (C > 65535) return FNORM_ERR_UNSUPPORTED;
  if ((gamma && !aligned(gamma, 4)) || (beta && !aligned(beta, 4)) ||
      (running_mean && !aligned(running_mean, 4)) || (running_var && !aligned(running_var, 4)) ||
      (save_mean && !aligned(save_mean, 4)) || (save_rstd && !aligned(save_rstd, 4)))
    return FNORM_ERR_ALIGNMENT;
  if (*total == 0) return FNORM_OK;
  if (!x || (y == nullptr && (gamma || beta))) return FNORM_ERR_INVALID_ARG;
  if (!aligned(x, 4) || (y && !aligned(y, 4))) return FNORM_ERR_ALIGNMENT;
  const size_t xb = static_cast<size_t>(*total) * 4, cb = static_cast<size_t>(C) * 4;
  if (y && x != y && overlaps(x, xb, y, xb)) return FNORM_ERR_INVALID_ARG;
  const void* outs[] = {running_mean, running_var, save_mean, save_rstd};
  for (const void* o : outs)
    if (overlaps(o, cb, x, xb) || (y && overlaps(o, cb, y, xb))) return FNORM_ERR_INVALID_ARG;
  return FNORM_OK;
}

void bn_fill(BnParams* p, const float* x, float* y, const float* gamma, const float* beta,
             float scale, float* running_mean, float* running_var, float momentum, float eps,
             float* save_mean, float* save_rstd, int64_t N, int64_t C, int64_t S, unsigned* err) {
  const BnLayout l = bn_layout(N, C, S);
  p->x = x;
  p->y = y;
  p->gamma = gamma;
  p->beta = beta;
  p->scale = scale;
  p->running_mean = running_mean;
  p->running_var = running_var;
  p->momentum = momentum;
  p->eps = eps;
  p->save_mean = save_mean;
  p->save_rstd = save_rstd;
  p->N = N;
  p->C = C;
  p->S = S;
  p->chunk = l.chunk;
  p->chunks = l.chunks;
  p->vec = aligned(x, 16) && (!y || aligned(y, 16)) && S % 4 == 0 && !env("FNORM_FORCE_SCALAR");
  const char* split = env("FNORM_BN_SPLIT");
  p->split = !(split && split[0] == '0');
  p->debug_timeout = force_timeout();
  p->err = err;
}

}  // namespace
}  // namespace fnorm

namespace fnorm {
namespace {

// Few fp32 slices too long for one cluster (the stream plan would keep most
// SMs idle): with a caller workspace, fnorm_instancenorm_ws runs them as a
// BatchNorm over the [1, N*C, S] view -- the per-(slice, 64 KiB chunk)
// statistics and apply launches spread every slice over all SMs; a slice's
// mean and rstd are the BatchNorm channel's saved statistics.
bool in_ws_shape(int64_t NC, int64_t S) {
  return S / 4 > int64_t(kMaxCluster) * 8192 && NC * 4 <= device_info().sm_count;
}

constexpr int64_t kInWsMergeFrom = 1024;   // chunks per slice (S >= 16 Mi values)

// Workspace of that route: the per-chunk partials, then one merged statistic
// per slice.
size_t in_ws_bytes(int64_t NC, int64_t S) {
  return bn_layout(1, NC, S).part_bytes + round256(static_cast<size_t>(NC) * 16);
}

// Validation and launch of the InstanceNorm entry points. `workspace` (may
// be null) is used only by the route above.
fnorm_status in_call(const char* name, const void* x, void* y, const float* gamma,
                     const float* beta, int64_t N, int64_t C, int64_t S, fnorm_dtype in_dtype,
                     fnorm_dtype out_dtype, float eps, float* mean_out, float* rstd_out,
                     void* workspace, size_t workspace_bytes, fnorm_stream_t stream) {
  if (N < 0 || C < 0 || S < 0) return FNORM_ERR_INVALID_ARG;
  if ((gamma && !aligned(gamma, 4)) || (beta && !aligned(beta, 4))) return FNORM_ERR_ALIGNMENT;
  if ((in_dtype != FNORM_F32 && in_dtype != FNORM_BF16) ||
      (out_dtype != FNORM_F32 && out_dtype != FNORM_BF16))
    return FNORM_ERR_INVALID_ARG;
  if (!finite_nonneg(eps)) return FNORM_ERR_INVALID_ARG;
  int64_t NC = 0, total = 0;
  if (!mul_ok(N, C, &NC) || !mul_ok(NC, S, &total)) return FNORM_ERR_INVALID_ARG;
  if (total == 0) return FNORM_OK;
  if (!x || !y) return FNORM_ERR_INVALID_ARG;
  const int tin = in_dtype == FNORM_F32 ? 0 : 1, tout = out_dtype == FNORM_F32 ? 0 : 1;
  const size_t es_in = tin == 0 ? 4 : 2, es_out = tout == 0 ? 4 : 2;
  if (!aligned(x, es_in) || !aligned(y, es_out) || (mean_out && !aligned(mean_out, 4)) ||
      (rstd_out && !aligned(rstd_out, 4)))
    return FNORM_ERR_ALIGNMENT;
  const size_t xb = static_cast<size_t>(total) * es_in, yb = static_cast<size_t>(total) * es_out;
  if (x != y && overlaps(x, xb, y, yb)) return FNORM_ERR_INVALID_ARG;
  if (x == y && es_in != es_out) return FNORM_ERR_INVALID_ARG;
  const size_t sb = static_cast<size_t>(NC) * 4;
  if (overlaps(mean_out, sb, x, xb) || overlaps(mean_out, sb, y, yb) ||
      overlaps(rstd_out, sb, x, xb) || overlaps(rstd_out, sb, y, yb) ||
      overlaps(mean_out, sb, rstd_out, sb))
    return FNORM_ERR_INVALID_ARG;
  const size_t cb = static_cast<size_t>(C) * 4;
  if (overlaps(gamma, cb, y, yb) || overlaps(beta, cb, y, yb) || overlaps(gamma, cb, mean_out, sb) ||
      overlaps(gamma, cb, rstd_out, sb) || overlaps(beta, cb, mean_out, sb) ||
      overlaps(beta, cb, rstd_out, sb))
    return FNORM_ERR_INVALID_ARG;

  const CallRange range(name);
  if (injected_launch_failure()) return FNORM_ERR_CUDA;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (workspace && tin == 0 && tout == 0 && in_ws_shape(NC, S) &&
      aligned(x, 16) && aligned(y, 16) && S % 4 == 0 && !env("FNORM_FORCE_PATH") &&
      !env("FNORM_FORCE_SCALAR")) {
    const BnLayout l = bn_layout(1, NC, S);
    const size_t wb = in_ws_bytes(NC, S);
    if (!aligned(workspace, 256)) return FNORM_ERR_ALIGNMENT;
    if (workspace_bytes < wb) return FNORM_ERR_INVALID_ARG;
    if (overlaps(workspace, wb, x, xb) || overlaps(workspace, wb, y, yb) ||
        overlaps(workspace, wb, mean_out, sb) || overlaps(workspace, wb, rstd_out, sb))
      return FNORM_ERR_INVALID_ARG;
    unsigned* err = err_word();
    if (!err) return FNORM_ERR_CUDA;
    BnParams p{};
    bn_fill(&p, static_cast<const float*>(x), static_cast<float*>(y), gamma, beta, 1.f,
            nullptr, nullptr, 0.f, eps, mean_out, rstd_out, 1, NC, S, err);
    p.affine_period = C;
    if (p.vec && p.split) {
      p.partials = static_cast<float4*>(workspace);
      p.stats = p.partials;
      p.stats_cstride = l.P;
      p.stats_istride = 1;
      p.stats_count = l.P;
      // up to kInWsMergeFrom chunks per slice, every apply CTA merges its
      // slice's partials (two launches); from there, one merge per slice
      // first (an extra launch, instead of each apply CTA reading thousands of
      // partials): measured [2,3,2048,2048] 256 chunks 3751 against 3527 GB/s,
      // [1,1,8192,8192] 4096 chunks 3157 against 3953 GB/s
      if (l.P < kInWsMergeFrom) return cuda_status(bn_launch(p, cs));
      p.local_out = reinterpret_cast<float4*>(static_cast<char*>(workspace) + l.part_bytes);
      cudaError_t e = bn_launch_local_stats(p, cs);
      if (e != cudaSuccess) return cuda_status(e);
      p.stats = p.local_out;
      p.stats_cstride = 1;
      p.stats_istride = NC;
      p.stats_count = 1;
      return cuda_status(bn_launch_apply(p, cs));
    }
  }

  // The same route without a workspace, for out-of-place calls: the output
  // buffer holds the per-unit statistics between the launches. Unit (q, k)
  // (slice q, 64 KiB chunk k) writes its partial into the first 16 bytes of
  // its own output range; one CTA per slice merges the slice's partials and
  // writes the result back into every one of those slots; the apply CTA of
  // each unit reads its own slot before it overwrites its range with outputs.
  // No CTA writes bytes another CTA still has to read.
  if (!workspace && tin == 0 && tout == 0 && x != y && in_ws_shape(NC, S) &&
      aligned(x, 16) && aligned(y, 16) && S % 4 == 0 && !env("FNORM_FORCE_PATH") &&
      !env("FNORM_FORCE_SCALAR")) {
    unsigned* err = err_word();
    if (!err) return FNORM_ERR_CUDA;
    BnParams p{};
    bn_fill(&p, static_cast<const float*>(x), static_cast<float*>(y), gamma, beta, 1.f,
            nullptr, nullptr, 0.f, eps, mean_out, rstd_out, 1, NC, S, err);
    p.affine_period = C;
    if (p.vec && p.split) {
      if (env("FNORM_DEBUG_PLAN"))
        std::fprintf(stderr, "fnorm_instancenorm plan: route=output_scratch NC=%lld S=%lld units=%lld\n",
                     static_cast<long long>(NC), static_cast<long long>(S),
                     static_cast<long long>(p.chunks));
      float4* slots = static_cast<float4*>(y);
      const int64_t slice4 = S / 4, unit4 = p.chunk / 4;
      p.partials = slots;
      p.part_cstride = slice4;
      p.part_kstride = unit4;
      p.stats = slots;
      p.stats_cstride = slice4;
      p.stats_istride = unit4;
      p.stats_count = p.chunks;
      p.local_out = slots;
      p.local_cstride = slice4;
      p.local_kstride = unit4;
      p.local_copies = p.chunks;
      cudaError_t e = bn_launch_local_stats(p, cs);
      if (e != cudaSuccess) return cuda_status(e);
      p.stats_istride = 0;
      p.stats_count = 1;
      p.stats_kstride = unit4;
      return cuda_status(bn_launch_apply(p, cs));
    }
  }

  InPlan plan;
  fnorm_status st = in_make_plan(tin, tout, x, y, NC, S, &plan);
  if (st != FNORM_OK) return st;
  unsigned* err = err_word();
  if (!err) return FNORM_ERR_CUDA;
  const InParams p{x,    y,     NC,   S, eps, mean_out, rstd_out, err, gamma, beta, C,
                   force_timeout()};
  return cuda_status(in_launch_dispatch(tin, tout, p, plan, cs));
}

}  // namespace
}  // namespace fnorm

using namespace fnorm;

extern "C" {

int fnorm_version(void) { return 100; }

void fnorm_tuning_reload(void) { load_knobs(); }

void fnorm_debug_force_timeout(int on) { g_force_timeout.store(on ? 1 : 0); }

void fnorm_debug_fail_launches(int n) { g_fail_launches.store(n > 0 ? n : 0); }

const char* fnorm_status_string(fnorm_status s) {
  switch (s) {
    case FNORM_OK: return "FNORM_OK";
    case FNORM_ERR_INVALID_ARG: return "FNORM_ERR_INVALID_ARG";
    case FNORM_ERR_UNSUPPORTED: return "FNORM_ERR_UNSUPPORTED";
    case FNORM_ERR_ALIGNMENT: return "FNORM_ERR_ALIGNMENT";
    case FNORM_ERR_CUDA: return "FNORM_ERR_CUDA";
    case FNORM_ERR_TIMEOUT: return "FNORM_ERR_TIMEOUT";
  }
  return "FNORM_ERR_UNKNOWN";
}

fnorm_status fnorm_get_last_error(void) {
  unsigned* w = err_word();
  if (!w) return FNORM_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return cuda_status(cudaErrorUnknown);
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fnorm_err_word, sizeof v) != cudaSuccess)
    return cuda_status(cudaErrorUnknown);
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_fnorm_err_word, &zero, sizeof zero) != cudaSuccess)
    return cuda_status(cudaErrorUnknown);
  return (v & kErrTimeout) ? FNORM_ERR_TIMEOUT : FNORM_OK;
}

fnorm_status fnorm_instancenorm_affine(const void* x, void* y, const float* gamma,
                                       const float* beta, int64_t N, int64_t C, int64_t S,
                                       fnorm_dtype in_dtype, fnorm_dtype out_dtype, float eps,
                                       float* mean_out, float* rstd_out, fnorm_stream_t stream) {
  return in_call("fnorm_instancenorm_affine", x, y, gamma, beta, N, C, S, in_dtype, out_dtype, eps,
                 mean_out, rstd_out, nullptr, 0, stream);
}

fnorm_status fnorm_instancenorm(const void* x, void* y, int64_t N, int64_t C, int64_t S,
                                fnorm_dtype in_dtype, fnorm_dtype out_dtype, float eps,
                                float* mean_out, float* rstd_out, fnorm_stream_t stream) {
  return in_call("fnorm_instancenorm", x, y, nullptr, nullptr, N, C, S, in_dtype, out_dtype, eps,
                 mean_out, rstd_out, nullptr, 0, stream);
}

size_t fnorm_instancenorm_workspace_size(int64_t N, int64_t C, int64_t S) {
  int64_t NC = 0, total = 0;
  if (N <= 0 || C <= 0 || S <= 0 || !mul_ok(N, C, &NC) || !mul_ok(NC, S, &total)) return 0;
  if (!in_ws_shape(NC, S)) return 0;
  return in_ws_bytes(NC, S);
}

fnorm_status fnorm_instancenorm_ws(const void* x, void* y, int64_t N, int64_t C, int64_t S,
                                   fnorm_dtype in_dtype, fnorm_dtype out_dtype, float eps,
                                   float* mean_out, float* rstd_out, void* workspace,
                                   size_t workspace_bytes, fnorm_stream_t stream) {
  return in_call("fnorm_instancenorm_ws", x, y, nullptr, nullptr, N, C, S, in_dtype, out_dtype,
                 eps, mean_out, rstd_out, workspace, workspace_bytes, stream);
}

fnorm_status fnorm_instancenorm_epilogue(const float* x, const float* m, float* y, int64_t* argmax,
                                         int64_t N, int64_t C, int64_t S, float eps,
                                         float clamp_lo, float clamp_hi, fnorm_stream_t stream) {
  if (N < 0 || C < 0 || S < 0) return FNORM_ERR_INVALID_ARG;
  if (!finite_nonneg(eps) || std::isnan(clamp_lo) || std::isnan(clamp_hi) || !(clamp_lo <= clamp_hi))
    return FNORM_ERR_INVALID_ARG;
  int64_t NS = 0, NC = 0, total = 0;
  if (!mul_ok(N, S, &NS) || !mul_ok(N, C, &NC) || !mul_ok(NC, S, &total))
    return FNORM_ERR_INVALID_ARG;
  if (NS == 0) return FNORM_OK;
  if (C == 0) return FNORM_ERR_INVALID_ARG;   // a max over no channels is undefined
  if (C > kEpiMaxChannels) return FNORM_ERR_UNSUPPORTED;
  if (!x || !m || !y) return FNORM_ERR_INVALID_ARG;
  if (!aligned(x, 4) || !aligned(m, 4) || !aligned(y, 4) || (argmax && !aligned(argmax, 8)))
    return FNORM_ERR_ALIGNMENT;
  const size_t xb = static_cast<size_t>(total) * 4, yb = static_cast<size_t>(NS) * 4,
               ab = argmax ? static_cast<size_t>(NS) * 8 : 0, mb = static_cast<size_t>(C) * 4;
  if (overlaps(y, yb, x, xb) || overlaps(y, yb, m, mb) || overlaps(argmax, ab, x, xb) ||
      overlaps(argmax, ab, m, mb) || overlaps(argmax, ab, y, yb))
    return FNORM_ERR_INVALID_ARG;

  const CallRange range("fnorm_instancenorm_epilogue");
  if (injected_launch_failure()) return FNORM_ERR_CUDA;
  EpiPlan plan;
  fnorm_status st = epi_make_plan(x, y, argmax, N, C, S, &plan);
  if (st != FNORM_OK) return st;
  unsigned* err = err_word();
  if (!err) return FNORM_ERR_CUDA;
  EpiParams p{};
  p.x = x;
  p.m = m;
  p.y = y;
  p.argmax = argmax;
  p.N = N;
  p.C = C;
  p.S = S;
  p.eps = eps;
  p.lo = clamp_lo;
  p.hi = clamp_hi;
  p.per = plan.per;
  p.debug_timeout = force_timeout();
  p.keep = plan.keep;
  p.err = err;
  return cuda_status(epi_launch(p, plan, reinterpret_cast<cudaStream_t>(stream)));
}

size_t fnorm_batchnorm_workspace_size(int64_t N, int64_t C, int64_t S) {
  if (N <= 0 || C <= 0 || S <= 0) return 0;
  int64_t t1 = 0, t2 = 0;
  if (!mul_ok(N, C, &t1) || !mul_ok(t1, S, &t2)) return 0;
  const BnLayout l = bn_layout(N, C, S);
  return l.ws_bytes;
}


}  // extern "C"

namespace fnorm {

// Every argument check of fnorm_batchnorm_train except those of the workspace
// (shared with fnorm_batchnorm_train_noalloc, which validates identically
// before looking at its scratch size). *total = N*C*S; total == 0 with FNORM_OK
// is a no-op.
fnorm_status bn_train_check(const float* x, const float* y, const float* gamma,
                            const float* beta, float scale, const float* running_mean,
                            const float* running_var, float momentum, float eps,
                            const float* save_mean, const float* save_rstd, int64_t N, int64_t C,
                            int64_t S, int64_t* total) {
  fnorm_status st = bn_check(x, y, gamma, beta, scale, running_mean, running_var, momentum, eps,
                             save_mean, save_rstd, N, C, S, total);
  if (st != FNORM_OK || *total == 0) return st;
  if (N * S < 2) return FNORM_ERR_INVALID_ARG;   // the unbiased estimate needs two values
  if (!y) return FNORM_ERR_INVALID_ARG;
  if (bn_layout(N, C, S).P > 0x7fffffffLL) return FNORM_ERR_UNSUPPORTED;
  return FNORM_OK;
}

}  // namespace fnorm

extern "C" {

fnorm_status fnorm_batchnorm_train(const float* x, float* y, const float* gamma, const float* beta,
                                   float scale, float* running_mean, float* running_var,
                                   float momentum, float eps, float* save_mean, float* save_rstd,
                                   int64_t N, int64_t C, int64_t S, void* workspace,
                                   size_t workspace_bytes, fnorm_stream_t stream) {
  int64_t total = 0;
  fnorm_status st = bn_train_check(x, y, gamma, beta, scale, running_mean, running_var, momentum,
                                   eps, save_mean, save_rstd, N, C, S, &total);
  if (st != FNORM_OK || total == 0) return st;
  if (!workspace) return FNORM_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return FNORM_ERR_ALIGNMENT;
  const BnLayout l = bn_layout(N, C, S);
  if (workspace_bytes < l.ws_bytes) return FNORM_ERR_INVALID_ARG;
  const size_t xb = static_cast<size_t>(total) * 4, cb = static_cast<size_t>(C) * 4,
               wb = l.ws_bytes;
  const void* outs[] = {running_mean, running_var, save_mean, save_rstd};
  for (const void* o : outs)
    if (overlaps(o, cb, workspace, wb)) return FNORM_ERR_INVALID_ARG;
  if (overlaps(workspace, wb, x, xb) || overlaps(workspace, wb, y, xb)) return FNORM_ERR_INVALID_ARG;

  const CallRange range("fnorm_batchnorm_train");
  if (injected_launch_failure()) return FNORM_ERR_CUDA;
  unsigned* err = err_word();
  if (!err) return FNORM_ERR_CUDA;
  BnParams p{};
  bn_fill(&p, x, y, gamma, beta, scale, running_mean, running_var, momentum, eps, save_mean,
          save_rstd, N, C, S, err);
  p.partials = static_cast<float4*>(workspace);
  p.stats = p.partials;
  p.stats_cstride = l.P;
  p.stats_istride = 1;
  p.stats_count = l.P;
  p.grid_counter = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + l.ws_bytes - 256);
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (l.col_part_bytes > 0 && !env("FNORM_BN_NO_COLUMNS")) {
    p.local_out = reinterpret_cast<float4*>(static_cast<char*>(workspace) + l.col_part_bytes);
    return cuda_status(bn_launch_columns(p, cs));
  }
  if (p.vec && p.split && env("FNORM_BN_RESIDENT")) {
    const cudaError_t e = bn_launch_resident(p, cs);
    if (e != cudaErrorCooperativeLaunchTooLarge) return cuda_status(e);
    cudaGetLastError();   // grid not co-resident here: the two-launch form
  }
  return cuda_status(bn_launch(p, cs));
}

fnorm_status fnorm_batchnorm_eval(const float* x, float* y, const float* gamma, const float* beta,
                                  float scale, const float* running_mean,
                                  const float* running_var, float eps, int64_t N, int64_t C,
                                  int64_t S, fnorm_stream_t stream) {
  if (!running_mean || !running_var) return FNORM_ERR_INVALID_ARG;
  int64_t total = 0;
  fnorm_status st = bn_check(x, y, gamma, beta, scale, running_mean, running_var, 0.f, eps,
                             nullptr, nullptr, N, C, S, &total);
  if (st != FNORM_OK || total == 0) return st;
  if (!y) return FNORM_ERR_INVALID_ARG;
  const BnLayout l = bn_layout(N, C, S);
  if (S >= kBnEvalFlatBelow && l.P > 0x7fffffffLL) return FNORM_ERR_UNSUPPORTED;
  const CallRange range("fnorm_batchnorm_eval");
  if (injected_launch_failure()) return FNORM_ERR_CUDA;
  unsigned* err = err_word();
  if (!err) return FNORM_ERR_CUDA;
  BnParams p{};
  bn_fill(&p, x, y, gamma, beta, scale, const_cast<float*>(running_mean),
          const_cast<float*>(running_var), 0.f, eps, nullptr, nullptr, N, C, S, err);
  return cuda_status(bn_launch_eval(p, reinterpret_cast<cudaStream_t>(stream)));
}

fnorm_status fnorm_batchnorm_local_stats(const float* x, float* stats_out, int64_t N, int64_t C,
                                         int64_t S, void* workspace, size_t workspace_bytes,
                                         fnorm_stream_t stream) {
  int64_t total = 0;
  fnorm_status st = bn_check(x, nullptr, nullptr, nullptr, 1.f, nullptr, nullptr, 0.f, 0.f,
                             nullptr, nullptr, N, C, S, &total);
  if (N < 0 || C < 0 || S < 0) return FNORM_ERR_INVALID_ARG;
  if (C == 0) return FNORM_OK;
  if (!stats_out) return FNORM_ERR_INVALID_ARG;
  if (!aligned(stats_out, 16)) return FNORM_ERR_ALIGNMENT;
  if (total == 0) {   // an empty shard contributes the merge identity
    if (st != FNORM_OK) return st;
    return cuda_status(cudaMemsetAsync(stats_out, 0, static_cast<size_t>(C) * 16,
                                       reinterpret_cast<cudaStream_t>(stream)));
  }
  if (st != FNORM_OK) return st;
  if (!workspace) return FNORM_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return FNORM_ERR_ALIGNMENT;
  const BnLayout l = bn_layout(N, C, S);
  if (l.P > 0x7fffffffLL) return FNORM_ERR_UNSUPPORTED;
  if (workspace_bytes < l.ws_bytes) return FNORM_ERR_INVALID_ARG;
  const size_t xb = static_cast<size_t>(total) * 4, sb = static_cast<size_t>(C) * 16;
  if (overlaps(stats_out, sb, x, xb) || overlaps(stats_out, sb, workspace, l.ws_bytes) ||
      overlaps(workspace, l.ws_bytes, x, xb))
    return FNORM_ERR_INVALID_ARG;
  const CallRange range("fnorm_batchnorm_local_stats");
  if (injected_launch_failure()) return FNORM_ERR_CUDA;
  unsigned* err = err_word();
  if (!err) return FNORM_ERR_CUDA;
  BnParams p{};
  bn_fill(&p, x, nullptr, nullptr, nullptr, 1.f, nullptr, nullptr, 0.f, 0.f, nullptr, nullptr, N, C,
          S, err);
  p.partials = static_cast<float4*>(workspace);
  p.stats = p.partials;
  p.stats_cstride = l.P;
  p.stats_istride = 1;
  p.stats_count = l.P;
  p.local_out = reinterpret_cast<float4*>(stats_out);
  if (l.col_part_bytes > 0 && !env("FNORM_BN_NO_COLUMNS"))
    return cuda_status(bn_launch_columns_local_stats(p, reinterpret_cast<cudaStream_t>(stream)));
  return cuda_status(bn_launch_local_stats(p, reinterpret_cast<cudaStream_t>(stream)));
}

fnorm_status fnorm_batchnorm_apply_stats(const float* x, float* y, const float* stats_all,
                                         int64_t R, const float* gamma, const float* beta,
                                         float scale, float* running_mean, float* running_var,
                                         float momentum, float eps, float* save_mean,
                                         float* save_rstd, int64_t N, int64_t C, int64_t S,
                                         fnorm_stream_t stream) {
  int64_t total = 0;
  fnorm_status st = bn_check(x, y, gamma, beta, scale, running_mean, running_var, momentum, eps,
                             save_mean, save_rstd, N, C, S, &total);
  if (st != FNORM_OK) return st;
  if (R < 1 || R > 65536) return FNORM_ERR_INVALID_ARG;
  // An empty shard still applies the gathered statistics to the running and
  // saved statistics (every rank of the group updates them alike).
  const bool stats_only = total == 0 && C > 0 && S >= 0 &&
                          (running_mean || save_mean || save_rstd);
  if (total == 0 && !stats_only) return FNORM_OK;
  if ((!y && !stats_only) || !stats_all) return FNORM_ERR_INVALID_ARG;
  if (!aligned(stats_all, 16)) return FNORM_ERR_ALIGNMENT;
  int64_t RC = 0;
  if (!mul_ok(R, C, &RC)) return FNORM_ERR_INVALID_ARG;
  const size_t xb = static_cast<size_t>(total) * 4, sb = static_cast<size_t>(RC) * 16;
  if (overlaps(stats_all, sb, y, xb)) return FNORM_ERR_INVALID_ARG;
  const CallRange range("fnorm_batchnorm_apply_stats");
  if (injected_launch_failure()) return FNORM_ERR_CUDA;
  unsigned* err = err_word();
  if (!err) return FNORM_ERR_CUDA;
  BnParams p{};
  bn_fill(&p, x, y, gamma, beta, scale, running_mean, running_var, momentum, eps, save_mean,
          save_rstd, stats_only ? 0 : N, C, S, err);
  if (stats_only) p.chunks = 1;
  p.stats = reinterpret_cast<const float4*>(stats_all);
  p.stats_cstride = 1;
  p.stats_istride = C;
  p.stats_count = R;
  if (!stats_only && S <= kBnColMaxS && !env("FNORM_BN_NO_COLUMNS"))
    return cuda_status(bn_launch_columns_apply_stats(p, reinterpret_cast<cudaStream_t>(stream)));
  return cuda_status(bn_launch_apply(p, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
