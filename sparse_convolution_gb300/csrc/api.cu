// Host-side runtime of the fvx C ABI: error reporting, the allocator hook,
// launch accounting and kernel timing, the device status word, handle views
// and destruction.  [DriveRT, "Inspection and debugging": errors name the
// failing item; "Measurement and reproducibility": kernel launches reported]
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "fvx_internal.cuh"
#include "../../include/fvx_testing.h"

namespace fvx {

static thread_local std::string g_last_error;

void set_error(const char* fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

fvx_status cuda_fail(cudaError_t e, const char* what, const char* file, int line) {
  const char* base = strrchr(file, '/');
  set_error("%s failed: %s (%s:%d)", what, cudaGetErrorString(e), base ? base + 1 : file, line);
  return FVX_ERR_CUDA;
}

// ---------------------------------------------------------------- allocator
static fvx_alloc_fn g_alloc = nullptr;
static fvx_free_fn g_free = nullptr;
static void* g_alloc_ctx = nullptr;

// The library's own stream-ordered pool per device.  Its release threshold is
// unbounded, so memory freed by one call is reused by the next instead of
// being returned to the driver at every synchronisation (the default pool's
// behaviour), without changing any pool the rest of the process uses.
static cudaMemPool_t library_pool() {
  static cudaMemPool_t pools[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!pools[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t p = nullptr;
    if (cudaMemPoolCreate(&p, &props) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    uint64_t thr = ~0ull;
    cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &thr);
    pools[dev] = p;
  }
  return pools[dev];
}

thread_local const char* t_entry = nullptr;

void* dalloc(size_t bytes, cudaStream_t s) {
  if (bytes == 0) bytes = 256;
  void* p = nullptr;
  if (g_alloc) {
    p = g_alloc(bytes, (fvx_stream)s, g_alloc_ctx);
  } else {
    cudaMemPool_t pool = library_pool();
    cudaError_t e = pool ? cudaMallocFromPoolAsync(&p, bytes, pool, s) : cudaMallocAsync(&p, bytes, s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      p = nullptr;
    }
  }
  if (!p) set_error("%s: device allocation of %zu bytes failed", t_entry ? t_entry : "fvx", bytes);
  return p;
}

void dfree(void* p, cudaStream_t s) {
  if (!p) return;
  if (g_free) g_free(p, (fvx_stream)s, g_alloc_ctx);
  else cudaFreeAsync(p, s);
}

void* pinned_staging(size_t bytes) {
  static thread_local void* buf = nullptr;
  static thread_local size_t cap = 0;
  if (bytes > cap) {
    if (buf) cudaFreeHost(buf);
    cap = bytes < 4096 ? 4096 : bytes;
    if (cudaMallocHost(&buf, cap) != cudaSuccess) {
      cudaGetLastError();
      buf = nullptr;
      cap = 0;
    }
  }
  return buf;
}

// ---------------------------------------------------------------- launches / profiling
static std::atomic<uint64_t> g_launches{0};
static std::mutex g_prof_mu;
static std::string g_prof_name;
static bool g_prof_on = false;
struct EvPair {
  cudaEvent_t a, b;
};
static std::vector<EvPair> g_prof_events;

LaunchScope::LaunchScope(const char* n, cudaStream_t s) : name(n), stream(s), ev0(nullptr) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_prof_on) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof_on && g_prof_name == name) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) == cudaSuccess) {
        cudaEventRecord(e, stream);
        ev0 = (void*)e;
      }
    }
  }
}

LaunchScope::~LaunchScope() {
  if (!ev0) return;
  cudaEvent_t e1;
  if (cudaEventCreate(&e1) == cudaSuccess) {
    cudaEventRecord(e1, stream);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_events.push_back(EvPair{(cudaEvent_t)ev0, e1});
  } else {
    cudaEventDestroy((cudaEvent_t)ev0);
  }
}

// After a sync: a nonzero status word (staged to the host with the sync's
// other values) means a bounded device-side wait gave up during the call.
fvx_status check_staged_status(const char* who, uint32_t staged, cudaStream_t s) {
  if (staged == 0u) return FVX_OK;
  uint32_t* w = device_status_word();
  if (w) cudaMemsetAsync(w, 0, 4, s);
  set_error("%s: a bounded device-side wait gave up in this or an earlier unchecked call (device status %u)", who,
            staged);
  return staged == DEV_TIMEOUT ? FVX_ERR_DEVICE_TIMEOUT : FVX_ERR_CHECK;
}

fvx_status device_sm_count(int* sms) {
  static int counts[64] = {0};
  int dev = 0;
  FVX_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) {
    set_error("device ordinal %d out of range", dev);
    return FVX_ERR_RANGE;
  }
  if (counts[dev] == 0) {
    int n = 0;
    FVX_CUDA(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev));
    counts[dev] = n;
  }
  *sms = counts[dev];
  return FVX_OK;
}

fvx_status check_launch(const char* name) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("launch of kernel %s failed: %s", name, cudaGetErrorString(e));
    return FVX_ERR_CUDA;
  }
  return FVX_OK;
}

// ---------------------------------------------------------------- device status word
uint32_t* device_status_word() {
  static uint32_t* words[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!words[dev]) {
    void* p = nullptr;
    if (cudaMalloc(&p, 256) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    cudaMemset(p, 0, 256);
    words[dev] = (uint32_t*)p;
  }
  return words[dev];
}

}  // namespace fvx

using namespace fvx;

extern "C" {

fvx_status fvx_set_allocator(fvx_alloc_fn alloc, fvx_free_fn free_fn, void* ctx) {
  if ((alloc == nullptr) != (free_fn == nullptr)) {
    set_error("fvx_set_allocator: alloc and free must both be set or both be NULL");
    return FVX_ERR_INVALID_ARG;
  }
  g_alloc = alloc;
  g_free = free_fn;
  g_alloc_ctx = ctx;
  return FVX_OK;
}

const char* fvx_status_string(fvx_status st) {
  switch (st) {
    case FVX_OK: return "FVX_OK";
    case FVX_ERR_INVALID_ARG: return "FVX_ERR_INVALID_ARG";
    case FVX_ERR_RANGE: return "FVX_ERR_RANGE";
    case FVX_ERR_CAPACITY: return "FVX_ERR_CAPACITY";
    case FVX_ERR_ALLOC: return "FVX_ERR_ALLOC";
    case FVX_ERR_CUDA: return "FVX_ERR_CUDA";
    case FVX_ERR_DEVICE_TIMEOUT: return "FVX_ERR_DEVICE_TIMEOUT";
    case FVX_ERR_CHECK: return "FVX_ERR_CHECK";
  }
  return "FVX_STATUS_UNKNOWN";
}

const char* fvx_last_error(void) { return g_last_error.c_str(); }

uint64_t fvx_launch_count(void) { return g_launches.load(); }

fvx_status fvx_profile_enable(const char* kernel_name) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& p : g_prof_events) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  g_prof_events.clear();
  if (kernel_name) {
    g_prof_name = kernel_name;
    g_prof_on = true;
  } else {
    g_prof_name.clear();
    g_prof_on = false;
  }
  return FVX_OK;
}

fvx_status fvx_profile_read(double* total_ms, int64_t* launches) {
  if (!total_ms || !launches) {
    set_error("fvx_profile_read: NULL output");
    return FVX_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lk(g_prof_mu);
  double tot = 0;
  for (auto& p : g_prof_events) {
    FVX_CUDA(cudaEventSynchronize(p.b));
    float ms = 0;
    FVX_CUDA(cudaEventElapsedTime(&ms, p.a, p.b));
    tot += ms;
  }
  *total_ms = tot;
  *launches = (int64_t)g_prof_events.size();
  return FVX_OK;
}

fvx_status fvx_profile_read_each(double* ms_each, int64_t cap, int64_t* launches) {
  if (!launches || cap < 0 || (cap > 0 && !ms_each)) {
    set_error("fvx_profile_read_each: NULL output or negative cap");
    return FVX_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lk(g_prof_mu);
  int64_t i = 0;
  for (auto& p : g_prof_events) {
    if (i < cap) {
      FVX_CUDA(cudaEventSynchronize(p.b));
      float ms = 0;
      FVX_CUDA(cudaEventElapsedTime(&ms, p.a, p.b));
      ms_each[i] = ms;
    }
    ++i;
  }
  *launches = (int64_t)g_prof_events.size();
  return FVX_OK;
}

fvx_status fvx_testing_bounded_wait(int32_t kind, uint64_t limit_ns, fvx_stream stream) {
  if ((kind != 0 && kind != 1) || limit_ns < 1000ull || limit_ns > 2000000000ull) {
    set_error("fvx_testing_bounded_wait: kind must be 0 or 1 and 1 us <= limit_ns <= 2 s (got %d, %llu)", kind,
              (unsigned long long)limit_ns);
    return FVX_ERR_INVALID_ARG;
  }
  uint32_t* w = device_status_word();
  if (!w) {
    set_error("fvx_testing_bounded_wait: could not set up the device status word");
    return FVX_ERR_CUDA;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (kind == 0) return testing_mbar_wait(limit_ns, w, s);
  // a word of the status block that is zeroed when the block is set up and
  // never written: a published flag that nothing sets
  return testing_flag_wait(reinterpret_cast<const uint64_t*>(w + 16), limit_ns, w, s);
}

fvx_status fvx_device_status(fvx_stream stream) {
  uint32_t* w = device_status_word();
  if (!w) {
    set_error("fvx_device_status: could not set up the device status word");
    return FVX_ERR_CUDA;
  }
  uint32_t h = 0;
  FVX_CUDA(cudaMemcpyAsync(&h, w, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream));
  FVX_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  FVX_CUDA(cudaMemsetAsync(w, 0, 4, (cudaStream_t)stream));
  FVX_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  if (h == DEV_TIMEOUT) {
    set_error("a bounded device-side wait gave up (device status word)");
    return FVX_ERR_DEVICE_TIMEOUT;
  }
  if (h != DEV_OK) {
    set_error("a device-side check failed (code %u)", h);
    return FVX_ERR_CHECK;
  }
  return FVX_OK;
}

fvx_status fvx_grid_counts(fvx_grid g, int64_t* n_upper, int64_t* n_lower, int64_t* n_leaf, int64_t* n_active) {
  if (!g) {
    set_error("fvx_grid_counts: NULL grid");
    return FVX_ERR_INVALID_ARG;
  }
  if (n_upper) *n_upper = g->n_upper;
  if (n_lower) *n_lower = g->n_lower;
  if (n_leaf) *n_leaf = g->n_leaf;
  if (n_active) *n_active = g->n_active;
  return FVX_OK;
}

fvx_status fvx_grid_view(fvx_grid g, fvx_grid_view_t* v) {
  if (!g || !v) {
    set_error("fvx_grid_view: NULL argument");
    return FVX_ERR_INVALID_ARG;
  }
  v->batch_size = g->B;
  v->n_rows = g->n_rows;
  v->n_upper = g->n_upper;
  v->n_lower = g->n_lower;
  v->n_leaf = g->n_leaf;
  v->n_active = g->n_active;
  v->ijk = g->ijk;
  v->row_to_index = g->row_to_index;
  v->voxel_batch_offsets = g->voxel_batch_offsets;
  v->leaf_origin = g->leaf_origin;
  v->leaf_batch = g->leaf_batch;
  v->leaf_records = g->leaf_rec;
  v->lower_origin = g->lower_origin;
  v->lower_batch = g->lower_batch;
  v->lower_mask = g->lower_mask;
  v->lower_prefix = g->lower_prefix;
  v->lower_first = g->lower_first;
  v->upper_origin = g->upper_origin;
  v->upper_batch = g->upper_batch;
  v->upper_mask = g->upper_mask;
  v->upper_prefix = g->upper_prefix;
  v->upper_first = g->upper_first;
  return FVX_OK;
}

fvx_status fvx_grid_batch_offsets(fvx_grid g, int64_t* host_out) {
  if (!g || !host_out) {
    set_error("fvx_grid_batch_offsets: NULL argument");
    return FVX_ERR_INVALID_ARG;
  }
  if (g->host_batch_offsets.empty()) {
    g->host_batch_offsets.resize((size_t)g->B + 1);
    FVX_CUDA(cudaMemcpyAsync(g->host_batch_offsets.data(), g->voxel_batch_offsets, sizeof(int64_t) * (g->B + 1),
                             cudaMemcpyDeviceToHost, g->stream));
    FVX_CUDA(cudaStreamSynchronize(g->stream));
  }
  memcpy(host_out, g->host_batch_offsets.data(), sizeof(int64_t) * (g->B + 1));
  return FVX_OK;
}

fvx_status fvx_kmap_view(fvx_kmap m, const int64_t** offsets_host, const int32_t** in_idx, const int32_t** out_idx,
                         const uint32_t** out_mask, int64_t* n_pairs, int64_t* n_out) {
  if (!m) {
    set_error("fvx_kmap_view: NULL kernel map");
    return FVX_ERR_INVALID_ARG;
  }
  if (offsets_host || n_pairs) FVX_TRY(kmap_read_totals(m, "fvx_kmap_view"));
  if (offsets_host) *offsets_host = m->offsets_host;
  if (in_idx) *in_idx = m->in_idx;
  if (out_idx) *out_idx = m->out_idx;
  if (out_mask) *out_mask = m->out_mask;
  if (n_pairs) *n_pairs = m->n_pairs;
  if (n_out) *n_out = m->n_out;
  return FVX_OK;
}

fvx_status fvx_grid_destroy(fvx_grid g) {
  if (!g) return FVX_OK;
  dfree(g->block, g->stream);
  delete g;
  return FVX_OK;
}

fvx_status fvx_kmap_destroy(fvx_kmap m) {
  if (!m) return FVX_OK;
  dfree(m->block, m->stream);
  dfree(m->block2, m->stream);
  delete m;
  return FVX_OK;
}

}  // extern "C"
