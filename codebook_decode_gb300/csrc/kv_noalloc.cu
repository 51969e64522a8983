// kv_noalloc.cu -- qtts_kv_write_noalloc: the KV-cache write of
// qtts_kv_write without any device allocation.
//
// qtts_kv_write stages K/V and the page list in buffers it cudaMallocs and
// cudaFrees on every call, and cudaFree waits for the whole device. A serving
// loop that places a new session's prompt KV while other sessions' frames run
// on another stream cannot pay for that wait, and code that runs under a
// framework-owned memory pool, or inside a region where the CUDA allocator may
// not be called, cannot allocate at all. This variant stages through a fixed
// array in the library's own static device memory instead, and orders its
// work on the caller's stream only.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "qtts_internal.h"

namespace {

// Largest K+V payload one call can stage: 4 MiB (K then V). At the 1.7B
// Talker's 8 kv heads x 128 dims that is 1024 tokens of one layer.
constexpr size_t kStageBytes = size_t(4) << 20;
constexpr int kStagePages = 1024;
constexpr int kMaxDevices = 64;

// Every GPU that loads the library holds these until the process exits.
static __device__ __align__(256) unsigned char g_kv_stage[kStageBytes];
static __device__ __align__(256) int32_t g_kv_stage_pages[kStagePages];

std::mutex g_mu;
bool g_ready[kMaxDevices];
void* g_stage_addr[kMaxDevices];
void* g_pages_addr[kMaxDevices];

// Device addresses of the static arrays for the current device (looked up once
// per device; the host-side names are only stand-ins for them).
int stage_addresses(int dev, void** stage, void** pages) {
  if (dev < 0 || dev >= kMaxDevices) return QTTS_E_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ready[dev]) {
    void* s = nullptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&s, g_kv_stage) != cudaSuccess) return QTTS_E_CUDA;
    if (cudaGetSymbolAddress(&p, g_kv_stage_pages) != cudaSuccess) return QTTS_E_CUDA;
    g_stage_addr[dev] = s;
    g_pages_addr[dev] = p;
    g_ready[dev] = true;
  }
  *stage = g_stage_addr[dev];
  *pages = g_pages_addr[dev];
  return QTTS_OK;
}

}  // namespace

extern "C" int qtts_kv_write_noalloc(qtts_model* m, int layer, int n_tok, const int32_t* pages_host,
                                     const uint16_t* k, const uint16_t* v, void* stream) {
  using namespace qtts;
  if (!m) return QTTS_E_INVALID;
  KvLayout L{};
  model_kv_layout(m, &L);
  if (layer < 0 || layer >= L.n_layers || n_tok < 0) return model_fail(m, QTTS_E_INVALID, "bad layer or token count");
  if (n_tok == 0) return QTTS_OK;
  if (!pages_host || !k || !v) return model_fail(m, QTTS_E_INVALID, "null argument");
  const size_t elems = (size_t)n_tok * L.nkv * L.d;
  const int np = (n_tok + kPage - 1) / kPage;
  if (elems * 2 * sizeof(uint16_t) > kStageBytes || np > kStagePages) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "qtts_kv_write_noalloc: %d tokens need %zu bytes of staging, the static buffer holds %zu; "
             "write fewer tokens per call",
             n_tok, elems * 2 * sizeof(uint16_t), kStageBytes);
    return model_fail(m, QTTS_E_INVALID, msg);
  }
  for (int i = 0; i < np; ++i)
    if (pages_host[i] < 0 || pages_host[i] >= L.pool_pages)
      return model_fail(m, QTTS_E_POOL, "qtts_kv_write_noalloc: page id outside the pool");
  int prev_dev = -1;
  if (cudaGetDevice(&prev_dev) != cudaSuccess) prev_dev = -1;
  if (cudaSetDevice(L.device) != cudaSuccess) return model_fail(m, QTTS_E_CUDA, "cudaSetDevice failed");
  // the caller's current device is put back on every path out
  struct Restore {
    int dev, model_dev;
    ~Restore() {
      if (dev >= 0 && dev != model_dev) cudaSetDevice(dev);
    }
  } restore{prev_dev, L.device};
  void* stage = nullptr;
  void* pages = nullptr;
  const int rc = stage_addresses(L.device, &stage, &pages);
  if (rc) return model_fail(m, rc, "qtts_kv_write_noalloc: cudaGetSymbolAddress failed");
  cudaStream_t s = (cudaStream_t)stream;
  uint16_t* kst = (uint16_t*)stage;
  uint16_t* vst = kst + elems;
  // every staged byte the scatter reads is written here first, so nothing
  // needs clearing between calls
  cudaError_t e = cudaMemcpyAsync(pages, pages_host, np * sizeof(int32_t), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(kst, k, elems * sizeof(uint16_t), cudaMemcpyDefault, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(vst, v, elems * sizeof(uint16_t), cudaMemcpyDefault, s);
  if (e == cudaSuccess)
    e = launch_kv_scatter(L.pool, L.pool_pages, L.nkv, L.d, layer, n_tok, (const int32_t*)pages, kst, vst, 1, s);
  if (e != cudaSuccess) return model_fail(m, QTTS_E_CUDA, cudaGetErrorString(e));
  return QTTS_OK;
}
