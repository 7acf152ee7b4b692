// libmoe C ABI: status strings, workspace query, status word, launch counter.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "router_bwd.cuh"

namespace moe {

static std::atomic<uint64_t> g_launches{0};

void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { (void)cudaGetLastError(); return 0; }
  return dev;
}

int sm_count() {
  static int cache[64] = {0};
  int dev = current_device();
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = 1;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace moe

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null/misaligned pointer or bad size";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: sizes outside what the kernels handle";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace null or too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or launch failed";
    default: return "unknown libmoe status";
  }
}

int moe_version(void) { return 100; }

uint64_t moe_launch_count(void) { return moe::g_launches.load(std::memory_order_relaxed); }

size_t moe_workspace_size(int T, int E, int k, int d, int h) {
  if (T < 0 || E <= 0 || k <= 0 || d <= 0) return 0;
  const size_t a = moe::workspace_bytes(T, E, k, d);
  const size_t b = moe::router_topk_scratch((long long)T * k, E, d).end;
  size_t r = a > b ? a : b;
  if (h > 0 && d % 128 == 0 && h % 128 == 0) {       // the MXFP8 forward's scale atoms
    const size_t c = moe::mx_scratch_end((long long)T * k, E, d, h);
    r = r > c ? r : c;
  }
  return r;
}

int moe_reset_status(void* ws, moe_stream_t stream) {
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), (cudaStream_t)stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int moe_get_status(const void* ws, int32_t* host_status, moe_stream_t stream) {
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  if (host_status == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(host_status, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // extern "C"
