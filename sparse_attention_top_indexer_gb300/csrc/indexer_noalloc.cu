// indexer_forward_noalloc: the whole indexer forward without a caller-provided
// workspace.
//
// Why it exists: some callers cannot allocate device memory when they call the
// indexer. Examples are a plugin whose host runtime owns all of the device's memory
// and hands out no scratch, and a server that fixes its memory budget at start-up and
// forbids allocation afterwards. indexer_forward needs a workspace from its caller;
// this entry point takes the same inputs and outputs but uses a fixed scratch array
// that lives in the library's own device memory instead.
//
// The scratch is a file-scope __device__ array of INDEXER_NOALLOC_SCRATCH_BYTES. Every
// GPU that loads this library holds that much memory until the process exits. Its
// device address is looked up once per device, on the first call made while that
// device is current, and kept for the life of the process (a cudaDeviceReset unloads the
// module that holds the array, so this entry point must not be used on a device after a
// reset). All calls share the one array, so calls that overlap on the GPU (different
// streams, or different host threads, without ordering between them) race on it and
// must not be issued. The array keeps what the last call left in it; each call that
// passes its argument checks clears the status word at its start, and every other byte
// it reads was written earlier in the same call. indexer_noalloc_status reads and clears
// that status word, so a caller can learn that a bounded device wait ran out.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/indexer.h"
#include "launch.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[INDEXER_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

int report(int code, const char* fmt, const char* what) {
  char msg[256];
  snprintf(msg, sizeof(msg), fmt, what);
  return indexer::set_last_error(code, msg);
}

// Device address of the scratch array on the current device (looked up once per device,
// with that device current). The host-side name of the array is not a device address.
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report(INDEXER_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return report(INDEXER_ERR_RANGE, "%s", "device index beyond 64");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return report(INDEXER_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return INDEXER_OK;
}

}  // namespace

extern "C" int indexer_forward_noalloc(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int B,
                                       int S, int start_pos, const float* rope_cs, int max_pos,
                                       const uint8_t* k_cache, int T_cap, const int32_t* cand_in,
                                       int32_t* cand_out, int32_t* topk_out, float* scores_out,
                                       indexer_stream_t stream) {
  const size_t need = indexer_workspace_size(dims, B, S, start_pos);
  if (need > (size_t)INDEXER_NOALLOC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "indexer_forward_noalloc: these sizes need %zu bytes of scratch; its static scratch holds %d "
             "bytes (use indexer_forward with a caller workspace)",
             need, INDEXER_NOALLOC_SCRATCH_BYTES);
    return indexer::set_last_error(INDEXER_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc != INDEXER_OK) return rc;
  // every argument check of the forward (including dims for which need == 0) runs before
  // anything is enqueued, so a rejected call leaves the shared array untouched
  rc = indexer::check_forward_args(dims, q, w, B, S, start_pos, rope_cs, max_pos, k_cache, T_cap, cand_in, cand_out,
                                   topk_out, scores_out, scratch, (size_t)INDEXER_NOALLOC_SCRATCH_BYTES);
  if (rc != INDEXER_OK) return rc;
  // the status word must start at zero; kernels only OR bits into it
  const cudaError_t e = cudaMemsetAsync(scratch, 0, INDEXER_STATUS_BYTES, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return report(INDEXER_ERR_CUDA, "clearing the static scratch status word: %s", cudaGetErrorString(e));
  return indexer_forward(dims, q, w, B, S, start_pos, rope_cs, max_pos, k_cache, T_cap, cand_in, cand_out,
                         topk_out, scores_out, scratch, (size_t)INDEXER_NOALLOC_SCRATCH_BYTES, stream);
}

// The status word of the last indexer_forward_noalloc call on the current device: waits for
// `stream`, reads the word from the static array, clears it and returns INDEXER_OK, or the
// error indexer_status would give for the same bits. Allocates nothing.
extern "C" int indexer_noalloc_status(indexer_stream_t stream) {
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != INDEXER_OK) return rc;
  return indexer_status(scratch, stream);
}
