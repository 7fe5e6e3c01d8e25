// static_ws.cu -- dsa_indexer_static: the fused paged indexer for callers that
// cannot give the library any device memory to work in.
//
// Some callers cannot allocate: plugin hosts that pass the library only its input
// and output tensors, and serving loops that reserve nearly all device memory up
// front and forbid allocation during a step (cudaMalloc / cudaFree may synchronise
// the device and stall every stream).  For them this entry point runs exactly the
// kernels of dsa_indexer, with their scratch -- work-list counters, work items and
// the fp32 score rows -- in one library-owned device array of
// DSA_STATIC_WORKSPACE_BYTES, which every GPU that loads this code holds until the
// process exits.
//
// In host code the array's name only stands for it: the device address is looked
// up per device, with that device current, by the first call made on it (and by
// later calls for as long as that lookup has not succeeded).
#include <mutex>

#include "dsa_indexer.h"

namespace {

constexpr size_t kStaticBytes = DSA_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 128;

// The scratch itself.  Calls share it and it keeps the last call's contents.  The
// work-list counters, the only part that must start at zero, are reset by every
// call: zeroed on the stream before the score kernel, or, for balanced per-CTA work
// lists (decode shapes), written in full (every CTA's count) by the list-building
// kernel.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

// Per device: the array's device address once a lookup has succeeded.  A failed
// lookup is not kept, so an error that an earlier, unrelated asynchronous launch left
// behind does not disable the entry point for the rest of the process.
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) == cudaSuccess) g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" dsa_status dsa_indexer_static(const dsa_indexer_args* args, dsa_stream_t stream) {
  if (!args) return DSA_ERR_INVALID_ARGUMENT;
  dsa_indexer_args a = *args;
  a.workspace = nullptr;
  a.workspace_bytes = 0;
  size_t need = 0;
  dsa_status st = dsa_indexer_workspace_size(&a, &need);
  if (st != DSA_OK) return st;
  if (need > kStaticBytes) return DSA_ERR_WORKSPACE;  // larger than the built-in scratch
  void* p = scratch_on_current_device();
  if (!p) return DSA_ERR_CUDA;
  a.workspace = p;
  a.workspace_bytes = kStaticBytes;
  return dsa_indexer(&a, stream);
}
