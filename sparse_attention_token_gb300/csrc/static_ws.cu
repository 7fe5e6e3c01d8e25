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
// up once per device, with that device current, by the first call made on it.
#include <mutex>

#include "dsa_indexer.h"

namespace {

constexpr size_t kStaticBytes = DSA_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 128;

// The scratch itself.  Calls share it and it keeps the last call's contents; the
// work-list counters, the only part that must start at zero, are cleared by every
// call (dsa_indexer zeroes them on the stream before its first kernel).
static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

struct DeviceScratch {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
DeviceScratch g_scratch[kMaxDevices];

// Device address of the scratch array on the current device (set up once per device).
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceScratch& s = g_scratch[dev];
  std::call_once(s.once, [&s]() {
    void* p = nullptr;
    s.err = cudaGetSymbolAddress(&p, g_static_scratch);
    s.ptr = s.err == cudaSuccess ? p : nullptr;
  });
  return s.err == cudaSuccess ? s.ptr : nullptr;
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
