// tq_decode_attention_noalloc: decode attention for callers that cannot
// allocate device memory.
//
// Some hosts of this library cannot call cudaMalloc at all: code running
// inside a CUDA-graph capture that must not allocate, embedded runtimes whose
// memory is fixed at start-up, and plugins of inference servers whose
// allocator belongs to the host process.  They can still pass their own
// input and output buffers, but not the scratch workspace that
// tq_decode_attention needs.  This entry point takes that workspace from one
// fixed device array, g_noalloc_scratch, compiled into the library.
//
// The array is TQ_NOALLOC_SCRATCH_BYTES long and lives on every GPU that
// loads the library until the process exits.  Host code cannot pass the
// array's name to a kernel (on the host it is only a stand-in symbol), so the
// first call on each device looks up its device address with
// cudaGetSymbolAddress while that device is current, and later calls reuse
// the cached address.  Every call shares the one array and the array keeps
// the previous call's contents; the decode kernels overwrite every scratch
// word they read before reading it, so nothing has to be cleared between
// calls.  Calls whose GPU work overlaps (different streams, no ordering) race
// on the array.
#include <mutex>

#include "tq_internal.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[TQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once).
tq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return TQ_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TQ_OK;
}

}  // namespace

extern "C" tq_status tq_decode_attention_noalloc(const tq_plan* plan, const void* q, tq_dtype q_dtype, int B, int Hq,
                                                 int Hkv, const tq_records* K, const tq_records* V,
                                                 const int32_t* ctx_len, int64_t ctx_stride, float scale, float* out,
                                                 tq_stream stream) {
  size_t need = 0;
  tq_status st = tq_decode_workspace_size(plan, B, Hq, Hkv, ctx_stride, &need);
  if (st != TQ_OK) return st;
  if (need > TQ_NOALLOC_SCRATCH_BYTES) return TQ_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != TQ_OK) return st;
  return tq_decode_attention(plan, q, q_dtype, B, Hq, Hkv, K, V, ctx_len, ctx_stride, scale, out, scratch,
                             TQ_NOALLOC_SCRATCH_BYTES, stream);
}
