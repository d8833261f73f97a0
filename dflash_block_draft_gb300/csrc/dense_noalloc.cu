// dense_noalloc.cu -- the dense entry point without a caller-supplied workspace.
//
// Some callers cannot hand the library a workspace: runtimes that plan all
// device memory once at start-up and forbid allocations while serving, or
// plugin interfaces whose fixed signature has no place for a scratch buffer.
// dflash_attn_dense_noalloc serves them by keeping the only scratch the dense
// path needs -- one tile-class byte per 128x128 tile of the mask -- in a
// file-scope device array of fixed size instead.  It calls no cudaMalloc,
// cudaFree or other allocating routine.
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace dflash {

// Scratch for the mask scan's tile classes.  Every GPU that loads the library
// holds these bytes until the process exits.
// Laid out like the dense workspace: 256 control bytes, then the class bytes.
static __device__ __align__(256) uint8_t g_noalloc_classes[DFLASH_NOALLOC_MAX_TILES + 256];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<uint8_t*> g_noalloc_ptr[kMaxDevices];

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
uint8_t* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  uint8_t* ptr = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_classes) != cudaSuccess || !addr) return nullptr;
    ptr = static_cast<uint8_t*>(addr);
    g_noalloc_ptr[dev].store(ptr, std::memory_order_release);
  }
  return ptr;
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" dflash_status_t dflash_attn_dense_noalloc(const dflash_dims_t* dims, dflash_dtype_t dtype,
                                                     const void* q, const void* k_nope, const void* k_rope,
                                                     const void* v, const void* mask, void* out, float* lse,
                                                     dflash_stream_t stream) {
  if (!dims) return DFLASH_ERR_INVALID;
  if (dims->B < 0 || dims->S < 0 || dims->Q < 0) return DFLASH_ERR_SHAPE;
  const long long nqt = ((long long)dims->Q + kTileM - 1) / kTileM;
  const long long nkt = ((long long)dims->S + dims->Q + kTileN - 1) / kTileN;
  if ((long long)dims->B * nqt * nkt > DFLASH_NOALLOC_MAX_TILES) return DFLASH_ERR_WORKSPACE;
  if (dims->B == 0 || dims->Q == 0) return DFLASH_OK;
  uint8_t* scratch = scratch_address();
  if (!scratch) return DFLASH_ERR_CUDA;
  // The mask scan overwrites every class byte this call reads, so nothing in
  // the shared array needs clearing first.
  return dflash_attn_dense(dims, dtype, q, k_nope, k_rope, v, mask, out, lse, scratch,
                           (size_t)DFLASH_NOALLOC_MAX_TILES + 256, stream);
}
