// mla_noalloc.cu — paged MLA decode for callers that cannot allocate device
// memory.
//
// mla_decode_paged and mla_combine_splits need scratch memory from the
// caller: a workspace (the split plan and a status word) and the per-split
// partial outputs.  Some callers have no way to provide it: an inference
// engine whose memory planner hands out every byte of the GPU before the
// first request, a plugin that runs inside a host program that owns all
// allocations, or a decode loop being recorded into a CUDA graph, where a
// cudaMalloc would break the capture.  mla_decode_attend_noalloc serves them:
// it takes only the inputs and the outputs, and carves every scratch buffer
// out of one fixed-size array that the library reserves on each GPU when it
// is loaded (and keeps until the process exits).
//
// The array is shared by every call on a device and keeps what the last call
// left in it; each call rewrites the parts it reads (the status word is
// cleared first).  Calls whose execution overlaps on the GPU — on two streams
// without ordering between them, or from two host threads — race on it.
#include <cstring>
#include <mutex>

#include "mla_internal.h"

namespace mla {
namespace {

// Upper bound on the scratch of one call: the split plan, the status word
// and the partial outputs (slots * Lq*H rows of 512 fp32 plus one fp32 lse),
// where slots = B + (number of SM clusters) - 1.
constexpr size_t kNoAllocScratchBytes = 32u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of the scratch array for the current device.  Looked up once
// per device (host code cannot use the symbol itself: on the host it names a
// stand-in object, not device memory).
// Devices past the cache are looked up on every call (as the decode's
// launch cache does).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return MLA_ERR_CUDA;
  if (dev >= kMaxDevices) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MLA_ERR_CUDA;
    *out = p;
    return MLA_OK;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_decode_attend_noalloc(const mla_dims* d, const void* q_cat, const void* kv_cache,
                                         const int32_t* block_table, const int32_t* seq_lens,
                                         void* o_lat, float* lse, int* device_status, void* stream) {
  if (!d) return MLA_ERR_INVALID_ARG;
  if (!q_cat || !kv_cache || !block_table || !seq_lens || !o_lat) return MLA_ERR_INVALID_ARG;
  // the same dims rules as mla_decode_paged (checked by asking it for a
  // workspace size, which validates and allocates nothing)
  size_t ws_bytes = 0;
  int rc = mla_decode_workspace_size(d, &ws_bytes);
  if (rc != MLA_OK) return rc;
  if ((reinterpret_cast<uintptr_t>(q_cat) | reinterpret_cast<uintptr_t>(kv_cache) |
       reinterpret_cast<uintptr_t>(o_lat)) & 15u)
    return MLA_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(block_table) | reinterpret_cast<uintptr_t>(seq_lens) |
       reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(device_status)) & 3u)
    return MLA_ERR_MISALIGNED;
  int slots = 0;
  if ((rc = mla_decode_num_slots(d, &slots)) != MLA_OK) return rc;
  const size_t rows = (size_t)d->Lq * d->H;
  const size_t lse_bytes = align256((size_t)slots * rows * sizeof(float));
  const size_t part_bytes = (size_t)slots * rows * kDc * sizeof(float);
  const size_t need = align256(ws_bytes) + lse_bytes + part_bytes;
  if (need > kNoAllocScratchBytes) return MLA_ERR_WORKSPACE;  // beyond the fixed scratch

  void* base = nullptr;
  if ((rc = scratch_address(&base)) != MLA_OK) return rc;
  unsigned char* p = static_cast<unsigned char*>(base);
  void* ws = p;
  float* lse_part = reinterpret_cast<float*>(p + align256(ws_bytes));
  float* o_part = reinterpret_cast<float*>(p + align256(ws_bytes) + lse_bytes);
  auto st = static_cast<cudaStream_t>(stream);

  // the status word must start at zero for this call's errors to be its own
  if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return MLA_ERR_CUDA;
  if ((rc = mla_decode_paged(d, q_cat, kv_cache, block_table, seq_lens, 0, o_part, lse_part, ws,
                             ws_bytes, stream)) != MLA_OK)
    return rc;
  if ((rc = mla_combine_splits(d, o_part, lse_part, ws, ws_bytes, o_lat, lse, stream)) != MLA_OK)
    return rc;
  if (device_status &&
      cudaMemcpyAsync(device_status, ws, sizeof(int), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}
