// permute_noalloc.cu -- moe_permute_noalloc: the expert grouping of
// moe_permute with its scratch held in a fixed device array of this library,
// so the caller passes only inputs and outputs and nothing is allocated.
//
// Who needs it: code that is handed only input and output buffers by a host
// framework -- for example a plugin or custom-operator interface that has no
// workspace argument -- and is not allowed to call cudaMalloc itself, because
// that framework owns all device memory or forbids allocations while a step
// is running.  Such a caller cannot provide the workspace moe_permute needs.
//
// The scratch is kNoAllocScratchInts int32 (512 KiB): two tables of
// [chunk][expert] counts, chunk = kPermuteChunk (256) assignments.  Every GPU
// that loads the library holds this array until the process exits.
#include <mutex>

#include "internal.h"

namespace moe {

// Per table: up to 65536 (chunk, expert) entries, i.e. ceil(T*K / 256) * n <= 65536
// (for n = 8 experts: T*K up to 2,097,152 assignments).
constexpr int kNoAllocTableInts = 65536;
constexpr int kNoAllocScratchInts = 2 * kNoAllocTableInts;

static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
int32_t* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_permute_scratch on the current device.  The host-side
// name of a __device__ array is only a stand-in, never a device address, so
// the address is looked up once per device, with that device current.
cudaError_t scratch_on_current_device(int32_t** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status moe_permute_noalloc(const moe_shape* shape, const moe_bf16* x,
                                                  const int32_t* ids, int32_t* offsets,
                                                  int32_t* perm_src, int32_t* slot_row,
                                                  moe_bf16* x_perm, void* stream) {
  if (shape == nullptr) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (offsets == nullptr || !aligned16(offsets)) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 &&
      (x == nullptr || ids == nullptr || perm_src == nullptr || slot_row == nullptr ||
       x_perm == nullptr || !aligned16(x) || !aligned16(ids) || !aligned16(perm_src) ||
       !aligned16(slot_row) || !aligned16(x_perm)))
    return MOE_ERR_INVALID_ARG;
  const int64_t R = (int64_t)shape->T * shape->top_k;
  const int64_t nchunks = (R + kPermuteChunk - 1) / kPermuteChunk;
  if (nchunks * shape->n_experts > kNoAllocTableInts) return MOE_ERR_WORKSPACE_TOO_SMALL;
  int32_t* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  // Both tables are fully overwritten (histogram, then chunk bases) before
  // they are read, so nothing left by an earlier call needs clearing.
  const cudaError_t e =
      launch_permute(*shape, x, ids, nullptr, offsets, scratch, scratch + kNoAllocTableInts,
                     perm_src, slot_row, x_perm, (int)nchunks, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
