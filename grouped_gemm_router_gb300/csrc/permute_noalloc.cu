// moe_permute_noalloc: the stable expert permutation for callers that cannot
// allocate device memory.
//
// moe_permute needs a scratch buffer for its per-block expert histogram, and
// the caller has to provide it.  Some callers cannot: code running inside a
// host framework that owns all device memory and gives its plugins no
// allocator, or a latency-critical path that must never call cudaMalloc
// (which can synchronise the device and can fail at run time).  This entry
// point takes the same inputs and outputs as moe_permute, but its scratch is
// a fixed array in the library's own device memory, so it allocates nothing.
//
// Properties of the shared scratch array:
//  * Size: kNoAllocHistEntries int32 (256 KB).  Every GPU that loads the
//    library holds it until the process exits.  A call needs ceil(T / TB) * E
//    entries, TB = moe_route_block_tokens(T) on the current device (16, 32 or
//    64 tokens); calls needing more than the array holds are rejected with
//    MOE_ERR_UNSUPPORTED_SHAPE.
//  * Every call on a device shares the one array, and it keeps the previous
//    call's contents.  Nothing in it has to start at zero: the histogram
//    kernel writes every entry the call reads.  Calls whose work overlaps on
//    the GPU (different streams, or different host threads) race on the
//    array and give wrong results; serialise them.
//  * The first call on each device resolves the array's device address with
//    cudaGetSymbolAddress while that device is current.  Make that first call
//    before any stream capture.
#include <mutex>

#include "moe_kernels.cuh"

namespace moe {
namespace {

constexpr size_t kNoAllocHistEntries = 64 * 1024;

// In host code `g_noalloc_hist` names a host-side stand-in, not device memory:
// only the address returned by cudaGetSymbolAddress may be given to a kernel.
static __device__ __align__(256) int32_t g_noalloc_hist[kNoAllocHistEntries];

constexpr int kMaxDevices = 64;
int32_t* g_hist_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set-up on the
// first call per device).
std::mutex g_scratch_mu;

cudaError_t scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_hist_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_hist);
    if (e != cudaSuccess) return e;
    g_hist_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_hist_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_permute_noalloc(const int32_t* ids, moe_dims d, int32_t* counts,
                                          int32_t* offsets, int32_t* perm, int32_t* inv,
                                          const void* x, void* x_sorted, void* stream) {
  const moe_status st = check_dims(d);  // the same shape limits as moe_permute
  if (st != MOE_OK) return st;
  if (!ids || !counts || !offsets || !perm || !inv) return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_sorted == nullptr)) return MOE_ERR_INVALID_ARG;
  if (x && ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(x_sorted)) & 15u))
    return MOE_ERR_INVALID_ARG;
  const size_t need = static_cast<size_t>(route_blocks(d.T)) * d.E;
  if (need > kNoAllocHistEntries) return MOE_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d.T == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * d.E, s) != cudaSuccess) return MOE_ERR_CUDA;
    return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d.E + 1), s) == cudaSuccess ? MOE_OK
                                                                                       : MOE_ERR_CUDA;
  }
  int32_t* hist = nullptr;
  if (scratch_address(&hist) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_hist(ids, d, hist, s) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_scatter(ids, hist, d, counts, offsets, perm, inv, static_cast<const uint16_t*>(x),
                                    static_cast<uint16_t*>(x_sorted), s));
}
