// moe_expert_ffn_noalloc: the grouped expert FFN with its scratch in a fixed, file-scope
// device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocator) at the point where
// they run the layer -- for example a plugin or custom operator inside a host framework
// that owns all device memory and hands its plugins no workspace, or a serving loop where
// allocation is forbidden after start-up because cudaMalloc may synchronise the device and
// stall every stream.  They still pass their own inputs and outputs.
//
// The scratch (the hidden activations H [S_max, f]) is one static __device__ array of
// kNoAllocScratchBytes.  Every GPU that loads this code keeps it until the process exits.
// All calls share it and it keeps the last call's contents, so calls that overlap on the GPU
// (different streams, or different host threads, without ordering between them) race on it;
// calls on one stream are ordered and safe.  H needs no clearing: every row that is read is
// written first by the same call.  There is no status word: the kernels' bounded waits still
// give up and return, but a timeout is not recorded anywhere the caller could read it.
#include <mutex>

#include "../../include/moe.h"
#include "launch.h"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;   // 64 MiB per device

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array for the current device, looked up once per device (with that
// device current) and kept for the life of the process.  The first call on a device does this
// set-up; make that first call outside any stream capture.  A device reset
// (cudaDeviceReset, or anything else that destroys the primary context) invalidates the kept
// address: do not call the entry point on that device after one.
uint8_t* scratch_address(cudaError_t* err) {
  static std::mutex mu;
  static uint8_t* addr[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<uint8_t*>(p);
  }
  return addr[dev];
}

}  // namespace

// Defined in api.cu: the shared implementation of moe_expert_ffn on a given scratch area.
moe_status expert_ffn_on_scratch(const void* tokens, const int32_t* perm, const int32_t* offsets,
                                 const void* W1, const void* W2, moe_dtype dtype, int T, int d,
                                 int f, int E, int S_max, void* expert_out, uint8_t* scratch,
                                 int* status, cudaStream_t s);
moe_status expert_ffn_check(const void* tokens, const int32_t* perm, const int32_t* offsets,
                            const void* W1, const void* W2, moe_dtype dtype, int T, int d, int f,
                            int E, int S_max, const void* expert_out);

}  // namespace moe

extern "C" moe_status moe_expert_ffn_noalloc(const void* tokens, const int32_t* perm,
                                             const int32_t* offsets, const void* W1,
                                             const void* W2, moe_dtype dtype, int T, int d, int f,
                                             int E, int S_max, void* expert_out,
                                             moe_stream_t stream) {
  using namespace moe;
  moe_status st = expert_ffn_check(tokens, perm, offsets, W1, W2, dtype, T, d, f, E, S_max,
                                   expert_out);
  if (st != MOE_OK) return st;
  if (T == 0 || S_max == 0) return MOE_OK;
  const size_t elt = dtype == MOE_F16 ? 2 : 4;
  if ((size_t)S_max * f * elt > kNoAllocScratchBytes)
    return MOE_ERR_WORKSPACE;                       // beyond the fixed scratch: rejected
  cudaError_t err;
  uint8_t* scratch = scratch_address(&err);
  if (!scratch) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // no status word: bounded waits still give up and return, but their MOE_ERR_TIMEOUT is
  // not recorded
  return expert_ffn_on_scratch(tokens, perm, offsets, W1, W2, dtype, T, d, f, E, S_max,
                               expert_out, scratch, nullptr, s);
}
