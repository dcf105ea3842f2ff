// ssm_linscan_fwd_noalloc: the scalar selective scan for callers that cannot allocate device
// memory.  The workspace the scan needs (a status/claim-counter header plus one 16-byte
// look-back descriptor per 4096-element tile) lives in a fixed array in device memory that
// is part of this library, so the call needs neither a caller-supplied workspace nor any
// allocation.  It launches exactly the kernel ssm_linscan_fwd launches.
#include <cstddef>

#include "ssm_internal.cuh"

namespace ssm {
namespace {

// Largest scan this entry point accepts: rows * len <= 2^26 elements (16384 tiles).
constexpr int64_t kNoAllocMaxElems = int64_t(1) << 26;
constexpr size_t kNoAllocScratchBytes = 256 + (size_t)(kNoAllocMaxElems / kLsTile) * sizeof(LsDesc);

// Every GPU that loads the library holds this array until the process exits.  All calls share
// it; it keeps the previous call's contents.
static __device__ __align__(256) unsigned char g_linscan_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device.  In host code the array's name is
// only a host-side stand-in, not a device address, so the address is looked up with the device
// current; it is looked up on every call (cheap once the library's module is loaded), so that it
// stays right after a cudaDeviceReset, which loads the module again, possibly elsewhere.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_linscan_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace ssm

using namespace ssm;

extern "C" ssm_status ssm_linscan_fwd_noalloc(const float* a, const float* b, float* h, int64_t rows, int64_t len,
                                              ssm_stream_t stream) {
  if (rows < 0 || len < 0) return SSM_ERR_INVALID_ARG;
  if (rows == 0 || len == 0) return SSM_OK;
  if (!a || !b || !h) return SSM_ERR_INVALID_ARG;
  if (len > kNoAllocMaxElems || rows > kNoAllocMaxElems / len) return SSM_ERR_UNSUPPORTED;  // above the fixed size
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) | reinterpret_cast<uintptr_t>(h)) % 16)
    return SSM_ERR_ALIGNMENT;
  const int64_t n = rows * len;
  const LinscanWorkspace layout = linscan_workspace_layout(n, nullptr);
  if (layout.total_bytes > kNoAllocScratchBytes) return SSM_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return SSM_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The status word and claim counters must start at zero.  The flag epoch after them is left
  // alone: each launch advances it, so descriptors an earlier call left are ignored.
  if (cudaMemsetAsync(scratch, 0, offsetof(WsHeader, epoch), s) != cudaSuccess) return SSM_ERR_CUDA;
  const LinscanWorkspace ws = linscan_workspace_layout(n, scratch);
  if (launch_linscan(a, b, h, rows, len, ws, next_lookback_ctl(), s) != cudaSuccess) return SSM_ERR_CUDA;
  return SSM_OK;
}
