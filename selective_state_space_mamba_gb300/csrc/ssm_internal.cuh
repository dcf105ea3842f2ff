// Internal declarations shared by the CUDA sources of the library (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ssm.h"

namespace ssm {

// ---------------------------------------------------------------------------------------
// Device status word: the first 8 bytes of every workspace.  High 32 bits hold the epoch
// of the call that failed, low 32 bits the ssm_status code.  Kernels treat a word whose
// epoch matches their own call as "abort all waits"; the host clears it in
// ssm_check_device_status().
// ---------------------------------------------------------------------------------------
struct WsHeader {
  unsigned long long status;  // (epoch << 32) | code
  uint32_t counter;           // look-back tile claim counter
  uint32_t done;              // tiles finished (the last one resets both counters)
};
constexpr size_t kHeaderBytes = 256;

// Look-back fault injection and wait limit (test hook), passed by value to each kernel.
struct LookbackCtl {
  uint32_t epoch;         // 30-bit call tag, never 0
  int64_t stall_tile;     // claim index that never publishes (-1: none)
  uint64_t spin_limit_ns; // per-wait limit
};
LookbackCtl next_lookback_ctl();

// Flag words carry the epoch so that flags left by earlier calls never look valid, and a
// fixed bit pattern so that stale non-flag data left in the workspace by a call of another
// size cannot pass for a flag: flag = (epoch << 32) | kFlagMagic | kind.
constexpr uint32_t kFlagAggregate = 1;  // tile aggregate published
constexpr uint32_t kFlagPrefix = 2;     // inclusive prefix published
constexpr uint32_t kFlagMagic = 0xA5A5A500u;
__host__ __device__ __forceinline__ unsigned long long make_flag(uint32_t epoch, uint32_t kind) {
  return ((unsigned long long)epoch << 32) | (kFlagMagic | kind);
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_relaxed_f2(const float2* p) {
  float2 v;
  asm volatile("ld.relaxed.gpu.global.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_relaxed_f4(const float4* p) {
  float4 v;
  asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Record a device error for this call (first writer wins) in the status word.
__device__ __forceinline__ void record_error(WsHeader* hdr, uint32_t epoch, uint32_t code) {
  atomicCAS(&hdr->status, 0ull, ((unsigned long long)epoch << 32) | code);
}
__device__ __forceinline__ bool call_aborted(const WsHeader* hdr, uint32_t epoch) {
  unsigned long long s = ld_relaxed_u64(&hdr->status);
  return s != 0ull && (uint32_t)(s >> 32) == epoch;
}

// Spin until *flag carries this call's epoch; returns the flag kind, or 0 when the wait
// gave up (limit reached, or another tile of this call already gave up).  Bounded.
__device__ __forceinline__ uint32_t wait_flag(const unsigned long long* flag, WsHeader* hdr, const LookbackCtl& ctl) {
  uint64_t t0 = 0;
  uint32_t spins = 0;
  const unsigned long long want = make_flag(ctl.epoch, 0);
  while (true) {
    const unsigned long long f = ld_acquire_u64(flag);
    if ((f & ~3ull) == want && (f & 3ull) != 0ull) return (uint32_t)(f & 3ull);
    if (++spins == 1) t0 = global_timer_ns();
    if ((spins & 63u) == 0u) {
      if (call_aborted(hdr, ctl.epoch)) return 0;
      if (global_timer_ns() - t0 > ctl.spin_limit_ns) {
        record_error(hdr, ctl.epoch, SSM_ERR_TIMEOUT);
        return 0;
      }
    }
    if (spins > 8) __nanosleep(spins > 256 ? 256 : 32);
  }
}

// Claim the next look-back tile (thread 0 only).
__device__ __forceinline__ uint32_t claim_tile(WsHeader* hdr) { return atomicAdd(&hdr->counter, 1u); }

// Called by thread 0 of every CTA after its last global access: the CTA that finishes last
// resets the claim counters so the workspace is ready for the next call.
__device__ __forceinline__ void retire_tile(WsHeader* hdr, uint32_t n_tiles) {
  __threadfence();
  uint32_t d = atomicAdd(&hdr->done, 1u);
  if (d == n_tiles - 1u) {
    atomicExch(&hdr->counter, 0u);
    atomicExch(&hdr->done, 0u);
  }
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------------------
// SSD problem description and workspace layout
// ---------------------------------------------------------------------------------------
struct SsdDims {
  int64_t batch, seqlen;
  int nheads, headdim, dstate, ngroups, chunk;
  int64_t nchunks;       // ceil(seqlen / chunk)
  int64_t lpad;          // nchunks * chunk
  ssm_dtype dtype;
};

// State passing tiling: a tile covers kSpElems state entries of one (batch, head) for up
// to kSpChunks consecutive chunks.
constexpr int kSpThreads = 256;
constexpr int kSpElems = kSpThreads * 4;  // one float4 per thread
constexpr int kSpChunks = 16;

struct SsdWorkspace {
  WsHeader* hdr;
  float* G;        // [batch, nheads, lpad] log2-scaled within-chunk cumsum of A*dt
  float* dtT;      // [batch, nheads, lpad] dt transposed to f32 (0 in the padding)
  float* Sc;       // [batch, nchunks, nheads, headdim, dstate] per-chunk state increments
  void* hin;       // [batch, nchunks, nheads, headdim, dstate] chunk-initial states (dtype)
  unsigned long long* flags; // [sp_tiles]
  float* agg;      // [sp_tiles, kSpElems]
  float* inc;      // [sp_tiles, kSpElems]
  int64_t sp_chains, sp_ctiles, sp_tiles;
  size_t total_bytes;
};
SsdWorkspace ssd_workspace_layout(const SsdDims& d, void* base);

struct LinscanWorkspace {
  WsHeader* hdr;
  unsigned long long* flags;  // [tiles]
  float2* agg;      // [tiles]
  float2* inc;      // [tiles]
  int64_t tiles;
  size_t total_bytes;
};
constexpr int kLsThreads = 256;
constexpr int kLsRuns = 4;                            // float4 runs per thread
constexpr int kLsTile = kLsThreads * 4 * kLsRuns;     // 4096 elements per tile
LinscanWorkspace linscan_workspace_layout(int64_t n, void* base);

// Launchers (return a CUDA error code; 0 = success).
cudaError_t launch_linscan(const float* a, const float* b, float* h, int64_t rows, int64_t len,
                           const LinscanWorkspace& ws, const LookbackCtl& ctl, cudaStream_t s);
cudaError_t launch_ssd_chunk_cumsum(const void* dt, const float* A, const SsdDims& d,
                                    const SsdWorkspace& ws, cudaStream_t s);
cudaError_t launch_ssd_chunk_state(const void* x, const void* B, const SsdDims& d,
                                   const SsdWorkspace& ws, cudaStream_t s);
cudaError_t launch_ssd_state_passing(const float* h0, float* h_final, const SsdDims& d,
                                     const SsdWorkspace& ws, const LookbackCtl& ctl, cudaStream_t s);
cudaError_t launch_ssd_chunk_scan(const void* x, const void* B, const void* C, const float* D,
                                  void* y, const SsdDims& d, const SsdWorkspace& ws, cudaStream_t s);

}  // namespace ssm
