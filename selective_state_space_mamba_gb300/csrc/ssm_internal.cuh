// Internal declarations shared by the CUDA sources of the library (not part of the ABI).
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only; the driver is reached through the runtime)
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
  uint32_t epoch;             // flag epoch of the next look-back launch on this workspace
  uint32_t pad;
};
constexpr size_t kHeaderBytes = 256;

// Look-back fault injection and wait limit (test hook), passed by value to each kernel.
struct LookbackCtl {
  uint32_t epoch;         // call tag (kernels with look-back flags replace it, see device_epoch)
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

// Scalar-scan tile descriptor: flag word and value in ONE 16-byte word, written and read
// with single 16-byte accesses, so a reader that sees the flag sees its value and the
// publisher needs no fence.  kind A: (a, b) = tile aggregate; kind P: b = inclusive prefix.
struct __align__(16) LsDesc {
  unsigned long long flag;
  float a, b;
};

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
__device__ __forceinline__ void st_relaxed_desc(LsDesc* p, unsigned long long flag, float a, float b) {
  const unsigned long long hi = ((unsigned long long)__float_as_uint(b) << 32) | __float_as_uint(a);
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(flag), "l"(hi) : "memory");
}
__device__ __forceinline__ void ld_relaxed_desc(const LsDesc* p, unsigned long long& flag, float& a, float& b) {
  unsigned long long hi;
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(flag), "=l"(hi) : "l"(p) : "memory");
  a = __uint_as_float((uint32_t)(hi & 0xffffffffull));
  b = __uint_as_float((uint32_t)(hi >> 32));
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

// Device index checks of debug builds (-DSSM_DEBUG).  SSM_CHECK(hdr, cond) is true when cond
// holds; otherwise it records SSM_ERR_BOUNDS in the workspace status word (reported by
// ssm_check_device_status; epoch 0, so that no wait of the call takes it for an abort) and
// the caller skips the access.  Release builds compile it to the constant true.
__device__ __forceinline__ bool debug_check(bool ok, WsHeader* hdr) {
  if (!ok) record_error(hdr, 0u, SSM_ERR_BOUNDS);
  return ok;
}
#ifdef SSM_DEBUG
#define SSM_CHECK(hdr, cond) ::ssm::debug_check((cond), (hdr))
#else
#define SSM_CHECK(hdr, cond) true
#endif
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

// ---- mbarrier + bulk-copy (TMA engine) helpers -----------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
// adds `bytes` to the barrier's expected transaction count without an arrive: the phase
// still needs its arrivals as well as the bytes
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Named barrier over `count` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also ORs `pred` over the participating threads: every thread gets the
// same answer, so a bounded wait that gave up in one thread makes all of them leave together
// (a thread that left alone would strand the others in the next barrier).
// ---- programmatic dependent launch ----
// A kernel started with launch_pdl may begin while the previous kernel of the stream is still
// running.  It lets its own successor start early (griddep_launch_dependents, at entry) and
// must pass griddep_wait (every thread that touches global memory) before it reads or writes
// anything in global memory: the previous kernel may be producing its inputs or still reading
// its outputs.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

__device__ __forceinline__ bool named_bar_any(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for a phase of an mbarrier; false when the limit passed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}
// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16), completing
// `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// ---- TMA tensor copies (cp.async.bulk.tensor), 2-D tiles -------------------------------
// Load box at (x = c0 inner, y = c1 outer) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
      : "memory");
}
// Store a shared-memory box to (c0, c1); elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(c0), "r"(c1)
               : "memory");
}
// L2 policy for data a kernel touches once (streamed in or out): its lines are evicted before
// lines of normal priority, so a stream does not push other data, such as dirty lines another
// kernel left behind, out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// L2 policy for a small input that many CTAs read again and again while a larger stream
// passes through L2: its lines are evicted after lines of normal and evict-first priority.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// tma_load_2d / tma_store_2d with an L2 cache policy
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, const void* src, int c0, int c1,
                                                  uint64_t pol) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(c0), "r"(c1), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups still READ shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most N of this thread's bulk groups are incomplete (writes done).
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Host: encode a 2-D tiled tensor map (inner dimension contiguous); returns a CUDA error code.
cudaError_t encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                                 uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                                 CUtensorMapSwizzle swizzle);

// Host: encode a 3-D tiled tensor map (dims[0] contiguous; strides of dims 1 and 2 in bytes).
cudaError_t encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, const uint64_t dims[3],
                                 const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle);

// Claim the next look-back tile (thread 0 only).
__device__ __forceinline__ uint32_t claim_tile(WsHeader* hdr) { return atomicAdd(&hdr->counter, 1u); }

// Called by thread 0 of every CTA after its last global access: the CTA that finishes last
// resets the claim counters so the workspace is ready for the next call, and moves the flag
// epoch on, so that the flags this launch left can never pass for the next launch's.
__device__ __forceinline__ void retire_tile(WsHeader* hdr, uint32_t n_tiles) {
  __threadfence();
  uint32_t d = atomicAdd(&hdr->done, 1u);
  if (d == n_tiles - 1u) {
    atomicExch(&hdr->counter, 0u);
    atomicExch(&hdr->done, 0u);
    atomicAdd(&hdr->epoch, 1u);
  }
}

// A look-back launch tags its flags with the epoch kept in the workspace, not with the host's
// per-call tag: a launch replayed from a CUDA graph then still gets a fresh epoch (the previous
// launch's last CTA advanced it after every CTA of that launch had read it).  Read after the
// previous kernel has finished (griddep_wait where the launch uses programmatic dependence).
__device__ __forceinline__ LookbackCtl device_epoch(LookbackCtl c, const WsHeader* hdr) {
  c.epoch = *reinterpret_cast<const volatile uint32_t*>(&hdr->epoch);
  return c;
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
  // plan (ssm_ssd_fwd_tune / ssm_ssd_fwd_set_plan); -1 / 0 leave the choice to the heuristics
  int plan_fused;        // 1: chunk states and state passing in one kernel, 0: two kernels
  int plan_seq;          // 1: sequential state passing, 0: look-back state passing
  int plan_scan_heads;   // chunk scan: heads per CTA (0: cost model)
  int plan_ring;         // fused state pass: 1 = 4 X + 3 B slots, 2 = 3 + 4, 3 = 5 + 2 (0: rule, 4 + 3)
  int64_t debug_shrink;  // debug builds: bound shortfall of the cumsum store check (test hook)
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
  LsDesc* desc;     // [tiles]
  int64_t tiles;
  size_t total_bytes;
};
#ifndef SSM_LS_LINES
#define SSM_LS_LINES 128
#endif
#ifndef SSM_LS_SPLIT
#define SSM_LS_SPLIT 2
#endif
#ifndef SSM_LS_STREAM_HINT  // a, b and h streamed through L2 with evict-first priority
#define SSM_LS_STREAM_HINT 1
#endif
constexpr int kLsLines = SSM_LS_LINES;                // 128-byte lines (32 floats) per tile
constexpr int kLsRow = 32;                            // elements per line
constexpr int kLsSplit = SSM_LS_SPLIT;                // consumer threads per line
constexpr int kLsElems = kLsRow / kLsSplit;           // consecutive elements per consumer thread
constexpr int kLsThreads = kLsLines * kLsSplit;       // consumer threads
constexpr int kLsTile = kLsLines * kLsRow;            // elements per tile
LinscanWorkspace linscan_workspace_layout(int64_t n, void* base);

// Raises `func`'s dynamic shared-memory limit to at least `bytes` on the current device, with
// one attribute call per device and size: later launches (for example while a stream is
// being captured into a CUDA graph) make none.
cudaError_t ensure_smem_limit(const void* func, size_t bytes);

// Launchers (return a CUDA error code; 0 = success).
// shape: the CTA shape (ssm_linscan_fwd_tune in ssm.h: 1 .. 4), 0 for the rule by row length
cudaError_t launch_linscan(const float* a, const float* b, float* h, int64_t rows, int64_t len,
                           const LinscanWorkspace& ws, const LookbackCtl& ctl, cudaStream_t s, int shape = 0);
constexpr int kLsShapes = 4;
// The chunk scan's CTA split: tier s covers the next tiles[s] tiles (batch, chunk, group, row
// tile; in that order, row tile fastest, the later row tile first) with items[s] CTAs per tile,
// a tile's heads split evenly between them.  plan_heads > 0 fixes runs of at most that many
// heads (one tier).
struct ScTiers {
  int64_t tiles[3];
  int items[3];
};
ScTiers sc_schedule(int64_t tiles, int row_tiles, int hpg, int sms, int plan_heads);

cudaError_t launch_ssd_chunk_cumsum(const void* dt, const float* A, const SsdDims& d,
                                    const SsdWorkspace& ws, cudaStream_t s);
cudaError_t launch_ssd_chunk_state(const void* x, const void* B, const SsdDims& d,
                                   const SsdWorkspace& ws, cudaStream_t s);
cudaError_t launch_ssd_state_passing(const float* h0, float* h_final, const SsdDims& d,
                                     const SsdWorkspace& ws, const LookbackCtl& ctl, cudaStream_t s);
cudaError_t launch_ssd_chunk_scan(const void* x, const void* B, const void* C, const float* D,
                                  void* y, const SsdDims& d, const SsdWorkspace& ws, cudaStream_t s);
size_t linscan_baseline_workspace(ssm_scan_algo algo, int64_t rows, int64_t len);
ssm_status linscan_baseline_check(ssm_scan_algo algo, int64_t rows, int64_t len);
cudaError_t launch_linscan_baseline(ssm_scan_algo algo, const float* a, const float* b, float* h, int64_t rows,
                                    int64_t len, void* workspace, const LookbackCtl& ctl, cudaStream_t s);
cudaError_t launch_ssd_step(const void* x, const void* dt, const float* A, const void* B, const void* C,
                            const float* D, const float* state_in, float* state_out, void* y, int64_t batch,
                            int nheads, int headdim, int dstate, int ngroups, ssm_dtype dtype, cudaStream_t s);

}  // namespace ssm
