// Host side of the C ABI declared in include/ssm.h: argument validation, workspace layout,
// and the launch sequence of each operation on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "ssm_internal.cuh"

namespace ssm {

cudaError_t launch_ssd_chunk_state_simt(const void* x, const void* B, const SsdDims& d, const SsdWorkspace& ws,
                                        cudaStream_t s);
cudaError_t launch_ssd_chunk_scan_simt(const void* x, const void* B, const void* C, const float* D, void* y,
                                       const SsdDims& d, const SsdWorkspace& ws, cudaStream_t s);
bool ssd_tc_supported(const SsdDims& d);
cudaError_t launch_ssd_chunk_state_tc(const void* x, const void* B, const SsdDims& d, const SsdWorkspace& ws,
                                      const LookbackCtl& ctl, cudaStream_t s);
bool ssd_scan_tc_supported(const SsdDims& d);
bool ssd_state_fused_supported(const SsdDims& d);
bool ssd_state_fused_possible(const SsdDims& d);
bool ssd_state_fused_split(const SsdDims& d);
int64_t ssd_fused_schedule(int64_t chains, int64_t nchunks, int sms, bool split, int64_t* rows, int64_t cap);
cudaError_t launch_ssd_state_fixup(float* h_final, const SsdDims& d, const SsdWorkspace& ws, cudaStream_t s);
cudaError_t launch_ssd_state_fused_tc(const void* x, const void* B, const float* h0, float* h_final,
                                      const SsdDims& d, const SsdWorkspace& ws, const LookbackCtl& ctl,
                                      cudaStream_t s);
cudaError_t launch_ssd_chunk_scan_tc(const void* x, const void* B, const void* C, const float* D, void* y,
                                     const SsdDims& d, const SsdWorkspace& ws, const LookbackCtl& ctl,
                                     cudaStream_t s);

namespace {

std::atomic<uint32_t> g_epoch{0};
std::atomic<int64_t> g_stall_tile{-1};
std::atomic<int64_t> g_bounds_shrink{0};  // debug builds: see ssm_debug_set_bounds_fault
std::atomic<uint64_t> g_spin_limit_ns{0};
constexpr uint64_t kDefaultSpinLimitNs = 1000000000ull;  // 1 s per wait

// ---- optional per-kernel timing (ssm_profile_begin / ssm_profile_end) ----
struct ProfRecord {
  int kernel;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
int g_prof_max = 0;
std::vector<ProfRecord> g_prof_records;
std::vector<cudaEvent_t> g_prof_pool;
int64_t g_prof_counts[SSM_PROFILE_KERNELS] = {0};

// Wraps one launch: records events around it on `s` while profiling is enabled.
template <typename F>
cudaError_t timed_launch(int kernel, cudaStream_t s, F&& launch) {
  ProfRecord rec{kernel, nullptr, nullptr};
  bool timed = false;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof_on) {
      g_prof_counts[kernel]++;
      if ((int)g_prof_records.size() < g_prof_max && g_prof_pool.size() >= 2) {
        rec.start = g_prof_pool.back();
        g_prof_pool.pop_back();
        rec.stop = g_prof_pool.back();
        g_prof_pool.pop_back();
        timed = true;
      }
    }
  }
  if (timed && cudaEventRecord(rec.start, s) != cudaSuccess) return cudaErrorUnknown;
  const cudaError_t e = launch();
  if (timed) {
    if (cudaEventRecord(rec.stop, s) != cudaSuccess) return cudaErrorUnknown;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_records.push_back(rec);
  }
  return e;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ssm_status check_ssd_dims(int64_t batch, int64_t seqlen, int nheads, int headdim, int dstate, int ngroups,
                          int chunk, ssm_dtype dtype) {
  if (batch < 0 || seqlen < 0 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1 || chunk < 1)
    return SSM_ERR_INVALID_ARG;
  if (nheads % ngroups != 0) return SSM_ERR_INVALID_ARG;
  if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
  if (headdim != 64) return SSM_ERR_UNSUPPORTED;
  if (dstate != 64 && dstate != 128) return SSM_ERR_UNSUPPORTED;
  if (chunk != 64 && chunk != 128 && chunk != 256) return SSM_ERR_UNSUPPORTED;
  // grid limits: chunks and batch go to grid.x / grid.z of some kernels
  const int64_t nchunks = (seqlen + chunk - 1) / chunk;
  if (nchunks * (chunk / 64) > 0x7fffffffLL || batch > 65535 || nheads > 65535) return SSM_ERR_UNSUPPORTED;
  return SSM_OK;
}

SsdDims make_dims(int64_t batch, int64_t seqlen, int nheads, int headdim, int dstate, int ngroups, int chunk,
                  ssm_dtype dtype) {
  SsdDims d;
  d.batch = batch;
  d.seqlen = seqlen;
  d.nheads = nheads;
  d.headdim = headdim;
  d.dstate = dstate;
  d.ngroups = ngroups;
  d.chunk = chunk;
  d.nchunks = (seqlen + chunk - 1) / chunk;
  d.lpad = d.nchunks * chunk;
  d.dtype = dtype;
  d.plan_fused = -1;
  d.plan_seq = -1;
  d.plan_scan_heads = 0;
  d.plan_ring = 0;
  d.debug_shrink = g_bounds_shrink.load(std::memory_order_relaxed);
  return d;
}

// Scratch that a tuner writes before each of its runs, outside the timed events: twice the
// L2 size, so that every candidate starts with its inputs out of L2 and dirty lines of other
// data in it, as a call does after other work, and not from the previous candidate's warm
// lines (which would favour, for inputs that fit in L2, plans that are slower from DRAM).
// Without the memory for it the runs go back to back.
struct TuneFlush {
  void* buf = nullptr;
  size_t bytes = 0;
  TuneFlush() {
    int dev = 0, l2 = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess ||
        l2 <= 0)
      return;
    if (cudaMalloc(&buf, 2 * (size_t)l2) != cudaSuccess) {
      buf = nullptr;
      (void)cudaGetLastError();  // clear the allocation error: the tuner runs on without it
      return;
    }
    bytes = 2 * (size_t)l2;
  }
  ~TuneFlush() {
    if (buf) cudaFree(buf);
  }
  TuneFlush(const TuneFlush&) = delete;
  TuneFlush& operator=(const TuneFlush&) = delete;
  cudaError_t run(cudaStream_t s, int r) const { return buf ? cudaMemsetAsync(buf, r & 0xff, bytes, s) : cudaSuccess; }
};

// ---- per-shape plans (ssm_ssd_fwd_tune / ssm_ssd_fwd_set_plan) ----
// A plan id packs (fused + 1) | (seq + 1) << 2 | scan_heads << 4 | ring << 20, with -1 (0 for
// scan_heads and ring) meaning "the heuristic"; fused 2 is the fused pass with split chains.
struct PlanKey {
  int dev;
  int64_t batch, seqlen;
  int nheads, headdim, dstate, ngroups, chunk, dtype;
  bool operator<(const PlanKey& o) const {
    return std::tie(dev, batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype) <
           std::tie(o.dev, o.batch, o.seqlen, o.nheads, o.headdim, o.dstate, o.ngroups, o.chunk, o.dtype);
  }
};
std::mutex g_plan_mu;
std::map<PlanKey, int> g_plans;

bool plan_key(const SsdDims& d, PlanKey* k) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  *k = PlanKey{dev, d.batch, d.seqlen, d.nheads, d.headdim, d.dstate, d.ngroups, d.chunk, (int)d.dtype};
  return true;
}
int plan_id(int fused, int seq, int heads, int ring = 0) {
  return (fused + 1) | ((seq + 1) << 2) | (heads << 4) | (ring << 20);
}
bool plan_valid(int id) { return id >= 0 && ((id >> 2) & 3) != 3 && (id >> 20) <= 3; }
void apply_plan(SsdDims& d, int id) {
  d.plan_fused = (id & 3) - 1;
  d.plan_seq = ((id >> 2) & 3) - 1;
  d.plan_scan_heads = (id >> 4) & 0xffff;
  d.plan_ring = (id >> 20) & 3;
}
// ---- per-size CTA shapes of the scalar scan (ssm_linscan_fwd_tune / ssm_linscan_set_shape) ----
std::mutex g_ls_mu;
std::map<std::tuple<int, int64_t, int64_t>, int> g_ls_shapes;
int cached_ls_shape(int64_t rows, int64_t len) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(g_ls_mu);
  const auto it = g_ls_shapes.find(std::make_tuple(dev, rows, len));
  return it == g_ls_shapes.end() ? 0 : it->second;
}

void apply_cached_plan(SsdDims& d) {
  PlanKey k;
  if (!plan_key(d, &k)) return;
  std::lock_guard<std::mutex> lk(g_plan_mu);
  const auto it = g_plans.find(k);
  if (it != g_plans.end()) apply_plan(d, it->second);
}

// Pointer, alignment and workspace checks of an SSD forward with tokens to process.
ssm_status check_ssd_buffers(const void* x, const void* dt, const float* A, const void* B, const void* C,
                             const float* D, const float* h0, const void* y, const float* h_final, const SsdDims& d,
                             const void* workspace, size_t workspace_bytes) {
  if (!x || !dt || !A || !B || !C || !D || !y) return SSM_ERR_INVALID_ARG;
  const void* ptrs[] = {x, dt, A, B, C, D, y};
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return SSM_ERR_ALIGNMENT;
  if ((h0 && !aligned(h0, 16)) || (h_final && !aligned(h_final, 16))) return SSM_ERR_ALIGNMENT;
  const SsdWorkspace need = ssd_workspace_layout(d, nullptr);
  if (!workspace || workspace_bytes < need.total_bytes) return SSM_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return SSM_ERR_ALIGNMENT;
  return SSM_OK;
}

}  // namespace

cudaError_t ensure_smem_limit(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  size_t& have = done[{dev, func}];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

LookbackCtl next_lookback_ctl() {
  LookbackCtl c;
  uint32_t e;
  do {
    e = (g_epoch.fetch_add(1, std::memory_order_relaxed) + 1) & 0x3fffffffu;
  } while (e == 0);
  c.epoch = e;
  c.stall_tile = g_stall_tile.load(std::memory_order_relaxed);
  const uint64_t lim = g_spin_limit_ns.load(std::memory_order_relaxed);
  c.spin_limit_ns = lim ? lim : kDefaultSpinLimitNs;
  return c;
}

SsdWorkspace ssd_workspace_layout(const SsdDims& d, void* base) {
  SsdWorkspace w{};
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* r = p ? p + off : nullptr;
    off = align_up(off + bytes, 256);
    return r;
  };
  const int64_t bh = d.batch * d.nheads;
  const int64_t HS = (int64_t)d.headdim * d.dstate;
  const size_t hin_elem = d.dtype == SSM_BF16 ? 2 : 4;
  w.sp_chains = bh * (HS / kSpElems);
  w.sp_ctiles = (d.nchunks + kSpChunks - 1) / kSpChunks;
  w.sp_tiles = w.sp_chains * w.sp_ctiles;
  w.hdr = reinterpret_cast<WsHeader*>(take(kHeaderBytes));
  w.flags = reinterpret_cast<unsigned long long*>(take(sizeof(unsigned long long) * w.sp_tiles));
  w.G = reinterpret_cast<float*>(take(sizeof(float) * bh * d.lpad));
  w.dtT = reinterpret_cast<float*>(take(sizeof(float) * bh * d.lpad));
  w.Sc = reinterpret_cast<float*>(take(sizeof(float) * d.batch * d.nchunks * d.nheads * HS));
  w.hin = take(hin_elem * d.batch * d.nchunks * d.nheads * HS);
  w.agg = reinterpret_cast<float*>(take(sizeof(float) * w.sp_tiles * kSpElems));
  w.inc = reinterpret_cast<float*>(take(sizeof(float) * w.sp_tiles * kSpElems));
  w.total_bytes = off;
  return w;
}

LinscanWorkspace linscan_workspace_layout(int64_t n, void* base) {
  LinscanWorkspace w{};
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* r = p ? p + off : nullptr;
    off = align_up(off + bytes, 256);
    return r;
  };
  w.tiles = (n + kLsTile - 1) / kLsTile;
  w.hdr = reinterpret_cast<WsHeader*>(take(kHeaderBytes));
  w.desc = reinterpret_cast<LsDesc*>(take(sizeof(LsDesc) * w.tiles));
  w.total_bytes = off;
  return w;
}

namespace {
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
cudaError_t get_encoder(EncodeFn* out) {
  static EncodeFn encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return e != cudaSuccess ? e : cudaErrorUnknown;
    encode = reinterpret_cast<EncodeFn>(fn);
  }
  *out = encode;
  return cudaSuccess;
}
}  // namespace

cudaError_t encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, const uint64_t dims[3],
                                 const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle) {
  EncodeFn encode;
  const cudaError_t e = get_encoder(&encode);
  if (e != cudaSuccess) return e;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(map, dtype, 3, const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                                 uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                                 CUtensorMapSwizzle swizzle) {
  EncodeFn encode;
  const cudaError_t ge = get_encoder(&encode);
  if (ge != cudaSuccess) return ge;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace ssm

namespace ssm {
namespace {

// The kernel sequence of one SSD forward on validated sizes, a sized workspace and d's plan.
ssm_status run_ssd(const void* x, const void* dt, const float* A, const void* B, const void* C, const float* D,
                   const float* h0, void* y, float* h_final, const SsdDims& d, void* workspace, cudaStream_t s) {
  const SsdWorkspace ws = ssd_workspace_layout(d, workspace);
  const LookbackCtl ctl = next_lookback_ctl();

  const bool state_tc = ssd_tc_supported(d);
  const bool scan_tc = ssd_scan_tc_supported(d);
  const bool fused = state_tc && ssd_state_fused_supported(d);
  if (timed_launch(1, s, [&] { return launch_ssd_chunk_cumsum(dt, A, d, ws, s); }) != cudaSuccess)
    return SSM_ERR_CUDA;
  if (fused) {
    // chunk states and the recurrence over chunks in one pass: S_c never goes to memory
    if (timed_launch(5, s, [&] { return launch_ssd_state_fused_tc(x, B, h0, h_final, d, ws, ctl, s); }) !=
        cudaSuccess)
      return SSM_ERR_CUDA;
    // split chains: add to every piece the state it enters with
    if (ssd_state_fused_split(d) &&
        timed_launch(8, s, [&] { return launch_ssd_state_fixup(h_final, d, ws, s); }) != cudaSuccess)
      return SSM_ERR_CUDA;
  } else {
    if (timed_launch(2, s, [&] {
          return state_tc ? launch_ssd_chunk_state_tc(x, B, d, ws, ctl, s)
                          : launch_ssd_chunk_state_simt(x, B, d, ws, s);
        }) != cudaSuccess)
      return SSM_ERR_CUDA;
    if (timed_launch(3, s, [&] { return launch_ssd_state_passing(h0, h_final, d, ws, ctl, s); }) != cudaSuccess)
      return SSM_ERR_CUDA;
  }
  if (timed_launch(4, s, [&] {
        return scan_tc ? launch_ssd_chunk_scan_tc(x, B, C, D, y, d, ws, ctl, s)
                  : launch_ssd_chunk_scan_simt(x, B, C, D, y, d, ws, s);
      }) != cudaSuccess)
    return SSM_ERR_CUDA;
  return SSM_OK;
}

}  // namespace
}  // namespace ssm

using namespace ssm;

extern "C" {

const char* ssm_status_string(ssm_status status) {
  switch (status) {
    case SSM_OK: return "SSM_OK";
    case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG: invalid argument";
    case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED: shape not supported by the kernels";
    case SSM_ERR_ALIGNMENT: return "SSM_ERR_ALIGNMENT: pointer not aligned as required";
    case SSM_ERR_WORKSPACE: return "SSM_ERR_WORKSPACE: workspace missing or too small";
    case SSM_ERR_CUDA: return "SSM_ERR_CUDA: CUDA runtime error";
    case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT: a look-back wait exceeded its limit";
    case SSM_ERR_BOUNDS: return "SSM_ERR_BOUNDS: a device index check of the debug build failed";
  }
  return "unknown ssm_status";
}

const char* ssm_version(void) { return "0.1.0"; }

size_t ssm_ssd_fwd_workspace_bytes(int64_t batch, int64_t seqlen, int nheads, int headdim, int dstate, int ngroups,
                                   int chunk, ssm_dtype dtype) {
  if (check_ssd_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype) != SSM_OK) return 0;
  return ssd_workspace_layout(make_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype), nullptr)
      .total_bytes;
}

ssm_status ssm_ssd_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C, const float* D,
                       const float* h0, void* y, float* h_final, int64_t batch, int64_t seqlen, int nheads,
                       int headdim, int dstate, int ngroups, int chunk, ssm_dtype dtype, void* workspace,
                       size_t workspace_bytes, ssm_stream_t stream) {
  ssm_status st = check_ssd_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype);
  if (st != SSM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  SsdDims d = make_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype);
  const size_t state_bytes = sizeof(float) * (size_t)batch * nheads * headdim * dstate;
  if (batch == 0 || seqlen == 0) {
    // no tokens: y is empty and the final state is the initial state
    if (h_final && state_bytes) {
      if (h0 && !aligned(h0, 16)) return SSM_ERR_ALIGNMENT;
      cudaError_t e = h0 ? cudaMemcpyAsync(h_final, h0, state_bytes, cudaMemcpyDeviceToDevice, s)
                         : cudaMemsetAsync(h_final, 0, state_bytes, s);
      if (e != cudaSuccess) return SSM_ERR_CUDA;
    }
    return SSM_OK;
  }
  st = check_ssd_buffers(x, dt, A, B, C, D, h0, y, h_final, d, workspace, workspace_bytes);
  if (st != SSM_OK) return st;
  apply_cached_plan(d);
  return run_ssd(x, dt, A, B, C, D, h0, y, h_final, d, workspace, s);
}

ssm_status ssm_ssd_fwd_tune(const void* x, const void* dt, const float* A, const void* B, const void* C,
                            const float* D, const float* h0, void* y, float* h_final, int64_t batch, int64_t seqlen,
                            int nheads, int headdim, int dstate, int ngroups, int chunk, ssm_dtype dtype,
                            void* workspace, size_t workspace_bytes, ssm_stream_t stream, int reps, int* plan_out,
                            float* ms_out) {
  ssm_status st = check_ssd_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype);
  if (st != SSM_OK) return st;
  if (reps < 1) return SSM_ERR_INVALID_ARG;
  if (plan_out) *plan_out = -1;
  if (ms_out) *ms_out = 0.f;
  if (batch == 0 || seqlen == 0) return SSM_OK;  // nothing to choose
  SsdDims d = make_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype);
  st = check_ssd_buffers(x, dt, A, B, C, D, h0, y, h_final, d, workspace, workspace_bytes);
  if (st != SSM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // candidates: the fused state path where it is possible (with split chains as well where
  // there are fewer chains than SMs), else the two state kernels with either state-passing
  // kernel; times the chunk scan's runs of heads per CTA
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SSM_ERR_CUDA;
  const bool split_cands = d.nchunks > 1 && batch * (int64_t)(nheads / 2) < sms;
  std::vector<int> cands;
  std::vector<int> heads = {0};
  if (ssd_scan_tc_supported(d)) {
    const int hpg = nheads / ngroups;
    for (int parts : {1, 2, 3, 4, 5, 6, 8}) heads.push_back((hpg + parts - 1) / parts);
    std::sort(heads.begin() + 1, heads.end());
    heads.erase(std::unique(heads.begin() + 1, heads.end()), heads.end());
  }
  for (int hd : heads) {
    if (ssd_tc_supported(d) && ssd_state_fused_possible(d))
      for (int ring = 1; ring <= 3; ++ring) {  // ring splits
        cands.push_back(plan_id(1, -1, hd, ring));
        if (split_cands) cands.push_back(plan_id(2, -1, hd, ring));  // the same with split chains
      }
    cands.push_back(plan_id(0, 1, hd));
    cands.push_back(plan_id(0, 0, hd));
  }
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return SSM_ERR_CUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return SSM_ERR_CUDA;
  }
  int best = -1;
  float best_ms = 0.f;
  st = SSM_OK;
  const TuneFlush flush;
  for (int id : cands) {
    SsdDims dc = d;
    apply_plan(dc, id);
    std::vector<float> t;
    for (int r = 0; r <= reps && st == SSM_OK; ++r) {  // one warm-up, then `reps` timed runs
      if (flush.run(s, r) != cudaSuccess || cudaEventRecord(e0, s) != cudaSuccess) st = SSM_ERR_CUDA;
      if (st == SSM_OK) st = run_ssd(x, dt, A, B, C, D, h0, y, h_final, dc, workspace, s);
      if (st == SSM_OK && cudaEventRecord(e1, s) != cudaSuccess) st = SSM_ERR_CUDA;
      float ms = 0.f;
      if (st == SSM_OK && (cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess))
        st = SSM_ERR_CUDA;
      if (r > 0) t.push_back(ms);
    }
    if (st != SSM_OK) break;
    // a device-side timeout in a candidate disqualifies nothing silently: report it
    unsigned long long word = 0;
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
      st = SSM_ERR_CUDA;
      break;
    }
    if (word != 0) {
      st = static_cast<ssm_status>(word & 0xffffffffu);
      break;
    }
    std::sort(t.begin(), t.end());
    const float med = t[t.size() / 2];
    if (best < 0 || med < best_ms) {
      best = id;
      best_ms = med;
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st != SSM_OK) return st;
  PlanKey k;
  if (!plan_key(d, &k)) return SSM_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    g_plans[k] = best;
  }
  if (plan_out) *plan_out = best;
  if (ms_out) *ms_out = best_ms;
  return SSM_OK;
}

ssm_status ssm_ssd_fwd_set_plan(int64_t batch, int64_t seqlen, int nheads, int headdim, int dstate, int ngroups,
                                int chunk, ssm_dtype dtype, int plan) {
  const ssm_status st = check_ssd_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype);
  if (st != SSM_OK) return st;
  if (plan != -1 && !plan_valid(plan)) return SSM_ERR_INVALID_ARG;
  PlanKey k;
  if (!plan_key(make_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype), &k)) return SSM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_plan_mu);
  if (plan == -1)
    g_plans.erase(k);
  else
    g_plans[k] = plan;
  return SSM_OK;
}

ssm_status ssm_ssd_fwd_get_plan(int64_t batch, int64_t seqlen, int nheads, int headdim, int dstate, int ngroups,
                                int chunk, ssm_dtype dtype, int* plan) {
  const ssm_status st = check_ssd_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype);
  if (st != SSM_OK) return st;
  if (!plan) return SSM_ERR_INVALID_ARG;
  *plan = -1;
  PlanKey k;
  if (!plan_key(make_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype), &k)) return SSM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_plan_mu);
  const auto it = g_plans.find(k);
  if (it != g_plans.end()) *plan = it->second;
  return SSM_OK;
}

void ssm_ssd_fwd_clear_plans(void) {
  std::lock_guard<std::mutex> lk(g_plan_mu);
  g_plans.clear();
}

ssm_status ssm_ssd_step(const void* x, const void* dt, const float* A, const void* B, const void* C,
                        const float* D, const float* state_in, float* state_out, void* y, int64_t batch, int nheads,
                        int headdim, int dstate, int ngroups, ssm_dtype dtype, ssm_stream_t stream) {
  if (batch < 0 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1 || nheads % ngroups != 0)
    return SSM_ERR_INVALID_ARG;
  if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_INVALID_ARG;
  if (headdim % 16 != 0 || (dstate != 64 && dstate != 128)) return SSM_ERR_UNSUPPORTED;
  if (batch == 0) return SSM_OK;
  if (!x || !dt || !A || !B || !C || !D || !state_out || !y) return SSM_ERR_INVALID_ARG;
  const void* ptrs[] = {x, dt, A, B, C, D, state_out, y};
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return SSM_ERR_ALIGNMENT;
  if (state_in && !aligned(state_in, 16)) return SSM_ERR_ALIGNMENT;
  const int64_t units = batch * nheads;
  if (units / nheads != batch) return SSM_ERR_INVALID_ARG;
  const int64_t state_elems = units * headdim * dstate;
  if (state_elems / ((int64_t)headdim * dstate) != units) return SSM_ERR_INVALID_ARG;
  if (state_in && state_in != state_out) {
    // in place is allowed; any other overlap of the two states is not
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(state_in), b0 = reinterpret_cast<uintptr_t>(state_out);
    const uintptr_t n = sizeof(float) * (uintptr_t)state_elems;
    if (a0 < b0 + n && b0 < a0 + n) return SSM_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (timed_launch(6, s, [&] {
        return launch_ssd_step(x, dt, A, B, C, D, state_in, state_out, y, batch, nheads, headdim, dstate, ngroups,
                               dtype, s);
      }) != cudaSuccess)
    return SSM_ERR_CUDA;
  return SSM_OK;
}

size_t ssm_linscan_workspace_bytes(int64_t rows, int64_t len) {
  if (rows < 0 || len < 0) return 0;
  return linscan_workspace_layout(rows * len, nullptr).total_bytes;
}

ssm_status ssm_linscan_fwd(const float* a, const float* b, float* h, int64_t rows, int64_t len, void* workspace,
                           size_t workspace_bytes, ssm_stream_t stream) {
  if (rows < 0 || len < 0) return SSM_ERR_INVALID_ARG;
  if (rows == 0 || len == 0) return SSM_OK;
  if (!a || !b || !h) return SSM_ERR_INVALID_ARG;
  if (!aligned(a, 16) || !aligned(b, 16) || !aligned(h, 16)) return SSM_ERR_ALIGNMENT;
  const int64_t n = rows * len;
  if (n / len != rows) return SSM_ERR_INVALID_ARG;
  const LinscanWorkspace need = linscan_workspace_layout(n, nullptr);
  if (need.tiles > 0x7fffffffLL) return SSM_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < need.total_bytes) return SSM_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return SSM_ERR_ALIGNMENT;
  const LinscanWorkspace ws = linscan_workspace_layout(n, workspace);
  const LookbackCtl ctl = next_lookback_ctl();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int shape = cached_ls_shape(rows, len);
  if (timed_launch(0, s, [&] { return launch_linscan(a, b, h, rows, len, ws, ctl, s, shape); }) != cudaSuccess)
    return SSM_ERR_CUDA;
  return SSM_OK;
}

ssm_status ssm_linscan_fwd_tune(const float* a, const float* b, float* h, int64_t rows, int64_t len, void* workspace,
                                size_t workspace_bytes, ssm_stream_t stream, int reps, int* shape_out, float* ms_out) {
  if (reps < 1) return SSM_ERR_INVALID_ARG;
  if (shape_out) *shape_out = -1;
  if (ms_out) *ms_out = 0.f;
  // the same argument checks as a call, by a call with the rule's shape
  ssm_status st = ssm_linscan_fwd(a, b, h, rows, len, workspace, workspace_bytes, stream);
  if (st != SSM_OK || rows == 0 || len == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const LinscanWorkspace ws = linscan_workspace_layout(rows * len, workspace);
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return SSM_ERR_CUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return SSM_ERR_CUDA;
  }
  int best = -1;
  float best_ms = 0.f;
  const TuneFlush flush;
  for (int shape = 1; shape <= kLsShapes && st == SSM_OK; ++shape) {
    std::vector<float> t;
    for (int r = 0; r <= reps && st == SSM_OK; ++r) {  // one warm-up, then `reps` timed runs
      if (flush.run(s, r) != cudaSuccess || cudaEventRecord(e0, s) != cudaSuccess ||
          launch_linscan(a, b, h, rows, len, ws, next_lookback_ctl(), s, shape) != cudaSuccess ||
          cudaEventRecord(e1, s) != cudaSuccess) {
        st = SSM_ERR_CUDA;
        break;
      }
      float ms = 0.f;
      if (cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) {
        st = SSM_ERR_CUDA;
        break;
      }
      if (r > 0) t.push_back(ms);
    }
    if (st != SSM_OK) break;
    unsigned long long word = 0;  // a device-side timeout in a candidate is reported, not skipped
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
      st = SSM_ERR_CUDA;
      break;
    }
    if (word != 0) {
      st = static_cast<ssm_status>(word & 0xffffffffu);
      break;
    }
    std::sort(t.begin(), t.end());
    if (best < 0 || t[t.size() / 2] < best_ms) {
      best = shape;
      best_ms = t[t.size() / 2];
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st != SSM_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_ls_mu);
    g_ls_shapes[std::make_tuple(dev, rows, len)] = best;
  }
  if (shape_out) *shape_out = best;
  if (ms_out) *ms_out = best_ms;
  return SSM_OK;
}

ssm_status ssm_linscan_set_shape(int64_t rows, int64_t len, int shape) {
  if (rows < 0 || len < 0 || shape < -1 || shape > kLsShapes) return SSM_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_ls_mu);
  if (shape <= 0)
    g_ls_shapes.erase(std::make_tuple(dev, rows, len));
  else
    g_ls_shapes[std::make_tuple(dev, rows, len)] = shape;
  return SSM_OK;
}

ssm_status ssm_linscan_get_shape(int64_t rows, int64_t len, int* shape) {
  if (!shape || rows < 0 || len < 0) return SSM_ERR_INVALID_ARG;
  *shape = cached_ls_shape(rows, len);
  if (*shape == 0) *shape = -1;
  return SSM_OK;
}

void ssm_linscan_clear_shapes(void) {
  std::lock_guard<std::mutex> lk(g_ls_mu);
  g_ls_shapes.clear();
}

size_t ssm_linscan_baseline_workspace_bytes(ssm_scan_algo algo, int64_t rows, int64_t len) {
  if (rows < 0 || len < 0 || linscan_baseline_check(algo, rows, len) == SSM_ERR_INVALID_ARG) return 0;
  return linscan_baseline_workspace(algo, rows, len);
}

ssm_status ssm_linscan_baseline(ssm_scan_algo algo, const float* a, const float* b, float* h, int64_t rows,
                                int64_t len, void* workspace, size_t workspace_bytes, ssm_stream_t stream) {
  if (rows < 0 || len < 0) return SSM_ERR_INVALID_ARG;
  const ssm_status st = linscan_baseline_check(algo, rows, len);
  if (st == SSM_ERR_INVALID_ARG) return st;
  if (rows == 0 || len == 0) return SSM_OK;
  if (st != SSM_OK) return st;
  if (!a || !b || !h) return SSM_ERR_INVALID_ARG;
  if (!aligned(a, 16) || !aligned(b, 16) || !aligned(h, 16)) return SSM_ERR_ALIGNMENT;
  if (rows * len / len != rows) return SSM_ERR_INVALID_ARG;
  const size_t need = linscan_baseline_workspace(algo, rows, len);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return SSM_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return SSM_ERR_ALIGNMENT;
  }
  const LookbackCtl ctl = next_lookback_ctl();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (timed_launch(7, s, [&] { return launch_linscan_baseline(algo, a, b, h, rows, len, workspace, ctl, s); }) !=
      cudaSuccess)
    return SSM_ERR_CUDA;
  return SSM_OK;
}

ssm_status ssm_check_device_status(void* workspace, ssm_stream_t stream) {
  if (!workspace) return SSM_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SSM_ERR_CUDA;
  unsigned long long word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return SSM_ERR_CUDA;
  if (word == 0) return SSM_OK;
  // a failed call may also have left the claim counters set: clear them, and move the flag
  // epoch on so that the failed call's flags never count for a later one
  WsHeader h{};
  if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return SSM_ERR_CUDA;
  const uint32_t next_epoch = h.epoch + 1u;
  h = WsHeader{};
  h.epoch = next_epoch;
  if (cudaMemcpy(workspace, &h, sizeof(h), cudaMemcpyHostToDevice) != cudaSuccess) return SSM_ERR_CUDA;
  const uint32_t code = (uint32_t)(word & 0xffffffffu);
  return code == 0 ? SSM_ERR_CUDA : static_cast<ssm_status>(code);
}

ssm_status ssm_profile_begin(int max_launches) {
  if (max_launches < 0) return SSM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof_records) {
    g_prof_pool.push_back(r.start);
    g_prof_pool.push_back(r.stop);
  }
  g_prof_records.clear();
  while ((int)g_prof_pool.size() < 2 * max_launches) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return SSM_ERR_CUDA;
    g_prof_pool.push_back(e);
  }
  for (auto& c : g_prof_counts) c = 0;
  g_prof_max = max_launches;
  g_prof_on = true;
  return SSM_OK;
}

ssm_status ssm_profile_end(double* ms_out, int64_t* launches_out) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = false;
  double ms[SSM_PROFILE_KERNELS] = {0};
  ssm_status st = SSM_OK;
  for (auto& r : g_prof_records) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      st = SSM_ERR_CUDA;
    ms[r.kernel] += t;
    g_prof_pool.push_back(r.start);
    g_prof_pool.push_back(r.stop);
  }
  g_prof_records.clear();
  for (int k = 0; k < SSM_PROFILE_KERNELS; ++k) {
    if (ms_out) ms_out[k] = ms[k];
    if (launches_out) launches_out[k] = g_prof_counts[k];
  }
  return st;
}

void ssm_debug_set_lookback_fault(int64_t stall_tile, uint64_t spin_limit_ns) {
  g_stall_tile.store(stall_tile < 0 ? -1 : stall_tile, std::memory_order_relaxed);
  g_spin_limit_ns.store(spin_limit_ns, std::memory_order_relaxed);
}

int ssm_debug_build(void) {
#ifdef SSM_DEBUG
  return 1;
#else
  return 0;
#endif
}

ssm_status ssm_debug_set_bounds_fault(int64_t shrink) {
#ifdef SSM_DEBUG
  if (shrink < 0) return SSM_ERR_INVALID_ARG;
  g_bounds_shrink.store(shrink, std::memory_order_relaxed);
  return SSM_OK;
#else
  (void)shrink;
  return SSM_ERR_UNSUPPORTED;
#endif
}

int64_t ssm_debug_fused_schedule(int64_t chains, int64_t nchunks, int sms, int split, int64_t* rows, int64_t cap) {
  return ssd_fused_schedule(chains, nchunks, sms, split != 0, rows, cap < 0 ? 0 : cap);
}

int64_t ssm_debug_scan_schedule(int64_t tiles, int row_tiles, int heads_per_group, int sms, int plan_heads,
                                int64_t* out) {
  if (tiles < 0 || (row_tiles != 1 && row_tiles != 2) || tiles % row_tiles || heads_per_group < 1 || sms < 1 ||
      plan_heads < 0)
    return -1;
  const ScTiers s = sc_schedule(tiles, row_tiles, heads_per_group, sms, plan_heads);
  int64_t grid = 0;
  for (int k = 0; k < 3; ++k) {
    if (out) {
      out[2 * k] = s.tiles[k];
      out[2 * k + 1] = s.items[k];
    }
    grid += s.tiles[k] * s.items[k];
  }
  return grid;
}

}  // extern "C"
