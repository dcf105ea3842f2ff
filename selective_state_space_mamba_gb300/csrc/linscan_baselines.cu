// Baseline scans of "Selective-scan CUDA kernels", section "The five kernels", rebuilt for
// GB300 so that its traffic-model study can be repeated here next to linscan_lookback (which
// is its Level 3c, redesigned).  All compute h[t] = a[t] h[t-1] + b[t] per row, h[-1] = 0,
// under the pair combine (a1,b1).(a2,b2) = (a1 a2, a2 b1 + b2) of the page's section "The
// problem".  They are deliberately the page's algorithms, not tuned variants:
//
//   Level 1   Blelloch: one CTA per row, the row's pairs in shared memory (padded against
//             bank conflicts), up-sweep then down-sweep for the exclusive prefixes; rows of
//             at most 2048 elements.  Traffic: a, b read, h written (3 arrays).
//   Level 2   three launches: (1) every 2048-element tile of a row is scanned from a zero
//             state, writing the local states and local decay products; (2) one CTA per row
//             scans the tiles' aggregates (the spine); (3) every element adds its local decay
//             product times the state entering its tile.  Traffic: 7 arrays (a, b; local h
//             and A written and read back; h).
//   Level 3   single pass, decoupled look-back over 256-element tiles claimed in counter
//             order, one element per thread; thread 0 walks the predecessors one at a time.
//   Level 3b  the same with a whole warp inspecting 32 predecessors at once.
//   Hillis-Steele  the page's PyTorch baseline algorithm, which it lists as future work in
//             CUDA: ceil(log2 L) passes over the whole array, pass d replacing every pair at
//             position t >= d of its row by (pair at t - d) . (pair at t); pairs ping-pong
//             between two workspace buffers, the last pass writes h (the b of the prefix).
//             Work-inefficient: L log L combines, ~24 bytes per element and pass.
//
// Levels 3 and 3b scan all rows as one flattened sequence with a reset at each row start
// (the combine selects the later b when its decay is 0), like linscan_lookback.  Their waits
// are bounded: past the limit the tile records SSM_ERR_TIMEOUT in the workspace status word
// and writes NaN.
#include "ssm_internal.cuh"

namespace ssm {
namespace {

struct Aff {
  float a, b;  // h -> a h + b; a == 0: absolute (a row start inside)
};
__device__ __forceinline__ Aff cat(Aff p, Aff q) {  // p first, then q
  return Aff{p.a * q.a, q.a == 0.f ? q.b : fmaf(q.a, p.b, q.b)};
}
__device__ __forceinline__ Aff shfl_up_aff(Aff v, int d) {
  return Aff{__shfl_up_sync(0xffffffffu, v.a, d), __shfl_up_sync(0xffffffffu, v.b, d)};
}
__device__ __forceinline__ Aff shfl_aff(Aff v, int src) {
  return Aff{__shfl_sync(0xffffffffu, v.a, src), __shfl_sync(0xffffffffu, v.b, src)};
}

// Scan of one Aff per thread over a CTA of kThreads threads (warp shuffles, then the warp
// totals through shared memory).  Returns the inclusive value; *excl gets the composition of
// the threads before this one, *total the CTA's.
template <int kThreads>
__device__ __forceinline__ Aff block_scan(Aff v, Aff* warp_tot, Aff* excl, Aff* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const Aff o = shfl_up_aff(v, d);
    if (lane >= d) v = cat(o, v);
  }
  Aff ex = shfl_up_aff(v, 1);
  if (lane == 0) ex = Aff{1.f, 0.f};
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  Aff before{1.f, 0.f};
  for (int w = 0; w < warp; ++w) before = cat(before, warp_tot[w]);
  Aff all = before;
  for (int w = warp; w < kThreads / 32; ++w) all = cat(all, warp_tot[w]);
  *total = all;
  *excl = cat(before, ex);
  return cat(before, v);
}

// ---------------------------------------------------------------- Level 1: Blelloch
constexpr int kBlMaxLen = 2048;
__device__ __forceinline__ int bl_pad(int i) { return i + (i >> 5); }

__global__ void __launch_bounds__(1024) scan_blelloch_kernel(const float* __restrict__ a, const float* __restrict__ b,
                                                             float* __restrict__ h, int64_t len, int n2) {
  extern __shared__ float bl_smem[];
  float* sa = bl_smem;
  float* sb = bl_smem + bl_pad(n2);
  const int64_t off = (int64_t)blockIdx.x * len;
  // each thread keeps the original elements it loaded, for the inclusive results
  float ea[2], eb[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = threadIdx.x + r * blockDim.x;
    const bool in = i < len;
    ea[r] = in ? a[off + i] : 1.f;  // identity past the end of the row
    eb[r] = in ? b[off + i] : 0.f;
    if (i < n2) {
      sa[bl_pad(i)] = ea[r];
      sb[bl_pad(i)] = eb[r];
    }
  }
  __syncthreads();
  // up-sweep: node r of level d holds the composition of its subtree (left subtree first)
  for (int d = 1; d < n2; d <<= 1) {
    for (int k = threadIdx.x; k < n2 / (2 * d); k += blockDim.x) {
      const int l = bl_pad(2 * d * k + d - 1), r = bl_pad(2 * d * k + 2 * d - 1);
      const Aff v = cat(Aff{sa[l], sb[l]}, Aff{sa[r], sb[r]});
      sa[r] = v.a;
      sb[r] = v.b;
    }
    __syncthreads();
  }
  // down-sweep: a node's value becomes the composition of everything before its subtree; its
  // left child gets that, its right child that followed by the left subtree
  if (threadIdx.x == 0) {
    sa[bl_pad(n2 - 1)] = 1.f;
    sb[bl_pad(n2 - 1)] = 0.f;
  }
  __syncthreads();
  for (int d = n2 >> 1; d >= 1; d >>= 1) {
    for (int k = threadIdx.x; k < n2 / (2 * d); k += blockDim.x) {
      const int l = bl_pad(2 * d * k + d - 1), r = bl_pad(2 * d * k + 2 * d - 1);
      const Aff left{sa[l], sb[l]}, par{sa[r], sb[r]};
      sa[l] = par.a;
      sb[l] = par.b;
      const Aff v = cat(par, left);
      sa[r] = v.a;
      sb[r] = v.b;
    }
    __syncthreads();
  }
  // exclusive prefix applied to h[-1] = 0 is the state before element i
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = threadIdx.x + r * blockDim.x;
    if (i < len) h[off + i] = fmaf(ea[r], sb[bl_pad(i)], eb[r]);
  }
}

// ---------------------------------------------------------------- Level 2: three passes
constexpr int kTpThreads = 256, kTpItems = 8, kTpTile = kTpThreads * kTpItems;  // 2048

// Pass 1: local scan of one tile from a zero state.  h <- local states, A <- local decay
// products, agg[row][tile] <- the tile's composition.
__global__ void __launch_bounds__(kTpThreads) scan3_local_kernel(const float* __restrict__ a,
                                                                 const float* __restrict__ b, float* __restrict__ h,
                                                                 float* __restrict__ A, Aff* __restrict__ agg,
                                                                 int64_t len, int tiles_per_row) {
  __shared__ Aff warp_tot[kTpThreads / 32];
  const int64_t row = blockIdx.y;
  const int tile = blockIdx.x;
  const int64_t base = row * len + (int64_t)tile * kTpTile;
  const int64_t n_here = len - (int64_t)tile * kTpTile;  // elements of the row from the tile on
  const int e0 = threadIdx.x * kTpItems;
  float va[kTpItems], vb[kTpItems];
#pragma unroll
  for (int j = 0; j < kTpItems; ++j) {
    const bool in = e0 + j < n_here;
    va[j] = in ? a[base + e0 + j] : 1.f;
    vb[j] = in ? b[base + e0 + j] : 0.f;
  }
  Aff t{1.f, 0.f};
#pragma unroll
  for (int j = 0; j < kTpItems; ++j) t = cat(t, Aff{va[j], vb[j]});
  Aff total, run;
  block_scan<kTpThreads>(t, warp_tot, &run, &total);  // run: the tile's elements before mine
#pragma unroll
  for (int j = 0; j < kTpItems; ++j) {
    run = cat(run, Aff{va[j], vb[j]});
    if (e0 + j < n_here) {
      h[base + e0 + j] = run.b;  // local state (zero entering the tile)
      A[base + e0 + j] = run.a;  // local product of decays
    }
  }
  if (threadIdx.x == 0) agg[row * tiles_per_row + tile] = total;
}

// Pass 2: one CTA per row scans its tiles' aggregates; agg[row][tile].b <- the state entering
// the tile.
__global__ void __launch_bounds__(kTpThreads) scan3_spine_kernel(Aff* __restrict__ agg, int tiles_per_row) {
  __shared__ Aff warp_tot[kTpThreads / 32];
  Aff* r = agg + (int64_t)blockIdx.x * tiles_per_row;
  const int e0 = threadIdx.x * kTpItems;  // tiles_per_row <= kTpTile
  Aff v[kTpItems];
  Aff t{1.f, 0.f};
#pragma unroll
  for (int j = 0; j < kTpItems; ++j) {
    v[j] = e0 + j < tiles_per_row ? r[e0 + j] : Aff{1.f, 0.f};
    t = cat(t, v[j]);
  }
  Aff total, run;
  block_scan<kTpThreads>(t, warp_tot, &run, &total);
  __syncthreads();  // every thread has read its aggregates before any is overwritten
#pragma unroll
  for (int j = 0; j < kTpItems; ++j) {
    if (e0 + j < tiles_per_row) r[e0 + j] = Aff{0.f, run.b};  // state entering tile e0 + j
    run = cat(run, v[j]);
  }
}

// Pass 3: h = local state + local decay product x state entering the tile.
__global__ void __launch_bounds__(kTpThreads) scan3_apply_kernel(float* __restrict__ h, const float* __restrict__ A,
                                                                 const Aff* __restrict__ agg, int64_t len,
                                                                 int tiles_per_row) {
  const int64_t row = blockIdx.y;
  const int tile = blockIdx.x;
  const int64_t base = row * len + (int64_t)tile * kTpTile;
  const int64_t n_here = len - (int64_t)tile * kTpTile;
  const float x = agg[row * tiles_per_row + tile].b;
#pragma unroll
  for (int j = 0; j < kTpItems; ++j) {
    const int e = threadIdx.x + j * kTpThreads;  // coalesced: consecutive threads, consecutive elements
    if (e < n_here) h[base + e] = fmaf(A[base + e], x, h[base + e]);
  }
}

// ---------------------------------------------------------------- Levels 3 / 3b: look-back
constexpr int kLbThreads = 256;  // one element per thread: a tile is 256 elements

// State before `tile`: thread 0 walks the predecessors one by one (serial), or warp 0
// inspects 32 at a time (warp).  Returns NaN after a wait that gave up.
template <bool kWarp>
__device__ float lb_prefix(int64_t tile, const LsDesc* desc, WsHeader* hdr, const LookbackCtl& ctl) {
  const unsigned long long want = make_flag(ctl.epoch, 0);
  const int lane = threadIdx.x & 31;
  Aff acc{1.f, 0.f};  // composition of the predecessors folded so far (newest last)
  uint64_t t0 = 0;
  uint32_t polls = 0;
  if (!kWarp) {
    for (int64_t j = tile - 1; j >= 0;) {
      unsigned long long f;
      float va, vb;
      ld_relaxed_desc(&desc[j], f, va, vb);
      if ((f & ~3ull) == want && (f & 3ull) != 0ull) {
        if ((f & 3ull) == kFlagPrefix) return fmaf(acc.a, vb, acc.b);  // acc applied to that state
        acc = cat(Aff{va, vb}, acc);
        --j;
        polls = 0;
        continue;
      }
      if (++polls == 1) t0 = global_timer_ns();
      if ((polls & 63u) == 0u) {
        if (call_aborted(hdr, ctl.epoch)) return __int_as_float(0x7fc00000);
        if (global_timer_ns() - t0 > ctl.spin_limit_ns) {
          record_error(hdr, ctl.epoch, SSM_ERR_TIMEOUT);
          return __int_as_float(0x7fc00000);
        }
      }
      if (polls > 64) __nanosleep(64);
    }
    return acc.b;  // reached the sequence start
  }
  int64_t newest = tile - 1;
  while (true) {
    const int64_t idx = newest - lane;
    bool valid = true, is_p = true;  // lanes before tile 0 count as a published zero state
    Aff v{0.f, 0.f};
    if (idx >= 0) {
      unsigned long long f;
      float va, vb;
      ld_relaxed_desc(&desc[idx], f, va, vb);
      valid = (f & ~3ull) == want && (f & 3ull) != 0ull;
      is_p = valid && (f & 3ull) == kFlagPrefix;
      v = is_p ? Aff{0.f, vb} : Aff{va, vb};
    }
    const unsigned invalid = __ballot_sync(0xffffffffu, !valid);
    const unsigned pmask = __ballot_sync(0xffffffffu, is_p);
    const int first_invalid = invalid ? __ffs(invalid) - 1 : 32;
    const int first_p = pmask ? __ffs(pmask) - 1 : 32;
    if (first_p < first_invalid || invalid == 0u) {
      const int last = first_p < 32 ? first_p : 31;  // lanes 0..last are folded, oldest first
      Aff win{1.f, 0.f};
      for (int l = last; l >= 0; --l) win = cat(win, shfl_aff(v, l));
      acc = cat(win, acc);
      if (first_p < 32) return acc.b;
      newest -= 32;
      polls = 0;
      continue;
    }
    if (++polls == 1) t0 = global_timer_ns();
    if ((polls & 31u) == 0u) {
      const bool aborted = call_aborted(hdr, ctl.epoch);
      const bool late = global_timer_ns() - t0 > ctl.spin_limit_ns;
      if (__any_sync(0xffffffffu, late) && lane == 0) record_error(hdr, ctl.epoch, SSM_ERR_TIMEOUT);
      if (__any_sync(0xffffffffu, aborted || late)) return __int_as_float(0x7fc00000);
    }
    if (polls > 64) __nanosleep(64);
  }
}

template <bool kWarp>
__global__ void __launch_bounds__(kLbThreads) scan_lookback_kernel(const float* __restrict__ a,
                                                                   const float* __restrict__ b, float* __restrict__ h,
                                                                   int64_t n, int64_t len, LsDesc* desc,
                                                                   WsHeader* hdr, LookbackCtl ctl_call) {
  const LookbackCtl ctl = device_epoch(ctl_call, hdr);
  __shared__ Aff warp_tot[kLbThreads / 32];
  __shared__ int64_t s_tile;
  __shared__ float s_x;
  if (threadIdx.x == 0) s_tile = claim_tile(hdr);  // counter order, not blockIdx (forward progress)
  __syncthreads();
  const int64_t tile = s_tile;
  const int64_t e = tile * kLbThreads + threadIdx.x;
  Aff v{1.f, 0.f};
  if (e < n) v = Aff{e % len == 0 ? 0.f : a[e], b[e]};  // a row start is a reset
  Aff total, excl;
  const Aff incl = block_scan<kLbThreads>(v, warp_tot, &excl, &total);
  // an absolute aggregate (a row start inside, or decays that underflow) is published as a
  // prefix at once; the elements before a row start still need the state entering the tile
  const bool absolute = tile == 0 || total.a == 0.f;
  const bool need_x = tile != 0 && (tile * kLbThreads) % len != 0;
  if (threadIdx.x == 0 && tile != ctl.stall_tile)
    st_relaxed_desc(&desc[tile], make_flag(ctl.epoch, absolute ? kFlagPrefix : kFlagAggregate),
                    absolute ? 0.f : total.a, total.b);
  if (need_x && (kWarp ? threadIdx.x < 32 : threadIdx.x == 0)) {
    const float x = lb_prefix<kWarp>(tile, desc, hdr, ctl);
    if (threadIdx.x == 0) {
      if (!absolute && tile != ctl.stall_tile)
        st_relaxed_desc(&desc[tile], make_flag(ctl.epoch, kFlagPrefix), 0.f, fmaf(total.a, x, total.b));
      s_x = x;
    }
  }
  __syncthreads();
  const float x = need_x ? s_x : 0.f;
  if (e < n) h[e] = incl.a == 0.f ? incl.b : fmaf(incl.a, x, incl.b);
  if (threadIdx.x == 0) retire_tile(hdr, gridDim.x);
}

// ---------------------------------------------------------------- Hillis-Steele
constexpr int kHsThreads = 256;

// One pass at distance d: out[t] = in[t - d] . in[t] where t - d is in the same row.
// bout == h and aout == nullptr on the last pass (only the states are needed).
__global__ void __launch_bounds__(kHsThreads) scan_hs_pass_kernel(const float* __restrict__ ain,
                                                                  const float* __restrict__ bin,
                                                                  float* __restrict__ aout, float* __restrict__ bout,
                                                                  int64_t n, int64_t len, int64_t d) {
  const int64_t e = (int64_t)blockIdx.x * kHsThreads + threadIdx.x;
  if (e >= n) return;
  Aff cur{ain[e], bin[e]};
  if (e % len >= d) cur = cat(Aff{ain[e - d], bin[e - d]}, cur);
  if (aout) aout[e] = cur.a;
  bout[e] = cur.b;
}

}  // namespace

size_t linscan_baseline_workspace(ssm_scan_algo algo, int64_t rows, int64_t len) {
  const int64_t n = rows * len;
  switch (algo) {
    case SSM_SCAN_BLELLOCH:
      return 0;
    case SSM_SCAN_THREE_PASS: {
      const int64_t tpr = (len + kTpTile - 1) / kTpTile;
      return (size_t)(sizeof(float) * n + 255) / 256 * 256 + sizeof(Aff) * (size_t)(rows * tpr);
    }
    case SSM_SCAN_LOOKBACK_SERIAL:
    case SSM_SCAN_LOOKBACK_WARP:
      return kHeaderBytes + sizeof(LsDesc) * (size_t)((n + kLbThreads - 1) / kLbThreads);
    case SSM_SCAN_HILLIS_STEELE:
      return 4 * ((sizeof(float) * (size_t)n + 255) / 256 * 256);  // two ping-pong pair buffers
  }
  return 0;
}

ssm_status linscan_baseline_check(ssm_scan_algo algo, int64_t rows, int64_t len) {
  if (algo == SSM_SCAN_BLELLOCH) return len <= kBlMaxLen && rows <= 0x7fffffff ? SSM_OK : SSM_ERR_UNSUPPORTED;
  if (algo == SSM_SCAN_THREE_PASS)
    return (len + kTpTile - 1) / kTpTile <= kTpTile && rows <= 65535 ? SSM_OK : SSM_ERR_UNSUPPORTED;
  if (algo == SSM_SCAN_LOOKBACK_SERIAL || algo == SSM_SCAN_LOOKBACK_WARP)
    return (rows * len + kLbThreads - 1) / kLbThreads <= 0x7fffffffLL ? SSM_OK : SSM_ERR_UNSUPPORTED;
  if (algo == SSM_SCAN_HILLIS_STEELE)
    return (rows * len + kHsThreads - 1) / kHsThreads <= 0x7fffffffLL ? SSM_OK : SSM_ERR_UNSUPPORTED;
  return SSM_ERR_INVALID_ARG;
}

cudaError_t launch_linscan_baseline(ssm_scan_algo algo, const float* a, const float* b, float* h, int64_t rows,
                                    int64_t len, void* workspace, const LookbackCtl& ctl, cudaStream_t s) {
  const int64_t n = rows * len;
  switch (algo) {
    case SSM_SCAN_BLELLOCH: {
      int n2 = 1;
      while (n2 < len) n2 <<= 1;
      const int threads = n2 / 2 < 32 ? 32 : n2 / 2;
      const size_t smem = 2 * sizeof(float) * (size_t)(n2 + (n2 >> 5));
      scan_blelloch_kernel<<<(unsigned)rows, threads, smem, s>>>(a, b, h, len, n2);
      return cudaGetLastError();
    }
    case SSM_SCAN_THREE_PASS: {
      const int tpr = (int)((len + kTpTile - 1) / kTpTile);
      float* A = static_cast<float*>(workspace);
      Aff* agg = reinterpret_cast<Aff*>(static_cast<char*>(workspace) + (sizeof(float) * n + 255) / 256 * 256);
      const dim3 grid((unsigned)tpr, (unsigned)rows);
      scan3_local_kernel<<<grid, kTpThreads, 0, s>>>(a, b, h, A, agg, len, tpr);
      scan3_spine_kernel<<<(unsigned)rows, kTpThreads, 0, s>>>(agg, tpr);
      scan3_apply_kernel<<<grid, kTpThreads, 0, s>>>(h, A, agg, len, tpr);
      return cudaGetLastError();
    }
    case SSM_SCAN_LOOKBACK_SERIAL:
    case SSM_SCAN_LOOKBACK_WARP: {
      WsHeader* hdr = static_cast<WsHeader*>(workspace);
      LsDesc* desc = reinterpret_cast<LsDesc*>(static_cast<char*>(workspace) + kHeaderBytes);
      const int64_t tiles = (n + kLbThreads - 1) / kLbThreads;
      if (algo == SSM_SCAN_LOOKBACK_SERIAL)
        scan_lookback_kernel<false><<<(unsigned)tiles, kLbThreads, 0, s>>>(a, b, h, n, len, desc, hdr, ctl);
      else
        scan_lookback_kernel<true><<<(unsigned)tiles, kLbThreads, 0, s>>>(a, b, h, n, len, desc, hdr, ctl);
      return cudaGetLastError();
    }
    case SSM_SCAN_HILLIS_STEELE: {
      if (len == 1) return cudaMemcpyAsync(h, b, sizeof(float) * (size_t)n, cudaMemcpyDeviceToDevice, s);
      const size_t arr = (sizeof(float) * (size_t)n + 255) / 256 * 256;
      char* w = static_cast<char*>(workspace);
      float* buf_a[2] = {reinterpret_cast<float*>(w), reinterpret_cast<float*>(w + 2 * arr)};
      float* buf_b[2] = {reinterpret_cast<float*>(w + arr), reinterpret_cast<float*>(w + 3 * arr)};
      const unsigned grid = (unsigned)((n + kHsThreads - 1) / kHsThreads);
      const float* ain = a;
      const float* bin = b;
      int nb = 0;
      for (int64_t d = 1; d < len; d <<= 1) {
        const bool last = 2 * d >= len;
        float* aout = last ? nullptr : buf_a[nb];
        float* bout = last ? h : buf_b[nb];
        scan_hs_pass_kernel<<<grid, kHsThreads, 0, s>>>(ain, bin, aout, bout, n, len, d);
        ain = buf_a[nb];
        bin = buf_b[nb];
        nb ^= 1;
      }
      return cudaGetLastError();
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace ssm
