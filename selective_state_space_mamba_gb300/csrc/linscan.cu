// linscan_lookback: the scalar selective scan h[t] = a[t] h[t-1] + b[t] ("Selective-scan
// CUDA kernels", section "The problem") as ONE single-pass decoupled look-back prefix scan
// (same page, "The five kernels", Levels 3 / 3b / 3c: tiles claimed with an atomic counter,
// aggregates published with flag A and inclusive prefixes with flag P, a whole warp
// inspecting 32 predecessors at once, several items per thread scanned in registers).
//
// GB300 layout choices (not on the page):
//   * all rows are scanned as ONE flattened sequence of rows*len elements, with a reset at
//     every row start.  Tiles then never straddle a misaligned row base, every load and
//     store is a 16-byte vector, and a tile that contains a row start publishes its prefix
//     immediately (its aggregate is absolute), which cuts the look-back chains at rows.
//   * within a tile, warp w owns 512 consecutive elements as 4 runs of 128; in each run lane
//     i owns 4 consecutive elements, so every float4 load/store instruction of a warp covers
//     512 contiguous bytes.
//   * a reset is an element whose decay is replaced by 0, and the combine SELECTS the later
//     operand's b when its decay is 0 instead of multiplying by 0, so an overflowed
//     predecessor can never turn a fresh row into NaN.
#include "ssm_internal.cuh"

namespace ssm {
namespace {

struct Pair {
  float a, b;  // the affine map h -> a*h + b; a == 0 marks "absolute" (reset inside)
};

// p is the earlier segment, q the later one: (a1,b1).(a2,b2) = (a1 a2, a2 b1 + b2).
__device__ __forceinline__ Pair combine(Pair p, Pair q) {
  Pair r;
  r.a = p.a * q.a;
  r.b = (q.a == 0.f) ? q.b : fmaf(q.a, p.b, q.b);
  return r;
}
__device__ __forceinline__ float apply(Pair p, float h_prev) { return (p.a == 0.f) ? p.b : fmaf(p.a, h_prev, p.b); }

__device__ __forceinline__ Pair shfl_up(Pair p, int d) {
  Pair r;
  r.a = __shfl_up_sync(0xffffffffu, p.a, d);
  r.b = __shfl_up_sync(0xffffffffu, p.b, d);
  return r;
}
__device__ __forceinline__ Pair shfl(Pair p, int src) {
  Pair r;
  r.a = __shfl_sync(0xffffffffu, p.a, src);
  r.b = __shfl_sync(0xffffffffu, p.b, src);
  return r;
}

__global__ void __launch_bounds__(kLsThreads) linscan_lookback_kernel(
    const float* __restrict__ a, const float* __restrict__ b, float* __restrict__ h, int64_t n, int64_t len,
    LinscanWorkspace ws, LookbackCtl ctl) {
  __shared__ uint32_t s_tile;
  __shared__ Pair s_warp[kLsThreads / 32];
  __shared__ Pair s_prefix;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_tile = claim_tile(ws.hdr);
  __syncthreads();
  const int64_t tile = s_tile;
  if (tile >= ws.tiles) {  // claim counter not reset (workspace not zero-filled): refuse
    if (threadIdx.x == 0) {
      record_error(ws.hdr, ctl.epoch, SSM_ERR_WORKSPACE);
      retire_tile(ws.hdr, (uint32_t)ws.tiles);
    }
    return;
  }
  const int64_t tile_base = tile * kLsTile;

  // ---- load 4 runs of 4 consecutive elements (16-byte vectors, coalesced per warp) ----
  float va[kLsRuns][4], vb[kLsRuns][4];
#pragma unroll
  for (int k = 0; k < kLsRuns; ++k) {
    const int64_t e0 = tile_base + warp * 512 + k * 128 + lane * 4;
    if (e0 + 3 < n) {
      const float4 fa = __ldcs(reinterpret_cast<const float4*>(a + e0));
      const float4 fb = __ldcs(reinterpret_cast<const float4*>(b + e0));
      va[k][0] = fa.x; va[k][1] = fa.y; va[k][2] = fa.z; va[k][3] = fa.w;
      vb[k][0] = fb.x; vb[k][1] = fb.y; vb[k][2] = fb.z; vb[k][3] = fb.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool in = e0 + j < n;
        va[k][j] = in ? a[e0 + j] : 1.f;  // identity beyond the end
        vb[k][j] = in ? b[e0 + j] : 0.f;
      }
    }
  }

  // ---- row starts become resets; per-lane inclusive scan of each run ----
  Pair ex[kLsRuns][4];  // element prefixes, relative to the start of the lane's run
  Pair lane_tot[kLsRuns];
#pragma unroll
  for (int k = 0; k < kLsRuns; ++k) {
    const int64_t e0 = tile_base + warp * 512 + k * 128 + lane * 4;
    int64_t m = e0 % len;  // position of the first element within its row
    Pair acc{1.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      Pair q{m == 0 ? 0.f : va[k][j], vb[k][j]};
      acc = (j == 0) ? q : combine(acc, q);
      ex[k][j] = acc;
      if (++m == len) m = 0;
    }
    lane_tot[k] = acc;
  }

  // ---- warp scan of each run, chained across the 4 runs ----
  Pair carry{1.f, 0.f};  // composition of the warp's earlier runs
#pragma unroll
  for (int k = 0; k < kLsRuns; ++k) {
    Pair inc = lane_tot[k];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      Pair o = shfl_up(inc, d);
      if (lane >= d) inc = combine(o, inc);
    }
    Pair excl = shfl_up(inc, 1);
    if (lane == 0) excl = Pair{1.f, 0.f};
    const Pair lane_prefix = combine(carry, excl);  // everything in the warp before this lane's run
#pragma unroll
    for (int j = 0; j < 4; ++j) ex[k][j] = combine(lane_prefix, ex[k][j]);
    carry = combine(carry, shfl(inc, 31));
  }
  if (lane == 0) s_warp[warp] = carry;
  __syncthreads();

  // ---- block scan of warp aggregates; thread 0 publishes the tile aggregate ----
  Pair warp_prefix{1.f, 0.f};
  Pair tile_agg{1.f, 0.f};
#pragma unroll
  for (int w = 0; w < kLsThreads / 32; ++w) {
    if (w == warp) warp_prefix = tile_agg;
    tile_agg = combine(tile_agg, s_warp[w]);
  }
  const bool stalled = (int64_t)tile == ctl.stall_tile;
  const bool absolute = (tile == 0) || (tile_agg.a == 0.f);
  if (threadIdx.x == 0 && !stalled) {
    if (absolute) {
      ws.inc[tile] = float2{0.f, tile_agg.b};
    } else {
      ws.agg[tile] = float2{tile_agg.a, tile_agg.b};
    }
    __threadfence();
    st_release_u64(&ws.flags[tile], make_flag(ctl.epoch, absolute ? kFlagPrefix : kFlagAggregate));
  }

  // ---- decoupled look-back by warp 0 (32 predecessors per step) ----
  // The first element of a tile that starts a row needs no prefix; neither does tile 0.
  const bool need_prefix = (tile != 0) && (tile_base % len != 0);
  if (warp == 0) {
    Pair acc{1.f, 0.f};  // composition of the predecessors inspected so far (newest last)
    if (need_prefix) {
      int64_t newest = tile - 1;
      while (true) {
        const int64_t idx = newest - lane;
        uint32_t kind = kFlagPrefix;
        Pair v{0.f, 0.f};
        if (idx >= 0) {
          kind = wait_flag(&ws.flags[idx], ws.hdr, ctl);
          if (kind == kFlagPrefix) {
            float2 f = ld_relaxed_f2(&ws.inc[idx]);
            v = Pair{0.f, f.y};
          } else if (kind == kFlagAggregate) {
            float2 f = ld_relaxed_f2(&ws.agg[idx]);
            v = Pair{f.x, f.y};
          } else {
            v = Pair{0.f, __int_as_float(0x7fc00000)};  // gave up: poison, flagged in status
            kind = kFlagPrefix;
          }
        }
        const unsigned pmask = __ballot_sync(0xffffffffu, kind == kFlagPrefix);
        const int last = pmask ? (__ffs(pmask) - 1) : 31;  // lanes 0..last are used
        // Fold lanes last..0 (oldest first) into the accumulated composition.
        Pair win{1.f, 0.f};
        for (int l = last; l >= 0; --l) win = combine(win, shfl(v, l));
        acc = combine(win, acc);
        if (pmask) break;
        newest -= 32;
      }
    }
    if (lane == 0) {
      s_prefix = acc;
      if (!stalled && !absolute) {
        const Pair incl = combine(acc, tile_agg);
        ws.inc[tile] = float2{0.f, incl.b};
        __threadfence();
        st_release_u64(&ws.flags[tile], make_flag(ctl.epoch, kFlagPrefix));
      }
    }
  }
  __syncthreads();
  const float h_in = s_prefix.b;  // state just before the tile (unused where not needed)

  // ---- apply and store ----
#pragma unroll
  for (int k = 0; k < kLsRuns; ++k) {
    const int64_t e0 = tile_base + warp * 512 + k * 128 + lane * 4;
    float o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = apply(combine(warp_prefix, ex[k][j]), h_in);
    if (e0 + 3 < n) {
      __stcs(reinterpret_cast<float4*>(h + e0), make_float4(o[0], o[1], o[2], o[3]));
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (e0 + j < n) h[e0 + j] = o[j];
    }
  }
  if (threadIdx.x == 0) retire_tile(ws.hdr, (uint32_t)ws.tiles);
}

}  // namespace

cudaError_t launch_linscan(const float* a, const float* b, float* h, int64_t rows, int64_t len,
                           const LinscanWorkspace& ws, const LookbackCtl& ctl, cudaStream_t s) {
  const int64_t n = rows * len;
  linscan_lookback_kernel<<<(unsigned)ws.tiles, kLsThreads, 0, s>>>(a, b, h, n, len, ws, ctl);
  return cudaGetLastError();
}

}  // namespace ssm
