// linscan_lookback: the scalar selective scan h[t] = a[t] h[t-1] + b[t] ("Selective-scan
// CUDA kernels", section "The problem") as ONE single-pass decoupled look-back prefix scan
// (same page, "The five kernels", Levels 3 / 3b / 3c: tiles claimed with an atomic counter,
// aggregates published with flag A and inclusive prefixes with flag P, a whole warp
// inspecting 32 predecessors at once, several items per thread scanned in registers).
//
// GB300 design choices (not on the page):
//   * all rows are scanned as ONE flattened sequence of rows*len elements, viewed as a 2-D
//     tensor of 128-byte lines (32 floats), with a reset at every row start.  A tile is
//     kLsLines consecutive lines; each consumer thread owns kLsElems consecutive elements of
//     one line, so a thread scans sequentially in registers and a warp needs one shuffle
//     scan per tile.
//   * tiles move by TMA: the producer warp loads a and b with 2-D tensor copies in 128-byte
//     swizzle mode (a thread reading its own line then hits 8 different bank groups per
//     quarter-warp: conflict-free), and h goes back to the same swizzled buffer and out with
//     a TMA tensor store.  Loads and stores are fully coalesced and asynchronous.
//   * persistent, warp-specialised CTAs: one producer warp claims tiles (atomic counter) and
//     fills a ring of shared-memory stages ("full" / "empty" mbarriers).  For rows of several
//     tiles (one CTA per SM, 7 stages) two groups of consumer warps take the CTA's tiles in
//     turn (for short rows, two CTAs per SM, 3 stages and one group); one look-back
//     warp resolves tile i's prefix while the group that owns it runs the first pass of its
//     next tile, i + 2 (its second pass then re-reads tile i from its stage), so the
//     look-back has two tiles' time and is off the consumers' path, and the two groups'
//     chains of waits overlap; one store warp issues the TMA store of each finished tile and
//     hands its stage back to the producer once the store has read it.  Claims stay in
//     counter order and each CTA consumes its claims in order (the groups alternate, the
//     look-back and store warps serve tiles in order), so the page's forward-progress
//     argument holds: the smallest
//     unfinished tile is always some CTA's current tile (its data arrives without waiting on
//     anything) and it waits only on smaller tiles.
//   * a tile's flag and value share one 16-byte descriptor (no fence between value and flag),
//     and the look-back stops at the nearest published prefix instead of waiting for all 32
//     inspected predecessors.  A tile holding a row start publishes its prefix at once (its
//     aggregate is absolute), which cuts look-back chains at rows.
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

struct LsStage {  // two [kLsLines x 32] float boxes in 128-byte swizzled layout
  float a[kLsTile];
  float b[kLsTile];  // h is written back over a
};
static_assert(kLsRow % (4 * kLsSplit) == 0, "a thread owns whole 16-byte chunks");
struct LsJob {        // consumer -> look-back warp, 2 x groups slots by tile index
  int64_t tile;      // >= tiles: stop
  int64_t r0;
  Pair agg;          // tile aggregate
  float prefix;      // look-back warp -> consumers: state before the tile
  int absolute;
};
// The CTA's shape: G consumer groups taking tiles in turn, an S-stage ring.  With one group a
// tile's second pass runs while the same warps scan the next tile; with two, while they scan
// the tile after that, so the look-back of a tile has two tiles' time.
template <int G, int S, int kCtasPerSm>
struct LsCfg {
  static constexpr int kGroups = G, kStages = S, kJobs = 2 * G, kMinBlocks = kCtasPerSm;
  static constexpr int kConsumers = G * kLsThreads;
  static constexpr int kBlock = kConsumers + 96;  // consumer warps + producer, look-back and store warps
};
#ifndef SSM_LS_LONG_STAGES
#define SSM_LS_LONG_STAGES 7
#endif
using LsLongRows = LsCfg<2, SSM_LS_LONG_STAGES, 1>;  // one CTA per SM (224 KB of stages)
using LsShortRows = LsCfg<1, 3, 2>;  // two CTAs per SM (96 KB of stages each)
// further CTA shapes the per-size tuner (ssm_linscan_fwd_tune) chooses among
using LsTwoGroups6 = LsCfg<2, 6, 1>;  // two groups, 6 stages, one CTA per SM
using LsOneGroup6 = LsCfg<1, 6, 1>;   // one group, 6 stages, one CTA per SM

template <class Cfg>
struct LsShared {
  LsStage stage[Cfg::kStages];   // first member: 1024-byte aligned (swizzle atom)
  uint64_t full[Cfg::kStages];   // producer -> consumers: tile id written, data landed
  uint64_t empty[Cfg::kStages];  // consumers -> producer: stage read and stored, may be refilled
  uint64_t lb_req[Cfg::kJobs];   // consumers -> look-back warp: job posted
  uint64_t lb_done[Cfg::kJobs];  // look-back warp -> consumers: prefix posted
  uint64_t st_req[Cfg::kStages]; // consumers -> store warp: stage holds a finished tile (or stop)
  int64_t st_line0[Cfg::kStages];// first line of that tile (< 0: stop)
  int64_t tile[Cfg::kStages];
  int64_t r0[Cfg::kStages];      // position of the tile's first element within its row
  LsJob job[Cfg::kJobs];
  Pair warp_agg[Cfg::kGroups][2][kLsThreads / 32];
};
static_assert(sizeof(LsStage) % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
static_assert(sizeof(LsShared<LsLongRows>) + 1024 <= 227 * 1024, "the long-row ring must fit one CTA's shared memory");

constexpr uint32_t kLsConsumerBar = 1;       // named barrier of consumer group g: 1 + g

struct LsArgs {
  const float* a;
  const float* b;
  float* h;
  int64_t n;      // rows * len
  int64_t len;
  int64_t lines;  // n / 32: full 128-byte lines covered by the tensor maps (0: no TMA)
};

// Position within its row of element e0 of a tile whose first element sits at r0 (< len):
// (r0 + e0) mod len, without a division when rows are at least a tile long.
__device__ __forceinline__ int64_t row_pos(int64_t r0, int e0, int64_t len) {
  if (len >= kLsTile) {
    const int64_t v = r0 + e0;
    return v >= len ? v - len : v;
  }
  return (r0 + e0) % len;
}

// Shared-memory word index of 16-byte chunk `chunk` (0..7) of line `line` in the 128-byte
// swizzled box.  The eight lanes of a quarter-warp read eight different bank groups.
__device__ __forceinline__ int swz(int line, int chunk) { return line * kLsRow + ((chunk ^ (line & 7)) << 2); }

// Producer (one thread): claim tiles in counter order and fill the stage ring; it ends after
// the first claim past the last tile, which it hands on as one sentinel per consumer group.  Each claim is made
// one tile ahead, so the atomic's round trip overlaps the wait for a free stage.  Progress is
// unchanged: the smallest unfinished tile, if it is only claimed, waits for a stage that
// holds smaller tiles, all of which are finished.
template <class Cfg>
__device__ void ls_producer(LsShared<Cfg>& sh, const LsArgs& p, const CUtensorMap* map_a, const CUtensorMap* map_b,
                            const LinscanWorkspace& ws, const LookbackCtl& ctl) {
  int64_t tile = claim_tile(ws.hdr);
  int stops = 0;
#if SSM_LS_STREAM_HINT
  const uint64_t pol = l2_evict_first_policy();
#endif
  for (int i = 0;; ++i) {
    const int st = i % Cfg::kStages;
    const int use = i / Cfg::kStages;
    if (use > 0 && !mbar_wait(&sh.empty[st], (uint32_t)(use - 1) & 1u, ctl.spin_limit_ns)) {
      record_error(ws.hdr, ctl.epoch, SSM_ERR_TIMEOUT);
      return;  // the consumers give up on their own bounded wait
    }
    sh.tile[st] = tile;
    if (tile >= ws.tiles) {
      mbar_arrive(&sh.full[st]);  // sentinel, no data
      if (++stops == Cfg::kGroups) return;  // every consumer group takes one
      continue;
    }
    sh.r0[st] = (tile * kLsTile) % p.len;
    const int64_t line0 = tile * kLsLines;
    if (line0 < p.lines) {
      // the whole box counts toward the transaction, rows past the tensor are zero-filled
      mbar_arrive_expect_tx(&sh.full[st], 2u * (uint32_t)sizeof(float) * kLsTile);
#if SSM_LS_STREAM_HINT
      tma_load_2d_hint(sh.stage[st].a, map_a, 0, (int)line0, &sh.full[st], pol);
      tma_load_2d_hint(sh.stage[st].b, map_b, 0, (int)line0, &sh.full[st], pol);
#else
      tma_load_2d(sh.stage[st].a, map_a, 0, (int)line0, &sh.full[st]);
      tma_load_2d(sh.stage[st].b, map_b, 0, (int)line0, &sh.full[st]);
#endif
    } else {
      mbar_arrive(&sh.full[st]);  // only the ragged tail: consumers read it directly
    }
    tile = claim_tile(ws.hdr);
  }
}

// Consumer warp 0: state just before `tile`, by decoupled look-back.  Lanes poll the
// descriptors of 32 predecessors; the window is complete once every lane up to the nearest
// published prefix (P) is valid, so a tile never waits on predecessors older than that P.
// Without a P in a complete window the 32 aggregates are folded in and the window moves
// back.  Bounded: past the limit it records SSM_ERR_TIMEOUT and yields NaN.
__device__ __forceinline__ float lookback(int64_t tile, const LinscanWorkspace& ws, const LookbackCtl& ctl,
                                          int lane) {
  Pair acc{1.f, 0.f};  // composition of the predecessors folded so far (newest last)
  int64_t newest = tile - 1;
  uint64_t t0 = 0;
  uint32_t polls = 0;
  const unsigned long long want = make_flag(ctl.epoch, 0);
  while (true) {
    const int64_t idx = newest - lane;
    bool valid = true, is_p = true;  // lanes before tile 0 count as a published zero prefix
    Pair v{0.f, 0.f};
    if (idx >= 0) {
      unsigned long long f;
      float va, vb;
      ld_relaxed_desc(&ws.desc[idx], f, va, vb);
      valid = (f & ~3ull) == want && (f & 3ull) != 0ull;
      is_p = valid && (f & 3ull) == kFlagPrefix;
      v = is_p ? Pair{0.f, vb} : Pair{va, vb};
    }
    const unsigned invalid = __ballot_sync(0xffffffffu, !valid);
    const unsigned pmask = __ballot_sync(0xffffffffu, is_p);
    const int first_invalid = invalid ? __ffs(invalid) - 1 : 32;
    const int first_p = pmask ? __ffs(pmask) - 1 : 32;
    if (first_p < first_invalid || invalid == 0u) {
      const int last = first_p < 32 ? first_p : 31;  // lanes 0..last are folded
      Pair win{1.f, 0.f};
      for (int l = last; l >= 0; --l) win = combine(win, shfl(v, l));
      acc = combine(win, acc);
      if (first_p < 32) return acc.b;
      newest -= 32;
      polls = 0;
      continue;
    }
    // a predecessor before the nearest prefix has not published yet: poll again (bounded)
    if (++polls == 1) t0 = global_timer_ns();
    if ((polls & 31u) == 0u) {
      const bool aborted = call_aborted(ws.hdr, ctl.epoch);
      const bool late = global_timer_ns() - t0 > ctl.spin_limit_ns;
      if (__any_sync(0xffffffffu, late) && lane == 0) record_error(ws.hdr, ctl.epoch, SSM_ERR_TIMEOUT);
      if (__any_sync(0xffffffffu, aborted || late)) return __int_as_float(0x7fc00000);
    }
    if (polls > 64) __nanosleep(64);
  }
}

// Look-back warp: serve the consumers' jobs in order until the stop job.
template <class Cfg>
__device__ void ls_lookback_warp(LsShared<Cfg>& sh, const LinscanWorkspace& ws, const LookbackCtl& ctl, int lane) {
  for (int j = 0;; ++j) {
    if (!mbar_wait(&sh.lb_req[j % Cfg::kJobs], (uint32_t)(j / Cfg::kJobs) & 1u, ctl.spin_limit_ns)) {
      if (lane == 0) record_error(ws.hdr, ctl.epoch, SSM_ERR_TIMEOUT);
      return;
    }
    LsJob& job = sh.job[j % Cfg::kJobs];
    const int64_t tile = job.tile;
    if (tile >= ws.tiles) return;
    const bool need_prefix = (tile != 0) && (job.r0 != 0);
    const float x = need_prefix ? lookback(tile, ws, ctl, lane) : 0.f;
    if (lane == 0) {
      if (tile != ctl.stall_tile && !job.absolute)
        st_relaxed_desc(&ws.desc[tile], make_flag(ctl.epoch, kFlagPrefix), 0.f, apply(job.agg, x));
      job.prefix = x;
      mbar_arrive(&sh.lb_done[j % Cfg::kJobs]);
    }
    __syncwarp();
  }
}

// Store warp (one thread): in tile order, TMA-store each finished stage, wait until the store
// has read it, and hand the stage back to the producer; stops at the stop job.
template <class Cfg>
__device__ void ls_store_warp(LsShared<Cfg>& sh, const CUtensorMap* map_h, const LinscanWorkspace& ws,
                              const LookbackCtl& ctl) {
#if SSM_LS_STREAM_HINT
  const uint64_t pol = l2_evict_first_policy();
#endif
  for (int j = 0;; ++j) {
    const int st = j % Cfg::kStages;
    if (!mbar_wait(&sh.st_req[st], (uint32_t)(j / Cfg::kStages) & 1u, ctl.spin_limit_ns)) {
      record_error(ws.hdr, ctl.epoch, SSM_ERR_TIMEOUT);
      break;
    }
    const int64_t line0 = sh.st_line0[st];
    if (line0 < 0) break;
    if (line0 < (int64_t)0x7fffffff && line0 >= 0) {
#if SSM_LS_STREAM_HINT
      tma_store_2d_hint(map_h, sh.stage[st].a, 0, (int)line0, pol);
#else
      tma_store_2d(map_h, sh.stage[st].a, 0, (int)line0);
#endif
      bulk_commit();
      bulk_wait_read<0>();
    }
    mbar_arrive(&sh.empty[st]);
  }
  bulk_wait<0>();  // every store of this CTA has completed
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kBlock, Cfg::kMinBlocks)
    linscan_lookback_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                            const __grid_constant__ CUtensorMap map_h, LsArgs p, LinscanWorkspace ws,
                            LookbackCtl ctl_call) {
  extern __shared__ unsigned char ls_smem_raw[];
  // align the stage ring to the 1024-byte swizzle atom (the launch adds 1 KB of slack)
  const uint32_t raw = smem_addr(ls_smem_raw);
  LsShared<Cfg>& sh = *reinterpret_cast<LsShared<Cfg>*>(ls_smem_raw + ((1024u - (raw & 1023u)) & 1023u));
  const LookbackCtl ctl = device_epoch(ctl_call, ws.hdr);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int grp = threadIdx.x / kLsThreads;            // consumer group: tiles it with it % Cfg::kGroups == grp
  const int t = threadIdx.x % kLsThreads;              // consumer thread within its group
  const uint32_t cbar = kLsConsumerBar + grp;
  const int my_line = t / kLsSplit;                    // line within the tile
  const int my_chunk0 = (t % kLsSplit) * (kLsElems / 4);  // first 16-byte chunk of the line

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int s = 0; s < Cfg::kJobs; ++s) {
      mbar_init(&sh.lb_req[s], 1);
      mbar_init(&sh.lb_done[s], 1);
    }
    for (int s = 0; s < Cfg::kStages; ++s) mbar_init(&sh.st_req[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == Cfg::kConsumers / 32) {  // producer warp
    if (lane == 0) ls_producer(sh, p, &map_a, &map_b, ws, ctl);
    return;
  }
  if (warp == Cfg::kConsumers / 32 + 1) {  // look-back warp
    ls_lookback_warp(sh, ws, ctl, lane);
    return;
  }
  if (warp == Cfg::kConsumers / 32 + 2) {  // store warp
    if (lane == 0) ls_store_warp(sh, &map_h, ws, ctl);
    return;
  }

  // per-thread results of pass 1 of the previous tile, consumed by its pass 2
  Pair prev_excl{1.f, 0.f}, prev_wp{1.f, 0.f};
  int64_t prev_tile = -1, prev_r0 = 0;
  for (int it = grp;; it += Cfg::kGroups) {
    const int st = it % Cfg::kStages;
    // A wait that gave up in any consumer stops all of them, so that none is left behind in
    // a later barrier.
    const bool got = mbar_wait(&sh.full[st], (uint32_t)(it / Cfg::kStages) & 1u, ctl.spin_limit_ns);
    const bool gave_up = named_bar_any(cbar, kLsThreads, !got);
    if (gave_up && t == 0) record_error(ws.hdr, ctl.epoch, SSM_ERR_TIMEOUT);
    const int64_t tile = gave_up ? ws.tiles : sh.tile[st];  // ws.tiles: stop
    const bool valid = tile < ws.tiles;  // uniform across the consumers
    Pair cur_excl{1.f, 0.f}, cur_wp{1.f, 0.f};
    int64_t cur_r0 = 0;

    // ================= pass 1 of this tile: aggregate, publish, post the look-back job =====
    if (valid) {
      cur_r0 = sh.r0[st];
      const int64_t tile_base = tile * kLsTile;
      const bool in_map = tile * kLsLines + my_line < p.lines;
      const int e0 = t * kLsElems;
      const int nv = (int)min(int64_t(kLsTile), p.n - tile_base);
      const float* sa = sh.stage[st].a;
      const float* sb = sh.stage[st].b;
      Pair tot{1.f, 0.f};
      int64_t m = row_pos(cur_r0, e0, p.len);  // position of my first element within its row
      // no row starts among my elements: the plain combine, without the per-element row logic
      const bool no_reset = m != 0 && m + kLsElems <= p.len;
#pragma unroll
      for (int c = 0; c < kLsElems / 4; ++c) {
        float va[4], vb[4];
        if (in_map) {
          const float4 fa = *reinterpret_cast<const float4*>(&sa[swz(my_line, my_chunk0 + c)]);
          const float4 fb = *reinterpret_cast<const float4*>(&sb[swz(my_line, my_chunk0 + c)]);
          va[0] = fa.x; va[1] = fa.y; va[2] = fa.z; va[3] = fa.w;
          vb[0] = fb.x; vb[1] = fb.y; vb[2] = fb.z; vb[3] = fb.w;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int e = e0 + 4 * c + j;
            va[j] = e < nv ? p.a[tile_base + e] : 1.f;  // identity past the end
            vb[j] = e < nv ? p.b[tile_base + e] : 0.f;
          }
        }
        if (no_reset) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const Pair q{va[j], vb[j]};
            tot = (c == 0 && j == 0) ? q : combine(tot, q);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const Pair q{m == 0 ? 0.f : va[j], vb[j]};
            tot = (c == 0 && j == 0) ? q : combine(tot, q);
            if (++m == p.len) m = 0;
          }
        }
      }
      Pair inc = tot;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const Pair o = shfl_up(inc, d);
        if (lane >= d) inc = combine(o, inc);
      }
      cur_excl = shfl_up(inc, 1);
      if (lane == 0) cur_excl = Pair{1.f, 0.f};
      const int gw = t >> 5;  // warp within the group
      if (lane == 31) sh.warp_agg[grp][(it / Cfg::kGroups) & 1][gw] = inc;
      named_bar_sync(cbar, kLsThreads);
      Pair tile_agg{1.f, 0.f};
#pragma unroll
      for (int w = 0; w < kLsThreads / 32; ++w) {
        if (w == gw) cur_wp = tile_agg;
        tile_agg = combine(tile_agg, sh.warp_agg[grp][(it / Cfg::kGroups) & 1][w]);
      }
      if (t == 0) {
        const bool absolute = (tile == 0) || (tile_agg.a == 0.f);
        if (tile != ctl.stall_tile)
          st_relaxed_desc(&ws.desc[tile], make_flag(ctl.epoch, absolute ? kFlagPrefix : kFlagAggregate),
                          absolute ? 0.f : tile_agg.a, tile_agg.b);
        LsJob& job = sh.job[it % Cfg::kJobs];
        job.tile = tile;
        job.r0 = cur_r0;
        job.agg = tile_agg;
        job.absolute = absolute;
        mbar_arrive(&sh.lb_req[it % Cfg::kJobs]);
      }
    } else if (t == 0) {
      sh.job[it % Cfg::kJobs].tile = ws.tiles;  // stop the look-back warp
      mbar_arrive(&sh.lb_req[it % Cfg::kJobs]);
    }

    // ======= pass 2 of this group's previous tile: apply its prefix, store ===================
    if (prev_tile >= 0) {
      const int pit = it - Cfg::kGroups;
      const int ps = pit % Cfg::kStages;
      const int pj = pit % Cfg::kJobs;
      float x = __int_as_float(0x7fc00000);
      if (mbar_wait(&sh.lb_done[pj], (uint32_t)(pit / Cfg::kJobs) & 1u, ctl.spin_limit_ns)) {
        x = sh.job[pj].prefix;
      } else if (t == 0) {
        record_error(ws.hdr, ctl.epoch, SSM_ERR_TIMEOUT);
      }
      const int64_t tile_base = prev_tile * kLsTile;
      const int64_t line0 = prev_tile * kLsLines;
      const bool in_map = line0 + my_line < p.lines;
      const int e0 = t * kLsElems;
      const int nv = (int)min(int64_t(kLsTile), p.n - tile_base);
      float* sa = sh.stage[ps].a;
      const float* sb = sh.stage[ps].b;
      float hcur = apply(prev_excl, apply(prev_wp, x));  // state before my line
      int64_t m = row_pos(prev_r0, e0, p.len);
      const bool no_reset = m != 0 && m + kLsElems <= p.len;
#pragma unroll
      for (int c = 0; c < kLsElems / 4; ++c) {
        float va[4], vb[4];
        if (in_map) {
          const float4 fa = *reinterpret_cast<const float4*>(&sa[swz(my_line, my_chunk0 + c)]);
          const float4 fb = *reinterpret_cast<const float4*>(&sb[swz(my_line, my_chunk0 + c)]);
          va[0] = fa.x; va[1] = fa.y; va[2] = fa.z; va[3] = fa.w;
          vb[0] = fb.x; vb[1] = fb.y; vb[2] = fb.z; vb[3] = fb.w;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int e = e0 + 4 * c + j;
            va[j] = e < nv ? p.a[tile_base + e] : 1.f;
            vb[j] = e < nv ? p.b[tile_base + e] : 0.f;
          }
        }
        float o[4];
        if (no_reset) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            hcur = fmaf(va[j], hcur, vb[j]);
            o[j] = hcur;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            hcur = (m == 0) ? vb[j] : fmaf(va[j], hcur, vb[j]);
            o[j] = hcur;
            if (++m == p.len) m = 0;
          }
        }
        if (in_map) {
          *reinterpret_cast<float4*>(&sa[swz(my_line, my_chunk0 + c)]) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (e0 + 4 * c + j < nv) p.h[tile_base + e0 + 4 * c + j] = o[j];
        }
      }
      if (in_map) fence_proxy_async_smem();
      named_bar_sync(cbar, kLsThreads);
      if (t == 0) {  // hand the stage to the store warp (no store for the tail-only tile)
        sh.st_line0[ps] = line0 < p.lines ? line0 : (int64_t)0x7fffffff;
        mbar_arrive(&sh.st_req[ps]);
      }
    }
    if (!valid) {
      if (t == 0) {  // stop the store warp through the (dataless) sentinel stage
        sh.st_line0[st] = -1;
        mbar_arrive(&sh.st_req[st]);
      }
      break;
    }
    prev_tile = tile;
    prev_r0 = cur_r0;
    prev_excl = cur_excl;
    prev_wp = cur_wp;
  }
  named_bar_sync(kLsConsumerBar + Cfg::kGroups, Cfg::kConsumers);  // every group is done
  if (threadIdx.x == 0) retire_tile(ws.hdr, gridDim.x);
}

// Grid (resident CTAs: every CTA of a launch runs at once) per device and CTA shape.
int g_ls_grid[4][64] = {};

template <class Cfg>
cudaError_t launch_cfg(int slot, int dev, const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_h,
                       const LsArgs& p, const LinscanWorkspace& ws, const LookbackCtl& ctl, cudaStream_t s) {
  cudaError_t e;
  const size_t smem = sizeof(LsShared<Cfg>) + 1024;  // + alignment slack
  if (g_ls_grid[slot][dev] == 0) {
    e = cudaFuncSetAttribute(linscan_lookback_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, linscan_lookback_kernel<Cfg>, Cfg::kBlock,
                                                           smem)) != cudaSuccess)
      return e;
    g_ls_grid[slot][dev] = sms * (per_sm > 0 ? per_sm : 1);
  }
  const int64_t cap = g_ls_grid[slot][dev];
  const unsigned grid = (unsigned)(ws.tiles < cap ? ws.tiles : cap);
  linscan_lookback_kernel<Cfg><<<grid, Cfg::kBlock, smem, s>>>(map_a, map_b, map_h, p, ws, ctl);
  return cudaGetLastError();
}

}  // namespace

// Rows of at least this many tiles take the long-row CTA shape.  Where rows hold several
// tiles, a tile's prefix comes from look-back over tiles that other CTAs are still scanning,
// and two tiles' time for it pays; where most tiles hold a row start, their prefixes are
// absolute at once and two CTAs per SM hide the loads better.
#ifndef SSM_LS_LONG_ROW_TILES
#define SSM_LS_LONG_ROW_TILES 4
#endif

cudaError_t launch_linscan(const float* a, const float* b, float* h, int64_t rows, int64_t len,
                           const LinscanWorkspace& ws, const LookbackCtl& ctl, cudaStream_t s, int shape) {
  LsArgs p{a, b, h, rows * len, len, (rows * len) / kLsRow};
  if (p.lines > 0x7fffffffLL) return cudaErrorInvalidValue;  // TMA coordinates are 32-bit
  CUtensorMap map_a{}, map_b{}, map_h{};
  if (p.lines > 0) {
    cudaError_t e;
    const uint64_t row_bytes = kLsRow * sizeof(float);
    if ((e = encode_tensor_map_2d(&map_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a, kLsRow, p.lines, row_bytes, kLsRow,
                                  kLsLines, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
      return e;
    if ((e = encode_tensor_map_2d(&map_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, b, kLsRow, p.lines, row_bytes, kLsRow,
                                  kLsLines, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
      return e;
    if ((e = encode_tensor_map_2d(&map_h, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, h, kLsRow, p.lines, row_bytes, kLsRow,
                                  kLsLines, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
      return e;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (shape == 0) shape = len >= (int64_t)SSM_LS_LONG_ROW_TILES * kLsTile ? 1 : 2;  // the rule
  switch (shape) {
    case 1: return launch_cfg<LsLongRows>(0, dev, map_a, map_b, map_h, p, ws, ctl, s);
    case 2: return launch_cfg<LsShortRows>(1, dev, map_a, map_b, map_h, p, ws, ctl, s);
    case 3: return launch_cfg<LsTwoGroups6>(2, dev, map_a, map_b, map_h, p, ws, ctl, s);
    case 4: return launch_cfg<LsOneGroup6>(3, dev, map_a, map_b, map_h, p, ws, ctl, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssm
