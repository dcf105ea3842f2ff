// ssd_chunk_scan_tc: the chunk output of "Accelerating Mamba-2 with High-Performance Forward
// Pass Kernels in NVIDIA CUDA Tile", "Kernel 3: compute_out",
//     Y = 2^G (C h_in^T) + ((C B^T) . 2^(G_i - G_j) dt_j . [i >= j]) X + D X,
// on the 5th-generation tensor cores for bf16 inputs (f32 accumulation).
//
// CTA = (batch, chunk, 128-row tile of the chunk starting at row i0, group, run of heads).  The
// CTAs take the tiles in order (the two row tiles of a chunk adjacent, the later one first, so
// that they run at the same time and share their x, h_in, G and dt reads in L2), in up to three
// tiers with a different number of CTAs per tile each: large runs of heads first, small ones
// last, so that the last wave of CTAs ends together (see ScTiers).
// The tile's columns j split into the rectangle j < i0 and the triangle i0 <= j < i0 + 128.
// In the rectangle every weight factors through the tile's first row:
//     2^(G_i - G_j) dt_j = u_i f_j,   u_i = 2^(G_i - G_i0) <= 1,   f_j = dt_j 2^(G_i0 - G_j) <= dt_j,
// so its part of Y is u_i (CB_rect (f . X_rect)): one MMA whose A operand (CB) is the same for
// all heads of the run and whose B operand is X with its rows scaled by f; u_i is applied in
// the f32 epilogue.  Only the 128 x 128 triangle needs a per-element weight matrix P.
//
// Warp roles (448 threads):
//   warp 0       TMA producer: the tile's C rows and B rows 0 .. i0+127 once; then, per head,
//                X rows 0 .. i0+127, the chunk-initial state h_in and the head's G and dt over
//                the chunk into a 2-stage ring (and the same tiles of later heads into L2)
//   warp 1       TMEM owner and MMA issuer (one thread): CB = C B^T once; per head
//                Y2 = C h_in^T as soon as the stage lands, then Ya = CB_rect (f . X_rect) and
//                Yt = P X_tri (P read from TMEM as the A operand) once the P warps are done
//   warps 2-9    P warps: CB once to bf16 in shared memory (the MMA operand layout); per head
//                the factor table, the rectangle's X rows scaled by f and the triangle P
//                (bf16, to TMEM)
//   warps 10-13  epilogue warps, one row per thread: x and G from the stage as it lands, then
//                y = Yt + 2^(G_i) Y2 + u_i Ya + D x (f32) -> bf16 -> swizzled stage -> TMA store
// P and the accumulators are double-buffered in TMEM, so the P warps build head k + 1 while
// the MMAs and the epilogue warps finish head k.

// Inside the triangle the same factoring is used per 32-row block I: w = 2^(G_i - G_r) *
// dt_j 2^(G_r - G_j), r = i0 + 32 I, both factors <= 1 for columns in earlier blocks.  In the
// diagonal 32 x 32 block the weight is 2^(G_i + c_j), c_j = log2(dt_j) - G_j, with the exponent
// set to -inf above the diagonal before the exponential (masking the exponent first never
// produces inf).  Weights are rounded to bf16 and multiplied into CB with one bf16x2 FMA.
//
// Every wait is bounded.  A math-warp wait that gives up is voted on (bar.red.or) so that all
// math warps leave together; the CTA then drains, frees its TMEM and returns.
#include "tc_common.cuh"

#include <algorithm>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#ifndef SSM_SCAN_Y_EVICT_FIRST  // y is written once: evict-first priority in L2
#define SSM_SCAN_Y_EVICT_FIRST 1
#endif

namespace ssm {
namespace {

constexpr int kScThreads = 448;  // warp 0 producer, warp 1 MMA, warps 2..9 P, warps 10..13 epilogue
constexpr int kScMath = 256;     // P warps
constexpr int kScEpi = 128;      // epilogue warps
constexpr uint32_t kScMathBar = 1, kScEpiBar = 2;
constexpr uint32_t kScTmemCols = 512;
constexpr int kRowB = 128;  // bytes per swizzled operand row (64 bf16)
constexpr int kCbBlock = 128 * kRowB;  // one 64-column block of CB (bf16) for the tile's 128 rows

// TMEM columns.  CB (f32) takes 0 .. i0+127 during the first phase only.  Afterwards P[b]
// (bf16 pairs, 64 columns) sits at 64 b, and accumulator set b at 320 (b = 0) or 128 (b = 1):
// Yt at +0, Y2 at +64, Ya at +128 (64 f32 columns each).  Set 1 overlaps CB; its first MMA
// is issued only after the math warps have signalled P of head 0, i.e. after CB was read.
constexpr uint32_t kColCB = 0;
__device__ __forceinline__ uint32_t col_p(int b) { return 64u * b; }
__device__ __forceinline__ uint32_t col_y(int b) { return b ? 128u : 320u; }

// Per-head factor table (floats):
//   [0, 192)    triangle: local row block I = 1..3 holds dt_j 2^(G_r - G_j) for the 32 I
//               columns i0 <= j < r, r = i0 + 32 I, at offset 16 I (I - 1)
//   [192, 320)  rectangle: f_j = dt_j 2^(G_i0 - G_j), j < i0 (tiles with i0 > 0)
//   [320, 448)  diagonal blocks: c_j = log2(dt_j) - G_j, i0 <= j < i0 + 128
constexpr int kVTri = 0, kVRect = 192, kVDiag = 320, kVFloats = 448;
__device__ __forceinline__ int v_off(int I) { return 16 * I * (I - 1); }

struct ScParams {
  const float* G;
  const float* dtT;
  const float* D;
  WsHeader* hdr;
  int64_t batch, lpad, nchunks;
  int nheads, ngroups, chunk, row_tiles;
  // CTAs in order: tier s covers the next tier_tiles[s] tiles with tier_items[s] CTAs per tile;
  // a tile's heads split evenly, tier_run[s] heads per CTA and one more for its first
  // tier_rem[s] CTAs (all below 2^31: the grid is)
  int tier_tiles[3], tier_items[3], tier_run[3], tier_rem[3];
  int first_wave;  // CTAs below this index (one per SM) may start while the previous kernel runs
};

// Shared memory (offsets from a 1024-byte aligned base), chunk size T:
//   C tile   2 s-blocks x 128 rows x 128 B                                        32 KB
//   B rows   2 s-blocks x T rows x 128 B; after CB: CB as bf16 in the K-major operand layout,
//            [column block of 64][128 rows][128 B], 16-byte chunks swizzled by row
//   stage[2] X: T rows x 128 B | h_in: 2 s-blocks x 64 rows x 128 B | G, dt: T floats each
//   y stage  128 rows x 128 B (swizzled, for the TMA store)
//   v[2]     the factor tables of two heads
struct ScLayout {
  uint32_t c0, b0, st0, st_bytes, hin_off, g_off, dt_off, y0, v0, bars, total;
  __host__ __device__ explicit ScLayout(int T) {
    c0 = 0;
    b0 = c0 + 2u * 128 * kRowB;
    st0 = b0 + 2u * T * kRowB;
    hin_off = (uint32_t)T * kRowB;
    g_off = hin_off + 2u * 64 * kRowB;
    dt_off = g_off + 4u * T;
    st_bytes = dt_off + 4u * T;
    y0 = st0 + 2u * st_bytes;
    v0 = y0 + 128u * kRowB;
    bars = v0 + 2u * 4u * kVFloats;
    total = bars + 16 * 8 + 16;
  }
};
enum ScBar {
  kInFull = 0, kCbDone = 1, kStFull = 2, kStEmpty = 4, kPFull = 6, kMmaDone = 8, kYFree = 10, kXRead = 12,
  kDone = 14, kScNumBars = 15
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
// (d0, d1) = (a0, a1) * (b0, b1) + (c0, c1), one f32x2 FMA
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                     float c1) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
// a * b on bf16 pairs, one rounding (fma with -0 keeps the sign of a zero product)
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(0x80008000u));
  return d;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// address of the 16-byte chunk holding columns 8 q .. 8 q + 7 of tile row r in the CB layout
__device__ __forceinline__ uint32_t cb_chunk(int r, int q) {
  return (uint32_t)((q >> 3) * kCbBlock + r * kRowB + (((q & 7) ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kScThreads, 1)
    ssd_chunk_scan_tc_kernel(const __grid_constant__ CUtensorMap map_c, const __grid_constant__ CUtensorMap map_b,
                             const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_hin,
                             const __grid_constant__ CUtensorMap map_y, ScParams p, LookbackCtl ctl) {
  extern __shared__ unsigned char sc_raw[];
  const uint32_t raw = smem_addr(sc_raw);
  unsigned char* base = sc_raw + ((1024u - (raw & 1023u)) & 1023u);
  const int T = p.chunk;
  const ScLayout L(T);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.bars + 16 * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L.bars + 16 * 8 + 4);
  float* v_all = reinterpret_cast<float*>(base + L.v0);

  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA -> tier -> (tile, run of heads) -> (batch, chunk, group, row tile), in 32 bits
  int item, run0, nh_run;
  {
    // constant parameter indices only (a runtime index would copy the parameters to the stack)
    const int n0 = p.tier_tiles[0] * p.tier_items[0], n1 = p.tier_tiles[1] * p.tier_items[1];
    const int cta = blockIdx.x;
    const bool t0 = cta < n0, t1 = !t0 && cta < n0 + n1;
    const int rel = t0 ? cta : (t1 ? cta - n0 : cta - n0 - n1);
    const int tile0 = t0 ? 0 : (t1 ? p.tier_tiles[0] : p.tier_tiles[0] + p.tier_tiles[1]);
    const int items = t0 ? p.tier_items[0] : (t1 ? p.tier_items[1] : p.tier_items[2]);
    const int run = t0 ? p.tier_run[0] : (t1 ? p.tier_run[1] : p.tier_run[2]);
    const int rem = t0 ? p.tier_rem[0] : (t1 ? p.tier_rem[1] : p.tier_rem[2]);
    item = tile0 + rel / items;
    const int k_item = rel % items;
    run0 = k_item * run + min(k_item, rem);
    nh_run = run + (k_item < rem ? 1 : 0);
  }
  // of a chunk's two row tiles the later one (with the rectangle, the longer CTA) comes first
  const int R = p.row_tiles - 1 - item % p.row_tiles;
  item /= p.row_tiles;
  const int g = item % p.ngroups;
  item /= p.ngroups;
  const int64_t c = item % (int)p.nchunks;
  const int64_t bi = item / (int)p.nchunks;
  const int hpg = p.nheads / p.ngroups;
  const int h_first = g * hpg + run0;
  const int i0 = R * 128;   // first chunk row of the tile (0 or 128)
  const int Nj = i0 + 128;  // columns 0 .. Nj-1 can be at or below the diagonal
  const int tok0 = (int)(c * T);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kScNumBars; ++i) mbar_init(&bars[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kScTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // Each role waits for the previous kernel (griddep_wait) only before its first use of what
  // that kernel or the cumsum wrote (h_in, G, dt) or of D, so that the C and B rows, CB and
  // the first two stages' x rows are loaded and built while the previous kernel ends.  The
  // forward's inputs are safe to read before the wait: the kernel before this one lets its
  // dependents launch only after its own wait, so by the time this grid runs every kernel
  // before that one (which may have written the inputs) has completed.
  auto fail = [&](void) {
    record_error(p.hdr, ctl.epoch, SSM_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------------------
    if (lane == 0 && nh_run > 0) {
      const uint32_t x_bytes = (uint32_t)Nj * kRowB, rest_bytes = 2u * 64 * kRowB + 8u * T;  // h_in, G, dt
      mbar_arrive_expect_tx(&bars[kInFull], 2u * 128 * kRowB + 2u * Nj * kRowB);
      for (int sb = 0; sb < 2; ++sb) {
        tc::tma_load_3d(base + L.c0 + sb * 128 * kRowB, &map_c, g * 128 + sb * 64, tok0 + i0, (int)bi, &bars[kInFull]);
        for (int rb = 0; rb < Nj / 128; ++rb)
          tc::tma_load_3d(base + L.b0 + sb * T * kRowB + rb * 128 * kRowB, &map_b, g * 128 + sb * 64, tok0 + rb * 128,
                          (int)bi, &bars[kInFull]);
      }
      // A stage is refilled only when the MMAs of the head two before it are done, about one
      // head's time before it is needed: too short for DRAM.  So the head's tiles are first
      // prefetched into L2, two heads ahead (measured: one or two heads ahead alike, three and
      // four slower, none 10 % slower); the stage load then reads L2.
      auto prefetch_head = [&](int kk) {
        if (kk >= nh_run) return;
        const int h = h_first + kk;
        for (int rb = 0; rb < Nj / 128; ++rb) tc::tma_prefetch_3d(&map_x, h * 64, tok0 + rb * 128, (int)bi);
        const int hin_row = (int)(((bi * p.nchunks + c) * p.nheads + h) * 64);
        for (int sb = 0; sb < 2; ++sb) tc::tma_prefetch_2d(&map_hin, sb * 64, hin_row);
        const int64_t grow = (bi * p.nheads + h) * p.lpad + tok0;
        tc::bulk_prefetch_l2(p.G + grow, 4u * T);
        tc::bulk_prefetch_l2(p.dtT + grow, 4u * T);
      };
      // A stage's phase completes on the producer's one arrive (issued with the h_in, G and dt
      // copies) and all of its bytes; the x rows' bytes are declared without an arrive, so that
      // the first two stages' x can be requested before the wait.
      auto load_x = [&](int k) {
        unsigned char* stage = base + L.st0 + (k & 1) * L.st_bytes;
        mbar_expect_tx(&bars[kStFull + (k & 1)], x_bytes);
        for (int rb = 0; rb < Nj / 128; ++rb)
          tc::tma_load_3d(stage + rb * 128 * kRowB, &map_x, (h_first + k) * 64, tok0 + rb * 128, (int)bi,
                          &bars[kStFull + (k & 1)]);
      };
      // x is an input: the first wave requests its first two stages' x before the wait, to
      // overlap the previous kernel's end.  Later CTAs start after it has ended and keep the
      // order below (the L2 prefetch two heads ahead first), which measured faster for them.
      const int x_early = (int)blockIdx.x < p.first_wave ? (nh_run < 2 ? nh_run : 2) : 0;
      for (int k = 0; k < x_early; ++k) load_x(k);
      griddep_wait();
      int issued = 0;
      for (int k = 0; k < nh_run && !*abort_flag; ++k) {
        const int st = k & 1;
        prefetch_head(k + 2);
        // the stage is free once the MMAs of head k - 2 are done and the epilogue warps have
        // taken its x and G
        if (k >= 2 && (!mbar_wait(&bars[kStEmpty + st], (uint32_t)((k >> 1) - 1) & 1u, ctl.spin_limit_ns) ||
                       !mbar_wait(&bars[kXRead + st], (uint32_t)((k >> 1) - 1) & 1u, ctl.spin_limit_ns))) {
          fail();
          break;
        }
        const int h = h_first + k;
        unsigned char* stage = base + L.st0 + st * L.st_bytes;
        if (k >= x_early) load_x(k);
        mbar_arrive_expect_tx(&bars[kStFull + st], rest_bytes);
        const int64_t hin_row = ((bi * p.nchunks + c) * p.nheads + h) * 64;
        // h_in rows [b x nc x nh x 64] and the [b, nh, lpad] G / dt^T rows of this head and chunk
        if (SSM_CHECK(p.hdr, h < p.nheads && hin_row + 64 <= p.batch * p.nchunks * p.nheads * 64))
          for (int sb = 0; sb < 2; ++sb)
            tma_load_2d(stage + L.hin_off + sb * 64 * kRowB, &map_hin, sb * 64, (int)hin_row, &bars[kStFull + st]);
        const int64_t grow = (bi * p.nheads + h) * p.lpad + tok0;
        if (SSM_CHECK(p.hdr, grow + T <= p.batch * p.nheads * p.lpad)) {
          bulk_g2s(stage + L.g_off, p.G + grow, 4u * T, &bars[kStFull + st]);
          bulk_g2s(stage + L.dt_off, p.dtT + grow, 4u * T, &bars[kStFull + st]);
        }
        issued = k + 1;
      }
      // a stage whose x was requested early but whose other copies were not (an abort) gets
      // its arrive now, so that its phase completes once the x rows have landed
      for (int k = issued; k < x_early; ++k) mbar_arrive(&bars[kStFull + k]);
      const int in_flight = issued > x_early ? issued : x_early;
      for (int k = max(0, in_flight - 2); k < in_flight; ++k)
        mbar_wait(&bars[kStFull + (k & 1)], (uint32_t)(k >> 1) & 1u, ctl.spin_limit_ns);
      mbar_wait(&bars[kInFull], 0, ctl.spin_limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ---------------------------------------------
    if (lane == 0 && nh_run > 0) {
      const uint32_t sbo = 8 * kRowB;
      const uint32_t c_addr = smem_addr(base + L.c0), b_addr = smem_addr(base + L.b0);
      bool ok = mbar_wait(&bars[kInFull], 0, ctl.spin_limit_ns);
      if (!ok) fail();
      if (ok) {
        // CB = C B^T: M = 128 tile rows, N = Nj columns, K = S = 128 (both K-major)
        const uint32_t id_cb = tc::idesc_bf16_f32(128, Nj, false, false);
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t ko = (ks & 3) * 32;  // 16 elements within the 64-element row
          const uint64_t a = tc::sdesc_sw128(c_addr + (ks >> 2) * 128 * kRowB + ko, 16, sbo);
          const uint64_t b = tc::sdesc_sw128(b_addr + (ks >> 2) * T * kRowB + ko, 16, sbo);
          tc::mma_bf16(tmem + kColCB, a, b, id_cb, ks > 0);
        }
        tc::mma_commit(&bars[kCbDone]);
      }
      griddep_wait();
      const uint32_t id_kk = tc::idesc_bf16_f32(128, 64, false, false);  // Y2: C, h_in both K-major
      const uint32_t id_kn = tc::idesc_bf16_f32(128, 64, false, true);   // Ya, Yt: X MN-major
      const uint32_t xlbo = (uint32_t)T * kRowB;
      int ndone = 0;  // heads whose MMAs were committed
      for (int k = 0; k < nh_run && ok && !*abort_flag; ++k) {
        const int st = k & 1, bf = k & 1;
        if (!mbar_wait(&bars[kStFull + st], (uint32_t)(k >> 1) & 1u, ctl.spin_limit_ns) ||
            (k >= 2 && !mbar_wait(&bars[kYFree + bf], (uint32_t)((k >> 1) - 1) & 1u, ctl.spin_limit_ns))) {
          fail();
          break;
        }
        tc::fence_after_sync();
        const uint32_t x_addr = smem_addr(base + L.st0 + st * L.st_bytes);
        const uint32_t h_addr = x_addr + L.hin_off;
        const uint32_t ycol = tmem + col_y(bf);
        // Y2 = C h_in^T: M = 128, N = 64 (p), K = S; runs while the math warps work
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t ko = (ks & 3) * 32;
          const uint64_t a = tc::sdesc_sw128(c_addr + (ks >> 2) * 128 * kRowB + ko, 16, sbo);
          const uint64_t b = tc::sdesc_sw128(h_addr + (ks >> 2) * 64 * kRowB + ko, 16, sbo);
          tc::mma_bf16(ycol + 64, a, b, id_kk, ks > 0);
        }
        if (!mbar_wait(&bars[kPFull + bf], (uint32_t)(k >> 1) & 1u, ctl.spin_limit_ns)) {
          fail();
          break;
        }
        tc::fence_after_sync();
        // Ya = CB_rect (f . X_rect): A = CB from shared memory (K = j < i0), B = scaled X rows
        for (int ks = 0; ks < i0 / 16; ++ks) {
          const uint64_t a = tc::sdesc_sw128(b_addr + (ks >> 2) * kCbBlock + (ks & 3) * 32, 16, sbo);
          const uint64_t b = tc::sdesc_sw128(x_addr + ks * 16 * kRowB, xlbo, sbo);
          tc::mma_bf16(ycol + 128, a, b, id_kn, ks > 0);
        }
        // Yt = P X_tri: A = P from TMEM (8 columns per 16 K), B = X rows i0 .. i0+127
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t b = tc::sdesc_sw128(x_addr + (i0 + ks * 16) * kRowB, xlbo, sbo);
          tc::mma_bf16_ts(ycol, tmem + col_p(bf) + ks * 8, b, id_kn, ks > 0);
        }
        tc::mma_commit(&bars[kStEmpty + st]);  // X, h_in, G, dt of this head are no longer needed
        tc::mma_commit(&bars[kMmaDone + bf]);
        ndone = k + 1;
      }
      tc::mma_commit(&bars[kDone]);
      mbar_wait(&bars[kDone], 0, ctl.spin_limit_ns);
      // A commit's arrive lands when its MMAs complete, in no fixed order with the others: wait
      // for the last phase of every committed barrier, so that no arrive is still due to this
      // CTA's shared memory when it exits.
      for (int x = 0; x < 2; ++x)
        if (ndone > x) {
          mbar_wait(&bars[kStEmpty + x], (uint32_t)(((ndone - 1 - x) / 2) & 1), ctl.spin_limit_ns);
          mbar_wait(&bars[kMmaDone + x], (uint32_t)(((ndone - 1 - x) / 2) & 1), ctl.spin_limit_ns);
        }
      if (ok) mbar_wait(&bars[kCbDone], 0, ctl.spin_limit_ns);
    }
  } else if (warp < 10) {
    // ------------------------------ P warps ------------------------------------------------
    const int mt = threadIdx.x - 64;   // 0..255
    const int quad = warp & 3;         // TMEM lanes 32*quad .. +31 = the row's 32-row block
    const int half = (warp - 2) >> 2;  // which interleaved 32-column blocks
    const int r = quad * 32 + lane;    // tile row
    const int i = i0 + r;              // chunk row
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    unsigned char* cb_smem = base + L.b0;
    bool ok = nh_run > 0;

    // ---- CB (f32, TMEM) -> bf16 in the K-major operand layout, over the B rows ----
    if (ok) {
      const bool bad = !mbar_wait(&bars[kCbDone], 0, ctl.spin_limit_ns);
      if (named_bar_any(kScMathBar, kScMath, bad)) {
        if (mt == 0) fail();
        ok = false;
      }
    }
    if (ok) {
      tc::fence_after_sync();
      for (int cb = half * 32; cb < Nj; cb += 64) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + lane_base + kColCB + cb, v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // four 16-byte chunks of 8 columns
          uint4 w;
          w.x = pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1]));
          w.y = pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
          w.z = pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
          w.w = pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
          *reinterpret_cast<uint4*>(cb_smem + cb_chunk(r, (cb >> 3) + q)) = w;
        }
      }
      fence_proxy_async_smem();  // the rectangle MMA reads CB through the async proxy
      tc::fence_before_sync();
    }
    griddep_wait();

    // Factor table of head k (layout at kVTri / kVRect / kVDiag).  Returns false (all threads
    // alike) when the head's stage never arrived.
    auto build_table = [&](int k) -> bool {
      const int st = k & 1;
      const bool bad = !mbar_wait(&bars[kStFull + st], (uint32_t)(k >> 1) & 1u, ctl.spin_limit_ns);
      if (named_bar_any(kScMathBar, kScMath, bad)) return false;
      const float* gq = reinterpret_cast<const float*>(base + L.st0 + st * L.st_bytes + L.g_off);
      const float* dq = reinterpret_cast<const float*>(base + L.st0 + st * L.st_bytes + L.dt_off);
      float* vq = v_all + (k & 1) * kVFloats;
      // at most three entries per thread, straight-line so that all their loads are issued
      // together: entry mt (triangle below kVRect, else rectangle), entry mt + 256 (rectangle,
      // tiles with i0 > 0) and the diagonal entry mt
      auto entry = [&](int e, int& j, int& ref) {
        if (e < kVRect) {  // triangle: local row block I, reference row i0 + 32 I
          const int I = e < 32 ? 1 : (e < 96 ? 2 : 3);
          j = i0 + e - v_off(I);
          ref = i0 + 32 * I;
        } else {  // rectangle: reference row i0
          j = e - kVRect;
          ref = i0;
        }
      };
      const int e0 = mt, e1 = mt + kScMath;
      const bool has0 = e0 < kVRect + i0, has1 = e1 < kVRect + i0, hasd = mt < 128;
      int j0 = 0, r0 = 0, j1 = 0, r1 = 0;
      entry(e0, j0, r0);
      entry(e1, j1, r1);
      const float d0 = has0 ? dq[j0] : 0.f, a0 = has0 ? gq[r0] - gq[j0] : 0.f;
      const float d1 = has1 ? dq[j1] : 0.f, a1 = has1 ? gq[r1] - gq[j1] : 0.f;
      const float dd = hasd ? dq[i0 + mt] : 1.f, gd = hasd ? gq[i0 + mt] : 0.f;
      if (has0) vq[e0] = d0 * tc::ex2_approx(a0);
      if (has1) vq[e1] = d1 * tc::ex2_approx(a1);
      if (hasd) vq[kVDiag + mt] = lg2_approx(dd) - gd;  // dt = 0 -> -inf
      return true;
    };

    if (ok && !build_table(0)) {
      if (mt == 0) fail();
      ok = false;
    }
    if (ok) {
      // The blocks above the diagonal are zero for every head: write them once into both P
      // buffers (every P warp has read its CB columns: build_table's barrier came after).
      tc::fence_after_sync();
      const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      for (int b = 0; b < 2; ++b)
        for (int Jp = quad + 1; Jp < 4; ++Jp) tc::tmem_st8(tmem + lane_base + col_p(b) + 16 * Jp + 8 * half, z);
    }
    for (int k = 0; k < nh_run && ok; ++k) {
      const int st = k & 1, bf = k & 1;
      // this head's table is complete, and P[bf] has been read by the MMAs of head k - 2
      const bool bad = k >= 2 && !mbar_wait(&bars[kMmaDone + bf], (uint32_t)((k - 2) >> 1) & 1u, ctl.spin_limit_ns);
      if (named_bar_any(kScMathBar, kScMath, bad)) {
        if (mt == 0) fail();
        break;
      }
      tc::fence_after_sync();
      unsigned char* stage = base + L.st0 + st * L.st_bytes;
      const float* g_s = reinterpret_cast<const float*>(stage + L.g_off);
      const float* v_s = v_all + (k & 1) * kVFloats;
      const float gi = g_s[i];
      const float ui = quad > 0 ? tc::ex2_approx(gi - g_s[i0 + 32 * quad]) : 0.f;  // triangle row factor

      // ---- rectangle: X rows j < i0 scaled by f_j in place, one row per thread of the warps
      // of row quads 0 and 1, whose triangle rows hold the fewest blocks ----
      if (i0 > 0 && quad < 2) {
        const int j = half * 64 + quad * 32 + lane;
        const float f = v_s[kVRect + j];
        const uint32_t f2 = pack_bf16(f, f);
        unsigned char* xrow = stage + j * kRowB;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint4* q = reinterpret_cast<uint4*>(xrow + (((cc + lane) & 7) << 4));  // rotated: spread over banks
          uint4 w = *q;
          w.x = mul_bf16x2(w.x, f2);
          w.y = mul_bf16x2(w.y, f2);
          w.z = mul_bf16x2(w.z, f2);
          w.w = mul_bf16x2(w.w, f2);
          *q = w;
        }
        fence_proxy_async_smem();
      }

      // ---- triangle P for my row: bf16 pairs into P[bf].  Blocks Jp <= quad are nonzero; the
      // two warps of a row quad take one 16-column half of each, so that both carry the same
      // work (one half of the diagonal block and quad halves of off-diagonal blocks each) ----
#pragma unroll
      for (int Jp = 0; Jp < 4; ++Jp) {
        if (Jp > quad) break;  // the same for the whole warp
        const int cb = i0 + 32 * Jp + 16 * half;  // first column of my half block
        uint32_t cw[8];  // CB row segment as bf16 pairs
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint4 w = *reinterpret_cast<const uint4*>(cb_smem + cb_chunk(r, (cb >> 3) + q));
          cw[4 * q] = w.x; cw[4 * q + 1] = w.y; cw[4 * q + 2] = w.z; cw[4 * q + 3] = w.w;
        }
        uint32_t pk[8];
        if (Jp < quad) {  // w = 2^(G_i - G_r) * dt_j 2^(G_r - G_j), both factors <= 1
          const float4* vv = reinterpret_cast<const float4*>(v_s + kVTri + v_off(quad) + 32 * Jp + 16 * half);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 f = vv[q];
            pk[2 * q] = mul_bf16x2(cw[2 * q], pack_bf16(ui * f.x, ui * f.y));
            pk[2 * q + 1] = mul_bf16x2(cw[2 * q + 1], pack_bf16(ui * f.z, ui * f.w));
          }
        } else {  // diagonal 32 x 32 block: 2^(G_i + c_j), exponent -inf above the diagonal
          const float4* cc4 = reinterpret_cast<const float4*>(v_s + kVDiag + 32 * Jp + 16 * half);
          const int c0 = 16 * half;  // my columns are cb .. cb + 15; my row is column 32 Jp + lane
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 cq = cc4[q];
            const float w0 = tc::ex2_approx(c0 + 4 * q <= lane ? gi + cq.x : -INFINITY);
            const float w1 = tc::ex2_approx(c0 + 4 * q + 1 <= lane ? gi + cq.y : -INFINITY);
            const float w2 = tc::ex2_approx(c0 + 4 * q + 2 <= lane ? gi + cq.z : -INFINITY);
            const float w3 = tc::ex2_approx(c0 + 4 * q + 3 <= lane ? gi + cq.w : -INFINITY);
            pk[2 * q] = mul_bf16x2(cw[2 * q], pack_bf16(w0, w1));
            pk[2 * q + 1] = mul_bf16x2(cw[2 * q + 1], pack_bf16(w2, w3));
          }
        }
        tc::tmem_st8(tmem + lane_base + col_p(bf) + 16 * Jp + 8 * half, pk);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      fence_proxy_async_smem();  // the stage's G and dt reads, before its TMA refill
      named_bar_sync(kScMathBar, kScMath);
      if (mt == 0) mbar_arrive(&bars[kPFull + bf]);

      // ---- the next head's table while the MMAs and the epilogue warps work ----
      if (k + 1 < nh_run && !build_table(k + 1)) {
        if (mt == 0) fail();
        break;
      }
    }
  } else {
    // ------------------------------ epilogue warps -----------------------------------------
    // y = Yt + 2^(G_i) Y2 + u_i Ya + D x for the tile's 128 rows (one per thread) x 64 p.
    // x and G are read from the stage as soon as it lands (the stage is refilled only after
    // this group has released it through kXRead); the accumulators once the MMAs are done.
    griddep_wait();  // D, and the stages' h_in, G and dt
    const int et = threadIdx.x - 320;  // 0..127
    const int quad = warp & 3;         // TMEM lanes 32*quad .. +31
    const int r = quad * 32 + lane;    // tile row
    const int i = i0 + r;              // chunk row
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    for (int k = 0; k < nh_run; ++k) {
      const int st = k & 1, b = k & 1;
      const int h = h_first + k;
      bool bad = !mbar_wait(&bars[kStFull + st], (uint32_t)(k >> 1) & 1u, ctl.spin_limit_ns);
      if (named_bar_any(kScEpiBar, kScEpi, bad)) {
        if (et == 0) fail();
        break;
      }
      const unsigned char* stage = base + L.st0 + st * L.st_bytes;
      const float* g_s = reinterpret_cast<const float*>(stage + L.g_off);
      const float gi = g_s[i];
      const float e_i = tc::ex2_approx(gi);
      const float u_i = i0 > 0 ? tc::ex2_approx(gi - g_s[i0]) : 0.f;
      const float Dh = SSM_CHECK(p.hdr, h < p.nheads) ? p.D[h] : 0.f;
      uint32_t xr[32];  // x(i, 0 .. 63) as bf16 pairs
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const uint4 w = *reinterpret_cast<const uint4*>(stage + i * kRowB + ((cc ^ (i & 7)) << 4));
        xr[4 * cc] = w.x; xr[4 * cc + 1] = w.y; xr[4 * cc + 2] = w.z; xr[4 * cc + 3] = w.w;
      }
      // these reads must be performed before the TMA (async proxy) may refill the stage
      fence_proxy_async_smem();
      named_bar_sync(kScEpiBar, kScEpi);
      if (et == 0) {
        mbar_arrive(&bars[kXRead + st]);  // x and G of this stage are in registers
        if (k > 0) bulk_wait_read<0>();   // the previous y store has read the y stage
      }
      bad = !mbar_wait(&bars[kMmaDone + b], (uint32_t)(k >> 1) & 1u, ctl.spin_limit_ns);
      if (named_bar_any(kScEpiBar, kScEpi, bad)) {
        if (et == 0) fail();
        break;
      }
      tc::fence_after_sync();
      const uint32_t ycol = tmem + lane_base + col_y(b);
      unsigned char* yrow = base + L.y0 + r * kRowB;
#pragma unroll
      for (int ps = 0; ps < 4; ++ps) {  // 16 p at a time
        uint32_t yt[16], y2[16], ya[16];
        tc::tmem_ld16(ycol + 16 * ps, yt);
        tc::tmem_ld16(ycol + 64 + 16 * ps, y2);
        if (i0 > 0) tc::tmem_ld16(ycol + 128 + 16 * ps, ya);
        tc::tmem_ld_wait();
        uint32_t out[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float o0, o1;
          fma2(o0, o1, e_i, e_i, __uint_as_float(y2[2 * q]), __uint_as_float(y2[2 * q + 1]),
               __uint_as_float(yt[2 * q]), __uint_as_float(yt[2 * q + 1]));
          if (i0 > 0)
            fma2(o0, o1, u_i, u_i, __uint_as_float(ya[2 * q]), __uint_as_float(ya[2 * q + 1]), o0, o1);
          const uint32_t xp = xr[8 * ps + q];
          fma2(o0, o1, Dh, Dh, bf_lo(xp), bf_hi(xp), o0, o1);
          out[q] = pack_bf16(o0, o1);
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int chunk = 2 * ps + cc;
          *reinterpret_cast<uint4*>(yrow + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(out[4 * cc], out[4 * cc + 1], out[4 * cc + 2], out[4 * cc + 3]);
        }
      }
      tc::fence_before_sync();
      fence_proxy_async_smem();
      named_bar_sync(kScEpiBar, kScEpi);
      if (et == 0) {
        mbar_arrive(&bars[kYFree + b]);  // accumulator set b may be overwritten
#if SSM_SCAN_Y_EVICT_FIRST
        tc::tma_store_3d_hint(&map_y, base + L.y0, h * 64, tok0 + i0, (int)bi, l2_evict_first_policy());
#else
        tc::tma_store_3d(&map_y, base + L.y0, h * 64, tok0 + i0, (int)bi);
#endif
        bulk_commit();
      }
    }
    if (et == 0) bulk_wait<0>();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kScTmemCols);
  }
}

}  // namespace

bool ssd_scan_tc_supported(const SsdDims& d) {
  return d.dtype == SSM_BF16 && d.headdim == 64 && d.dstate == 128 && (d.chunk == 128 || d.chunk == 256);
}

// ---- the chunk scan's work split -------------------------------------------------------
// The CTAs take the tiles (batch, chunk, group, row tile) in order, a tile's heads split evenly
// between its CTAs.  With one CTA per SM the hardware hands each CTA, in index order, to the SM
// that frees first, so the split decides how the last wave ends: tiers of large runs of heads
// first and small ones last end it more evenly than one split for all tiles, and large runs
// pay the per-CTA set-up (C and B rows, CB, the first stage, the drain) less often.

// Greedy list scheduling over `sms` SMs, the model of that dispatch.  Costs in units of a head
// of a first row tile: a head of a later row tile (which adds the rectangle) 1.25, a CTA's
// set-up and drain 4.7 (per-role timings at b4 L8192 nh80: 1.18 us, 1.47 us and ~5.5 us).
double sc_model_makespan(const ScTiers& s, int row_tiles, int hpg, int sms) {
  std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
  for (int i = 0; i < sms; ++i) free_at.push(0.0);
  double end = 0.0;
  int64_t tile = 0;
  for (int k = 0; k < 3; ++k)
    for (int64_t tt = 0; tt < s.tiles[k]; ++tt, ++tile) {
      const double per_head = (row_tiles == 2 && tile % 2 == 0) ? 1.25 : 1.0;  // the later row tile first
      for (int j = 0; j < s.items[k]; ++j) {
        const int nh = hpg / s.items[k] + (j < hpg % s.items[k] ? 1 : 0);
        const double t0 = free_at.top();
        free_at.pop();
        free_at.push(t0 + nh * per_head + 4.7);
        end = std::max(end, t0 + nh * per_head + 4.7);
      }
    }
  return end;
}

int64_t sc_ctas(const ScTiers& s) { return s.tiles[0] * s.items[0] + s.tiles[1] * s.items[1] + s.tiles[2] * s.items[2]; }

ScTiers sc_uniform(int64_t tiles, int items) {
  ScTiers s{};
  s.tiles[0] = tiles;
  s.items[0] = items;
  s.items[1] = s.items[2] = 1;
  return s;
}

// The split for `tiles` tiles of `hpg` heads.  plan_heads > 0 (a plan): runs of at most that
// many heads, one tier.  0: the split the model finds fastest among one tier of up to 8 CTAs per
// tile and three tiers around the best of those (the first f chunks with a CTAs per tile, the
// last m with c, the rest with b; a <= b < c), all with runs of at most 40 heads, kept only
// where the model gains 2 % (its error is larger than that), fewer CTAs deciding between equal
// model times; computed once per shape and SM count.  Searched only up to 8 waves: beyond, the
// last wave weighs little.
ScTiers sc_schedule(int64_t tiles, int row_tiles, int hpg, int sms, int plan_heads) {
  if (plan_heads > 0) {
    const int run = plan_heads < hpg ? plan_heads : hpg;
    return sc_uniform(tiles, (hpg + run - 1) / run);
  }
  static std::mutex mu;
  static std::map<std::tuple<int64_t, int, int, int>, ScTiers> cache;
  const auto key = std::make_tuple(tiles, row_tiles, hpg, sms);
  {
    std::lock_guard<std::mutex> lk(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  // Runs of at most 40 heads: the later row tile takes ~25 % longer per head, so over a longer
  // run the two row tiles of a chunk drift apart by more than their shared lines stay in L2
  // (measured at b4 L8192 nh80: runs of 80 heads first cost 1-20 us against runs of 40).
  const int min_items = (hpg + 39) / 40;
  int b_best = min_items;
  double t_best = -1.0;
  for (int b = min_items; b <= std::max(min_items, std::min(hpg, 8)); ++b) {
    if (tiles * b > 8LL * sms && b > min_items) break;
    const double tm = sc_model_makespan(sc_uniform(tiles, b), row_tiles, hpg, sms);
    if (t_best < 0 || tm < t_best) {
      t_best = tm;
      b_best = b;
    }
  }
  ScTiers best = sc_uniform(tiles, b_best);
  const int64_t chunks = tiles / row_tiles;  // tiles of one (batch, chunk, group), adjacent
  if (tiles * b_best <= 8LL * sms && chunks >= 8) {
    const double uniform_time = t_best;
    for (int b = std::max(min_items, b_best - 1); b <= std::min(hpg, b_best + 1); ++b)
      for (int a = std::max(min_items, b - 1); a <= b; ++a)
        for (int cm : {2, 4}) {
          const int c = std::min(hpg, cm * b);
          if (c <= b) continue;
          for (int fq : {0, 1, 2, 3, 4})       // first chunks: 0 .. 1/2 of them
            for (int mq = 0; mq <= 8; ++mq) {  // last chunks: 0 .. 1/8 of them, in 64ths
              const int64_t f = chunks * fq / 8, m = chunks * mq / 64;
              if ((fq && !f) || (mq && !m) || f + m > chunks) continue;
              ScTiers s{};
              s.tiles[0] = f * row_tiles;
              s.items[0] = a;
              s.tiles[1] = (chunks - f - m) * row_tiles;
              s.items[1] = b;
              s.tiles[2] = m * row_tiles;
              s.items[2] = c;
              const double tm = sc_model_makespan(s, row_tiles, hpg, sms);
              // the model's makespan moves in steps: of equal ones, the split with fewer CTAs
              // (fewer set-ups) measured faster
              if (tm < 0.98 * uniform_time &&
                  (tm < t_best - 1e-9 || (tm <= t_best + 1e-9 && sc_ctas(s) < sc_ctas(best)))) {
                t_best = tm;
                best = s;
              }
            }
        }
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = best;
  return best;
}

cudaError_t launch_ssd_chunk_scan_tc(const void* x, const void* B, const void* C, const float* D, void* y,
                                     const SsdDims& d, const SsdWorkspace& ws, const LookbackCtl& ctl,
                                     cudaStream_t s) {
  CUtensorMap map_c, map_b, map_x, map_hin, map_y;
  const uint64_t bcd[3] = {(uint64_t)d.ngroups * 128, (uint64_t)d.seqlen, (uint64_t)d.batch};
  const uint64_t bcs[2] = {(uint64_t)d.ngroups * 128 * 2, (uint64_t)d.seqlen * d.ngroups * 128 * 2};
  const uint64_t xd[3] = {(uint64_t)d.nheads * 64, (uint64_t)d.seqlen, (uint64_t)d.batch};
  const uint64_t xs[2] = {(uint64_t)d.nheads * 64 * 2, (uint64_t)d.seqlen * d.nheads * 64 * 2};
  const uint32_t box[3] = {64, 128, 1};
  cudaError_t e;
  if ((e = encode_tensor_map_3d(&map_c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, bcd, bcs, box, CU_TENSOR_MAP_SWIZZLE_128B)) !=
      cudaSuccess)
    return e;
  if ((e = encode_tensor_map_3d(&map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, bcd, bcs, box, CU_TENSOR_MAP_SWIZZLE_128B)) !=
      cudaSuccess)
    return e;
  if ((e = encode_tensor_map_3d(&map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, xd, xs, box, CU_TENSOR_MAP_SWIZZLE_128B)) !=
      cudaSuccess)
    return e;
  if ((e = encode_tensor_map_3d(&map_y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, y, xd, xs, box, CU_TENSOR_MAP_SWIZZLE_128B)) !=
      cudaSuccess)
    return e;
  const uint64_t hin_rows = (uint64_t)d.batch * d.nchunks * d.nheads * 64;
  if ((e = encode_tensor_map_2d(&map_hin, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws.hin, 128, hin_rows, 256, 64, 64,
                                CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  ScParams p;
  p.G = ws.G;
  p.dtT = ws.dtT;
  p.D = D;
  p.hdr = ws.hdr;
  p.batch = d.batch;
  p.lpad = d.lpad;
  p.nchunks = d.nchunks;
  p.nheads = d.nheads;
  p.ngroups = d.ngroups;
  p.chunk = d.chunk;
  p.row_tiles = d.chunk / 128;
  const int hpg = d.nheads / d.ngroups;
  int dev = 0, sms = 148;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t tiles = d.batch * d.nchunks * d.ngroups * p.row_tiles;
  const ScTiers tiers = sc_schedule(tiles, p.row_tiles, hpg, sms, d.plan_scan_heads);
  int64_t grid = 0;
  for (int k = 0; k < 3; ++k) grid += tiers.tiles[k] * tiers.items[k];
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  p.first_wave = sms;
  for (int k = 0; k < 3; ++k) {
    p.tier_tiles[k] = (int)tiers.tiles[k];
    p.tier_items[k] = tiers.items[k];
    p.tier_run[k] = hpg / tiers.items[k];
    p.tier_rem[k] = hpg % tiers.items[k];
  }
  const ScLayout L(d.chunk);
  const size_t smem = L.total + 1024;
  if ((e = ensure_smem_limit(reinterpret_cast<const void*>(ssd_chunk_scan_tc_kernel), smem)) != cudaSuccess)
    return e;
  return launch_pdl(ssd_chunk_scan_tc_kernel, dim3((unsigned)grid), dim3(kScThreads), smem, s, map_c, map_b, map_x,
                    map_hin, map_y, p, ctl);
}

}  // namespace ssm
