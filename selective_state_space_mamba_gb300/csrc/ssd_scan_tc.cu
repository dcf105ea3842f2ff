// ssd_chunk_scan_tc: the chunk output of "Accelerating Mamba-2 with High-Performance Forward
// Pass Kernels in NVIDIA CUDA Tile", "Kernel 3: compute_out",
//     Y = 2^G (C h_in^T) + ((C B^T) . 2^(G_i - G_j) dt_j . [i >= j]) X + D X,
// on the 5th-generation tensor cores for bf16 inputs (f32 accumulation).
//
// CTA = (batch, chunk, 128-row tile of the chunk, group, run of heads), warp-specialised:
//   warp 0     TMA producer: the tile's C rows and the chunk's B rows once; then, per head,
//              X, the chunk-initial state h_in and the head's G and dt over the chunk into a
//              2-stage ring
//   warp 1     TMEM owner and MMA issuer (one thread): CB = C B^T once (M = 128 rows,
//              N = columns up to the tile's end, K = S; shared by all heads of the run: the
//              post recomputes it per head); per head Y2 = C h_in^T as soon as the stage lands,
//              and Y1 = P X once P is ready (P read from TMEM as the A operand)
//   warps 2-9  math: CB once to bf16 in shared memory; per head, P = CB . w with
//              w(i, j) = dt_j 2^(G_i - G_j) for j <= i, written to TMEM as bf16, and the row's
//              x values kept in registers; then the previous head's epilogue
//              y = Y1 + 2^(G_i) Y2 + D x (f32) -> bf16 -> swizzled stage -> TMA store
// P and the accumulators are double-buffered in TMEM, so the MMA of head k runs while the
// math warps finish head k-1.
//
// The decay weight is a product of two factors that are both <= 1 wherever row i lies in a
// later 32-token block than column j: w = 2^(G_i - G_r) * dt_j 2^(G_r - G_j), r the first token
// of i's block (G is non-increasing).  Only in the diagonal 32 x 32 block of a warp's rows is
// 2^(G_i - G_j) evaluated per element, with the exponent set to -inf above the diagonal before
// the exponential (the post masks after exp2; masking the exponent first never produces inf).
//
// Every wait is bounded.  A math-warp wait that gives up is voted on (bar.red.or) so that all
// math warps leave together; the CTA then drains, frees its TMEM and returns.
#include "tc_common.cuh"

namespace ssm {
namespace {

constexpr int kScThreads = 320;  // warp 0 producer, warp 1 MMA, warps 2..9 math
constexpr int kScMath = 256;
constexpr uint32_t kScMathBar = 1;
constexpr uint32_t kScTmemCols = 512;
// TMEM columns: CB (f32, first phase only) 0..Nj-1; then P[b] at 128 b (bf16 pairs, 128 columns)
// and Y1[b] / Y2[b] at 256 + 128 b / 320 + 128 b (64 f32 columns each).
constexpr uint32_t kColCB = 0;
__device__ __forceinline__ uint32_t col_p(int b) { return 128u * b; }
__device__ __forceinline__ uint32_t col_y1(int b) { return 256u + 128u * b; }
__device__ __forceinline__ uint32_t col_y2(int b) { return 320u + 128u * b; }
constexpr int kRowB = 128;  // bytes per swizzled operand row (64 bf16)

struct ScParams {
  const float* G;
  const float* dtT;
  const float* D;
  WsHeader* hdr;
  int64_t lpad, nchunks;
  int nheads, ngroups, chunk, row_tiles;
  int heads_per_item, items_per_tile;
};

// Shared memory (offsets from a 1024-byte aligned base), chunk size T:
//   C tile   2 s-blocks x 128 rows x 128 B                                      32 KB
//   B rows   2 s-blocks x T rows x 128 B; after CB: CB as bf16 [128 rows][Nj] (16-byte chunks
//            swizzled within each row)
//   stage[2] X: T rows x 128 B | h_in: 2 s-blocks x 64 rows x 128 B | G, dt: T floats each
//   y stage  128 rows x 128 B (swizzled, for the TMA store)
//   v[2]     the off-diagonal factor tables of two heads, packed by 32-row block
struct ScLayout {
  uint32_t c0, b0, st0, st_bytes, hin_off, g_off, dt_off, y0, v0, v_floats, bars, total;
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
    v_floats = 16u * 8 * 7;  // row blocks 1..7 hold 32 * block entries: 32 * 28
    bars = v0 + 2u * 4u * v_floats;
    total = bars + 16 * 8 + 16;
  }
};
enum ScBar {
  kInFull = 0, kCbDone = 1, kStFull = 2, kStEmpty = 4, kPFull = 6, kMmaDone = 8, kYFree = 10, kDone = 12,
  kScNumBars = 13
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
// offset of row block I's factors in a packed table (block I >= 1 holds 32 I entries)
__device__ __forceinline__ int v_off(int I) { return 16 * I * (I - 1); }

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

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work item -> (batch, chunk, group, row tile, run of heads)
  int64_t item = blockIdx.x;
  const int k_item = (int)(item % p.items_per_tile);
  item /= p.items_per_tile;
  const int R = (int)(item % p.row_tiles);
  item /= p.row_tiles;
  const int g = (int)(item % p.ngroups);
  item /= p.ngroups;
  const int64_t c = item % p.nchunks;
  const int64_t bi = item / p.nchunks;
  const int hpg = p.nheads / p.ngroups;
  const int h_first = g * hpg + k_item * p.heads_per_item;
  const int nh_run = min(p.heads_per_item, hpg - k_item * p.heads_per_item);
  const int i0 = R * 128;   // first chunk row of the tile
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
  auto fail = [&](void) {
    record_error(p.hdr, ctl.epoch, SSM_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------------------
    if (lane == 0 && nh_run > 0) {
      mbar_arrive_expect_tx(&bars[kInFull], 2u * 128 * kRowB + 2u * Nj * kRowB);
      for (int sb = 0; sb < 2; ++sb) {
        tc::tma_load_3d(base + L.c0 + sb * 128 * kRowB, &map_c, g * 128 + sb * 64, tok0 + i0, (int)bi, &bars[kInFull]);
        for (int rb = 0; rb < Nj / 128; ++rb)
          tc::tma_load_3d(base + L.b0 + sb * T * kRowB + rb * 128 * kRowB, &map_b, g * 128 + sb * 64, tok0 + rb * 128,
                          (int)bi, &bars[kInFull]);
      }
      int issued = 0;
      for (int k = 0; k < nh_run && !*abort_flag; ++k) {
        const int st = k & 1;
        if (k >= 2 && !mbar_wait(&bars[kStEmpty + st], (uint32_t)((k >> 1) - 1) & 1u, ctl.spin_limit_ns)) {
          fail();
          break;
        }
        const int h = h_first + k;
        unsigned char* stage = base + L.st0 + st * L.st_bytes;
        mbar_arrive_expect_tx(&bars[kStFull + st], (uint32_t)Nj * kRowB + 2u * 64 * kRowB + 8u * T);
        for (int rb = 0; rb < Nj / 128; ++rb)
          tc::tma_load_3d(stage + rb * 128 * kRowB, &map_x, h * 64, tok0 + rb * 128, (int)bi, &bars[kStFull + st]);
        const int hin_row = (int)(((bi * p.nchunks + c) * p.nheads + h) * 64);
        for (int sb = 0; sb < 2; ++sb)
          tma_load_2d(stage + L.hin_off + sb * 64 * kRowB, &map_hin, sb * 64, hin_row, &bars[kStFull + st]);
        const int64_t grow = (bi * p.nheads + h) * p.lpad + tok0;
        bulk_g2s(stage + L.g_off, p.G + grow, 4u * T, &bars[kStFull + st]);
        bulk_g2s(stage + L.dt_off, p.dtT + grow, 4u * T, &bars[kStFull + st]);
        issued = k + 1;
      }
      for (int k = max(0, issued - 2); k < issued; ++k)
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
      const uint32_t id_y2 = tc::idesc_bf16_f32(128, 64, false, false);
      const uint32_t id_y1 = tc::idesc_bf16_f32(128, 64, false, true);
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
        // Y2 = C h_in^T: M = 128, N = 64 (p), K = S (both K-major); runs while P is being formed
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t ko = (ks & 3) * 32;
          const uint64_t a = tc::sdesc_sw128(c_addr + (ks >> 2) * 128 * kRowB + ko, 16, sbo);
          const uint64_t b = tc::sdesc_sw128(h_addr + (ks >> 2) * 64 * kRowB + ko, 16, sbo);
          tc::mma_bf16(tmem + col_y2(bf), a, b, id_y2, ks > 0);
        }
        if (!mbar_wait(&bars[kPFull + bf], (uint32_t)(k >> 1) & 1u, ctl.spin_limit_ns)) {
          fail();
          break;
        }
        tc::fence_after_sync();
        // Y1 = P X: A = P from TMEM (8 columns per 16 K), B = X rows (MN-major, p contiguous)
        for (int ks = 0; ks < Nj / 16; ++ks) {
          const uint64_t b = tc::sdesc_sw128(x_addr + ks * 16 * kRowB, (uint32_t)T * kRowB, sbo);
          tc::mma_bf16_ts(tmem + col_y1(bf), tmem + col_p(bf) + ks * 8, b, id_y1, ks > 0);
        }
        tc::mma_commit(&bars[kStEmpty + st]);  // X, h_in, G, dt of this head are no longer needed
        tc::mma_commit(&bars[kMmaDone + bf]);
      }
      tc::mma_commit(&bars[kDone]);
      mbar_wait(&bars[kDone], 0, ctl.spin_limit_ns);
    }
  } else {
    // ------------------------------ math warps ---------------------------------------------
    const int mt = threadIdx.x - 64;   // 0..255
    const int quad = warp & 3;         // TMEM lanes 32*quad .. +31
    const int half = (warp - 2) >> 2;  // which interleaved 32-column blocks
    const int r = quad * 32 + lane;    // tile row
    const int i = i0 + r;              // chunk row
    const int I = i >> 5;              // 32-token block of the row (warp-uniform)
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int row_bytes = Nj * 2;      // CB row in bf16
    unsigned char* cb_smem = base + L.b0;
    bool ok = nh_run > 0;

    // ---- CB (f32, TMEM) -> bf16 rows in shared memory over the dead B rows ----
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
          const int chunk = (cb >> 3) + q;
          uint4 w;
          w.x = pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1]));
          w.y = pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
          w.z = pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
          w.w = pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
          *reinterpret_cast<uint4*>(cb_smem + r * row_bytes + ((chunk ^ (r & 7)) << 4)) = w;
        }
      }
      tc::fence_before_sync();
    }

    // Off-diagonal factors of head k for the tile's row blocks: v[I][j] = dt_j 2^(G_{32I} - G_j),
    // j < 32 I.  Returns false (all threads alike) when the head's stage never arrived.
    auto build_table = [&](int k) -> bool {
      const int st = k & 1;
      const bool bad = !mbar_wait(&bars[kStFull + st], (uint32_t)(k >> 1) & 1u, ctl.spin_limit_ns);
      if (named_bar_any(kScMathBar, kScMath, bad)) return false;
      const float* gq = reinterpret_cast<const float*>(base + L.st0 + st * L.st_bytes + L.g_off);
      const float* dq = reinterpret_cast<const float*>(base + L.st0 + st * L.st_bytes + L.dt_off);
      float* vq = v_all + (k & 1) * L.v_floats;
      const int Ilo = max(1, i0 >> 5), Ihi = (i0 + 128) >> 5;  // row blocks of this tile
      for (int e = v_off(Ilo) + mt; e < v_off(Ihi); e += kScMath) {
        int II = Ilo;
        while (v_off(II + 1) <= e) ++II;
        const int j = e - v_off(II);
        vq[e] = dq[j] * tc::ex2_approx(gq[32 * II] - gq[j]);
      }
      return true;
    };

    // y = Y1 + 2^(G_i) Y2 + D x of head kk -> swizzled stage -> TMA store.  False (all alike)
    // on a wait that gave up.
    auto epilogue = [&](int kk, float e_i, float Dk, const uint32_t (&xk)[16]) -> bool {
      const int b2 = kk & 1;
      const bool bad = !mbar_wait(&bars[kMmaDone + b2], (uint32_t)(kk >> 1) & 1u, ctl.spin_limit_ns);
      if (named_bar_any(kScMathBar, kScMath, bad)) return false;
      tc::fence_after_sync();
      uint32_t y1[32], y2[32];
      tc::tmem_ld32(tmem + lane_base + col_y1(b2) + half * 32, y1);
      tc::tmem_ld32(tmem + lane_base + col_y2(b2) + half * 32, y2);
      tc::tmem_ld_wait();
      uint32_t outp[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        outp[q] = pack_bf16(__uint_as_float(y1[2 * q]) + e_i * __uint_as_float(y2[2 * q]) + Dk * bf_lo(xk[q]),
                            __uint_as_float(y1[2 * q + 1]) + e_i * __uint_as_float(y2[2 * q + 1]) + Dk * bf_hi(xk[q]));
      tc::fence_before_sync();
      if (mt == 0) bulk_wait_read<0>();  // the previous y store has read the stage
      named_bar_sync(kScMathBar, kScMath);
      if (mt == 0) mbar_arrive(&bars[kYFree + b2]);  // Y[b2] may be overwritten
      unsigned char* yrow = base + L.y0 + r * kRowB;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int chunk = half * 4 + cc;
        *reinterpret_cast<uint4*>(yrow + ((chunk ^ (r & 7)) << 4)) =
            make_uint4(outp[cc * 4], outp[cc * 4 + 1], outp[cc * 4 + 2], outp[cc * 4 + 3]);
      }
      fence_proxy_async_smem();
      named_bar_sync(kScMathBar, kScMath);
      if (mt == 0) {
        tc::tma_store_3d(&map_y, base + L.y0, (h_first + kk) * 64, tok0 + i0, (int)bi);
        bulk_commit();
      }
      return true;
    };

    if (ok && !build_table(0)) {
      if (mt == 0) fail();
      ok = false;
    }
    // 2^(G_i), D and the row's x values of the previous head, taken before its stage is released
    float prev_e = 0.f, prev_D = 0.f;
    uint32_t prev_x[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) prev_x[q] = 0u;
    for (int k = 0; k < nh_run && ok; ++k) {
      const int st = k & 1, bf = k & 1;
      const int h = h_first + k;
      named_bar_sync(kScMathBar, kScMath);  // CB (first head) and this head's table are complete
      const float* g_s = reinterpret_cast<const float*>(base + L.st0 + st * L.st_bytes + L.g_off);
      const float* dt_s = reinterpret_cast<const float*>(base + L.st0 + st * L.st_bytes + L.dt_off);
      const float* v_s = v_all + (k & 1) * L.v_floats + (I >= 1 ? v_off(I) : 0);
      const float gi = g_s[i];
      const float ui = I > 0 ? tc::ex2_approx(gi - g_s[32 * I]) : 0.f;
      const float cur_D = p.D[h];
      const float cur_e = tc::ex2_approx(gi);
      uint32_t cur_x[16];  // x(i, 32 half .. 32 half + 31) as bf16 pairs
      {
        const unsigned char* xrow = base + L.st0 + st * L.st_bytes + i * kRowB;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint4 w = *reinterpret_cast<const uint4*>(xrow + (((half * 4 + cc) ^ (i & 7)) << 4));
          cur_x[4 * cc] = w.x; cur_x[4 * cc + 1] = w.y; cur_x[4 * cc + 2] = w.z; cur_x[4 * cc + 3] = w.w;
        }
      }

      // ---- P = CB . w for my row: bf16 pairs into P[bf] ----
      for (int J = half; J < Nj / 32; J += 2) {
        const int cb = J * 32;
        uint32_t pk[16];
        if (J > I) {  // entirely above the diagonal
#pragma unroll
          for (int q = 0; q < 16; ++q) pk[q] = 0u;
        } else {
          uint32_t cw[16];  // CB row segment as bf16 pairs
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 w = *reinterpret_cast<const uint4*>(cb_smem + r * row_bytes + ((((cb >> 3) + q) ^ (r & 7)) << 4));
            cw[4 * q] = w.x; cw[4 * q + 1] = w.y; cw[4 * q + 2] = w.z; cw[4 * q + 3] = w.w;
          }
          if (J < I) {  // w = 2^(G_i - G_r) * dt_j 2^(G_r - G_j), both factors <= 1
            const float4* vv = reinterpret_cast<const float4*>(v_s + cb);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 f = vv[q];
              pk[2 * q] = pack_bf16(bf_lo(cw[2 * q]) * (ui * f.x), bf_hi(cw[2 * q]) * (ui * f.y));
              pk[2 * q + 1] = pack_bf16(bf_lo(cw[2 * q + 1]) * (ui * f.z), bf_hi(cw[2 * q + 1]) * (ui * f.w));
            }
          } else {  // diagonal 32 x 32 block: per-element 2^(G_i - G_j), exponent -inf above it
            const float4* gg = reinterpret_cast<const float4*>(g_s + cb);
            const float4* dd = reinterpret_cast<const float4*>(dt_s + cb);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 gq = gg[q], dq = dd[q];
              const int j = cb + 4 * q;
              const float p0 = bf_lo(cw[2 * q]) * dq.x * tc::ex2_approx(j <= i ? gi - gq.x : -INFINITY);
              const float p1 = bf_hi(cw[2 * q]) * dq.y * tc::ex2_approx(j + 1 <= i ? gi - gq.y : -INFINITY);
              const float p2 = bf_lo(cw[2 * q + 1]) * dq.z * tc::ex2_approx(j + 2 <= i ? gi - gq.z : -INFINITY);
              const float p3 = bf_hi(cw[2 * q + 1]) * dq.w * tc::ex2_approx(j + 3 <= i ? gi - gq.w : -INFINITY);
              pk[2 * q] = pack_bf16(p0, p1);
              pk[2 * q + 1] = pack_bf16(p2, p3);
            }
          }
        }
        tc::tmem_st16(tmem + lane_base + col_p(bf) + (cb >> 1), pk);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      named_bar_sync(kScMathBar, kScMath);
      if (mt == 0) mbar_arrive(&bars[kPFull + bf]);

      // ---- the previous head's epilogue while the MMA multiplies this one ----
      if (k >= 1 && !epilogue(k - 1, prev_e, prev_D, prev_x)) {
        if (mt == 0) fail();
        ok = false;
        break;
      }
      prev_e = cur_e;
      prev_D = cur_D;
#pragma unroll
      for (int q = 0; q < 16; ++q) prev_x[q] = cur_x[q];
      // ---- the next head's table while the MMA works ----
      if (k + 1 < nh_run && !build_table(k + 1)) {
        if (mt == 0) fail();
        ok = false;
        break;
      }
    }
    if (ok && !epilogue(nh_run - 1, prev_e, prev_D, prev_x) && mt == 0) fail();
    if (mt == 0) bulk_wait<0>();
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
  // split each (batch, chunk, group, row tile)'s heads into runs: about three CTAs per SM or more
  const int64_t tiles = d.batch * d.nchunks * d.ngroups * p.row_tiles;
  int runs = (int)((3 * (int64_t)sms + tiles - 1) / tiles);
  runs = runs < 1 ? 1 : (runs > hpg ? hpg : runs);
  p.heads_per_item = (hpg + runs - 1) / runs;
  p.items_per_tile = (hpg + p.heads_per_item - 1) / p.heads_per_item;
  const ScLayout L(d.chunk);
  const size_t smem = L.total + 1024;
  if ((e = cudaFuncSetAttribute(ssd_chunk_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
      cudaSuccess)
    return e;
  const int64_t grid = tiles * p.items_per_tile;
  ssd_chunk_scan_tc_kernel<<<(unsigned)grid, kScThreads, smem, s>>>(map_c, map_b, map_x, map_hin, map_y, p, ctl);
  return cudaGetLastError();
}

}  // namespace ssm
