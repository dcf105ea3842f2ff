// ssd_chunk_scan_tc: the chunk output of "Accelerating Mamba-2 with High-Performance Forward
// Pass Kernels in NVIDIA CUDA Tile", "Kernel 3: compute_out",
//     Y = 2^G (C h_in^T) + ((C B^T) . 2^(G_i - G_j) dt_j . [i >= j]) X + D X,
// on the 5th-generation tensor cores for bf16 inputs (f32 accumulation).
//
// CTA = (batch, chunk, 128-row tile of the chunk, group, run of heads), warp-specialised:
//   warp 0     TMA producer: the tile's C rows and the chunk's B rows once; then, per head,
//              X (rows 0 .. end of the tile) and the chunk-initial state h_in into a 2-stage ring
//   warp 1     TMEM owner and MMA issuer (one thread): CB = C B^T once (M = 128 rows,
//              N = columns up to the tile's end, K = S, f32 in TMEM, shared by all heads of the
//              run: the post recomputes it per head); per head Y2 = C h_in^T (K = S) and
//              Y1 = P X (K = columns), with P read from TMEM
//   warps 2-9  math: per head, P = CB . w with w(i, j) = dt_j 2^(G_i - G_j) for j <= i, written
//              to TMEM as bf16 (the MMA's A operand; the post's register-resident masked tile);
//              then the epilogue y = Y1 + 2^(G_i) Y2 + D x -> bf16 -> swizzled stage -> TMA store
//
// The decay weight is a product of two factors that are both <= 1 wherever row i and column j
// lie in different 64-token blocks: w = 2^(G_i - G_r) * dt_j 2^(G_r - G_j) with r the first
// token of i's block (G is non-increasing).  Only inside a diagonal 64 x 64 block is
// 2^(G_i - G_j) evaluated per element, with the exponent set to -inf above the diagonal before
// the exponential (the post masks after exp2; masking the exponent first never produces inf).
#include "tc_common.cuh"

namespace ssm {
namespace {

constexpr int kScThreads = 320;  // warp 0 producer, warp 1 MMA, warps 2..9 math
constexpr int kScMath = 256;
constexpr uint32_t kScMathBar = 1;
constexpr uint32_t kScTmemCols = 512;
constexpr uint32_t kColCB = 0, kColP = 256, kColY1 = 384, kColY2 = 448;
constexpr int kRowB = 128;  // bytes per swizzled row (64 bf16)

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
//   C tile   2 s-blocks x 128 rows x 128 B                         32 KB
//   B rows   2 s-blocks x T rows x 128 B
//   stage[2] X: T rows x 128 B, then h_in: 2 s-blocks x 64 rows x 128 B
//   y stage  128 rows x 128 B (swizzled, for the TMA store)
//   G, dt: T floats each; v: 4 x T floats; barriers
struct ScLayout {
  uint32_t c0, b0, st0, st_bytes, hin_off, y0, g0, dt0, v0, bars, total;
  __host__ __device__ explicit ScLayout(int T) {
    c0 = 0;
    b0 = c0 + 2u * 128 * kRowB;
    st0 = b0 + 2u * T * kRowB;
    hin_off = (uint32_t)T * kRowB;
    st_bytes = hin_off + 2u * 64 * kRowB;
    y0 = st0 + 2u * st_bytes;
    g0 = y0 + 128u * kRowB;
    dt0 = g0 + 4u * T;
    v0 = dt0 + 4u * T;
    bars = v0 + 16u * T;
    total = bars + 16 * 8 + 16;
  }
};
enum ScBar { kInFull = 0, kCbDone = 1, kStFull = 2, kStEmpty = 4, kPFull = 6, kMmaDone = 7, kYFree = 8, kDone = 9,
             kScNumBars = 10 };

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
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
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.bars + kScNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L.bars + kScNumBars * 8 + 4);
  float* g_s = reinterpret_cast<float*>(base + L.g0);
  float* dt_s = reinterpret_cast<float*>(base + L.dt0);
  float* v_s = reinterpret_cast<float*>(base + L.v0);  // [I][j]: dt_j 2^(G_{64 I} - G_j)

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
        mbar_arrive_expect_tx(&bars[kStFull + st], (uint32_t)Nj * kRowB + 2u * 64 * kRowB);
        for (int rb = 0; rb < Nj / 128; ++rb)
          tc::tma_load_3d(stage + rb * 128 * kRowB, &map_x, h * 64, tok0 + rb * 128, (int)bi, &bars[kStFull + st]);
        const int hin_row = (int)(((bi * p.nchunks + c) * p.nheads + h) * 64);
        for (int sb = 0; sb < 2; ++sb)
          tma_load_2d(stage + L.hin_off + sb * 64 * kRowB, &map_hin, sb * 64, hin_row, &bars[kStFull + st]);
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
        const int st = k & 1;
        if (!mbar_wait(&bars[kPFull], (uint32_t)k & 1u, ctl.spin_limit_ns) ||
            !mbar_wait(&bars[kStFull + st], (uint32_t)(k >> 1) & 1u, ctl.spin_limit_ns) ||
            (k >= 1 && !mbar_wait(&bars[kYFree], (uint32_t)(k - 1) & 1u, ctl.spin_limit_ns))) {
          fail();
          break;
        }
        tc::fence_after_sync();
        const uint32_t x_addr = smem_addr(base + L.st0 + st * L.st_bytes);
        const uint32_t h_addr = x_addr + L.hin_off;
        // Y2 = C h_in^T: M = 128, N = 64 (p), K = S (both K-major)
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t ko = (ks & 3) * 32;
          const uint64_t a = tc::sdesc_sw128(c_addr + (ks >> 2) * 128 * kRowB + ko, 16, sbo);
          const uint64_t b = tc::sdesc_sw128(h_addr + (ks >> 2) * 64 * kRowB + ko, 16, sbo);
          tc::mma_bf16(tmem + kColY2, a, b, id_y2, ks > 0);
        }
        // Y1 = P X: A = P from TMEM (8 columns per 16 K), B = X rows (MN-major, p contiguous)
        for (int ks = 0; ks < Nj / 16; ++ks) {
          const uint64_t b = tc::sdesc_sw128(x_addr + ks * 16 * kRowB, (uint32_t)T * kRowB, sbo);
          tc::mma_bf16_ts(tmem + kColY1, tmem + kColP + ks * 8, b, id_y1, ks > 0);
        }
        tc::mma_commit(&bars[kMmaDone]);
      }
      tc::mma_commit(&bars[kDone]);
      mbar_wait(&bars[kDone], 0, ctl.spin_limit_ns);
    }
  } else {
    // ------------------------------ math warps ---------------------------------------------
    const int mt = threadIdx.x - 64;        // 0..255
    const int quad = warp & 3;              // TMEM lanes 32*quad .. +31
    const int half = (warp - 2) >> 2;       // column half
    const int r = quad * 32 + lane;         // tile row
    const int i = i0 + r;                   // chunk row
    const int I = i >> 6;                   // 64-token block of the row
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    bool ok = true;
    if (!mbar_wait(&bars[kCbDone], 0, ctl.spin_limit_ns)) {
      if (mt == 0) fail();
      ok = false;
    }
    for (int k = 0; k < nh_run && ok; ++k) {
      const int st = k & 1;
      const int h = h_first + k;
      const int64_t grow = (bi * p.nheads + h) * p.lpad + tok0;
      // ---- per-head tables: G, dt over the chunk; v[I][j] = dt_j 2^(G_{64I} - G_j), j < 64 I ----
      for (int t = mt; t < T; t += kScMath) {
        g_s[t] = p.G[grow + t];
        dt_s[t] = p.dtT[grow + t];
      }
      named_bar_sync(kScMathBar, kScMath);
      for (int e = mt; e < 3 * T; e += kScMath) {
        const int II = 1 + e / T, j = e % T;
        if (j < 64 * II && 64 * II < T) v_s[II * T + j] = dt_s[j] * exp2f(g_s[64 * II] - g_s[j]);
      }
      named_bar_sync(kScMathBar, kScMath);
      const float gi = g_s[i];
      const float ui = I > 0 ? exp2f(gi - g_s[64 * I]) : 0.f;
      // ---- P = CB . w for my row and my half of the columns, written to TMEM as bf16 pairs ----
      const int cols = Nj / 2;
      for (int cb = half * cols; cb < (half + 1) * cols; cb += 32) {
        uint32_t cbv[32];
        tc::tmem_ld32(tmem + lane_base + kColCB + cb, cbv);
        tc::tmem_ld_wait();
        const int J = cb >> 6;  // 64-block of these 32 columns (warp-uniform)
        uint32_t pk[16];
#pragma unroll
        for (int jj = 0; jj < 32; jj += 2) {
          float pv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int j = cb + jj + u;
            const float cbf = __uint_as_float(cbv[jj + u]);
            if (J < I) {
              pv[u] = cbf * ui * v_s[I * T + j];
            } else if (J == I) {
              const float ex = j <= i ? gi - g_s[j] : -INFINITY;
              pv[u] = cbf * dt_s[j] * exp2f(ex);
            } else {
              pv[u] = 0.f;
            }
          }
          pk[jj >> 1] = pack_bf16(pv[0], pv[1]);
        }
        tc::tmem_st16(tmem + lane_base + kColP + (cb >> 1), pk);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      named_bar_sync(kScMathBar, kScMath);
      if (mt == 0) mbar_arrive(&bars[kPFull]);

      // ---- epilogue: y = Y1 + 2^(G_i) Y2 + D x for my row, p in [32 half, 32 half + 32) ----
      if (!mbar_wait(&bars[kMmaDone], (uint32_t)k & 1u, ctl.spin_limit_ns)) {
        if (mt == 0) fail();
        break;
      }
      tc::fence_after_sync();
      uint32_t y1[32], y2[32];
      tc::tmem_ld32(tmem + lane_base + kColY1 + half * 32, y1);
      tc::tmem_ld32(tmem + lane_base + kColY2 + half * 32, y2);
      tc::tmem_ld_wait();
      const float ei = exp2f(gi);
      const float Dh = p.D[h];
      const unsigned char* xrow = base + L.st0 + st * L.st_bytes + i * kRowB;
      uint32_t outp[16];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int chunk = half * 4 + cc;  // 8 p-values
        const uint4 xv = *reinterpret_cast<const uint4*>(xrow + ((chunk ^ (i & 7)) << 4));
        const __nv_bfloat162* xe = reinterpret_cast<const __nv_bfloat162*>(&xv);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 xf = __bfloat1622float2(xe[q]);
          const int col = cc * 8 + q * 2;
          const float o0 = __uint_as_float(y1[col]) + ei * __uint_as_float(y2[col]) + Dh * xf.x;
          const float o1 = __uint_as_float(y1[col + 1]) + ei * __uint_as_float(y2[col + 1]) + Dh * xf.y;
          outp[cc * 4 + q] = pack_bf16(o0, o1);
        }
      }
      tc::fence_before_sync();
      if (mt == 0) bulk_wait_read<0>();  // the previous head's y store has read the stage
      named_bar_sync(kScMathBar, kScMath);
      if (mt == 0) {
        mbar_arrive(&bars[kYFree]);          // Y1 / Y2 may be overwritten
        mbar_arrive(&bars[kStEmpty + st]);   // X and h_in of this head are no longer needed
      }
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
        tc::tma_store_3d(&map_y, base + L.y0, h * 64, tok0 + i0, (int)bi);
        bulk_commit();
      }
    }
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
