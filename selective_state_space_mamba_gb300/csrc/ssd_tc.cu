// Tensor-core (tcgen05 / TMEM / TMA) kernels for the bf16 chunk contractions of the Mamba-2
// SSD forward.
//
// ssd_chunk_state_tc: the decayed jump term of "Accelerating Mamba-2 with High-Performance
// Forward Pass Kernels in NVIDIA CUDA Tile", "Kernel 2: fwd_pass_state":
//     S_c = X^T (w . B),  w_t = dt_t 2^(G_last - G_t)          (H x S per batch, chunk, head)
// computed per chunk in parallel (the chunk loop of the post's kernel becomes the separate
// state-passing scan).  The weighted X is split into bf16 hi + lo parts (lo = the rounding
// remainder) and both are multiplied, so the weighting costs no bf16 rounding (2^-18 instead of
// 2^-9 relative): the chunk states feed h_final, whose tolerance a single bf16 rounding of
// x * w exceeds.  One MMA tile covers TWO heads of the same B/C group: M = 128 rows
// (64 p-values of each head), N = S = 128, K = the chunk's tokens.  B (the group's B, s
// contiguous) is read from shared memory as TMA lands it; the weighted X is the A operand and
// is read from TENSOR MEMORY: the scaler threads write hi and lo straight into TMEM (a thread
// owns one row p, i.e. one TMEM lane, and packs two tokens per 32-bit column), so neither the
// split halves nor the MMA's reads of them touch shared memory.  The per-token weight goes on
// X (the post scales B instead; B is shared by the heads of a group here, so the per-head
// weight goes on X — the "swap A/B" idea of the post's optimisation section read the other
// way round).
//
// The weighted X and its remainder come from three bf16x2 FMAs per pair of values, each with
// one rounding: w is split into w_hi + w_lo (bf16 each); hi = x w_hi rounded; hi - x w_hi is
// then exact (a 16-bit product minus its own 8-bit rounding); lo = x w - hi is that remainder
// plus x w_lo, rounded once.  hi + lo equals x w to about 2^-17 relative.
//
// Work unit = (batch, chunk, group, head pair).  The units are split into one contiguous
// range per CTA (one CTA per SM, so every SM gets the same number of units, give or take
// one); a CTA reloads B only where its range crosses into the next (batch, chunk, group).
// CTA warps:
//   warp 0      TMA producer: B when the group changes (two buffers, so the next group's B
//               lands while the current group's MMAs run); X of the pair's two heads, 64 tokens
//               at a time, with those tokens' G and dt and the chunk's last G, into a 4-stage
//               ring
//   warp 1      TMEM owner and MMA issuer (one thread): 2 x 4 MMAs (hi, lo) per stage, A from
//               TMEM, into one of two 128-column f32 accumulators; tcgen05.commit frees the
//               stage (its X in shared memory and its hi/lo columns in TMEM), and after the
//               last stage of a unit hands the accumulator to the epilogue
//   warps 2-9   two groups of four warps that take alternate stages, so that one group's
//               chain (wait, table, loads, split, TMEM store) overlaps the other's; in a group
//               one row p of one head per thread (its TMEM lane): 64 threads first tabulate
//               the bf16 weight pairs of the stage's token pairs, then every thread turns its
//               64 values of X into 32 hi and 32 lo columns
//   warps 10-13 epilogue: TMEM -> registers -> a swizzled 32 x 32 f32 block per warp in shared
//               memory -> TMA store into S_c; the accumulator is freed after its last TMEM load
// Every wait is bounded; on expiry the CTA records SSM_ERR_TIMEOUT, drains, frees its TMEM
// and returns.
#include "tc_common.cuh"

namespace ssm {
namespace {

constexpr int kCsWarps = 14;  // 0 producer, 1 MMA, 2-9 scalers, 10-13 epilogue
constexpr int kCsThreads = kCsWarps * 32;
constexpr int kCsMaxT = 256;
constexpr int kCsKH = 64;         // tokens per stage
constexpr int kCsStages = 4;   // X ring in shared memory (released once the scalers have read it)
constexpr int kCsBBufs = 2;    // B of two groups: the next group's B lands while this one's MMAs run
constexpr int kCsAStages = 4;  // hi/lo ring in TMEM (released when the MMAs have read it)
constexpr int kCsRowBytes = 128;  // 64 bf16 per swizzled row
constexpr uint32_t kCsScaleBar = 1, kCsEpiBar = 2;  // scaler group g uses named barrier 1 + 2 g
constexpr uint32_t kCsTmemCols = 512;  // two 128-column accumulators, then 64 A columns per stage
constexpr uint32_t kCsTmemA = 256;     // hi of A stage a at kCsTmemA + 64 a, lo 32 columns later
// per stage and head: G of the stage's tokens, dt of the stage's tokens, the chunk's last 4 G
constexpr uint32_t kCsGdHead = (2 * kCsKH + 4) * 4;

struct CsParams {
  const float* G;
  const float* dtT;
  float* Sc;
  WsHeader* hdr;
  int64_t batch, lpad, nchunks, units;
  int nheads, ngroups, chunk;
};

// Shared-memory layout (offsets from a 1024-byte aligned base), chunk size T:
//   stage[8] = X[2 heads][64 rows][128 B]                                      swizzled
//   bm[s block][T rows][128 B]                                                 swizzled
//   epi[4 warps][32 rows][128 B]   S_c staging for the TMA store (swizzled)
//   gd[8 stages][2 heads] = { G[64], dt[64], G[T-4 .. T-1] }
//   wt[4 A stages][2 heads][32 token pairs] = { w_hi pair, -w_hi pair, -w_lo pair } (bf16x2)
//   barriers, TMEM base, abort flag
struct CsLayout {
  uint32_t stage_bytes, bm0, epi0, gd0, wt0, bars, total;
  __host__ __device__ explicit CsLayout(int T) {
    stage_bytes = 2u * kCsKH * kCsRowBytes;
    bm0 = kCsStages * stage_bytes;
    epi0 = bm0 + kCsBBufs * 2u * T * kCsRowBytes;
    gd0 = epi0 + 4u * 32 * kCsRowBytes;
    wt0 = gd0 + kCsStages * 2u * kCsGdHead;
    bars = wt0 + kCsAStages * 2u * (kCsKH / 2) * 16u;
    total = bars + 32 * 8 + 16;
  }
};
enum CsBar {
  kBFull = 0, kBEmpty = kBFull + kCsBBufs, kXFull = kBEmpty + kCsBBufs, kXEmpty = kXFull + kCsStages, kAFull = kXEmpty + kCsStages, kAEmpty = kAFull + kCsAStages,
  kAccFull = kAEmpty + kCsAStages, kAccEmpty = kAccFull + 2, kDone = kAccEmpty + 2, kNumBars = kDone + 1
};

// d = a * b + c on bf16 pairs, one rounding
__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

struct CsUnit {
  int64_t bi, c, grp;
  int g, h;  // group, first head of the pair
};
__device__ __forceinline__ CsUnit cs_unit(const CsParams& p, int64_t u) {
  const int hpg = p.nheads / p.ngroups, ppg = hpg / 2;
  CsUnit r;
  r.grp = u / ppg;
  const int pair = (int)(u % ppg);
  r.g = (int)(r.grp % p.ngroups);
  const int64_t t = r.grp / p.ngroups;
  r.c = t % p.nchunks;
  r.bi = t / p.nchunks;
  r.h = r.g * hpg + 2 * pair;
  return r;
}

__global__ void __launch_bounds__(kCsThreads, 1)
    ssd_chunk_state_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_b,
                              const __grid_constant__ CUtensorMap map_sc, CsParams p, LookbackCtl ctl) {
  extern __shared__ unsigned char cs_raw[];
  const uint32_t raw = smem_addr(cs_raw);
  unsigned char* base = cs_raw + ((1024u - (raw & 1023u)) & 1023u);
  const int T = p.chunk;
  const CsLayout L(T);
  const int nk = T / kCsKH;  // stages per unit
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bars);
  static_assert(kNumBars <= 32, "barrier area");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.bars + 32 * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L.bars + 32 * 8 + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch_dependents();
  const int64_t u_begin = (int64_t)blockIdx.x * p.units / gridDim.x;
  const int64_t u_end = (int64_t)(blockIdx.x + 1) * p.units / gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], 1);  // every barrier has one arriving thread
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kCsTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // set-up above touched no global memory; G and dt come from the previous kernel
  auto fail = [&](void) {
    record_error(p.hdr, ctl.epoch, SSM_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------------------
    if (lane == 0 && u_end > u_begin) {
      int64_t cur_grp = -1;
      int64_t i = 0;  // stage step
      int nreload = 0;
      bool ok = true;
      for (int64_t u = u_begin; u < u_end && ok && !*abort_flag; ++u) {
        const CsUnit w = cs_unit(p, u);
        for (int kh = 0; kh < nk; ++kh, ++i) {
          const int st = (int)(i % kCsStages);
          if (i >= kCsStages &&
              !mbar_wait(&bars[kXEmpty + st], (uint32_t)((i / kCsStages) - 1) & 1u, ctl.spin_limit_ns)) {
            ok = false;
            break;
          }
          if (w.grp != cur_grp) {
            // B is read by every MMA of the previous group: the MMA thread releases it when it
            // moves on (this producer may be up to three rings ahead of the MMAs, so it waits on
            // a barrier of its own rather than on a ring's)
            // buffer nreload % 2 last held the B of reload nreload - 2
            const int bb = nreload % kCsBBufs;
            if (nreload >= kCsBBufs && !mbar_wait(&bars[kBEmpty + bb], (uint32_t)((nreload / kCsBBufs) - 1) & 1u,
                                                  ctl.spin_limit_ns)) {
              ok = false;
              break;
            }
            ++nreload;
            unsigned char* bdst = base + L.bm0 + bb * 2u * T * kCsRowBytes;
            mbar_arrive_expect_tx(&bars[kBFull + bb], 2u * T * kCsRowBytes);
            for (int sb = 0; sb < 2; ++sb)
              tc::tma_load_3d(bdst + sb * T * kCsRowBytes, &map_b, w.g * 128 + sb * 64, (int)(w.c * T), (int)w.bi,
                              &bars[kBFull + bb]);
            cur_grp = w.grp;
          }
          unsigned char* gd = base + L.gd0 + st * 2 * kCsGdHead;
          mbar_arrive_expect_tx(&bars[kXFull + st], L.stage_bytes + 2u * kCsGdHead);
          for (int hh = 0; hh < 2; ++hh) {
            tc::tma_load_3d(base + st * L.stage_bytes + hh * kCsKH * kCsRowBytes, &map_x, (w.h + hh) * 64,
                            (int)(w.c * T + kh * kCsKH), (int)w.bi, &bars[kXFull + st]);
            const int64_t row = (w.bi * p.nheads + w.h + hh) * p.lpad + w.c * T;
            // G and dt^T are [b, nh, lpad]: the chunk's T entries of this head
            if (!SSM_CHECK(p.hdr, w.h + hh < p.nheads && row + T <= p.batch * p.nheads * p.lpad)) continue;
            bulk_g2s(gd + hh * kCsGdHead, p.G + row + kh * kCsKH, 4u * kCsKH, &bars[kXFull + st]);
            bulk_g2s(gd + hh * kCsGdHead + 4u * kCsKH, p.dtT + row + kh * kCsKH, 4u * kCsKH, &bars[kXFull + st]);
            bulk_g2s(gd + hh * kCsGdHead + 8u * kCsKH, p.G + row + T - 4, 16u, &bars[kXFull + st]);
          }
        }
      }
      if (!ok) fail();
      // leave no copy in flight: the last loads of each stage have landed (bounded)
      for (int64_t j = (i > kCsStages ? i - kCsStages : 0); j < i; ++j)
        mbar_wait(&bars[kXFull + (int)(j % kCsStages)], (uint32_t)(j / kCsStages) & 1u, ctl.spin_limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ---------------------------------------------
    if (lane == 0 && u_end > u_begin) {
      const uint32_t idesc = tc::idesc_bf16_f32(128, 128, /*a_mn=*/false, /*b_mn=*/true);  // A from TMEM
      const uint32_t b_lbo = T * kCsRowBytes;      // s 0..63 block -> s 64..127 block
      const uint32_t sbo = 8 * kCsRowBytes;        // next 8-token group
      int64_t cur_grp = -1, i = 0;  // i: steps whose MMAs were committed
      int nb = 0, q = 0, nacc = 0;  // nacc: accumulators handed to the epilogue
      bool ok = true;
      for (int64_t u = u_begin; u < u_end && ok && !*abort_flag; ++u, ++q) {
        const CsUnit w = cs_unit(p, u);
        const int acc = q & 1;
        if (w.grp != cur_grp) {
          // the previous group's B buffer, once its MMAs are done
          if (nb > 0) tc::mma_commit(&bars[kBEmpty + (nb - 1) % kCsBBufs]);
          ++nb;
          cur_grp = w.grp;
          ok = mbar_wait(&bars[kBFull + (nb - 1) % kCsBBufs], (uint32_t)((nb - 1) / kCsBBufs) & 1u,
                         ctl.spin_limit_ns);
        }
        if (ok && q >= 2) ok = mbar_wait(&bars[kAccEmpty + acc], (uint32_t)((q >> 1) - 1) & 1u, ctl.spin_limit_ns);
        for (int kh = 0; kh < nk && ok; ++kh, ++i) {
          const int as = (int)(i % kCsAStages);
          if (!mbar_wait(&bars[kAFull + as], (uint32_t)(i / kCsAStages) & 1u, ctl.spin_limit_ns)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a_hi = tmem + kCsTmemA + 64u * as, a_lo = a_hi + 32;
          const uint32_t b0 =
              smem_addr(base + L.bm0) + ((nb - 1) % kCsBBufs) * 2u * T * kCsRowBytes + kh * kCsKH * kCsRowBytes;
#pragma unroll
          for (int ks = 0; ks < kCsKH / 16; ++ks) {
            const uint32_t koff = ks * 16 * kCsRowBytes;  // 16 tokens = two 8-row groups of B
            const uint64_t bdesc = tc::sdesc_sw128(b0 + koff, b_lbo, sbo);
            // 16 tokens of A = 8 TMEM columns (two tokens per column)
            tc::mma_bf16_ts(tmem + acc * 128, a_hi + ks * 8, bdesc, idesc, kh > 0 || ks > 0);
            tc::mma_bf16_ts(tmem + acc * 128, a_lo + ks * 8, bdesc, idesc, true);
          }
          tc::mma_commit(&bars[kAEmpty + as]);  // the A stage's TMEM columns may be rewritten
        }
        if (ok) {
          tc::mma_commit(&bars[kAccFull + acc]);  // the accumulator is ready
          ++nacc;
        }
      }
      if (!ok) fail();
      tc::mma_commit(&bars[kDone]);
      mbar_wait(&bars[kDone], 0, ctl.spin_limit_ns);  // every MMA has completed
      // A commit's arrive lands when its MMAs complete, in no fixed order with the others: wait
      // for the last phase of every committed barrier, so that no arrive is still due to this
      // CTA's shared memory when it exits.
      for (int x = 0; x < kCsAStages; ++x)
        if (i > x) mbar_wait(&bars[kAEmpty + x], (uint32_t)(((i - 1 - x) / kCsAStages) & 1), ctl.spin_limit_ns);
      for (int x = 0; x < 2; ++x)
        if (nacc > x) mbar_wait(&bars[kAccFull + x], (uint32_t)(((nacc - 1 - x) / 2) & 1), ctl.spin_limit_ns);
      // kBEmpty commits were made for groups 0 .. nb - 2, group j's on buffer j % 2
      for (int x = 0; x < kCsBBufs; ++x) {
        const int j = (nb - 2) - (((nb - 2) - x) % kCsBBufs + kCsBBufs) % kCsBBufs;
        if (nb >= 2 && j >= 0) mbar_wait(&bars[kBEmpty + x], (uint32_t)(j / kCsBBufs) & 1u, ctl.spin_limit_ns);
      }
    }
  } else if (warp < 10) {
    // ---------------- scale X by w, split into bf16 hi + lo parts, into TMEM ----------------
    const int grp = (warp - 2) >> 2;       // this group takes the steps i with i % 2 == grp
    const int gt = threadIdx.x - 64 - 128 * grp;  // 0..127 within the group
    const uint32_t gbar = kCsScaleBar + 2 * grp;
    const int quad = warp & 3;             // TMEM lanes 32 quad .. +31
    const int hh = quad >> 1;              // rows 0..63: head 0, rows 64..127: head 1
    const int prow = (quad & 1) * 32 + lane;  // this thread's p within its head
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    int64_t i = 0;
    bool ok = true;
    for (int64_t u = u_begin; u < u_end && ok; ++u) {
      for (int kh = 0; kh < nk; ++kh, ++i) {
        if ((int)(i & 1) != grp) continue;
        const int st = (int)(i % kCsStages), as = (int)(i % kCsAStages);
        // X of step i has landed, and the MMAs of step i - 4 have read this A stage's columns
        const bool bad =
            !mbar_wait(&bars[kXFull + st], (uint32_t)(i / kCsStages) & 1u, ctl.spin_limit_ns) ||
            (i >= kCsAStages &&
             !mbar_wait(&bars[kAEmpty + as], (uint32_t)((i / kCsAStages) - 1) & 1u, ctl.spin_limit_ns));
        if (named_bar_any(gbar, 128, bad)) {  // leave together, or not at all
          if (gt == 0) fail();
          ok = false;
          break;
        }
        tc::fence_after_sync();
        uint4* wt = reinterpret_cast<uint4*>(base + L.wt0) + as * 2 * (kCsKH / 2);
        if (gt < 2 * (kCsKH / 2)) {  // the bf16 weight pairs of (head, token pair)
          const int wh = gt / (kCsKH / 2), pr = gt % (kCsKH / 2);
          const float* gd = reinterpret_cast<const float*>(base + L.gd0 + (st * 2 + wh) * kCsGdHead);
          const float glast = gd[2 * kCsKH + 3];
          const float w0 = gd[kCsKH + 2 * pr] * tc::ex2_approx(glast - gd[2 * pr]);
          const float w1 = gd[kCsKH + 2 * pr + 1] * tc::ex2_approx(glast - gd[2 * pr + 1]);
          const __nv_bfloat162 whi = __floats2bfloat162_rn(w0, w1);
          const __nv_bfloat162 nwlo =
              __floats2bfloat162_rn(__bfloat162float(whi.x) - w0, __bfloat162float(whi.y) - w1);
          const uint32_t whi2 = *reinterpret_cast<const uint32_t*>(&whi);
          wt[wh * (kCsKH / 2) + pr] = make_uint4(whi2, whi2 ^ 0x80008000u, *reinterpret_cast<const uint32_t*>(&nwlo), 0u);
        }
        named_bar_sync(gbar, 128);
        // my row p of head hh: tokens 2 j and 2 j + 1 form TMEM column j of the A stage
        const unsigned char* xh = base + st * L.stage_bytes + hh * kCsKH * kCsRowBytes;
        const int cpos = (prow >> 3), cin = (prow & 7) * 2;  // 16-byte chunk and byte within it
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t0 = 32 * half + 2 * j, t1 = t0 + 1;
            const uint32_t x0 = *reinterpret_cast<const uint16_t*>(xh + t0 * kCsRowBytes + ((cpos ^ (t0 & 7)) << 4) + cin);
            const uint32_t x1 = *reinterpret_cast<const uint16_t*>(xh + t1 * kCsRowBytes + ((cpos ^ (t1 & 7)) << 4) + cin);
            const uint32_t x2 = x0 | (x1 << 16);
            const uint4 w = wt[hh * (kCsKH / 2) + 16 * half + j];
            const uint32_t h2 = fma_bf16x2(x2, w.x, 0x80008000u);  // x w_hi, rounded
            const uint32_t d2 = fma_bf16x2(x2, w.y, h2);           // hi - x w_hi, exact
            lo[j] = fma_bf16x2(x2, w.z, d2) ^ 0x80008000u;         // x w - hi, rounded
            hi[j] = h2;
          }
          const uint32_t a_hi = tmem + lane_base + kCsTmemA + 64u * as + 16u * half;
          tc::tmem_st16(a_hi, hi);
          tc::tmem_st16(a_hi + 32, lo);
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        fence_proxy_async_smem();  // the X and G/dt reads, before the stage's TMA refill
        named_bar_sync(gbar, 128);
        if (gt == 0) {
          mbar_arrive(&bars[kXEmpty + st]);  // X and G/dt of step i are read: refill the stage
          mbar_arrive(&bars[kAFull + as]);   // hi and lo of step i are in TMEM
        }
      }
    }
  } else {
    // ------------------------------ epilogue: TMEM -> S_c ----------------------------------
    const int quad = warp & 3;  // TMEM lanes 32*quad .. +31 = accumulator rows
    unsigned char* stg = base + L.epi0 + quad * 32 * kCsRowBytes;
    int q = 0;
    bool stored = false;
    for (int64_t u = u_begin; u < u_end; ++u, ++q) {
      const CsUnit w = cs_unit(p, u);
      const int acc = q & 1;
      const bool bad = !mbar_wait(&bars[kAccFull + acc], (uint32_t)(q >> 1) & 1u, ctl.spin_limit_ns);
      if (named_bar_any(kCsEpiBar, 128, bad)) {  // leave together, or not at all
        if (threadIdx.x == 320) fail();
        break;
      }
      tc::fence_after_sync();
      // the unit's 128 accumulator rows are 128 consecutive rows of S_c (two heads x 64 p)
      const int row0 = (int)(((w.bi * p.nchunks + w.c) * p.nheads + w.h) * 64) + quad * 32;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + acc * 128 + cb * 32, r);
        tc::tmem_ld_wait();
        if (cb == 3) {  // the accumulator has been read
          tc::fence_before_sync();
          named_bar_sync(kCsEpiBar, 128);
          if (threadIdx.x == 320) mbar_arrive(&bars[kAccEmpty + acc]);
        }
        if (stored) {  // the previous block's store has read the staging rows
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<float4*>(stg + lane * kCsRowBytes + ((j ^ (lane & 7)) << 4)) =
              make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]), __uint_as_float(r[4 * j + 2]),
                          __uint_as_float(r[4 * j + 3]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&map_sc, stg, cb * 32, row0);
          bulk_commit();
        }
        stored = true;
      }
    }
    if (lane == 0) bulk_wait<0>();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kCsTmemCols);
  }
}

}  // namespace

bool ssd_tc_supported(const SsdDims& d) {
  return d.dtype == SSM_BF16 && d.headdim == 64 && d.dstate == 128 && (d.nheads / d.ngroups) % 2 == 0 &&
         d.chunk <= kCsMaxT;
}

cudaError_t launch_ssd_chunk_state_tc(const void* x, const void* B, const SsdDims& d, const SsdWorkspace& ws,
                                      const LookbackCtl& ctl, cudaStream_t s) {
  CUtensorMap map_x, map_b;
  const uint64_t xd[3] = {(uint64_t)d.nheads * 64, (uint64_t)d.seqlen, (uint64_t)d.batch};
  const uint64_t xs[2] = {(uint64_t)d.nheads * 64 * 2, (uint64_t)d.seqlen * d.nheads * 64 * 2};
  const uint64_t bd[3] = {(uint64_t)d.ngroups * 128, (uint64_t)d.seqlen, (uint64_t)d.batch};
  const uint64_t bs[2] = {(uint64_t)d.ngroups * 128 * 2, (uint64_t)d.seqlen * d.ngroups * 128 * 2};
  const uint32_t xbox[3] = {64, (uint32_t)kCsKH, 1};
  const uint32_t bbox[3] = {64, (uint32_t)d.chunk, 1};
  cudaError_t e;
  if ((e = encode_tensor_map_3d(&map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, xd, xs, xbox, CU_TENSOR_MAP_SWIZZLE_128B)) !=
      cudaSuccess)
    return e;
  if ((e = encode_tensor_map_3d(&map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, bd, bs, bbox, CU_TENSOR_MAP_SWIZZLE_128B)) !=
      cudaSuccess)
    return e;
  CUtensorMap map_sc;  // S_c as rows (batch, chunk, head, p) x 128 s, f32
  const uint64_t sc_rows = (uint64_t)d.batch * d.nchunks * d.nheads * 64;
  if ((e = encode_tensor_map_2d(&map_sc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ws.Sc, 128, sc_rows, 512, 32, 32,
                                CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  CsParams p;
  p.G = ws.G;
  p.dtT = ws.dtT;
  p.Sc = ws.Sc;
  p.hdr = ws.hdr;
  p.batch = d.batch;
  p.lpad = d.lpad;
  p.nchunks = d.nchunks;
  p.nheads = d.nheads;
  p.ngroups = d.ngroups;
  p.chunk = d.chunk;
  p.units = d.batch * d.nchunks * d.ngroups * (d.nheads / d.ngroups / 2);
  int dev = 0, sms = 148;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const CsLayout L(d.chunk);
  const size_t smem = L.total + 1024;
  if ((e = ensure_smem_limit(reinterpret_cast<const void*>(ssd_chunk_state_tc_kernel), smem)) != cudaSuccess)
    return e;
  // one CTA per SM (shared memory allows no second), each with an equal share of the units
  const int64_t grid = p.units < sms ? p.units : sms;
  return launch_pdl(ssd_chunk_state_tc_kernel, dim3((unsigned)grid), dim3(kCsThreads), smem, s, map_x, map_b, map_sc, p,
                    ctl);
}

}  // namespace ssm
