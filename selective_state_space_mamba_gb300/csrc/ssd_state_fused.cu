// ssd_state_fused_tc: the chunk states and the inter-chunk recurrence of the Mamba-2 SSD
// forward in one pass, for bf16 inputs ("Accelerating Mamba-2 with High-Performance Forward
// Pass Kernels in NVIDIA CUDA Tile", "Kernel 2: fwd_pass_state": the chunk loop runs inside one
// program and every chunk-initial state is written once):
//     h_in[0] = h0,   h_in[c+1] = 2^(G_last[c]) h_in[c] + X_c^T (w_c . B_c),   h_final = h_in[nc]
// with w_t = dt_t 2^(G_last - G_t) inside chunk c.
//
// A chain is the chunks of one (batch, head pair), walked in order.  The CTAs take contiguous,
// equal ranges of the (chain, chunk) units, chain-major: one chain each when there are no more
// chains than SMs, else one CTA per SM and ranges of at least one chain's length, so that a
// range holds at most the tail of one chain, whole chains and the head of one more.  A CTA
// runs the head first and publishes the state where it stops (f32, with a flag), then the
// whole chains, then the tail, which starts from the state the previous CTA published for
// that chain: the previous CTA ran that head first, and its head is shorter than what this
// CTA runs before its tail by the range length minus the chain length, so the wait is short.
// With few long chains (fewer than half as many as SMs) one CTA per chain leaves most SMs idle,
// so the pass can instead split them ("split chains"): one CTA per SM runs an equal range of
// units at once, every segment that starts inside its chain from a zero state, and each range
// publishes the state where it stops into its own slot; ssd_state_fixup (below) then adds to
// every such piece's h_in, and to h_final, the state the piece enters with.  The recurrence is
// linear in the state, so this gives the chain's states exactly (h_in is rounded to bf16 once
// more).
// The pair's rows (2 heads x 64 p = 128 TMEM lanes, x 128 s columns, f32) have three TMEM
// homes: the running state h and two accumulators S[0], S[1].  The MMAs add the weighted X^T B
// of the CTA's q-th chunk c into S[q & 1] without waiting for the state; the state warps then
// write h out as h_in[c] (bf16), fold S[q & 1] in (h = 2^(G_last) h + S) and release the
// accumulator for the chunk run two later.  The weighted X is split
// into bf16 hi + lo halves exactly as in ssd_chunk_state_tc, so the state keeps f32 accuracy.
// The per-chunk increments S_c never go to memory: against the chunk-state + state-passing
// pair this saves writing and re-reading them (f32) entirely.
//
// Warps (480 threads):
//   warp 0     TMA producer of X: per 64-token step, X of the pair's two heads with the step's
//              G and dt and the chunk's last G into the X ring
//   warp 1     TMEM owner and MMA issuer (one thread): per chunk, once S[q & 1] is free,
//              2 x 4 MMAs (hi, lo) per step accumulating into it, A from the operand ring
//   warp 2     TMA producer of B: the step's rows of the group's B into the B ring
//   warps 3-6  scalers, a token row per thread: the row to registers, the X slot handed back at
//              once, x w -> hi + lo into the operand ring.  X is thus held only from its load
//              to the scalers' read, and B and the operand from their fill to the MMAs'
//              completion, instead of one stage holding all three from the load to the MMAs
//   warps 7-14 state warps, two threads per state row: h0 or the published state in, h_in out
//              per chunk, the decay and S folded in, h_final at a chain's end, the state
//              published where a head ends
// Every wait is bounded; on expiry the CTA records SSM_ERR_TIMEOUT, drains, frees its TMEM and
// returns.
#include "tc_common.cuh"

#ifndef SSM_SF_SPLIT_MIN_CHUNKS  // the rule splits chains of at least this many chunks
#define SSM_SF_SPLIT_MIN_CHUNKS 32
#endif

namespace ssm {
namespace {

constexpr int kSfScalers = 128;      // warps 3-6: one token row of one head per thread
constexpr int kSfStateThreads = 256; // warps 7-14: two threads per state row
constexpr int kSfScaler0 = 96;       // first scaler thread (warps 0-2: X producer, MMA, B producer)
constexpr int kSfThreads = kSfScaler0 + kSfScalers + kSfStateThreads;
constexpr int kSfKH = 64;         // tokens per step
// Ring depths: X slots and B slots are template parameters (the plan picks the split: 4 + 3,
// 3 + 4 or 5 + 2; B comes from L2, shared by every head of a group); operand (hi + lo) slots:
constexpr int kSfOS = 2;
constexpr int kSfRowBytes = 128;  // 64 bf16 per swizzled row
constexpr uint32_t kSfScaleBar = 1, kSfStateBar = 2;
constexpr uint32_t kSfTmemCols = 512;  // h at 0, S[0] at 128, S[1] at 256
constexpr uint32_t kSfGdHead = (2 * kSfKH + 4) * 4;  // G[64], dt[64], G[T-4 .. T-1] of one head

struct SfParams {
  const float* G;
  const float* dtT;
  const float* h0;   // [b, nh, 64, 128] f32 or null (zeros)
  __nv_bfloat16* hin;  // [b, nc, nh, 64, 128]
  float* h_final;    // [b, nh, 64, 128] or null
  float* carry;      // [chains][128 rows][128] f32: the state where a chain's head ends
  unsigned long long* flags;  // [chains]: carry published (epoch-tagged)
  WsHeader* hdr;
  int64_t batch, lpad, nchunks, units;  // units = chains x nchunks
  int nheads, ngroups, chunk;
  int b_keep;  // B is small next to L2: load it with evict-last priority
  int split;   // chains split into independent pieces (see ssd_state_fixup below)
};

// This CTA's units [u0, u1) of (chain, chunk), chain-major, as segments in the order they run:
// the head that ends inside the range (publishes its final state), whole chains, the tail
// that starts inside the range (starts from the published state).  A range is never inside
// one chain (ranges are at least one chain long where a chain is split).
struct SfRange {
  int64_t first_chain, last_chain, full_begin;
  int c_first, c_last_end, nfull, nseg;
  bool has_tail, has_head, single;  // single: the range lies inside one chain (one segment)
};
struct SfSeg {
  int64_t chain;
  int c0, c1;
  bool from_carry, to_carry;
};
__host__ __device__ __forceinline__ SfRange sf_range(int64_t u0, int64_t u1, int64_t nc) {
  SfRange r;
  r.first_chain = u0 / nc;
  r.c_first = (int)(u0 % nc);
  r.last_chain = (u1 - 1) / nc;
  r.c_last_end = (int)((u1 - 1) % nc) + 1;
  r.has_tail = r.c_first > 0;
  r.has_head = r.c_last_end < nc;
  r.full_begin = r.first_chain + (r.has_tail ? 1 : 0);
  const int64_t full_end = r.last_chain + (r.has_head ? 0 : 1);
  r.nfull = full_end > r.full_begin ? (int)(full_end - r.full_begin) : 0;
  r.nseg = (r.has_head ? 1 : 0) + r.nfull + (r.has_tail ? 1 : 0);
  r.single = r.first_chain == r.last_chain;
  if (r.single) r.nseg = 1;  // a whole chain, or (split chains) a piece inside one
  return r;
}
__host__ __device__ __forceinline__ SfSeg sf_seg(const SfRange& r, int s, int64_t nc) {
  SfSeg g;
  if (r.single) {
    g.chain = r.first_chain;
    g.c0 = r.c_first;
    g.c1 = r.c_last_end;
    g.from_carry = r.c_first > 0;
    g.to_carry = r.c_last_end < nc;
    return g;
  }
  if (r.has_head) {
    if (s == 0) {
      g.chain = r.last_chain;
      g.c0 = 0;
      g.c1 = r.c_last_end;
      g.from_carry = false;
      g.to_carry = true;
      return g;
    }
    --s;
  }
  if (s < r.nfull) {
    g.chain = r.full_begin + s;
    g.c0 = 0;
    g.c1 = (int)nc;
  } else {
    g.chain = r.first_chain;
    g.c0 = r.c_first;
    g.c1 = (int)nc;
  }
  g.from_carry = s >= r.nfull;
  g.to_carry = false;
  return g;
}

// Shared memory (offsets from a 1024-byte aligned base), three rings:
//   X[XS]      X of the pair's two heads for one step: [2 heads][64 rows][128 B], swizzled;
//              released as soon as the scalers hold it in registers
//   B[BS]      the step's rows of the group's B: [2 s blocks][64 rows][128 B], swizzled;
//              released when the step's MMAs complete
//   Op[kSfOS]  the weighted X of one step as bf16 hi and lo halves, each laid out like X;
//              written by the scalers, released when the step's MMAs complete
//   Hs         h_in of one chunk as bf16, [2 s blocks][128 rows][128 B], swizzled: the state
//              warps write it here and one TMA store per s block takes it to memory, so
//              that their 256-byte rows do not reach the load/store unit as scattered
//              16-byte stores (these held up the scalers' shared-memory accesses)
//   gd[XS][2 heads]  G, dt and the chunk's last G of the step (travels with X)
//   barriers, TMEM base, abort flag
template <int XS, int BS>
struct SfLayout {
  uint32_t x_bytes, b0, op0, op_bytes, hs0, gd0, bars, total;
  __host__ __device__ SfLayout() {
    x_bytes = 2u * kSfKH * kSfRowBytes;  // 16 KB
    b0 = XS * x_bytes;
    op0 = b0 + BS * x_bytes;
    op_bytes = 2u * x_bytes;
    hs0 = op0 + kSfOS * op_bytes;
    gd0 = hs0 + 2u * 128 * kSfRowBytes;
    bars = gd0 + XS * 2u * kSfGdHead;
    total = bars + 32 * 8 + 16;
  }
};

// d = a * b + c on bf16 pairs, one rounding
__device__ __forceinline__ uint32_t sf_fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t sf_bf16_pair(float v) {
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return h | (h << 16);
}
__device__ __forceinline__ uint32_t sf_pack(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int XS, int BS>
__global__ void __launch_bounds__(kSfThreads, 1)
    ssd_state_fused_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_b,
                              const __grid_constant__ CUtensorMap map_hin, SfParams p, LookbackCtl ctl_call) {
  constexpr int kSfXS = XS, kSfBS = BS;
  // mbarriers: X full / empty, B full / empty, operand full / empty, S ready / free, done
  constexpr int kXFull = 0, kXEmpty = kXFull + kSfXS, kBFull = kXEmpty + kSfXS, kBEmpty = kBFull + kSfBS;
  constexpr int kOpFull = kBEmpty + kSfBS, kOpEmpty = kOpFull + kSfOS, kSReady = kOpEmpty + kSfOS;
  constexpr int kSFree = kSReady + 2, kDone = kSFree + 2, kSfNumBars = kDone + 1;
  static_assert(kSfNumBars <= 32, "barrier area");
  extern __shared__ unsigned char sf_raw[];
  const uint32_t raw = smem_addr(sf_raw);
  unsigned char* base = sf_raw + ((1024u - (raw & 1023u)) & 1023u);
  const int T = p.chunk;
  const SfLayout<XS, BS> L;
  const int nk = T / kSfKH;  // steps per chunk
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.bars + 32 * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L.bars + 32 * 8 + 4);
  volatile uint32_t* claim_slot = reinterpret_cast<volatile uint32_t*>(base + L.bars + 32 * 8 + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hpg = p.nheads / p.ngroups, ppg = hpg / 2;
  const int64_t nc = p.nchunks;
  // chain -> (batch, group, first head of the pair)
  auto chain_bi = [&](int64_t z) { return z / ((int64_t)ppg * p.ngroups); };
  auto chain_g = [&](int64_t z) { return (int)((z / ppg) % p.ngroups); };
  auto chain_h = [&](int64_t z) { return chain_g(z) * hpg + 2 * (int)(z % ppg); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSfNumBars; ++i)
      mbar_init(&bars[i], (i >= kXEmpty && i < kXEmpty + kSfXS) || (i >= kOpFull && i < kOpFull + kSfOS)
                              ? (uint32_t)kSfScalers
                              : 1u);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kSfTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // G and dt come from the previous kernel (which also zeroed the claim counter)
  // Dependents may launch only now: the chunk scan loads the forward's inputs (C, B, x) before
  // its own wait, which is safe because this point is reached only after the cumsum, and so
  // every kernel before it, has completed.
  griddep_launch_dependents();
  // The CTA's range index is claimed in order from the workspace counter, not taken from
  // blockIdx: the CTA it may wait for (range index - 1) has then claimed first, so it is
  // running, and its first segment waits for nobody.  No CTA needs another to be resident.
  if (threadIdx.x == 0) *claim_slot = atomicAdd(&p.hdr->counter, 1u);
  __syncthreads();
  const int64_t vb = *claim_slot;
  const int64_t u0 = vb * p.units / gridDim.x;
  const int64_t u1 = (vb + 1) * p.units / gridDim.x;
  const SfRange rg = nc > 0 && u1 > u0 ? sf_range(u0, u1, nc) : SfRange{0, 0, 0, 0, 0, 0, 0, false, false, false};
  // published states carry this launch's epoch (the last CTA to finish moves it on)
  const LookbackCtl ctl = device_epoch(ctl_call, p.hdr);
  auto fail = [&](void) {
    record_error(p.hdr, ctl.epoch, SSM_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------------------
    if (lane == 0) {
      int64_t i = 0, nx = 0;  // steps and X copies issued
      bool ok = true;
      for (int s = 0; s < rg.nseg && ok; ++s) {
        const SfSeg sg = sf_seg(rg, s, nc);
        const int64_t bi = chain_bi(sg.chain);
        const int g = chain_g(sg.chain), h = chain_h(sg.chain);
        for (int64_t c = sg.c0; c < sg.c1 && ok && !*abort_flag; ++c) {
          for (int kh = 0; kh < nk; ++kh, ++i) {
            const int xs = (int)(i % kSfXS);
            const int tok = (int)(c * T + kh * kSfKH);
            // X and the step's G / dt: the slot is free once the scalers hold step i - kSfXS
            if (i >= kSfXS && !mbar_wait(&bars[kXEmpty + xs], (uint32_t)((i / kSfXS) - 1) & 1u, ctl.spin_limit_ns)) {
              ok = false;
              break;
            }
            unsigned char* xst = base + xs * L.x_bytes;
            unsigned char* gd = base + L.gd0 + xs * 2 * kSfGdHead;
            mbar_arrive_expect_tx(&bars[kXFull + xs], L.x_bytes + 2u * kSfGdHead);
            // x is read once: evict-first, so that its stream does not push B out of L2
            for (int hh = 0; hh < 2; ++hh)
              tc::tma_load_3d_hint(xst + hh * kSfKH * kSfRowBytes, &map_x, (h + hh) * 64, tok, (int)bi, &bars[kXFull + xs],
                                   l2_evict_first_policy());
            for (int hh = 0; hh < 2; ++hh) {
              const int64_t row = (bi * p.nheads + h + hh) * p.lpad + c * T;
              // G and dt^T are [b, nh, lpad]: the chunk's T entries of this head
              if (!SSM_CHECK(p.hdr, h + hh < p.nheads && row + T <= p.batch * p.nheads * p.lpad)) continue;
              bulk_g2s(gd + hh * kSfGdHead, p.G + row + kh * kSfKH, 4u * kSfKH, &bars[kXFull + xs]);
              bulk_g2s(gd + hh * kSfGdHead + 4u * kSfKH, p.dtT + row + kh * kSfKH, 4u * kSfKH, &bars[kXFull + xs]);
              bulk_g2s(gd + hh * kSfGdHead + 8u * kSfKH, p.G + row + T - 4, 16u, &bars[kXFull + xs]);
            }
            ++nx;
          }
        }
      }
      if (!ok) fail();
      // leave no copy in flight (bounded): the last copies into every slot of both rings
      for (int64_t j = (nx > kSfXS ? nx - kSfXS : 0); j < nx; ++j)
        mbar_wait(&bars[kXFull + (int)(j % kSfXS)], (uint32_t)(j / kSfXS) & 1u, ctl.spin_limit_ns);
    }
  } else if (warp == 2) {
    // ------------------------------ TMA producer of B --------------------------------------
    // Its own thread, so that a B slot, held until the MMAs of its step complete, never holds
    // back the X loads, which come from DRAM and need the longer lead.
    if (lane == 0) {
      int64_t i = 0, nb = 0;  // steps and B copies issued
      bool ok = true;
      for (int s = 0; s < rg.nseg && ok; ++s) {
        const SfSeg sg = sf_seg(rg, s, nc);
        const int64_t bi = chain_bi(sg.chain);
        const int g = chain_g(sg.chain);
        for (int64_t c = sg.c0; c < sg.c1 && ok && !*abort_flag; ++c) {
          for (int kh = 0; kh < nk; ++kh, ++i) {
            const int bs = (int)(i % kSfBS);
            // the slot is free once the MMAs of step i - kSfBS have completed
            if (i >= kSfBS && !mbar_wait(&bars[kBEmpty + bs], (uint32_t)((i / kSfBS) - 1) & 1u, ctl.spin_limit_ns)) {
              ok = false;
              break;
            }
            unsigned char* bst = base + L.b0 + bs * L.x_bytes;
            mbar_arrive_expect_tx(&bars[kBFull + bs], L.x_bytes);
            // B is read by every head pair of its group: where all of it fits well inside L2
            // (8 MB at b4 L8192), evict-last keeps it there against the x stream
            for (int sb = 0; sb < 2; ++sb) {
              if (p.b_keep)
                tc::tma_load_3d_hint(bst + sb * kSfKH * kSfRowBytes, &map_b, g * 128 + sb * 64, (int)(c * T + kh * kSfKH),
                                     (int)bi, &bars[kBFull + bs], l2_evict_last_policy());
              else
                tc::tma_load_3d(bst + sb * kSfKH * kSfRowBytes, &map_b, g * 128 + sb * 64, (int)(c * T + kh * kSfKH),
                                (int)bi, &bars[kBFull + bs]);
            }
            ++nb;
          }
        }
      }
      if (!ok) fail();
      for (int64_t j = (nb > kSfBS ? nb - kSfBS : 0); j < nb; ++j)
        mbar_wait(&bars[kBFull + (int)(j % kSfBS)], (uint32_t)(j / kSfBS) & 1u, ctl.spin_limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ---------------------------------------------
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(128, 128, /*a_mn=*/true, /*b_mn=*/true);
      const uint32_t ab_lbo = kSfKH * kSfRowBytes;  // head 0 -> head 1 block, s 0..63 -> s 64..127 block
      const uint32_t sbo = 8 * kSfRowBytes;         // next 8-token group
      bool ok = true;
      int64_t i = 0, nready = 0;  // steps whose MMAs were committed, chunks handed to the state warps
      const int64_t nq = u1 - u0;  // chunks this CTA runs, in order (the accumulators alternate)
      for (int64_t q = 0; q < nq && ok && !*abort_flag; ++q) {
        const int sb = (int)(q & 1);
        const uint32_t acc = tmem + 128u + 128u * sb;
        // the state warps have folded S[sb] (the chunk run two before) into the state
        if (q >= 2 && !mbar_wait(&bars[kSFree + sb], (uint32_t)(((q - 2) >> 1) & 1), ctl.spin_limit_ns)) {
          ok = false;
          break;
        }
        for (int kh = 0; kh < nk; ++kh, ++i) {
          const int os = (int)(i % kSfOS), bs = (int)(i % kSfBS);
          if (!mbar_wait(&bars[kOpFull + os], (uint32_t)(i / kSfOS) & 1u, ctl.spin_limit_ns) ||
              !mbar_wait(&bars[kBFull + bs], (uint32_t)(i / kSfBS) & 1u, ctl.spin_limit_ns)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t hi0 = smem_addr(base + L.op0 + os * L.op_bytes);
          const uint32_t lo0 = hi0 + L.x_bytes;
          const uint32_t b0 = smem_addr(base + L.b0 + bs * L.x_bytes);
#pragma unroll
          for (int ks = 0; ks < kSfKH / 16; ++ks) {
            const uint32_t koff = ks * 16 * kSfRowBytes;  // 16 tokens = two 8-row groups
            const uint64_t bdesc = tc::sdesc_sw128(b0 + koff, ab_lbo, sbo);
            tc::mma_bf16(acc, tc::sdesc_sw128(hi0 + koff, ab_lbo, sbo), bdesc, idesc, kh > 0 || ks > 0);
            tc::mma_bf16(acc, tc::sdesc_sw128(lo0 + koff, ab_lbo, sbo), bdesc, idesc, true);
          }
          tc::mma_commit(&bars[kOpEmpty + os]);  // the operand slot may take a later step
          tc::mma_commit(&bars[kBEmpty + bs]);   // the B slot may be refilled
        }
        if (ok) {
          tc::mma_commit(&bars[kSReady + sb]);  // S[sb] holds chunk q
          ++nready;
        }
      }
      if (!ok) fail();
      tc::mma_commit(&bars[kDone]);
      mbar_wait(&bars[kDone], 0, ctl.spin_limit_ns);  // every MMA has completed
      // A commit's arrive lands when its MMAs complete, in no fixed order with the others: wait
      // for the last phase of every committed barrier, so that no arrive is still due to this
      // CTA's shared memory when it exits.
      for (int x = 0; x < kSfOS; ++x)
        if (i > x) mbar_wait(&bars[kOpEmpty + x], (uint32_t)(((i - 1 - x) / kSfOS) & 1), ctl.spin_limit_ns);
      for (int x = 0; x < kSfBS; ++x)
        if (i > x) mbar_wait(&bars[kBEmpty + x], (uint32_t)(((i - 1 - x) / kSfBS) & 1), ctl.spin_limit_ns);
      for (int x = 0; x < 2; ++x)
        if (nready > x) mbar_wait(&bars[kSReady + x], (uint32_t)(((nready - 1 - x) / 2) & 1), ctl.spin_limit_ns);
    }
  } else if (warp < (kSfScaler0 + kSfScalers) / 32) {
    // ---------------- scale X by w, split into bf16 hi + lo parts --------------------------
    // One token row of one head per thread: the row's eight 16-byte pieces go to registers,
    // the X slot is handed back, then hi and lo are written to the operand slot.
    const int t = threadIdx.x - kSfScaler0;  // token row of the step: head t / 64, token t % 64
    const int hh = t / kSfKH, tok = t % kSfKH;
    const int64_t nsteps = (u1 - u0) * nk;
    for (int64_t i = 0; i < nsteps; ++i) {
      const int xs = (int)(i % kSfXS), os = (int)(i % kSfOS);
      const bool bad = !mbar_wait(&bars[kXFull + xs], (uint32_t)(i / kSfXS) & 1u, ctl.spin_limit_ns) ||
                       (i >= kSfOS && !mbar_wait(&bars[kOpEmpty + os], (uint32_t)((i / kSfOS) - 1) & 1u,
                                                 ctl.spin_limit_ns));
      if (named_bar_any(kSfScaleBar, kSfScalers, bad)) {  // leave together, or not at all
        if (t == 0) fail();
        break;
      }
      const float* gd = reinterpret_cast<const float*>(base + L.gd0 + (xs * 2 + hh) * kSfGdHead);
      const float wv = gd[kSfKH + tok] * tc::ex2_approx(gd[2 * kSfKH + 3] - gd[tok]);
      const unsigned char* xrow = base + xs * L.x_bytes + t * kSfRowBytes;
      // the row's pieces in an order rotated by the row, so that a warp's accesses spread over
      // the banks; each piece keeps its swizzled position in the operand slot
      uint4 xv[8];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) xv[cc] = *reinterpret_cast<const uint4*>(xrow + ((cc ^ (t & 7)) << 4));
      // these reads are performed before the TMA (async proxy) refills the slot
      fence_proxy_async_smem();
      mbar_arrive(&bars[kXEmpty + xs]);
      const __nv_bfloat16 w_hi = __float2bfloat16_rn(wv);
      const float w_lo = wv - __bfloat162float(w_hi);
      const uint32_t whi2 = sf_bf16_pair(__bfloat162float(w_hi));
      const uint32_t nwhi2 = whi2 ^ 0x80008000u;
      const uint32_t nwlo2 = sf_bf16_pair(-w_lo);
      unsigned char* hrow = base + L.op0 + os * L.op_bytes + t * kSfRowBytes;
      unsigned char* lrow = hrow + L.x_bytes;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const int pc = cc ^ (t & 7);  // the piece's position in the row (X's swizzled layout)
        uint32_t* e = reinterpret_cast<uint32_t*>(&xv[cc]);
        uint4 hv, lv;
        uint32_t* fh = reinterpret_cast<uint32_t*>(&hv);
        uint32_t* fl = reinterpret_cast<uint32_t*>(&lv);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t x2 = e[k];
          const uint32_t h2 = sf_fma_bf16x2(x2, whi2, 0x80008000u);  // x w_hi, rounded
          const uint32_t d2 = sf_fma_bf16x2(x2, nwhi2, h2);           // hi - x w_hi, exact
          fl[k] = sf_fma_bf16x2(x2, nwlo2, d2) ^ 0x80008000u;          // x w - hi, rounded
          fh[k] = h2;
        }
        *reinterpret_cast<uint4*>(hrow + (pc << 4)) = hv;
        *reinterpret_cast<uint4*>(lrow + (pc << 4)) = lv;
      }
      fence_proxy_async_smem();  // the MMAs read the operand through the async proxy
      mbar_arrive(&bars[kOpFull + os]);
    }
  } else {
    // ------------------------------ state warps --------------------------------------------
    // Two threads per state row (TMEM lane), 64 of its 128 columns each.
    const int sw = warp - (kSfScaler0 + kSfScalers) / 32;  // 0 .. 7
    const int quad = warp & 3;                  // TMEM lanes 32*quad .. +31
    const int half = sw >> 2;                   // columns 64*half .. +63
    const int m = quad * 32 + lane;             // state row: head h + m / 64, p = m % 64
    const int hh = m >> 6, pp = m & 63;
    const int col0 = 64 * half;
    const bool leader = half == 0 && m == 0;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    int64_t q = 0;  // chunks run so far (the accumulators alternate)
    bool ok = true;
    for (int s = 0; s < rg.nseg && ok; ++s) {
      const SfSeg sg = sf_seg(rg, s, nc);
      const int64_t bi = chain_bi(sg.chain);
      const int h = chain_h(sg.chain);
      const int64_t bh = bi * p.nheads + h + hh;
      // the state rows of both heads (h0, h_final, G) and the chain's published state and flag;
      // the same answer in every state thread, so that they leave together
      if (!SSM_CHECK(p.hdr, bi * p.nheads + h + 1 < p.batch * p.nheads && sg.chain < p.units / nc)) {
        ok = false;
        break;
      }
      const float* h0r = p.h0 ? p.h0 + (bh * 64 + pp) * 128 + col0 : nullptr;
      // this row of the published state: the chain's slot, or with split chains the range's
      // (a range ends inside at most one chain)
      float* cr = p.carry + ((p.split ? vb : sg.chain) * 128 + m) * 128 + col0;
      const float* Glast = p.G + bh * p.lpad + (T - 1);  // G_last of chunk c at Glast[c * T]
      if (sg.from_carry && !p.split) {
        // the previous CTA ran this chain's head first and published where it stopped
        bool bad = false;
        if (leader) bad = wait_flag(&p.flags[sg.chain], p.hdr, ctl) != kFlagPrefix;
        if (named_bar_any(kSfStateBar, kSfStateThreads, bad)) {
          if (leader) fail();
          ok = false;
          break;
        }
      }
      for (int64_t c = sg.c0; c < sg.c1; ++c, ++q) {
        const int sb = (int)(q & 1);
        const bool bad = !mbar_wait(&bars[kSReady + sb], (uint32_t)((q >> 1) & 1), ctl.spin_limit_ns);
        if (leader) bulk_wait_read<0>();  // the previous chunk's h_in store has read the staging buffer
        if (named_bar_any(kSfStateBar, kSfStateThreads, bad)) {  // S[sb] holds chunk c
          if (leader) fail();
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const float dec = exp2f(Glast[c * T]);  // decay over chunk c
        unsigned char* hsrow = base + L.hs0 + half * (128 * kSfRowBytes) + m * kSfRowBytes;
        const bool chain_end = c == nc - 1, publish = sg.to_carry && c == sg.c1 - 1;
        const bool first = c == sg.c0;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {  // 16 columns (s) at a time
          const uint32_t col = (uint32_t)(col0 + 16 * qq);
          float v[16];
          uint32_t sv[16];
          tc::tmem_ld16(tmem + lane_base + 128u + 128u * sb + col, sv);
          if (first && !sg.from_carry) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float4 f = h0r ? reinterpret_cast<const float4*>(h0r + 16 * qq)[j] : make_float4(0.f, 0.f, 0.f, 0.f);
              v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
            }
          } else if (first && p.split) {  // a piece of a split chain: from zero, fixed up later
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.f;
          } else if (first) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float4 f = ld_relaxed_f4(reinterpret_cast<const float4*>(cr + 16 * qq) + j);
              v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
            }
          } else {
            uint32_t r[16];
            tc::tmem_ld16(tmem + lane_base + col, r);
            tc::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
          }
          tc::tmem_ld_wait();
          // h_in[c] (bf16): the state entering chunk c, to the staging buffer (16-byte piece
          // 2 qq + j of the row's s block, swizzled)
#pragma unroll
          for (int j = 0; j < 2; ++j)
            *reinterpret_cast<uint4*>(hsrow + (((2 * qq + j) ^ (m & 7)) << 4)) =
                make_uint4(sf_pack(v[8 * j], v[8 * j + 1]), sf_pack(v[8 * j + 2], v[8 * j + 3]),
                           sf_pack(v[8 * j + 4], v[8 * j + 5]), sf_pack(v[8 * j + 6], v[8 * j + 7]));
          // the state after chunk c
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = fmaf(dec, v[j], __uint_as_float(sv[j]));
          if (chain_end) {
            if (p.h_final) {
              float4* f = reinterpret_cast<float4*>(p.h_final + (bh * 64 + pp) * 128 + col0 + 16 * qq);
#pragma unroll
              for (int j = 0; j < 4; ++j) f[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
          } else if (publish) {  // h_in[c + 1] for the CTA that runs the rest of this chain
            float4* f = reinterpret_cast<float4*>(cr + 16 * qq);
#pragma unroll
            for (int j = 0; j < 4; ++j) f[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
            uint32_t s0[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) s0[j] = __float_as_uint(v[j]);
            tc::tmem_st16(tmem + lane_base + col, s0);
          }
        }
        tc::tmem_st_wait();
        if (publish && !p.split) __threadfence();  // this thread's part of the published state, before the flag
        fence_proxy_async_smem();      // the staged h_in, before the TMA store reads it
        tc::fence_before_sync();
        named_bar_sync(kSfStateBar, kSfStateThreads);
        if (leader) {
          const int64_t row0 = ((bi * nc + c) * p.nheads + h) * 64;  // the pair's 128 rows of h_in[c]
          if (SSM_CHECK(p.hdr, c < nc && row0 + 128 <= p.batch * nc * p.nheads * 64))
            for (int s2 = 0; s2 < 2; ++s2)
              tma_store_2d(&map_hin, base + L.hs0 + s2 * (128 * kSfRowBytes), 64 * s2, (int)row0);
          bulk_commit();
          mbar_arrive(&bars[kSFree + sb]);  // S[sb] may take the chunk run two later
          if (publish && !p.split) st_release_u64(&p.flags[sg.chain], make_flag(ctl.epoch, kFlagPrefix));
        }
      }
    }
    if (leader) bulk_wait<0>();  // every h_in store has completed
    if (nc == 0 && p.h_final) {  // no chunks: the final state is the initial one (one chain per CTA)
      const int64_t bh = chain_bi(vb) * p.nheads + chain_h(vb) + hh;
      const float* h0r = p.h0 ? p.h0 + (bh * 64 + pp) * 128 + col0 : nullptr;
      float4* f = reinterpret_cast<float4*>(p.h_final + (bh * 64 + pp) * 128 + col0);
#pragma unroll 4
      for (int j = 0; j < 16; ++j) f[j] = h0r ? reinterpret_cast<const float4*>(h0r)[j] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kSfTmemCols);
  }
  if (threadIdx.x == 0) retire_tile(p.hdr, gridDim.x);  // the last CTA moves the epoch on
}

// ---------------------------------------------------------------------------------------------
// ssd_state_fixup: with split chains the fused pass runs all pieces of a chain at once, every
// piece that starts inside its chain from a zero state, and each range leaves the state where
// its last segment ends in its own slot E[j] (j = the range index).  The state entering the
// piece that range k starts at unit u_k (inside chain z, which starts at unit zc) follows the
// chain's own recurrence taken over pieces:
//     H(u_k) = E[k-1] + 2^(D(u_(k-1), u_k)) H(u_(k-1))   if u_(k-1) > zc,  else  H(u_k) = E[k-1]
// with D(a, b) the decay exponent (the sum of G_last) over the chunks a .. b-1.  This kernel
// forms H(u_k) in f32 and adds 2^(D(u_k, c)) H(u_k) to h_in[c] for every chunk c of the piece,
// and to h_final where the piece ends its chain; what the fused pass wrote there is the
// piece's own part, exact by linearity of the recurrence.  One CTA per (piece, block of 16
// state rows of one head), eight consecutive entries per thread.
constexpr int kFxThreads = 256;
constexpr int kFxRows = 16;
constexpr int kFxPieces = 256;  // earlier pieces whose decay sums are formed together
constexpr int kFxBatch = 8;     // chunks whose h_in loads are in flight together
constexpr int kFxFold = 2;      // earlier pieces' end states in flight together

struct FxParams {
  const float* G;
  __nv_bfloat16* hin;  // [b, nc, nh, 64, 128]
  float* h_final;      // [b, nh, 64, 128] or null
  const float* carry;  // [ranges][128 rows][128]: E
  int64_t units, ranges, nchunks, lpad;
  int nheads, chunk;
};

// eight bf16 (w) += f * acc, rounded back to bf16
__device__ __forceinline__ void fx_apply(uint4& w, float f, const float* acc) {
  uint32_t* u = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(u[i] << 16), hi = __uint_as_float(u[i] & 0xffff0000u);
    const __nv_bfloat162 r = __floats2bfloat162_rn(fmaf(f, acc[2 * i], lo), fmaf(f, acc[2 * i + 1], hi));
    u[i] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

__global__ void __launch_bounds__(kFxThreads, 3) ssd_state_fixup_kernel(FxParams p) {
  __shared__ float s_piece[kFxPieces];  // decay exponents of the pieces walked back over
  griddep_wait();               // h_in, h_final and E come from the fused pass
  griddep_launch_dependents();  // after the wait: the chunk scan reads the forward's inputs early
  const int64_t nc = p.nchunks;
  constexpr int kBlocks = 128 / kFxRows;
  const int64_t k = 1 + blockIdx.x / kBlocks;  // the range that starts the piece
  const int rb = (int)(blockIdx.x % kBlocks);
  auto u = [&](int64_t j) { return j * p.units / p.ranges; };
  const int64_t uk = u(k);
  if (k >= p.ranges || uk % nc == 0) return;  // a piece that starts its chain began from h0
  const int64_t z = uk / nc, zc = z * nc;
  const int b = (int)(uk - zc);  // the piece's chunks [b, e) of the chain (below 2^31)
  const int e = (int)((u(k + 1) < zc + nc ? u(k + 1) : zc + nc) - zc);
  const int pairs = p.nheads / 2;
  const int64_t bi = z / pairs;
  const int m = rb * kFxRows + (int)threadIdx.x / 16;  // state row of the pair, 0 .. 127
  const int h = 2 * (int)(z % pairs) + m / 64, pp = m & 63;
  const int s0 = ((int)threadIdx.x % 16) * 8;
  const int warp = (int)threadIdx.x >> 5, lane = (int)threadIdx.x & 31;
  const int64_t bh = bi * p.nheads + h;
  const float* Glast = p.G + bh * p.lpad + (p.chunk - 1);  // G_last of chunk c at Glast[c * chunk]
  const float* slot = p.carry + m * 128 + s0;             // E[j] at slot + j * 16384
  auto load8 = [&](int64_t j, float* v) {
    const float4* q = reinterpret_cast<const float4*>(slot + j * 16384);
    const float4 a0 = q[0], a1 = q[1];
    v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w;
    v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
  };
  // H(u_k) = E[k-1] + sum over the pieces j < k of this chain that start inside it (u(j) > zc)
  // of 2^(D(u(j), u_k)) E[j-1], unrolled from the recurrence above
  float acc[8];
  load8(k - 1, acc);
  int64_t j_lo = k;
  while (j_lo > 1 && u(j_lo - 1) > zc) --j_lo;  // pieces j_lo .. k-1 started inside the chain
  float lg = 0.f;                               // D(u(j), u_k), accumulated newest first
  for (int64_t jb = k - 1; jb >= j_lo; jb -= kFxPieces) {
    const int nb = (int)(jb - j_lo + 1 < kFxPieces ? jb - j_lo + 1 : kFxPieces);  // pieces jb, jb-1, ..
    __syncthreads();  // s_piece of the previous batch has been read
    for (int i = warp; i < nb; i += kFxThreads / 32) {  // a warp per piece: its decay exponent
      const int64_t j = jb - i;
      float t = 0.f;
      for (int64_t c = u(j) - zc + lane; c < u(j + 1) - zc; c += 32) t += Glast[c * p.chunk];
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      if (lane == 0) s_piece[i] = t;
    }
    __syncthreads();
    for (int i0 = 0; i0 < nb; i0 += kFxFold) {  // kFxFold pieces' end states in flight at a time
      float v[kFxFold][8];
#pragma unroll
      for (int i = 0; i < kFxFold; ++i)
        if (i0 + i < nb) load8(jb - (i0 + i) - 1, v[i]);
#pragma unroll
      for (int i = 0; i < kFxFold; ++i) {
        if (i0 + i < nb) {
          lg += s_piece[i0 + i];
          const float f = exp2f(lg);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = fmaf(f, v[i][q], acc[q]);
        }
      }
    }
  }
  // h_in[c] += 2^(D(b, c)) H over the piece, kFxBatch chunks per step so that their loads overlap
  const int64_t cstride = (int64_t)p.nheads * 8192;
  __nv_bfloat16* q = p.hin + ((bi * nc + b) * p.nheads + h) * 8192 + pp * 128 + s0;  // chunk b
  const float* gq = Glast + (int64_t)b * p.chunk;
  float lgc = 0.f;
  int c = b;
  for (; c + kFxBatch <= e; c += kFxBatch, q += kFxBatch * cstride, gq += kFxBatch * p.chunk) {
    uint4 w[kFxBatch];
    float g[kFxBatch];
#pragma unroll
    for (int i = 0; i < kFxBatch; ++i) {
      w[i] = *reinterpret_cast<const uint4*>(q + i * cstride);
      g[i] = gq[i * p.chunk];
    }
#pragma unroll
    for (int i = 0; i < kFxBatch; ++i) {
      fx_apply(w[i], exp2f(lgc), acc);
      *reinterpret_cast<uint4*>(q + i * cstride) = w[i];
      lgc += g[i];
    }
  }
  for (; c < e; ++c, q += cstride, gq += p.chunk) {
    uint4 w = *reinterpret_cast<const uint4*>(q);
    fx_apply(w, exp2f(lgc), acc);
    *reinterpret_cast<uint4*>(q) = w;
    lgc += *gq;
  }
  if ((int64_t)e == nc && p.h_final) {
    const float f = exp2f(lgc);
    float4* q = reinterpret_cast<float4*>(p.h_final + (bh * 64 + pp) * 128 + s0);
    float4 a0 = q[0], a1 = q[1];
    a0.x = fmaf(f, acc[0], a0.x); a0.y = fmaf(f, acc[1], a0.y); a0.z = fmaf(f, acc[2], a0.z); a0.w = fmaf(f, acc[3], a0.w);
    a1.x = fmaf(f, acc[4], a1.x); a1.y = fmaf(f, acc[5], a1.y); a1.z = fmaf(f, acc[6], a1.z); a1.w = fmaf(f, acc[7], a1.w);
    q[0] = a0;
    q[1] = a1;
  }
}

// CTAs of a launch: one per chain, or one per SM (ranges of at least one chain) when there are
// more chains than SMs.  With split chains, as many equal pieces of every chain as fit the SMs
// (at most one per chunk), so that the pieces of the two head pairs that share a group's B run
// the same chunks at the same time and read B once from DRAM; with more chains than SMs, one
// range per SM.
__host__ __forceinline__ int64_t sf_grid(int64_t chains, int64_t nchunks, int sms, bool split) {
  if (nchunks == 0) return chains;
  if (split) {
    if (chains <= sms) {
      const int64_t per = (int64_t)sms / chains;
      return chains * (per < nchunks ? per : nchunks);
    }
    return sms;
  }
  return chains <= sms ? chains : sms;
}

}  // namespace

int64_t ssd_fused_schedule(int64_t chains, int64_t nchunks, int sms, bool split, int64_t* rows, int64_t cap) {
  if (chains < 0 || nchunks < 0 || sms < 1) return -1;
  const int64_t grid = sf_grid(chains, nchunks, sms, split), units = chains * nchunks;
  int64_t n = 0;
  for (int64_t k = 0; k < grid; ++k) {
    const int64_t u0 = k * units / grid, u1 = (k + 1) * units / grid;
    if (nchunks == 0 || u1 <= u0) continue;
    const SfRange rg = sf_range(u0, u1, nchunks);
    for (int s = 0; s < rg.nseg; ++s, ++n) {
      const SfSeg g = sf_seg(rg, s, nchunks);
      if (rows && n < cap) {
        int64_t* r = rows + 6 * n;
        r[0] = k;
        r[1] = g.chain;
        r[2] = g.c0;
        r[3] = g.c1;
        r[4] = g.from_carry ? 1 : 0;
        r[5] = g.to_carry ? 1 : 0;
      }
    }
  }
  return n;
}

// Per 64-token step the fused pass does the same work as ssd_chunk_state_tc, so against the
// chunk-state + state-passing pair it saves the f32 chunk states' round trip and the second
// launch.  With no more chains than SMs each CTA runs one chain (b8 L2048 nh24: 42 us against
// ~49 us); with more, one CTA per SM runs an equal range of chunks, splitting chains where the
// ranges meet.
// Shapes the fused kernel computes correctly (any number of chains and chunks).
bool ssd_state_fused_possible(const SsdDims& d) {
  return d.dtype == SSM_BF16 && d.headdim == 64 && d.dstate == 128 && (d.nheads / d.ngroups) % 2 == 0 &&
         d.chunk % kSfKH == 0 && d.chunk <= 256;
}

namespace {
int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}
// The rule for split chains: few chains (at most half the SMs) of at least 32 chunks, but at
// most 16 pieces per chain, since the fix-up of a piece composes the end states of every
// earlier piece of its chain (measured, forward: 16 chains of 512 chunks 855 us against 943 us
// for chunk states + look-back state passing, 16 of 128 chunks 243 against 259 us, 20 of 128
// 247 against 272 us, 32 of 32 114 against 120 us; 8 chains of 64 chunks 87 against 77 us, 4
// of 64 79 against 50 us, 2 of 256 138 against 91 us).
bool sf_split_rule(int64_t chains, int64_t nchunks, int sms) {
  return 2 * chains <= sms && 16 * chains >= sms && nchunks >= SSM_SF_SPLIT_MIN_CHUNKS;
}
}  // namespace

// Whether the fused kernel is the faster state path: the plan's choice, else either more
// chains than SMs (ranges split across CTAs: b4 L8192 nh80, 160 chains, 158 us against 207 us
// for chunk states + state passing), one wave of short chains (a long chain is one CTA's
// serial work), or few long chains, split into pieces (see ssd_state_fused_split).
bool ssd_state_fused_supported(const SsdDims& d) {
  if (!ssd_state_fused_possible(d)) return false;
  if (d.plan_fused >= 0) return d.plan_fused != 0;
  const int sms = device_sms();
  if (sms < 1) return false;
  const int64_t chains = d.batch * (int64_t)(d.nheads / 2);
  return chains > sms || d.nchunks <= 16 || sf_split_rule(chains, d.nchunks, sms);
}

// Whether the fused pass splits its chains into independent pieces (one range per SM, every
// piece after a chain's first from a zero state) and ssd_state_fixup then adds the state each
// piece enters with: the plan's choice (fused = 2), else the rule above.
bool ssd_state_fused_split(const SsdDims& d) {
  if (!ssd_state_fused_possible(d) || d.nchunks == 0) return false;
  if (d.plan_fused >= 0) return d.plan_fused == 2;
  const int sms = device_sms();
  return sms > 0 && sf_split_rule(d.batch * (int64_t)(d.nheads / 2), d.nchunks, sms);
}

cudaError_t launch_ssd_state_fused_tc(const void* x, const void* B, const float* h0, float* h_final,
                                      const SsdDims& d, const SsdWorkspace& ws, const LookbackCtl& ctl,
                                      cudaStream_t s) {
  CUtensorMap map_x, map_b;
  const uint64_t xd[3] = {(uint64_t)d.nheads * 64, (uint64_t)d.seqlen, (uint64_t)d.batch};
  const uint64_t xs[2] = {(uint64_t)d.nheads * 64 * 2, (uint64_t)d.seqlen * d.nheads * 64 * 2};
  const uint64_t bd[3] = {(uint64_t)d.ngroups * 128, (uint64_t)d.seqlen, (uint64_t)d.batch};
  const uint64_t bs[2] = {(uint64_t)d.ngroups * 128 * 2, (uint64_t)d.seqlen * d.ngroups * 128 * 2};
  const uint32_t box[3] = {64, (uint32_t)kSfKH, 1};
  cudaError_t e;
  if ((e = encode_tensor_map_3d(&map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, xd, xs, box, CU_TENSOR_MAP_SWIZZLE_128B)) !=
      cudaSuccess)
    return e;
  if ((e = encode_tensor_map_3d(&map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, bd, bs, box, CU_TENSOR_MAP_SWIZZLE_128B)) !=
      cudaSuccess)
    return e;
  // h_in as [batch x chunks x heads x 64 rows][128 s] bf16; boxes of 64 s x one pair's 128 rows
  CUtensorMap map_hin = {};
  const uint64_t hin_rows = (uint64_t)d.batch * d.nchunks * d.nheads * 64;
  if (hin_rows > 0 && (e = encode_tensor_map_2d(&map_hin, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws.hin, 128, hin_rows, 256,
                                                64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  SfParams p;
  p.G = ws.G;
  p.dtT = ws.dtT;
  p.h0 = h0;
  p.hin = static_cast<__nv_bfloat16*>(ws.hin);
  p.h_final = h_final;
  p.carry = ws.Sc;  // the chunk-state buffer is free on this path: one state per split chain
  p.flags = ws.flags;
  p.hdr = ws.hdr;
  p.batch = d.batch;
  p.lpad = d.lpad;
  p.nchunks = d.nchunks;
  p.nheads = d.nheads;
  p.ngroups = d.ngroups;
  p.chunk = d.chunk;
  // B's lines keep evict-last priority after the pass (until read again with another policy),
  // so the hint is given only where all of B takes at most a quarter of L2
  p.b_keep = (uint64_t)d.batch * (uint64_t)d.seqlen * (uint64_t)d.ngroups * 128u * 2u <= (32ull << 20);
  const int64_t chains = d.batch * (int64_t)(d.nheads / 2);
  p.units = chains * d.nchunks;
  const int sms = device_sms();
  if (sms < 1) return cudaErrorInvalidDevice;
  const bool split = ssd_state_fused_split(d);
  p.split = split ? 1 : 0;
  // one chain per CTA, or one CTA per SM with ranges of at least one chain (chains > SMs), so
  // that a range never lies inside one chain; the CTAs claim their ranges in order, so the CTA
  // whose published state a range waits for is already running.  With split chains one range
  // per SM, each publishing into its own slot of the (otherwise unused) chunk-state buffer,
  // which holds a 128 x 128 state per unit.
  const int64_t grid = sf_grid(chains, d.nchunks, sms, split);
  if (split ? grid > p.units : (grid > chains || ws.sp_tiles < chains)) return cudaErrorInvalidValue;
  // the plan's ring split (X slots + B slots); the rule is 4 + 3
  auto go = [&](auto kernel, size_t total) -> cudaError_t {
    const size_t smem = total + 1024;
    cudaError_t e2 = ensure_smem_limit(reinterpret_cast<const void*>(kernel), smem);
    if (e2 != cudaSuccess) return e2;
    return launch_pdl(kernel, dim3((unsigned)grid), dim3(kSfThreads), smem, s, map_x, map_b, map_hin, p, ctl);
  };
  switch (d.plan_ring) {
    case 2: return go(ssd_state_fused_tc_kernel<3, 4>, SfLayout<3, 4>().total);
    case 3: return go(ssd_state_fused_tc_kernel<5, 2>, SfLayout<5, 2>().total);
    default: return go(ssd_state_fused_tc_kernel<4, 3>, SfLayout<4, 3>().total);
  }
}

cudaError_t launch_ssd_state_fixup(float* h_final, const SsdDims& d, const SsdWorkspace& ws, cudaStream_t s) {
  const int64_t chains = d.batch * (int64_t)(d.nheads / 2);
  const int sms = device_sms();
  if (sms < 1) return cudaErrorInvalidDevice;
  FxParams p;
  p.G = ws.G;
  p.hin = static_cast<__nv_bfloat16*>(ws.hin);
  p.h_final = h_final;
  p.carry = ws.Sc;
  p.units = chains * d.nchunks;
  p.ranges = sf_grid(chains, d.nchunks, sms, true);  // as the fused pass split them
  p.nchunks = d.nchunks;
  p.lpad = d.lpad;
  p.nheads = d.nheads;
  p.chunk = d.chunk;
  const int64_t grid = (p.ranges - 1) * (128 / kFxRows);
  if (grid <= 0) return cudaSuccess;  // one range: every chain ran whole
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(ssd_state_fixup_kernel, dim3((unsigned)grid), dim3(kFxThreads), 0, s, p);
}

}  // namespace ssm
