// ssd_state_passing: the inter-chunk scan of the Mamba-2 SSD forward.
//
// With S_c the state increment of chunk c (computed in parallel by ssd_chunk_state) and
// d_c = exp(sum of a over chunk c) = 2^(G_last of chunk c), the chunk-initial states are
//     h_in[0] = h0,   h_in[c+1] = d_c h_in[c] + S_c,   h_final = h_in[nchunks]
// ("Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA CUDA Tile",
// "Kernel 2: fwd_pass_state": the jump h_{t+T} = exp(G_last) h_t + X^T(exp(G_last - G) B),
// whose chunk loop runs sequentially inside one program there).
//
// Here the loop over chunks is a scan under the same affine pair combine as the scalar scan
// ("Selective-scan CUDA kernels", "The problem"), run as a decoupled look-back: each tile is
// kSpElems state entries of one (batch, head) across up to kSpChunks chunks, whose increments
// it stages in shared memory.  A tile publishes its aggregate state vector (flag A), looks
// back over predecessor tiles of the same chain (a warp inspects 32 flags at once, atomic
// claim order guarantees progress), publishes its inclusive state (flag P), then writes h_in
// for each of its chunks.  The decay of an aggregate is not published: every tile recomputes
// it from G.
//
// When there are enough state entries to fill the GPU without splitting the chunk axis (the
// usual case: batch x heads x H x S in the millions), the recurrence runs as written instead:
// ssd_state_passing_seq_kernel gives each thread four entries of one (batch, head) and walks
// all chunks in order, with the chunk increments of the next kSeqAhead chunks already in
// flight (copied into shared memory).  No flags, fences or workspace beyond S_c and h_in.
#include "ssm_internal.cuh"

namespace ssm {
namespace {

__device__ __forceinline__ float4 f4_fma(float s, float4 x, float4 y) {
  return make_float4(fmaf(s, x.x, y.x), fmaf(s, x.y, y.y), fmaf(s, x.z, y.z), fmaf(s, x.w, y.w));
}

template <typename T> __device__ __forceinline__ void store4(T* p, float4 v);
template <> __device__ __forceinline__ void store4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <> __device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

// The tile's chunk increments (kSpChunks rows of kSpElems floats, 64 KB) are staged in shared
// memory by bulk copies rather than held in registers, so three CTAs fit an SM and their
// copies, look-backs and h_in stores overlap.
constexpr int kSpMinBlocks = 3;
constexpr size_t kSpSmem = sizeof(float) * kSpChunks * kSpElems;

template <typename HinT>
__global__ void __launch_bounds__(kSpThreads, kSpMinBlocks)
    ssd_state_passing_kernel(const float* __restrict__ h0, float* __restrict__ h_final, SsdDims d, SsdWorkspace ws,
                             LookbackCtl ctl_call) {
  extern __shared__ float4 sp_sc[];  // [kSpChunks][kSpThreads]: chunk k, this thread's 4 entries
  __shared__ uint64_t s_bar;
  __shared__ uint32_t s_tile;
  __shared__ int s_last, s_found;
  griddep_wait();  // S_c, G and the claim counter come from the previous kernels
  // after the wait: the chunk scan that follows loads the forward's inputs before its own
  // wait, which is safe once this grid's start implies that every earlier kernel has ended
  griddep_launch_dependents();
  const LookbackCtl ctl = device_epoch(ctl_call, ws.hdr);

  if (threadIdx.x == 0) {
    s_tile = claim_tile(ws.hdr);
    mbar_init(&s_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t tile = s_tile;
  if (tile >= ws.sp_tiles) {  // claim counter not reset: refuse rather than index past the workspace
    if (threadIdx.x == 0) {
      record_error(ws.hdr, ctl.epoch, SSM_ERR_WORKSPACE);
      retire_tile(ws.hdr, (uint32_t)ws.sp_tiles);
    }
    return;
  }
  const int64_t chain = tile % ws.sp_chains;
  const int64_t ctile = tile / ws.sp_chains;
  const int HS = d.headdim * d.dstate;
  const int nslices = HS / kSpElems;
  const int64_t bh = chain / nslices;  // bi * nheads + h
  const int slice = (int)(chain % nslices);
  const int64_t bi = bh / d.nheads;
  const int h = (int)(bh % d.nheads);
  const int64_t nc = d.nchunks;
  const int64_t c0 = ctile * kSpChunks;
  const int nk = (int)(nc - c0 < kSpChunks ? nc - c0 : kSpChunks);
  const int e = slice * kSpElems + threadIdx.x * 4;
  const float* Grow = ws.G + bh * d.lpad + (d.chunk - 1);  // G_last of chunk c at Grow[c * chunk]

  // ---- this tile's chunk increments (shared memory) and decays (registers) ----
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&s_bar, (uint32_t)(nk * kSpElems * sizeof(float)));
    for (int k = 0; k < nk; ++k)
      bulk_g2s(sp_sc + k * kSpThreads, ws.Sc + ((bi * nc + c0 + k) * d.nheads + h) * HS + slice * kSpElems,
               (uint32_t)(kSpElems * sizeof(float)), &s_bar);
  }
  float lg[kSpChunks];
#pragma unroll
  for (int k = 0; k < kSpChunks; ++k)
    if (k < nk) lg[k] = Grow[(c0 + k) * d.chunk];
  if (!mbar_wait(&s_bar, 0, ctl.spin_limit_ns)) {
    record_error(ws.hdr, ctl.epoch, SSM_ERR_TIMEOUT);
    mbar_wait(&s_bar, 0, ctl.spin_limit_ns);  // the copies land in this CTA's shared memory: wait for them
  }
  const float4* sc = sp_sc + threadIdx.x;  // chunk k at sc[k * kSpThreads]
  float4 agg = make_float4(0.f, 0.f, 0.f, 0.f);
  float lg_tile = 0.f;
#pragma unroll
  for (int k = 0; k < kSpChunks; ++k) {
    if (k < nk) {
      agg = f4_fma(exp2f(lg[k]), agg, sc[k * kSpThreads]);
      lg_tile += lg[k];
    }
  }

  const bool stalled = (int64_t)tile == ctl.stall_tile;
  float* my_agg = ws.agg + tile * kSpElems + threadIdx.x * 4;
  float* my_inc = ws.inc + tile * kSpElems + threadIdx.x * 4;
  float4 X;  // state entering the tile's first chunk
  if (ctile == 0) {
    X = h0 ? *reinterpret_cast<const float4*>(h0 + bh * HS + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (!stalled) *reinterpret_cast<float4*>(my_inc) = f4_fma(exp2f(lg_tile), X, agg);
    // The CTA barrier orders every thread's store before thread 0's release store of the flag,
    // and a release is cumulative: a reader that acquires the flag sees all of them.  (No
    // fence per thread: each would wait for its own store to reach L2.)
    __syncthreads();
    if (threadIdx.x == 0 && !stalled) st_release_u64(&ws.flags[tile], make_flag(ctl.epoch, kFlagPrefix));
  } else {
    if (!stalled) *reinterpret_cast<float4*>(my_agg) = agg;
    __syncthreads();  // as above: barrier, then one release store
    if (threadIdx.x == 0 && !stalled) st_release_u64(&ws.flags[tile], make_flag(ctl.epoch, kFlagAggregate));

    // ---- look-back: compose predecessors newest to oldest until a published prefix ----
    float4 acc_b = make_float4(0.f, 0.f, 0.f, 0.f);  // map h -> 2^acc_lg h + acc_b
    float acc_lg = 0.f;
    int64_t newest = ctile - 1;
    while (true) {
      if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int64_t ct = newest - lane;
        uint32_t kind = kFlagPrefix;
        if (ct >= 0) {
          kind = wait_flag(&ws.flags[ct * ws.sp_chains + chain], ws.hdr, ctl);
          if (kind == 0) kind = 3;  // gave up: use as a (poisoned) prefix
        }
        const unsigned pmask = __ballot_sync(0xffffffffu, kind != kFlagAggregate);
        const int last = pmask ? (__ffs(pmask) - 1) : 31;  // lanes 0..last are composed
        const uint32_t kind_last = __shfl_sync(0xffffffffu, kind, last);
        if (lane == 0) {
          s_last = last;
          s_found = pmask ? (int)kind_last : 0;
        }
      }
      __syncthreads();
      // The lanes of warp 0 acquired the flags; the CTA barrier above carries that ordering to
      // every thread of the CTA, whose loads below then see the published vectors.
      const int last = s_last;
      const int found = s_found;  // 0: all 32 were aggregates, 2: prefix, 3: gave up
      for (int l = 0; l <= last; ++l) {
        const int64_t ct = newest - l;
        const int64_t t = ct * ws.sp_chains + chain;
        if (l == last && found != 0) {
          float4 v;
          if (found == kFlagPrefix) {
            v = ld_relaxed_f4(reinterpret_cast<const float4*>(ws.inc + t * kSpElems + threadIdx.x * 4));
          } else {
            const float nan = __int_as_float(0x7fc00000);
            v = make_float4(nan, nan, nan, nan);
          }
          acc_b = f4_fma(exp2f(acc_lg), v, acc_b);
        } else {
          const float4 v = ld_relaxed_f4(reinterpret_cast<const float4*>(ws.agg + t * kSpElems + threadIdx.x * 4));
          acc_b = f4_fma(exp2f(acc_lg), v, acc_b);
          float lq = 0.f;
          const int64_t cb = ct * kSpChunks;
          const int nq = (int)(nc - cb < kSpChunks ? nc - cb : kSpChunks);
          for (int k = 0; k < nq; ++k) lq += Grow[(cb + k) * d.chunk];
          acc_lg += lq;
        }
      }
      if (found != 0) break;
      newest -= 32;
      __syncthreads();  // warp 0 rewrites s_last / s_found
    }
    X = acc_b;
    if (!stalled) *reinterpret_cast<float4*>(my_inc) = f4_fma(exp2f(lg_tile), X, agg);
    __syncthreads();  // as above: barrier, then one release store
    if (threadIdx.x == 0 && !stalled) st_release_u64(&ws.flags[tile], make_flag(ctl.epoch, kFlagPrefix));
  }

  // ---- chunk-initial states of this tile, then the final state ----
  HinT* hin = static_cast<HinT*>(ws.hin);
#pragma unroll
  for (int k = 0; k < kSpChunks; ++k) {
    if (k < nk) {
      const int64_t c = c0 + k;
      store4<HinT>(hin + ((bi * nc + c) * d.nheads + h) * HS + e, X);
      X = f4_fma(exp2f(lg[k]), X, sc[k * kSpThreads]);
    }
  }
  if (h_final && c0 + nk == nc) *reinterpret_cast<float4*>(h_final + bh * HS + e) = X;
  if (threadIdx.x == 0) retire_tile(ws.hdr, (uint32_t)ws.sp_tiles);
}

constexpr int kSeqThreads = 256;
constexpr int kSeqAhead = 8;             // chunk increments in flight per thread
// Fewer four-entry groups than this: the look-back kernel.  A thread of the sequential kernel
// takes about 0.5 us per chunk (its chain of dependent steps), so the kernel needs about
// 6.8 TB/s x 0.5 us / 24 B (S_c read + h_in written per entry and chunk) ~ 140 K groups to
// run at HBM speed; with fewer it is latency bound (b1 L131072 nh32: 65,536 groups, 268 us
// against 178 us for the look-back kernel).
constexpr int64_t kSeqMinGroups = 131072;

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Each thread streams its own four entries of S_c for chunk c + kSeqAhead into its own
// 16-byte slot of a shared-memory ring while it combines chunk c, so the loads in flight cost
// no registers; a thread only ever reads slots it filled itself (cp.async.wait_group).
template <typename HinT>
__global__ void __launch_bounds__(kSeqThreads) ssd_state_passing_seq_kernel(const float* __restrict__ h0,
                                                                            float* __restrict__ h_final, SsdDims d,
                                                                            SsdWorkspace ws) {
  __shared__ float4 ring[kSeqAhead][kSeqThreads];
  griddep_wait();  // S_c and G come from the previous kernels
  griddep_launch_dependents();  // after the wait, as in the look-back kernel above
  const int HS = d.headdim * d.dstate;
  const int64_t q4 = HS / 4;
  const int64_t gidx = (int64_t)blockIdx.x * kSeqThreads + threadIdx.x;
  if (gidx >= d.batch * d.nheads * q4) return;
  const int64_t bh = gidx / q4;  // bi * nheads + h
  const int e = (int)(gidx % q4) * 4;
  const int64_t bi = bh / d.nheads;
  const int h = (int)(bh % d.nheads);
  const int64_t nc = d.nchunks;
  const float* Grow = ws.G + bh * d.lpad + (d.chunk - 1);  // G_last of chunk c at Grow[c * chunk]
  const int64_t step = (int64_t)d.nheads * HS;              // chunk c -> c + 1 in S_c and h_in
  // S_c and h_in are [b, nc, nh, H, S]: this thread's four entries over every chunk; G is
  // [b, nh, lpad]: this head's last G of every chunk
  if (!SSM_CHECK(ws.hdr, (bi * nc * d.nheads + h) * (int64_t)HS + e + (nc > 0 ? nc - 1 : 0) * (int64_t)d.nheads * HS + 4 <=
                             d.batch * nc * d.nheads * (int64_t)HS &&
                             bh * d.lpad + nc * d.chunk <= d.batch * d.nheads * d.lpad))
    return;
  const float* src = ws.Sc + (bi * nc * d.nheads + h) * (int64_t)HS + e;
  HinT* hin = static_cast<HinT*>(ws.hin) + (bi * nc * d.nheads + h) * (int64_t)HS + e;
  float4* slot = &ring[0][threadIdx.x];

  float lg[kSeqAhead];
#pragma unroll
  for (int u = 0; u < kSeqAhead; ++u) {
    if (u < nc) {
      cp_async16(slot + u * kSeqThreads, src + u * step);
      lg[u] = Grow[u * d.chunk];
    }
    cp_async_commit();  // one group per chunk, empty past the end
  }
  const float* next = src + kSeqAhead * step;
  float4 X = h0 ? *reinterpret_cast<const float4*>(h0 + bh * HS + e) : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t c0 = 0; c0 < nc; c0 += kSeqAhead) {
#pragma unroll
    for (int u = 0; u < kSeqAhead; ++u) {
      const int64_t c = c0 + u;
      if (c < nc) {
        cp_async_wait<kSeqAhead - 1>();  // chunk c's group (the oldest) has landed
        const float4 v = slot[u * kSeqThreads];
        store4<HinT>(hin, X);  // state entering chunk c
        hin += step;
        X = f4_fma(exp2f(lg[u]), X, v);
        if (c + kSeqAhead < nc) {
          cp_async16(slot + u * kSeqThreads, next);
          lg[u] = Grow[(c + kSeqAhead) * d.chunk];
        }
        next += step;
        cp_async_commit();
      }
    }
  }
  cp_async_wait<0>();
  if (h_final) *reinterpret_cast<float4*>(h_final + bh * HS + e) = X;
}

}  // namespace

bool ssd_state_passing_sequential(const SsdDims& d) {
  if (d.plan_seq >= 0) return d.plan_seq != 0;
  return d.batch * d.nheads * (int64_t)(d.headdim * d.dstate / 4) >= kSeqMinGroups;
}

cudaError_t launch_ssd_state_passing(const float* h0, float* h_final, const SsdDims& d, const SsdWorkspace& ws,
                                     const LookbackCtl& ctl, cudaStream_t s) {
  if (ssd_state_passing_sequential(d)) {
    const int64_t groups = d.batch * d.nheads * (int64_t)(d.headdim * d.dstate / 4);
    const unsigned grid = (unsigned)((groups + kSeqThreads - 1) / kSeqThreads);
    if (d.dtype == SSM_BF16)
      return launch_pdl(ssd_state_passing_seq_kernel<__nv_bfloat16>, dim3(grid), dim3(kSeqThreads), 0, s, h0, h_final,
                        d, ws);
    return launch_pdl(ssd_state_passing_seq_kernel<float>, dim3(grid), dim3(kSeqThreads), 0, s, h0, h_final, d, ws);
  }
  cudaError_t e;
  if (d.dtype == SSM_BF16) {
    if ((e = ensure_smem_limit(reinterpret_cast<const void*>(ssd_state_passing_kernel<__nv_bfloat16>), kSpSmem)) !=
        cudaSuccess)
      return e;
    return launch_pdl(ssd_state_passing_kernel<__nv_bfloat16>, dim3((unsigned)ws.sp_tiles), dim3(kSpThreads), kSpSmem,
                      s, h0, h_final, d, ws, ctl);
  }
  if ((e = ensure_smem_limit(reinterpret_cast<const void*>(ssd_state_passing_kernel<float>), kSpSmem)) != cudaSuccess)
    return e;
  return launch_pdl(ssd_state_passing_kernel<float>, dim3((unsigned)ws.sp_tiles), dim3(kSpThreads), kSpSmem, s, h0,
                    h_final, d, ws, ctl);
}

}  // namespace ssm
