// ssd_chunk_cumsum: per-chunk inclusive cumulative sums of a_t = A[h] dt[b,t,h], scaled by
// log2(e) so that every later decay is an exp2 ("Accelerating Mamba-2 with High-Performance
// Forward Pass Kernels in NVIDIA CUDA Tile", "Kernel 1: Computing cumulative sums").  The
// decay matrix of a chunk is then L[i,j] = exp(sum_{k=j+1..i} a_k) = 2^(G_i - G_j), j <= i.
//
// Output layout is [batch, head, token] (the post's "GMEM layout" optimisation): the later
// kernels read one head's G and dt as contiguous runs.  dt is written out transposed as f32
// at the same time, with 0 in the padding of the last chunk (decay 1, no input: exact).
//
// One CTA per (chunk, block of 8 heads, batch): the dt tile [chunk, 8 heads] is staged
// through shared memory so both the read (heads contiguous) and the writes (tokens
// contiguous) are coalesced: each warp scans whole head rows in registers and writes each
// row of dt^T and G straight from them.  The tile is stored head-major with one padding word after every 8 tokens
// and a row stride of 4 (mod 32) words, so that both the scan's reads (each lane reads a run
// of consecutive tokens of one head) and the initial writes (8 heads x 4 tokens per warp) see
// at most 2-way bank conflicts.
#include "ssm_internal.cuh"

namespace ssm {
namespace {

constexpr int kCsHeads = 8;
constexpr int kCsThreads = 256;
constexpr int kCsMaxChunk = 256;
constexpr int kCsWarps = kCsThreads / 32;
constexpr int kCsHeadsPerWarp = kCsHeads / kCsWarps;
constexpr int kCsLoads = kCsMaxChunk * kCsHeads / kCsThreads;

// Raw bits of one dt value.  The loads are volatile asm so that all of a thread's loads are
// issued, in order, before the first conversion waits on one of them.  (Not the read-only
// path: under programmatic dependent launch the previous kernel may have just written dt.)
__device__ __forceinline__ uint32_t ld_bits(const __nv_bfloat16* p) {
  unsigned short v;
  asm volatile("ld.global.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return (uint32_t)v << 16;  // bf16 bits in the top half are the f32 bits
}
__device__ __forceinline__ uint32_t ld_bits(const float* p) {
  uint32_t v;
  asm volatile("ld.global.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// shared-memory word of (token t, local head h); row stride T + T / 8 + 4
__device__ __forceinline__ int sidx(int t, int h, int row) { return h * row + t + (t >> 3); }
__host__ __device__ __forceinline__ int s_row(int T) { return T + T / 8 + 4; }

template <typename DtT>
__global__ void __launch_bounds__(kCsThreads) ssd_chunk_cumsum_kernel(const DtT* __restrict__ dt,
                                                                       const float* __restrict__ A, SsdDims d,
                                                                       float* __restrict__ G, float* __restrict__ dtT,
                                                                       WsHeader* hdr) {
  extern __shared__ float s_dt[];  // [kCsHeads][chunk + chunk / 8 + 4], see sidx
  griddep_launch_dependents();
  griddep_wait();  // dt may come from, and G / dtT may still be read by, the previous kernel
  const int c = blockIdx.x, hblk = blockIdx.y;
  const int64_t bi = blockIdx.z;
  const int T = d.chunk, nh = d.nheads;
  const int srow = s_row(T);
  const int h0 = hblk * kCsHeads;
  const int nhb = min(kCsHeads, nh - h0);
  const int64_t t0 = (int64_t)c * T;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  if (c == 0 && hblk == 0 && bi == 0 && threadIdx.x == 0) {
    // the state-passing kernel runs after this one on the same stream: start its claims at 0
    hdr->counter = 0u;
    hdr->done = 0u;
  }

  // element k of this thread: head threadIdx % kCsHeads, token threadIdx / kCsHeads +
  // (threads / kCsHeads) k: a warp reads whole tokens' head blocks
  constexpr int kTokStride = kCsThreads / kCsHeads;
  const int lh = threadIdx.x % kCsHeads, lt = threadIdx.x / kCsHeads;
  const int tmax = d.seqlen - t0 < T ? (int)(d.seqlen - t0) : T;  // real tokens in this chunk
  const bool head_ok = lh < nhb;
  const int64_t src0 = (bi * d.seqlen + t0 + lt) * nh + h0 + (head_ok ? lh : 0);
  const DtT* src = dt + src0;
  uint32_t raw[kCsLoads];
#pragma unroll
  for (int k = 0; k < kCsLoads; ++k) {
    const int t = lt + kTokStride * k;
    raw[k] = 0u;
    if (head_ok && t < tmax &&
        SSM_CHECK(hdr, src0 + (int64_t)kTokStride * k * nh < d.batch * d.seqlen * nh))  // dt [b, L, nh]
      raw[k] = ld_bits(src + (int64_t)kTokStride * k * nh);
  }
  float Ah[kCsHeadsPerWarp];
#pragma unroll
  for (int q = 0; q < kCsHeadsPerWarp; ++q) {
    const int hh = warp + q * kCsWarps;
    Ah[q] = hh < nhb && SSM_CHECK(hdr, h0 + hh < nh) ? A[h0 + hh] : 0.f;
  }
#pragma unroll
  for (int k = 0; k < kCsLoads; ++k) {
    const int t = lt + kTokStride * k;
    if (t < T && SSM_CHECK(hdr, sidx(t, lh, srow) < kCsHeads * srow)) s_dt[sidx(t, lh, srow)] = __uint_as_float(raw[k]);
  }
  __syncthreads();

  // Each warp scans whole head rows: lane l holds tokens l * per_lane .. + per_lane - 1, so
  // after the scan it writes its run of the dt^T row and of the G row directly (8 to 32
  // contiguous bytes per lane, one contiguous row per warp).
  const int per_lane = T / 32;  // chunk is a multiple of 64 and at most 256
#pragma unroll
  for (int q = 0; q < kCsHeadsPerWarp; ++q) {
    const int hh = warp + q * kCsWarps;
    float dv[8], gv[8];
    float run = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      dv[k] = 0.f;
      if (k < per_lane) {
        dv[k] = s_dt[sidx(lane * per_lane + k, hh, srow)];
        run += Ah[q] * dv[k];
        gv[k] = run;
      }
    }
    // exclusive prefix of the lane totals
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    const float excl = incl - run;
#pragma unroll
    for (int k = 0; k < 8; ++k) gv[k] = (excl + gv[k]) * kLog2e;
    // G and dt^T are [b, nh, lpad]; debug builds check each lane's run against that size (less
    // the test hook's shortfall)
    if (hh < nhb && SSM_CHECK(hdr, (bi * nh + h0 + hh) * d.lpad + t0 + (lane + 1) * per_lane <=
                                       d.batch * nh * d.lpad - d.debug_shrink)) {
      const int64_t off = (bi * nh + h0 + hh) * d.lpad + t0 + lane * per_lane;
      if (per_lane == 2) {
        *reinterpret_cast<float2*>(dtT + off) = make_float2(dv[0], dv[1]);
        *reinterpret_cast<float2*>(G + off) = make_float2(gv[0], gv[1]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; k += 4) {
          if (k < per_lane) {
            *reinterpret_cast<float4*>(dtT + off + k) = make_float4(dv[k], dv[k + 1], dv[k + 2], dv[k + 3]);
            *reinterpret_cast<float4*>(G + off + k) = make_float4(gv[k], gv[k + 1], gv[k + 2], gv[k + 3]);
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_ssd_chunk_cumsum(const void* dt, const float* A, const SsdDims& d, const SsdWorkspace& ws,
                                    cudaStream_t s) {
  dim3 grid((unsigned)d.nchunks, (unsigned)((d.nheads + kCsHeads - 1) / kCsHeads), (unsigned)d.batch);
  const size_t smem = sizeof(float) * kCsHeads * s_row(d.chunk);
  if (d.dtype == SSM_BF16)
    return launch_pdl(ssd_chunk_cumsum_kernel<__nv_bfloat16>, grid, dim3(kCsThreads), smem, s,
                      static_cast<const __nv_bfloat16*>(dt), A, d, ws.G, ws.dtT, ws.hdr);
  return launch_pdl(ssd_chunk_cumsum_kernel<float>, grid, dim3(kCsThreads), smem, s, static_cast<const float*>(dt),
                    A, d, ws.G, ws.dtT, ws.hdr);
}

}  // namespace ssm
