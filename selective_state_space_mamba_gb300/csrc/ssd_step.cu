// ssd_step: the Mamba-2 recurrence applied to ONE new token per sequence, with the state
// carried from the previous call (decode).  "Accelerating Mamba-2 with High-Performance
// Forward Pass Kernels in NVIDIA CUDA Tile", section "Mamba-2 architecture": per head,
//     h' = exp(A dt) h + x (dt B)^T        (state H x S, S contiguous)
//     y  = h' c + D x                       (inclusive reading, as in the chunked forward)
// The post sets this recurrent form against the chunked one: one state update per token,
// no matrix products, so the whole cost is reading and writing the f32 state once
// (8 H S bytes per head and token).  It is a pure HBM stream; tensor cores have nothing
// to contract here.
//
// Work split: the state is a list of rows (b, h, p) of S floats.  A warp "item" is 1024
// consecutive floats (8 rows for S = 128, 16 rows for S = 64, always inside one head since
// H is a multiple of 16).  Lane l reads float4 number l + 32 k (k = 0..7): every load
// instruction of the warp covers 512 contiguous bytes, and all eight are issued before the
// first is used.  Each lane keeps the same four columns s of B and C for all its rows.
// The 8 per-row partial dot products of a lane are reduced across the lanes of their row
// with a halving butterfly (each exchange halves the values a lane still holds), 5 shuffle
// rounds and 9 shuffles in all instead of 8 x 5.
//
// state_out may be state_in (in place): every float4 is read and written by the same lane,
// its load before its store, and the pointers are not declared __restrict__.
#include "ssm_internal.cuh"

namespace ssm {
namespace {

constexpr int kStepThreads = 256;
constexpr int kStepWarps = kStepThreads / 32;
constexpr int kStepLoads = 8;                         // float4 per lane per item
constexpr int kStepItemFloats = 32 * 4 * kStepLoads;  // 1024

__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ void from_f(float v, __nv_bfloat16* p) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void from_f(float v, float* p) { *p = v; }

// four consecutive elements as f32
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xffff0000u));
}

template <typename T, int S>
__global__ void __launch_bounds__(kStepThreads, 4)
    ssd_step_kernel(const T* x, const T* dt, const float* A, const T* B, const T* C, const float* D,
                    const float* state_in, float* state_out, T* y, int64_t items, int nheads, int headdim,
                    int heads_per_group, int ngroups) {
  constexpr int kLanesPerRow = S / 4;            // 32 (S = 128) or 16 (S = 64)
  constexpr int kRowsPerLoad = 32 / kLanesPerRow;  // rows one warp load instruction covers
  griddep_launch_dependents();
  griddep_wait();  // the state may come from the previous kernel on the stream
  const int lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * kStepWarps + (threadIdx.x >> 5);
  if (item >= items) return;
  const int64_t row0 = item * (kStepItemFloats / S);  // first state row (b, h, p) of the item
  const int64_t bh = row0 / headdim;                  // every row of the item is in head bh
  const int p0 = (int)(row0 - bh * headdim);
  const int h = (int)(bh % nheads);
  const int64_t bi = bh / nheads;
  const int64_t grow = (bi * ngroups + h / heads_per_group) * S;
  const int col = 4 * (lane % kLanesPerRow);  // this lane's four state columns
  const int rsub = lane / kLanesPerRow;       // row offset of the lane inside one load

  const int64_t base = row0 * S + 4 * lane;  // float offset of load k: base + 128 k
  float4 hv[kStepLoads];
#pragma unroll
  for (int k = 0; k < kStepLoads; ++k)
    hv[k] = state_in ? ld4(state_in + base + 128 * k) : make_float4(0.f, 0.f, 0.f, 0.f);
  const float dtv = to_f(dt[bh]);
  const float decay = expf(A[h] * dtv);
  const float4 bv = ld4(B + grow + col);
  const float4 cv = ld4(C + grow + col);
  const T* xrow = x + bh * headdim + p0;
  float xdt[kStepLoads];
#pragma unroll
  for (int k = 0; k < kStepLoads; ++k) xdt[k] = to_f(xrow[k * kRowsPerLoad + rsub]) * dtv;

  float part[kStepLoads];
#pragma unroll
  for (int k = 0; k < kStepLoads; ++k) {
    float4 n;
    n.x = fmaf(decay, hv[k].x, xdt[k] * bv.x);
    n.y = fmaf(decay, hv[k].y, xdt[k] * bv.y);
    n.z = fmaf(decay, hv[k].z, xdt[k] * bv.z);
    n.w = fmaf(decay, hv[k].w, xdt[k] * bv.w);
    *reinterpret_cast<float4*>(state_out + base + 128 * k) = n;
    part[k] = fmaf(n.w, cv.w, fmaf(n.z, cv.z, fmaf(n.y, cv.y, n.x * cv.x)));
  }

  // Halving butterfly over the lanes of a row: in round `bit`, the lane with that bit set
  // keeps the upper half of its values and sends the lower half, its partner the reverse.
  // The lanes of one row are the low log2(kLanesPerRow) bits, so the rounds run over those.
  int kf = 0;  // which of the 8 loads the single value left at the end belongs to
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int bit = (kLanesPerRow / 2) >> r;
    const int half = kStepLoads >> (r + 1);
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = up ? part[j] : part[j + half];
      const float keep = up ? part[j + half] : part[j];
      part[j] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
    if (up) kf += half;
  }
#pragma unroll
  for (int bit = (kLanesPerRow / 16); bit >= 1; bit >>= 1) part[0] += __shfl_xor_sync(0xffffffffu, part[0], bit);

  if ((lane & (kLanesPerRow / 8 - 1)) == 0) {  // one lane per row writes y
    const int p = kf * kRowsPerLoad + rsub;
    from_f(part[0] + D[h] * to_f(xrow[p]), y + bh * headdim + p0 + p);
  }
}

template <typename T, int S>
cudaError_t launch_step(const void* x, const void* dt, const float* A, const void* B, const void* C, const float* D,
                        const float* state_in, float* state_out, void* y, int64_t batch, int nheads, int headdim,
                        int ngroups, cudaStream_t s) {
  const int64_t items = batch * nheads * (int64_t)headdim * S / kStepItemFloats;
  const int64_t blocks = (items + kStepWarps - 1) / kStepWarps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(ssd_step_kernel<T, S>, dim3((unsigned)blocks), dim3(kStepThreads), 0, s,
                    static_cast<const T*>(x), static_cast<const T*>(dt), A, static_cast<const T*>(B),
                    static_cast<const T*>(C), D, state_in, state_out, static_cast<T*>(y), items, nheads, headdim,
                    nheads / ngroups, ngroups);
}

}  // namespace

cudaError_t launch_ssd_step(const void* x, const void* dt, const float* A, const void* B, const void* C,
                            const float* D, const float* state_in, float* state_out, void* y, int64_t batch,
                            int nheads, int headdim, int dstate, int ngroups, ssm_dtype dtype, cudaStream_t s) {
  if (dtype == SSM_BF16)
    return dstate == 128 ? launch_step<__nv_bfloat16, 128>(x, dt, A, B, C, D, state_in, state_out, y, batch, nheads,
                                                           headdim, ngroups, s)
                         : launch_step<__nv_bfloat16, 64>(x, dt, A, B, C, D, state_in, state_out, y, batch, nheads,
                                                          headdim, ngroups, s);
  return dstate == 128
             ? launch_step<float, 128>(x, dt, A, B, C, D, state_in, state_out, y, batch, nheads, headdim, ngroups, s)
             : launch_step<float, 64>(x, dt, A, B, C, D, state_in, state_out, y, batch, nheads, headdim, ngroups, s);
}

}  // namespace ssm
