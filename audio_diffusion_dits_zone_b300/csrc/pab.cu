// The difference measure of attention broadcast across diffusion steps.
//
// "Real-time video generation with pyramid attention broadcast" (method): attention
// outputs of consecutive diffusion steps differ little through the middle of the
// schedule (a U-shaped difference curve), so a step there may reuse (broadcast) an
// earlier step's output; the mean squared error between consecutive steps' attention
// outputs is what chooses how far each attention's outputs are broadcast.
//
//   mse[h] = (1 / (N d)) sum_{n, c} (a[n][h][c] - b[n][h][c])^2
//
// attn_mse_partial  grid (chunks, heads): a CTA sums the squared differences of its
//                   head over a contiguous range of token rows (16-byte vector loads,
//                   a head row read by d / 8 consecutive threads: coalesced), reduces
//                   in a fixed order and writes one fp32 partial.  HBM-bound: reads
//                   both tensors once.
// attn_mse_final    sums each head's partials in chunk order in fp64 (deterministic).
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

constexpr int kMseThreads = 256;

template <typename T, int EV>
struct Vec16;
template <>
struct Vec16<__nv_bfloat16, 8> {
  __device__ static float sqdiff(const uint4& x, const uint4& y) {
    const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(&x);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&y);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 u = __bfloat1622float2(a[k]), v = __bfloat1622float2(b[k]);
      const float d0 = u.x - v.x, d1 = u.y - v.y;
      s = fmaf(d0, d0, fmaf(d1, d1, s));
    }
    return s;
  }
};
template <>
struct Vec16<float, 4> {
  __device__ static float sqdiff(const uint4& x, const uint4& y) {
    const float* a = reinterpret_cast<const float*>(&x);
    const float* b = reinterpret_cast<const float*>(&y);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float d0 = a[k] - b[k];
      s = fmaf(d0, d0, s);
    }
    return s;
  }
};

template <typename T, int EV>
__global__ void __launch_bounds__(kMseThreads) attn_mse_partial_kernel(const T* __restrict__ a, const T* __restrict__ b,
                                                                      int64_t ld, int N, int d, int chunk_rows,
                                                                      float* __restrict__ part) {
  __shared__ float red[kMseThreads / 32];
  const int h = blockIdx.y, chunk = blockIdx.x;
  const int vpr = d / EV;               // 16-byte vectors per head row
  const int rpi = kMseThreads / vpr;    // rows per iteration
  const int tv = threadIdx.x % vpr, tr = threadIdx.x / vpr;
  const int r0 = chunk * chunk_rows, r1 = min(N, r0 + chunk_rows);
  float acc = 0.f;
  if (tr < rpi) {
    const int64_t col = (int64_t)h * d + (int64_t)tv * EV;
#pragma unroll 4
    for (int r = r0 + tr; r < r1; r += rpi) {
      const int64_t off = (int64_t)r * ld + col;
      const uint4 x = __ldcs(reinterpret_cast<const uint4*>(a + off));
      const uint4 y = __ldcs(reinterpret_cast<const uint4*>(b + off));
      acc += Vec16<T, EV>::sqdiff(x, y);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kMseThreads / 32; ++w) s += red[w];
    part[(size_t)h * gridDim.x + chunk] = s;
  }
}

// Scalar fallback for layouts without 16-byte vectors.
template <typename T>
__global__ void __launch_bounds__(kMseThreads) attn_mse_scalar_kernel(const T* __restrict__ a, const T* __restrict__ b,
                                                                     int64_t ld, int N, int d, int chunk_rows,
                                                                     float* __restrict__ part) {
  __shared__ float red[kMseThreads / 32];
  const int h = blockIdx.y, chunk = blockIdx.x;
  const int r0 = chunk * chunk_rows, r1 = min(N, r0 + chunk_rows);
  float acc = 0.f;
  for (int64_t e = threadIdx.x; e < (int64_t)(r1 - r0) * d; e += kMseThreads) {
    const int64_t r = r0 + e / d, c = e % d;
    const int64_t off = r * ld + (int64_t)h * d + c;
    const float x = to_f32<T>(a[off]) - to_f32<T>(b[off]);
    acc = fmaf(x, x, acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < kMseThreads / 32; ++w) s += red[w];
    part[(size_t)h * gridDim.x + chunk] = s;
  }
}

__global__ void attn_mse_final_kernel(const float* __restrict__ part, int chunks, int Hh, double inv,
                                      float* __restrict__ mse) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= Hh) return;
  double s = 0.0;
  for (int c = 0; c < chunks; ++c) s += (double)part[(size_t)h * chunks + c];
  mse[h] = (float)(s * inv);
}

}  // namespace

int attn_mse_chunks(int N, int Hh) {
  const int want = (148 * 8 + Hh - 1) / Hh;  // about eight CTAs per SM in all
  return std::max(1, std::min(want, N));
}

cudaError_t attn_mse_launch(const void* a, const void* b, int dtype, int64_t ld, int N, int Hh, int d, float* mse,
                            float* part, cudaStream_t st) {
  const int chunks = attn_mse_chunks(N, Hh);
  const int chunk_rows = (N + chunks - 1) / chunks;
  const dim3 grid(chunks, Hh);
  const bool al = ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15) == 0;
  {
    HookScope hs("attn_mse", st);
    if (dtype == PRISM_BF16) {
      if (al && d % 8 == 0 && ld % 8 == 0 && d / 8 <= kMseThreads)
        attn_mse_partial_kernel<__nv_bfloat16, 8><<<grid, kMseThreads, 0, st>>>(
            static_cast<const __nv_bfloat16*>(a), static_cast<const __nv_bfloat16*>(b), ld, N, d, chunk_rows, part);
      else
        attn_mse_scalar_kernel<__nv_bfloat16><<<grid, kMseThreads, 0, st>>>(
            static_cast<const __nv_bfloat16*>(a), static_cast<const __nv_bfloat16*>(b), ld, N, d, chunk_rows, part);
    } else {
      if (al && d % 4 == 0 && ld % 4 == 0 && d / 4 <= kMseThreads)
        attn_mse_partial_kernel<float, 4><<<grid, kMseThreads, 0, st>>>(
            static_cast<const float*>(a), static_cast<const float*>(b), ld, N, d, chunk_rows, part);
      else
        attn_mse_scalar_kernel<float><<<grid, kMseThreads, 0, st>>>(static_cast<const float*>(a),
                                                                    static_cast<const float*>(b), ld, N, d,
                                                                    chunk_rows, part);
    }
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  HookScope hs("attn_mse_final", st);
  attn_mse_final_kernel<<<(Hh + 127) / 128, 128, 0, st>>>(part, chunks, Hh, 1.0 / ((double)N * d), mse);
  return cudaGetLastError();
}

}  // namespace prism
