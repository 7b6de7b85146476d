// The A2V field: the audio-to-video cross-attention and its per-token feature norm.
//
// "Prism: dynamic sparse attention for 2K joint video-audio generation training",
// section "Region-adapted block construction", paragraph 1: besides the video
// features' channel variance, each macro-zone uses the feature norm of the
// audio-to-video cross-attention, which measures how strongly the audio drives that
// part of the video.
//
// Reading (the page gives no formula): for every video token n and head h,
//   O[n][h] = sum_m softmax_m(Qv[n][h] . Ka[m][h] / sqrt(d)) Va[m][h],
//   a2v[n]  = sqrt(sum_h |O[n][h]|^2),
// the L2 norm of the token's whole cross-attention output feature (Hh * d channels).
//
// The cross-attention is the forward attention kernel with no kept lists (every audio
// key block is visited) and an epilogue that writes |O[n][h]|^2 in fp32 before the
// output is rounded; this file adds the reduction over heads.
#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

// One thread per token; consecutive threads read consecutive tokens of each head's row
// (coalesced), heads summed in a fixed order.
__global__ void __launch_bounds__(256) a2v_reduce_kernel(const float* __restrict__ sqn, int N, int Hh,
                                                         float* __restrict__ a2v) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  float s = 0.f;
  for (int h = 0; h < Hh; ++h) s += sqn[(size_t)h * N + n];
  a2v[n] = sqrtf(s);
}

}  // namespace

cudaError_t a2v_reduce_launch(const float* sqn, int N, int Hh, float* a2v, cudaStream_t st) {
  HookScope hs("a2v_reduce", st);
  a2v_reduce_kernel<<<(unsigned)((N + 255) / 256), 256, 0, st>>>(sqn, N, Hh, a2v);
  return cudaGetLastError();
}

}  // namespace prism
