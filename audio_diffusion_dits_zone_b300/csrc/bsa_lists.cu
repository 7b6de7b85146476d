// Helpers of the block-sparse attention backward.
//
// transpose_lists: for every (head h, key block j) the query blocks i whose kept
//   list contains j, ascending.  A bit matrix bits[h][j][i / 32] is set from the
//   kept lists (atomicOr), then one warp per (h, j) emits the set bits in order
//   (popcount + warp scan), so the result is deterministic.
// row_dot: D[h][r] = sum_c dO[r, h, c] * O[r, h, c] (fp32), the softmax-gradient
//   row term of dS = P * (dP - D).
// order_rows: the launch order of the attention kernels' CTAs.  A CTA's work is its
//   list length; under the CDF rule lengths differ by up to two orders of magnitude
//   within a head, so a long row started late leaves the GPU idle at the end of the
//   launch.  Within each head the rows are ordered by list length, longest first
//   (equal lengths by index, so the order is deterministic); heads stay in sequence,
//   which keeps the CTAs in flight on one or two heads' K and V (L2-resident).
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

__global__ void set_bits_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ idx, int Hh, int nb,
                                uint32_t* __restrict__ bits, uint32_t* status) {
  const int words = (nb + 31) / 32;
  const int row = blockIdx.x;  // h * nb + i
  const int h = row / nb, i = row - h * nb;
  const int cnt = counts[row];
  const int32_t* lst = idx + (size_t)row * nb;
  for (int t = threadIdx.x; t < cnt && t < nb; t += blockDim.x) {
    const int j = lst[t];
    if (j < 0 || j >= nb) {
      flag_error(status, PRISM_DEV_BAD_INDEX);
      continue;
    }
    atomicOr(&bits[((size_t)h * nb + j) * words + (i >> 5)], 1u << (i & 31));
  }
  if (threadIdx.x == 0 && (cnt < 0 || cnt > nb)) flag_error(status, PRISM_DEV_BAD_INDEX);
}

__global__ void emit_lists_kernel(const uint32_t* __restrict__ bits, int Hh, int nb, int32_t* __restrict__ tcounts,
                                  int32_t* __restrict__ tidx) {
  const int words = (nb + 31) / 32;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= Hh * nb) return;
  const uint32_t* bw = bits + (size_t)warp * words;
  int32_t* out = tidx + (size_t)warp * nb;
  int base = 0;
  for (int w0 = 0; w0 < words; w0 += 32) {
    const uint32_t word = (w0 + lane < words) ? bw[w0 + lane] : 0u;
    const int c = __popc(word);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int pos = base + incl - c;
    uint32_t x = word;
    while (x) {
      const int b = __ffs(x) - 1;
      out[pos++] = (w0 + lane) * 32 + b;
      x &= x - 1;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) tcounts[warp] = base;
}

template <typename T>
__global__ void row_dot_kernel(const T* __restrict__ o, const T* __restrict__ dO, int64_t ld, int N, int Hh, int d,
                               float* __restrict__ D) {
  // one warp per (token, head)
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (int64_t)N * Hh) return;
  const int64_t n = wid / Hh;
  const int h = (int)(wid - n * Hh);
  const T* a = o + n * ld + (int64_t)h * d;
  const T* b = dO + n * ld + (int64_t)h * d;
  float s = 0.f;
  for (int c = lane; c < d; c += 32) s = fmaf(to_f32<T>(a[c]), to_f32<T>(b[c]), s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) D[(size_t)h * N + n] = s;
}


// One warp per head: counting sort of the head's rows by list length, descending and
// stable.  hist[0..nb] in dynamic shared memory.
__global__ void __launch_bounds__(32) order_rows_kernel(const int32_t* __restrict__ counts, int nb,
                                                        int32_t* __restrict__ order) {
  extern __shared__ int32_t hist[];
  const int h = blockIdx.x, lane = threadIdx.x;
  const int32_t* c = counts + (size_t)h * nb;
  auto key = [&](int i) { return min(max(c[i], 0), nb); };
  for (int b = lane; b <= nb; b += 32) hist[b] = 0;
  __syncwarp();
  for (int i = lane; i < nb; i += 32) atomicAdd(&hist[key(i)], 1);
  __syncwarp();
  // hist[b] <- rows whose length exceeds b (their start in the order)
  int run = 0;
  for (int b0 = nb; b0 >= 0; b0 -= 32) {
    const int b = b0 - lane;
    const int v = b >= 0 ? hist[b] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (b >= 0) hist[b] = run + incl - v;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncwarp();
  const uint32_t lt = (1u << lane) - 1u;
  for (int i0 = 0; i0 < nb; i0 += 32) {
    const int i = i0 + lane;
    const int k = i < nb ? key(i) : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, k);
    const int rank = __popc(peers & lt);
    const int base = i < nb ? hist[k] : 0;
    __syncwarp();
    if (i < nb) {
      order[(size_t)h * nb + base + rank] = h * nb + i;
      if (rank == 0) hist[k] = base + __popc(peers);
    }
    __syncwarp();
  }
}

}  // namespace

size_t lists_ws_bytes(int Hh, int nb) {
  const size_t words = (size_t)(nb + 31) / 32;
  return a256((size_t)Hh * nb * words * 4) + a256((size_t)Hh * nb * 4) + a256((size_t)Hh * nb * nb * 4);
}

cudaError_t transpose_lists_launch(const int32_t* counts, const int32_t* idx, int Hh, int nb, void* ws,
                                   int32_t** tcounts, int32_t** tidx, cudaStream_t st, uint32_t* status) {
  const size_t words = (size_t)(nb + 31) / 32;
  char* p = static_cast<char*>(ws);
  uint32_t* bits = reinterpret_cast<uint32_t*>(p);
  p += a256((size_t)Hh * nb * words * 4);
  *tcounts = reinterpret_cast<int32_t*>(p);
  p += a256((size_t)Hh * nb * 4);
  *tidx = reinterpret_cast<int32_t*>(p);
  cudaError_t e = cudaMemsetAsync(bits, 0, (size_t)Hh * nb * words * 4, st);
  if (e != cudaSuccess) return e;
  {
    HookScope hs("lists_set_bits", st);
    set_bits_kernel<<<Hh * nb, 128, 0, st>>>(counts, idx, Hh, nb, bits, status);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t threads = (int64_t)Hh * nb * 32;
  HookScope hs("lists_emit", st);
  emit_lists_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(bits, Hh, nb, *tcounts, *tidx);
  return cudaGetLastError();
}

bool order_rows_supported(int nb) { return nb >= 1 && (size_t)(nb + 1) * 4 <= kOrderSmemMax; }

cudaError_t order_rows_launch(const int32_t* counts, int Hh, int nb, int32_t* order, const char* name,
                              cudaStream_t st) {
  if (!order_rows_supported(nb)) return cudaErrorInvalidValue;
  HookScope hs(name, st);
  order_rows_kernel<<<Hh, 32, (size_t)(nb + 1) * 4, st>>>(counts, nb, order);
  return cudaGetLastError();
}

cudaError_t row_dot_launch(const void* o, const void* dO, int dtype, int64_t ld, int N, int Hh, int d, float* Drow,
                           cudaStream_t st) {
  const int64_t threads = (int64_t)N * Hh * 32;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  HookScope hs("row_dot", st);
  if (dtype == PRISM_BF16)
    row_dot_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(o),
                                                          static_cast<const __nv_bfloat16*>(dO), ld, N, Hh, d, Drow);
  else
    row_dot_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(o), static_cast<const float*>(dO), ld, N,
                                                  Hh, d, Drow);
  return cudaGetLastError();
}

}  // namespace prism
