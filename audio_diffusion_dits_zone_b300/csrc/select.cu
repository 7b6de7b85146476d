// Step 3 of the path: hybrid block selection.
//
// "Prism: dynamic sparse attention for 2K joint video-audio generation training",
// section "Region-adapted block construction", paragraph 2: a hybrid block
// selection makes each query's sparsity dynamic; settings use sparsity
// 0.75 / 0.80 / 0.85 / 0.93 and a CDF threshold of 0.20.
//
// Reading: order the row's blocks by score, largest first (equal scores: smaller
// index first); keep the top k = ceil((1 - s) nb) and also the shortest prefix
// whose softmax mass reaches the threshold; both are prefixes of one order, so
// the kept set is the first max(k, m) blocks; emit them in ascending index order.
//
// One CTA per (head, query block).  The row (nb <= 4096) is sorted in shared memory
// as 64-bit keys (inverted order-preserving score bits : index), so the sort order
// is exactly (score descending, index ascending) and deterministic.  The softmax
// mass prefix is a deterministic block scan in fp32; the kept flags are compacted
// in ascending index order with a second scan.
#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

constexpr int kSelThreads = 256;
constexpr int kMaxNb = 4096;

__device__ __forceinline__ uint32_t order_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending uint order == ascending float order
}

// Exclusive scan over the block of one value per thread; returns the prefix and
// writes the block total to *total.  `tmp` holds 32 values.
template <typename V>
__device__ __forceinline__ V block_exclusive_scan(V x, V* tmp, V* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  V incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const V y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    V w = lane < nw ? tmp[lane] : V(0);
    V wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const V y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) tmp[lane] = wi - w;
    if (lane == nw - 1) tmp[31] = wi;
  }
  __syncthreads();
  const V res = tmp[warp] + incl - x;
  *total = tmp[31];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const float* __restrict__ scores, int nb, int P,
                                                             int k_top, float tau, int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ idx) {
  __shared__ unsigned long long keys[kMaxNb];
  __shared__ float tmpf[32];
  __shared__ int tmpi[32];
  __shared__ int mcut;
  __shared__ unsigned int flags[kMaxNb / 32];
  const size_t row = blockIdx.x;
  const float* s = scores + row * nb;
  for (int t = threadIdx.x; t < P; t += kSelThreads) {
    unsigned long long key = ~0ull;
    if (t < nb) key = ((unsigned long long)(~order_bits(s[t])) << 32) | (unsigned)t;
    keys[t] = key;
  }
  if (threadIdx.x == 0) mcut = nb;
  __syncthreads();
  // bitonic sort, ascending
  for (int kk = 2; kk <= P; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int t = threadIdx.x; t < (P >> 1); t += kSelThreads) {
        const int lo = ((t / j) * 2 * j) + (t % j);
        const int hi = lo + j;
        const bool up = (lo & kk) == 0;
        const unsigned long long a = keys[lo], b = keys[hi];
        if ((a > b) == up) {
          keys[lo] = b;
          keys[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  // softmax mass prefix in sorted order: each thread owns a contiguous run
  const int per = (nb + kSelThreads - 1) / kSelThreads;
  const int beg = min(nb, (int)threadIdx.x * per), end = min(nb, beg + per);
  const float smax = s[(unsigned)(keys[0] & 0xffffffffu)];
  float local = 0.f;
  for (int t = beg; t < end; ++t) local += expf(s[(unsigned)(keys[t] & 0xffffffffu)] - smax);
  float Z;
  float run = block_exclusive_scan<float>(local, tmpf, &Z);
  const float target = tau * Z;
  for (int t = beg; t < end; ++t) {
    run += expf(s[(unsigned)(keys[t] & 0xffffffffu)] - smax);
    if (run >= target) {
      atomicMin(&mcut, t + 1);
      break;
    }
  }
  __syncthreads();
  const int r = max(k_top, mcut);
  // kept flags by block index, then compaction in ascending index order
  for (int w = threadIdx.x; w < (nb + 31) / 32; w += kSelThreads) flags[w] = 0u;
  __syncthreads();
  for (int t = threadIdx.x; t < r; t += kSelThreads) {
    const unsigned j = (unsigned)(keys[t] & 0xffffffffu);
    atomicOr(&flags[j >> 5], 1u << (j & 31));
  }
  __syncthreads();
  int cnt = 0;
  for (int t = beg; t < end; ++t) cnt += (flags[t >> 5] >> (t & 31)) & 1u;
  int tot;
  int pos = block_exclusive_scan<int>(cnt, tmpi, &tot);
  int32_t* out = idx + row * nb;
  for (int t = beg; t < end; ++t)
    if ((flags[t >> 5] >> (t & 31)) & 1u) out[pos++] = t;
  if (threadIdx.x == 0) counts[row] = tot;
}

}  // namespace

cudaError_t select_launch(const float* scores, int Hh, int nb, int k_top, float tau, int32_t* counts, int32_t* idx,
                          cudaStream_t st) {
  int P = 1;
  while (P < nb) P <<= 1;
  if (P < 2) P = 2;
  HookScope hs("select", st);
  select_kernel<<<(unsigned)Hh * nb, kSelThreads, 0, st>>>(scores, nb, P, k_top, tau, counts, idx);
  return cudaGetLastError();
}

}  // namespace prism
