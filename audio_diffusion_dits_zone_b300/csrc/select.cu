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
// the kept set is the shortest prefix that holds at least k blocks AND at least
// tau of the mass; emit it in ascending index order.
//
// One warp per (head, query block) for rows of up to 768 blocks, one CTA of four
// warps per row for longer ones; no sort.  The row is read once into shared memory,
// then:
//   1. drops every block into one of 256 equal-width buckets of [min, max] score
//      (a monotone map), with a histogram of counts and softmax masses;
//   2. scans the buckets from the top to the first one at which both conditions
//      hold: everything above it is kept, nothing below it;
//   3. ranks that bucket's blocks exactly (score descending, index ascending) and
//      keeps the shortest prefix of them that completes both conditions;
//   4. writes the kept indices in ascending order with ballots.
// Masses are fixed-point integers, q = round(exp(s - max) * 2^40), so every sum is
// exact and independent of the order the lanes add in: the lists are
// deterministic, and the sums are closer to the exact softmax mass than an fp32
// running sum would be (the only rounding is in exp and in q, <= 2^-41 per block).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

constexpr int kSelThreads = 128;  // select_row_kernel: one CTA of 4 warps per row
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelWarpsMax = 4;   // select_warp_kernel: rows (one per warp) per CTA
constexpr int kWarpRowMaxNb = 768;  // rows up to this many blocks go one per warp
constexpr int kBins = 256;
constexpr float kMassScale = 1099511627776.0f;  // 2^40

__device__ __forceinline__ uint32_t order_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 and +0 are the same score
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending uint order == ascending float order
}
__device__ __forceinline__ unsigned long long mass_of(float s, float smax) {
  return __float2ull_rn(expf(s - smax) * kMassScale);
}
__device__ __forceinline__ int bucket_of(float s, float smin, float scale) {
  return min(kBins - 1, max(0, __float2int_rz((s - smin) * scale)));
}

struct RowBins {
  uint32_t cnt[kBins];
  unsigned long long mass[kBins];
};

// Shared memory of a row: its scores, a kept flag per block, the crossing bucket's
// block indices (in index order), then the histogram.
__host__ __device__ constexpr size_t row_bytes(int nb) {
  return ((size_t)nb * (4 + 1 + 4) + 15) / 16 * 16 + sizeof(RowBins);
}

// One warp per row, each warp with its own shared-memory row: short rows, where many
// rows in flight per SM matter more than the latency of one.
__global__ void __launch_bounds__(kSelWarpsMax * 32) select_warp_kernel(const float* __restrict__ scores, int rows,
                                                                    int nb, int k_top, double tau,
                                                                    int32_t* __restrict__ counts,
                                                                    int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.x * (blockDim.x >> 5) + warp;
  if (row >= rows) return;  // whole warp; nothing below synchronises across warps
  uint8_t* base = smem + warp * row_bytes(nb);
  float* sv = reinterpret_cast<float*>(base);
  int32_t* cand = reinterpret_cast<int32_t*>(base + (size_t)nb * 4);
  uint8_t* kept = base + (size_t)nb * 8;
  RowBins& B = *reinterpret_cast<RowBins*>(base + ((size_t)nb * 9 + 15) / 16 * 16);
  const float* s = scores + (size_t)row * nb;

  // ---- 1. read the row; min and max
  float mx = -INFINITY, mn = INFINITY;
  for (int t = lane; t < nb; t += 32) {
    const float v = s[t];
    sv[t] = v;
    kept[t] = 0;
    mx = fmaxf(mx, v);
    mn = fminf(mn, v);
  }
  for (int b = lane; b < kBins; b += 32) {
    B.cnt[b] = 0u;
    B.mass[b] = 0ull;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  const float range = mx - mn;
  const float scale = range > 0.f ? (float)kBins / range : 0.f;
  __syncwarp();
  // ---- histogram of counts and masses
  for (int t = lane; t < nb; t += 32) {
    const float v = sv[t];
    const int b = bucket_of(v, mn, scale);
    atomicAdd(&B.cnt[b], 1u);
    atomicAdd(&B.mass[b], mass_of(v, mx));
  }
  __syncwarp();
  // ---- 2. scan from the top bucket; lane l owns buckets 255 - 8l ... 248 - 8l
  uint32_t c8[8];
  unsigned long long m8[8];
  uint32_t cl = 0u;
  unsigned long long ml = 0ull;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int b = kBins - 1 - 8 * lane - e;
    c8[e] = B.cnt[b];
    m8[e] = B.mass[b];
    cl += c8[e];
    ml += m8[e];
  }
  uint32_t ci = cl;
  unsigned long long mi = ml;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t cy = __shfl_up_sync(0xffffffffu, ci, o);
    const unsigned long long my = __shfl_up_sync(0xffffffffu, mi, o);
    if (lane >= o) {
      ci += cy;
      mi += my;
    }
  }
  const unsigned long long ztot = __shfl_sync(0xffffffffu, mi, 31);
  // integer sums reach tau * total exactly when they reach its ceiling
  unsigned long long target;
  {
    const double tq = ceil(tau * (double)ztot);
    target = tq >= (double)ztot ? ztot : (unsigned long long)tq;
  }
  const uint32_t kneed = (uint32_t)k_top;
  uint32_t c_run = ci - cl;
  unsigned long long m_run = mi - ml;
  int hit = -1;
  uint32_t hit_cb = 0u, hit_c = 0u;
  unsigned long long hit_mb = 0ull;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (hit < 0 && c8[e] > 0u && c_run + c8[e] >= kneed && m_run + m8[e] >= target) {
      hit = e;
      hit_cb = c_run;
      hit_mb = m_run;
      hit_c = c8[e];
    }
    c_run += c8[e];
    m_run += m8[e];
  }
  // both conditions hold once every block is counted (nb >= k, total >= target), so
  // some lane hits; its bucket is the crossing one
  const uint32_t hits = __ballot_sync(0xffffffffu, hit >= 0);
  const int src = hits ? __ffs(hits) - 1 : 31;
  const int bstar = __shfl_sync(0xffffffffu, kBins - 1 - 8 * lane - (hit < 0 ? 7 : hit), src);
  const uint32_t above = __shfl_sync(0xffffffffu, hit_cb, src);
  const unsigned long long above_m = __shfl_sync(0xffffffffu, hit_mb, src);
  const uint32_t L = __shfl_sync(0xffffffffu, hit_c, src);

  // ---- 3. the crossing bucket's blocks in index order; everything above is kept
  uint32_t nc = 0u, kmin = 0xffffffffu, kmax = 0u;
  for (int t0 = 0; t0 < nb; t0 += 32) {
    const int t = t0 + lane;
    int b = -1;
    if (t < nb) b = bucket_of(sv[t], mn, scale);
    if (b > bstar) kept[t] = 1;
    const bool in = b == bstar;
    const uint32_t bal = __ballot_sync(0xffffffffu, in);
    if (in) {
      cand[nc + __popc(bal & ((1u << lane) - 1u))] = t;
      const uint32_t key = order_bits(sv[t]);
      kmin = min(kmin, key);
      kmax = max(kmax, key);
    }
    nc += __popc(bal);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  __syncwarp();
  // rank r of a candidate = candidates before it in (score desc, index asc) order;
  // keep the r-th (0-based) and all before it for the smallest r that completes
  // both conditions: take = r + 1
  uint32_t best = L;  // take; L keeps the whole bucket (never needed when a lane hits)
  if (kmin == kmax) {
    // one score value: the order is the index order and every mass is equal
    const unsigned long long qv = mass_of(sv[cand[0]], mx);
    const uint32_t tk = kneed > above ? kneed - above : 0u;
    uint32_t tm = 0u;
    if (above_m < target) tm = qv > 0ull ? (uint32_t)min((unsigned long long)L, (target - above_m + qv - 1ull) / qv) : L;
    best = min(L, max(tk, tm));
  } else {
    for (uint32_t c0 = 0; c0 < L; c0 += 32) {
      const uint32_t c = c0 + lane;
      uint32_t take = 0xffffffffu;
      if (c < L) {
        const int ti = cand[c];
        const uint32_t key = order_bits(sv[ti]);
        uint32_t rank = 0u;
        unsigned long long pre = 0ull;
        for (uint32_t d = 0; d < L; ++d) {
          const int td = cand[d];
          const float vd = sv[td];
          const uint32_t kd = order_bits(vd);
          if (kd > key || (kd == key && td < ti)) {
            ++rank;
            pre += mass_of(vd, mx);
          }
        }
        if (above + rank + 1u >= kneed && above_m + pre + mass_of(sv[ti], mx) >= target) take = rank + 1u;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) take = min(take, __shfl_xor_sync(0xffffffffu, take, o));
      best = min(best, take);
    }
    // mark the candidates whose rank is below `best`
    for (uint32_t c0 = 0; c0 < L; c0 += 32) {
      const uint32_t c = c0 + lane;
      if (c < L) {
        const int ti = cand[c];
        const uint32_t key = order_bits(sv[ti]);
        uint32_t rank = 0u;
        for (uint32_t d = 0; d < L; ++d) {
          const int td = cand[d];
          const uint32_t kd = order_bits(sv[td]);
          rank += (kd > key || (kd == key && td < ti)) ? 1u : 0u;
        }
        if (rank < best) kept[ti] = 1;
      }
    }
  }
  if (kmin == kmax)
    for (uint32_t c = lane; c < best; c += 32) kept[cand[c]] = 1;
  __syncwarp();

  // ---- 4. ascending output
  int32_t* out = idx + (size_t)row * nb;
  uint32_t n = 0u;
  for (int t0 = 0; t0 < nb; t0 += 32) {
    const int t = t0 + lane;
    const bool k = t < nb && kept[t];
    const uint32_t bal = __ballot_sync(0xffffffffu, k);
    if (k) out[n + __popc(bal & ((1u << lane) - 1u))] = t;
    n += __popc(bal);
  }
  if (lane == 0) counts[row] = (int32_t)n;
}

// One CTA per row (long rows, where one warp's latency per row would dominate):
// block-wide scalars of the row.
struct RowShared {
  float wmax[kSelWarps], wmin[kSelWarps];
  uint32_t wcnt[kSelWarps], wkmin[kSelWarps], wkmax[kSelWarps], wtake[kSelWarps];
  int bstar;
  uint32_t above, L;
  unsigned long long above_m, target;
};

__global__ void __launch_bounds__(kSelThreads) select_row_kernel(const float* __restrict__ scores, int nb, int k_top,
                                                             double tau, int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ RowShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  float* sv = reinterpret_cast<float*>(smem);
  int32_t* cand = reinterpret_cast<int32_t*>(smem + (size_t)nb * 4);
  uint8_t* kept = smem + (size_t)nb * 8;
  RowBins& B = *reinterpret_cast<RowBins*>(smem + ((size_t)nb * 9 + 15) / 16 * 16);
  const float* s = scores + (size_t)row * nb;
  // each warp owns a contiguous range of whole 32-block chunks (for the ordered passes)
  const int per = (nb + kSelThreads - 1) / kSelThreads * 32;
  const int r0 = min(nb, warp * per), r1 = min(nb, r0 + per);
  const uint32_t lt_mask = (1u << lane) - 1u;

  // ---- 1. read the row; min and max; clear the histogram
  float mx = -INFINITY, mn = INFINITY;
  for (int t = tid; t < nb; t += kSelThreads) {
    const float v = s[t];
    sv[t] = v;
    kept[t] = 0;
    mx = fmaxf(mx, v);
    mn = fminf(mn, v);
  }
  for (int b = tid; b < kBins; b += kSelThreads) {
    B.cnt[b] = 0u;
    B.mass[b] = 0ull;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  if (lane == 0) {
    sh.wmax[warp] = mx;
    sh.wmin[warp] = mn;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    mx = fmaxf(mx, sh.wmax[w]);
    mn = fminf(mn, sh.wmin[w]);
  }
  const float range = mx - mn;
  const float scale = range > 0.f ? (float)kBins / range : 0.f;
  // ---- histogram of counts and masses
  for (int t = tid; t < nb; t += kSelThreads) {
    const float v = sv[t];
    const int b = bucket_of(v, mn, scale);
    atomicAdd(&B.cnt[b], 1u);
    atomicAdd(&B.mass[b], mass_of(v, mx));
  }
  __syncthreads();
  // ---- 2. warp 0 scans from the top bucket; lane l owns buckets 255 - 8l ... 248 - 8l
  if (warp == 0) {
    uint32_t c8[8];
    unsigned long long m8[8];
    uint32_t cl = 0u;
    unsigned long long ml = 0ull;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int b = kBins - 1 - 8 * lane - e;
      c8[e] = B.cnt[b];
      m8[e] = B.mass[b];
      cl += c8[e];
      ml += m8[e];
    }
    uint32_t ci = cl;
    unsigned long long mi = ml;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t cy = __shfl_up_sync(0xffffffffu, ci, o);
      const unsigned long long my = __shfl_up_sync(0xffffffffu, mi, o);
      if (lane >= o) {
        ci += cy;
        mi += my;
      }
    }
    const unsigned long long ztot = __shfl_sync(0xffffffffu, mi, 31);
    // integer sums reach tau * total exactly when they reach its ceiling
    unsigned long long target;
    {
      const double tq = ceil(tau * (double)ztot);
      target = tq >= (double)ztot ? ztot : (unsigned long long)tq;
    }
    const uint32_t kneed = (uint32_t)k_top;
    uint32_t c_run = ci - cl;
    unsigned long long m_run = mi - ml;
    int hit = -1;
    uint32_t hit_cb = 0u, hit_c = 0u;
    unsigned long long hit_mb = 0ull;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (hit < 0 && c8[e] > 0u && c_run + c8[e] >= kneed && m_run + m8[e] >= target) {
        hit = e;
        hit_cb = c_run;
        hit_mb = m_run;
        hit_c = c8[e];
      }
      c_run += c8[e];
      m_run += m8[e];
    }
    // both conditions hold once every block is counted (nb >= k, total >= target), so
    // some lane hits; its bucket is the crossing one
    const uint32_t hits = __ballot_sync(0xffffffffu, hit >= 0);
    const int src = hits ? __ffs(hits) - 1 : 31;
    const int bstar = __shfl_sync(0xffffffffu, kBins - 1 - 8 * lane - (hit < 0 ? 7 : hit), src);
    const uint32_t above = __shfl_sync(0xffffffffu, hit_cb, src);
    const unsigned long long above_m = __shfl_sync(0xffffffffu, hit_mb, src);
    const uint32_t L = __shfl_sync(0xffffffffu, hit_c, src);
    if (lane == 0) {
      sh.bstar = bstar;
      sh.above = above;
      sh.above_m = above_m;
      sh.L = L;
      sh.target = target;
    }
  }
  __syncthreads();
  const int bstar = sh.bstar;
  const uint32_t above = sh.above, L = sh.L, kneed = (uint32_t)k_top;
  const unsigned long long above_m = sh.above_m, target = sh.target;

  // ---- 3. the crossing bucket's blocks in index order; everything above is kept
  uint32_t nc = 0u, kmin = 0xffffffffu, kmax = 0u;
  for (int t0 = r0; t0 < r1; t0 += 32) {
    const int t = t0 + lane;
    int b = -1;
    if (t < r1) b = bucket_of(sv[t], mn, scale);
    if (b > bstar) kept[t] = 1;
    const bool in = b == bstar;
    nc += __popc(__ballot_sync(0xffffffffu, in));
    if (in) {
      const uint32_t key = order_bits(sv[t]);
      kmin = min(kmin, key);
      kmax = max(kmax, key);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    sh.wcnt[warp] = nc;
    sh.wkmin[warp] = kmin;
    sh.wkmax[warp] = kmax;
  }
  __syncthreads();
  uint32_t off = 0u;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    if (w < warp) off += sh.wcnt[w];
    kmin = min(kmin, sh.wkmin[w]);
    kmax = max(kmax, sh.wkmax[w]);
  }
  for (int t0 = r0; t0 < r1; t0 += 32) {  // write this range's candidates at its offset
    const int t = t0 + lane;
    const bool in = t < r1 && bucket_of(sv[t], mn, scale) == bstar;
    const uint32_t bal = __ballot_sync(0xffffffffu, in);
    if (in) cand[off + __popc(bal & lt_mask)] = t;
    off += __popc(bal);
  }
  __syncthreads();
  // rank r of a candidate = candidates before it in (score desc, index asc) order;
  // keep the r-th (0-based) and all before it for the smallest r that completes
  // both conditions: take = r + 1
  if (kmin == kmax) {
    // one score value: the order is the index order and every mass is equal
    const unsigned long long qv = mass_of(sv[cand[0]], mx);
    const uint32_t tk = kneed > above ? kneed - above : 0u;
    uint32_t tm = 0u;
    if (above_m < target) tm = qv > 0ull ? (uint32_t)min((unsigned long long)L, (target - above_m + qv - 1ull) / qv) : L;
    const uint32_t best = min(L, max(tk, tm));
    for (uint32_t c = tid; c < best; c += kSelThreads) kept[cand[c]] = 1;
  } else {
    uint32_t take = 0xffffffffu;
    for (uint32_t c = tid; c < L; c += kSelThreads) {
      const int ti = cand[c];
      const uint32_t key = order_bits(sv[ti]);
      uint32_t rank = 0u;
      unsigned long long pre = 0ull;
      for (uint32_t d = 0; d < L; ++d) {
        const int td = cand[d];
        const float vd = sv[td];
        const uint32_t kd = order_bits(vd);
        if (kd > key || (kd == key && td < ti)) {
          ++rank;
          pre += mass_of(vd, mx);
        }
      }
      if (above + rank + 1u >= kneed && above_m + pre + mass_of(sv[ti], mx) >= target) take = min(take, rank + 1u);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) take = min(take, __shfl_xor_sync(0xffffffffu, take, o));
    if (lane == 0) sh.wtake[warp] = take;
    __syncthreads();
    uint32_t best = L;  // L keeps the whole bucket (never needed when the scan hits)
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) best = min(best, sh.wtake[w]);
    // mark the candidates whose rank is below `best`
    for (uint32_t c = tid; c < L; c += kSelThreads) {
      const int ti = cand[c];
      const uint32_t key = order_bits(sv[ti]);
      uint32_t rank = 0u;
      for (uint32_t d = 0; d < L; ++d) {
        const int td = cand[d];
        const uint32_t kd = order_bits(sv[td]);
        rank += (kd > key || (kd == key && td < ti)) ? 1u : 0u;
      }
      if (rank < best) kept[ti] = 1;
    }
  }
  __syncthreads();

  // ---- 4. ascending output: each warp counts its range, then writes at its offset
  uint32_t kc = 0u;
  for (int t0 = r0; t0 < r1; t0 += 32) {
    const int t = t0 + lane;
    kc += __popc(__ballot_sync(0xffffffffu, t < r1 && kept[t]));
  }
  if (lane == 0) sh.wcnt[warp] = kc;
  __syncthreads();
  uint32_t n = 0u, total = 0u;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    if (w < warp) n += sh.wcnt[w];
    total += sh.wcnt[w];
  }
  int32_t* out = idx + (size_t)row * nb;
  for (int t0 = r0; t0 < r1; t0 += 32) {
    const int t = t0 + lane;
    const bool k = t < r1 && kept[t];
    const uint32_t bal = __ballot_sync(0xffffffffu, k);
    if (k) out[n + __popc(bal & lt_mask)] = t;
    n += __popc(bal);
  }
  if (tid == 0) counts[row] = (int32_t)total;
}

}  // namespace

cudaError_t select_launch(const float* scores, int Hh, int nb, int k_top, double tau, int32_t* counts, int32_t* idx,
                          cudaStream_t st) {
  const size_t per = row_bytes(nb);
  const int rows = Hh * nb;
  cudaError_t e;
  if (nb <= kWarpRowMaxNb) {
    const int warps = (int)std::max<size_t>(1, std::min<size_t>(kSelWarpsMax, (200u * 1024u) / per));
    const size_t smem = per * warps;
    if ((e = cudaFuncSetAttribute(select_warp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    HookScope hs("select", st);
    select_warp_kernel<<<(unsigned)((rows + warps - 1) / warps), warps * 32, smem, st>>>(scores, rows, nb, k_top, tau,
                                                                                        counts, idx);
  } else {
    if ((e = cudaFuncSetAttribute(select_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)per)) !=
        cudaSuccess)
      return e;
    HookScope hs("select", st);
    select_row_kernel<<<(unsigned)rows, kSelThreads, per, st>>>(scores, nb, k_top, tau, counts, idx);
  }
  return cudaGetLastError();
}

}  // namespace prism
