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
// One CTA of 128 threads per (head, query block); no sort.  The row is read once
// into shared memory as order-preserving 32-bit keys.  The end of the kept prefix
// is found by a radix descent over the key bits (4 digits of 8 bits, most
// significant first): at each digit a 256-bin histogram of the candidates' counts
// and softmax masses picks the first bin, from the top, at which both conditions
// hold, and the descent continues inside it.  After the last digit the cut is one
// exact score value; equal scores there are taken in index order.
//
// Masses are fixed-point integers, q = round(exp(s - max) * 2^40), so every sum is
// exact and independent of the order the threads add in: the lists are
// deterministic, and the sums are closer to the exact softmax mass than an fp32
// running sum would be (the only rounding is in exp and in q, <= 2^-41 per block).
#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

constexpr int kSelThreads = 128;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBins = 256;
constexpr float kMassScale = 1099511627776.0f;  // 2^40

__device__ __forceinline__ uint32_t order_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 and +0 are the same score
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending uint order == ascending float order
}
__device__ __forceinline__ float from_order_bits(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
__device__ __forceinline__ unsigned long long mass_of(uint32_t key, float smax) {
  return __float2ull_rn(expf(from_order_bits(key) - smax) * kMassScale);
}

struct SelShared {
  uint32_t cnt[kBins];
  unsigned long long mass[kBins];
  float fmax[kSelWarps];
  unsigned long long usum[kSelWarps];
  uint32_t scan[kSelWarps];
  // descent state, written by warp 0
  uint32_t prefix, above_cnt, pick_cnt;
  unsigned long long above_mass;
  int done;
};

// Inclusive scan of v over the block; every thread gets its inclusive prefix and
// the block total.
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t* tmp, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    const uint32_t t = tmp[w];
    before += w < warp ? t : 0u;
    tot += t;
  }
  *total = tot;
  __syncthreads();
  return before + x;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const float* __restrict__ scores, int nb, int k_top,
                                                             double tau, int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ idx) {
  extern __shared__ uint32_t keys[];  // [nb]
  __shared__ SelShared sh;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t row = blockIdx.x;
  const float* s = scores + row * nb;

  // ---- read the row once: keys and the row max
  float mx = -INFINITY;
  for (int t = threadIdx.x; t < nb; t += kSelThreads) {
    const float v = s[t];
    keys[t] = order_bits(v);
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) sh.fmax[warp] = mx;
  __syncthreads();
  float smax = sh.fmax[0];
#pragma unroll
  for (int w = 1; w < kSelWarps; ++w) smax = fmaxf(smax, sh.fmax[w]);

  // ---- total mass (integer, exact)
  unsigned long long z = 0;
  for (int t = threadIdx.x; t < nb; t += kSelThreads) z += mass_of(keys[t], smax);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane == 0) sh.usum[warp] = z;
  if (threadIdx.x == 0) {
    sh.prefix = 0u;
    sh.above_cnt = 0u;
    sh.above_mass = 0ull;
    sh.done = 0;
  }
  __syncthreads();
  unsigned long long ztot = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) ztot += sh.usum[w];
  const double target = tau * (double)ztot;
  const uint32_t kneed = (uint32_t)k_top;

  // ---- radix descent: 4 digits of 8 bits
  uint32_t mask = 0u;
  for (int level = 0; level < 4; ++level) {
    const int shift = 24 - 8 * level;
    for (int b = threadIdx.x; b < kBins; b += kSelThreads) {
      sh.cnt[b] = 0u;
      sh.mass[b] = 0ull;
    }
    __syncthreads();
    const uint32_t prefix = sh.prefix;
    // warp-aggregated histogram: lanes that hit the same bin add once
    for (int t0 = 0; t0 < nb; t0 += kSelThreads) {
      const int t = t0 + threadIdx.x;
      uint32_t key = 0u;
      bool cand = false;
      if (t < nb) {
        key = keys[t];
        cand = (key & mask) == prefix;
      }
      const uint32_t act = __ballot_sync(0xffffffffu, cand);
      if (!act) continue;
      const uint32_t bin = cand ? (key >> shift) & 0xffu : 0x100u + lane;  // non-candidates never match a bin
      const uint32_t grp = __match_any_sync(0xffffffffu, bin);
      const unsigned long long q = cand ? mass_of(key, smax) : 0ull;
      const uint32_t qhi = (uint32_t)(q >> 20), qlo = (uint32_t)(q & 0xfffffu);  // q <= 2^40
      const uint32_t shi = __reduce_add_sync(grp, qhi), slo = __reduce_add_sync(grp, qlo);
      if (cand && lane == __ffs(grp) - 1) {
        atomicAdd(&sh.cnt[bin], (uint32_t)__popc(grp));
        atomicAdd(&sh.mass[bin], ((unsigned long long)shi << 20) + (unsigned long long)slo);
      }
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255 - 8l ... 248 - 8l (descending score order)
      uint32_t c8[8];
      unsigned long long m8[8];
      uint32_t cl = 0u;
      unsigned long long ml = 0ull;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int b = kBins - 1 - 8 * lane - e;
        c8[e] = sh.cnt[b];
        m8[e] = sh.mass[b];
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
      uint32_t c_run = sh.above_cnt + (ci - cl);
      unsigned long long m_run = sh.above_mass + (mi - ml);
      // first bin (from the top) at which both conditions hold; also the lane's last
      // non-empty bin, the fallback should no bin qualify (only with NaN scores)
      int hit = -1, last = -1;
      uint32_t hit_cb = 0u, hit_c = 0u, last_cb = 0u, last_c = 0u;
      unsigned long long hit_mb = 0ull, last_mb = 0ull;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (c8[e] > 0u) {
          if (hit < 0 && c_run + c8[e] >= kneed && (double)(m_run + m8[e]) >= target) {
            hit = e;
            hit_cb = c_run;
            hit_mb = m_run;
            hit_c = c8[e];
          }
          last = e;
          last_cb = c_run;
          last_mb = m_run;
          last_c = c8[e];
        }
        c_run += c8[e];
        m_run += m8[e];
      }
      const uint32_t hits = __ballot_sync(0xffffffffu, hit >= 0);
      const uint32_t nonempty = __ballot_sync(0xffffffffu, last >= 0);
      const int src = hits ? __ffs(hits) - 1 : (nonempty ? 31 - __clz(nonempty) : -1);
      if (lane == src) {
        const bool h = hits != 0u;
        const uint32_t b = (uint32_t)(kBins - 1 - 8 * lane - (h ? hit : last));
        sh.prefix = prefix | (b << shift);
        sh.above_cnt = h ? hit_cb : last_cb;
        sh.above_mass = h ? hit_mb : last_mb;
        sh.pick_cnt = h ? hit_c : last_c;
      }
    }
    mask |= 0xffu << shift;
    __syncthreads();
  }

  // ---- the cut: keys above V are kept; of the keys equal to V (one score value,
  // equal masses), the first `take` in index order
  const uint32_t V = sh.prefix;
  const uint32_t above = sh.above_cnt, neq = sh.pick_cnt;
  const unsigned long long above_m = sh.above_mass;
  uint32_t take;
  {
    const unsigned long long qv = mass_of(V, smax);
    const uint32_t tk = kneed > above ? kneed - above : 0u;
    uint32_t tm = 0u;
    if ((double)above_m < target) {
      tm = neq;
      if (qv > 0ull) {
        const double need = (target - (double)above_m) / (double)qv;
        uint32_t t = (uint32_t)fmin(ceil(need), (double)neq);
        // settle the rounding of the division on the integer sums themselves
        while (t > 0u && (double)(above_m + (unsigned long long)(t - 1u) * qv) >= target) --t;
        while (t < neq && (double)(above_m + (unsigned long long)t * qv) < target) ++t;
        tm = t;
      }
    }
    take = min(neq, max(tk, tm));
  }

  // ---- compaction in ascending index order; each thread owns a contiguous run
  const int per = (nb + kSelThreads - 1) / kSelThreads;
  const int beg = min(nb, (int)threadIdx.x * per), end = min(nb, beg + per);
  uint32_t n_tie = 0u, n_hi = 0u;
  for (int t = beg; t < end; ++t) {
    const uint32_t key = keys[t];
    n_hi += key > V;
    n_tie += key == V;
  }
  // one scan of both counts, packed (each <= 4096)
  uint32_t tot;
  const uint32_t incl = block_incl_scan((n_tie << 16) | n_hi, sh.scan, &tot);
  const uint32_t excl = incl - ((n_tie << 16) | n_hi);
  const uint32_t tie_before = excl >> 16, hi_before = excl & 0xffffu;
  uint32_t pos = hi_before + min(tie_before, take);
  uint32_t tie_rank = tie_before;
  int32_t* out = idx + row * nb;
  for (int t = beg; t < end; ++t) {
    const uint32_t key = keys[t];
    if (key > V) {
      out[pos++] = t;
    } else if (key == V) {
      if (tie_rank < take) out[pos++] = t;
      ++tie_rank;
    }
  }
  if (threadIdx.x == 0) counts[row] = (int32_t)((tot & 0xffffu) + take);
}

}  // namespace

cudaError_t select_launch(const float* scores, int Hh, int nb, int k_top, double tau, int32_t* counts, int32_t* idx,
                          cudaStream_t st) {
  HookScope hs("select", st);
  select_kernel<<<(unsigned)Hh * nb, kSelThreads, (size_t)nb * sizeof(uint32_t), st>>>(scores, nb, k_top, tau,
                                                                                        counts, idx);
  return cudaGetLastError();
}

}  // namespace prism
