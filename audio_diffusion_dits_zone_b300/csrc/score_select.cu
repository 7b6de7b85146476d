// Steps 2b + 3 fused: block scores and hybrid block selection in one kernel; the
// [Hh][nb][nb] score matrix never reaches global memory.
//
// "Prism: dynamic sparse attention for 2K joint video-audio generation training",
// section "Region-adapted block construction", paragraph 2: a hybrid selection of
// key blocks per query block, sparsity 0.75 / 0.80 / 0.85 / 0.93, CDF threshold 0.20.
// Same readings and the same arithmetic as the separate scores and select kernels:
//   S[h][i][j] = qbar[h][i] . kbar[h][j] / sqrt(d), accumulated in fp32 over d in
//   ascending order (bit-identical to the scores kernel), and the kept set = the
//   first max(k, m) blocks in (score desc, index asc) order with k = the top-(1 - s)
//   count and m the shortest prefix whose softmax mass reaches tau; softmax masses as
//   exact fixed-point integers q = round(exp(s - max) * 2^40) (the select kernels'
//   definition), so the lists equal theirs bit for bit.
//
// One CTA of R warps per (head, R consecutive query blocks):
//   1. score rows: the R rows of qbar (transposed in shared memory) against every key
//      block, 512 keys per tile, kbar staged 8 channels at a time (double-buffered);
//      a thread owns 4 rows x 4 keys (16 fp32 accumulators), so each channel step is
//      two 16-byte shared loads for 16 FMAs, and two CTAs fit on an SM (one CTA's
//      selection overlaps the other's score rows).  The R score rows stay in shared
//      memory.
//   2. selection: warp w selects row w.  Blocks are dropped into 256 equal-width
//      buckets of [min, max] with fixed-point mass histograms; the scan from the top
//      finds the bucket where both conditions are first met; everything above it is
//      kept.  If that bucket holds at most 256 blocks they are ranked exactly; if its
//      blocks all have one score, the first ones by index are kept; otherwise its
//      value range is bucketed again (each level narrows the range 256-fold, so a few
//      levels end with a small or single-valued bucket).  Kept blocks are bit flags,
//      written out in ascending order with ballots.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

constexpr int kSsKeys = 512;    // keys per score tile
constexpr int kSsSlice = 8;     // channels per staged slice of kbar
constexpr int kBins = 256;
constexpr int kCandCap = 256;   // candidates ranked exactly per level
constexpr int kMaxLevels = 8;
constexpr float kMassScale = 1099511627776.0f;  // 2^40

__device__ __forceinline__ uint32_t order_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 and +0 are the same score
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ unsigned long long mass_of(float s, float smax) {
  return __float2ull_rn(expf(s - smax) * kMassScale);
}
__device__ __forceinline__ int bucket_of(float s, float lo, float scale) {
  return min(kBins - 1, max(0, __float2int_rz((s - lo) * scale)));
}

// Per-warp selection state: histogram, candidates and two bit sets over the row.
__host__ __device__ constexpr size_t sel_bytes(int nb) {
  return (size_t)kBins * 4 + (size_t)kBins * 8 + (size_t)kCandCap * 2 + 2 * (size_t)((nb + 31) / 32) * 4;
}

// A warp selects one row sv[0, nb) (shared memory).  Writes idx_row[0, count) ascending
// and returns the count (lane 0's value is the one to store).
__device__ int select_row(const float* sv, int nb, int k_top, double tau, uint8_t* state) {
  const int lane = threadIdx.x & 31;
  const int nw = (nb + 31) / 32;
  uint32_t* cnt = reinterpret_cast<uint32_t*>(state);
  unsigned long long* mass = reinterpret_cast<unsigned long long*>(state + kBins * 4);
  uint16_t* cand = reinterpret_cast<uint16_t*>(state + kBins * 12);
  uint32_t* mem = reinterpret_cast<uint32_t*>(state + kBins * 12 + kCandCap * 2);  // still undecided
  uint32_t* kept = mem + nw;

  float mx = -INFINITY, mn = INFINITY;
  for (int t = lane; t < nb; t += 32) {
    const float v = sv[t];
    mx = fmaxf(mx, v);
    mn = fminf(mn, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  for (int w = lane; w < nw; w += 32) {
    const int rem = nb - 32 * w;
    mem[w] = rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
    kept[w] = 0u;
  }
  const uint32_t kneed = (uint32_t)k_top;
  uint32_t above = 0u;                 // blocks kept so far
  unsigned long long above_m = 0ull;   // their mass
  unsigned long long target = 0ull;
  float lo = mn, hi = mx;
  bool done = false;
  for (int level = 0; level < kMaxLevels && !done; ++level) {
    const float range = hi - lo;
    const float scale = range > 0.f ? (float)kBins / range : 0.f;
    for (int b = lane; b < kBins; b += 32) {
      cnt[b] = 0u;
      mass[b] = 0ull;
    }
    __syncwarp();
    for (int t = lane; t < nb; t += 32) {
      if ((mem[t >> 5] >> (t & 31)) & 1u) {
        const float v = sv[t];
        const int b = bucket_of(v, lo, scale);
        atomicAdd(&cnt[b], 1u);
        atomicAdd(&mass[b], mass_of(v, mx));
      }
    }
    __syncwarp();
    // scan from the top bucket; lane l owns buckets 255 - 8l ... 248 - 8l
    uint32_t c8[8];
    unsigned long long m8[8];
    uint32_t cl = 0u;
    unsigned long long ml = 0ull;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int b = kBins - 1 - 8 * lane - e;
      c8[e] = cnt[b];
      m8[e] = mass[b];
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
    if (level == 0) {
      // integer sums reach tau * total exactly when they reach its ceiling
      const unsigned long long ztot = __shfl_sync(0xffffffffu, mi, 31);
      const double tq = ceil(tau * (double)ztot);
      target = tq >= (double)ztot ? ztot : (unsigned long long)tq;
    }
    uint32_t c_run = above + ci - cl;
    unsigned long long m_run = above_m + mi - ml;
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
    // the members' totals meet both conditions, so some lane hits
    const uint32_t hits = __ballot_sync(0xffffffffu, hit >= 0);
    const int src = hits ? __ffs(hits) - 1 : 31;
    const int bstar = __shfl_sync(0xffffffffu, kBins - 1 - 8 * lane - (hit < 0 ? 7 : hit), src);
    above = __shfl_sync(0xffffffffu, hit_cb, src);
    above_m = __shfl_sync(0xffffffffu, hit_mb, src);
    const uint32_t L = __shfl_sync(0xffffffffu, hit_c, src);
    // buckets above the crossing one are kept; the crossing bucket's blocks stay undecided
    uint32_t nc = 0u, kmin = 0xffffffffu, kmax = 0u;
    float vmin = INFINITY, vmax = -INFINITY;
    for (int t0 = 0; t0 < nb; t0 += 32) {
      const int t = t0 + lane;
      int b = -1;
      float v = 0.f;
      if (t < nb && ((mem[t0 >> 5] >> lane) & 1u)) {
        v = sv[t];
        b = bucket_of(v, lo, scale);
      }
      const uint32_t up = __ballot_sync(0xffffffffu, b > bstar);
      const uint32_t in = __ballot_sync(0xffffffffu, b == bstar);
      if (lane == 0) {
        kept[t0 >> 5] |= up;
        mem[t0 >> 5] = in;
      }
      if (b == bstar) {
        const uint32_t pos = nc + __popc(in & ((1u << lane) - 1u));
        if (pos < (uint32_t)kCandCap) cand[pos] = (uint16_t)t;
        const uint32_t key = order_bits(v);
        kmin = min(kmin, key);
        kmax = max(kmax, key);
        vmin = fminf(vmin, v);
        vmax = fmaxf(vmax, v);
      }
      nc += __popc(in);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
      vmin = fminf(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
      vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    }
    __syncwarp();
    if (kmin == kmax) {
      // one score value: the order is the index order and every mass is equal; keep the
      // first `take` undecided blocks by index
      int first = -1;
      for (int w = 0; w < nw && first < 0; ++w)
        if (mem[w]) first = 32 * w + __ffs(mem[w]) - 1;
      const unsigned long long qv = mass_of(sv[first], mx);
      const uint32_t tk = kneed > above ? kneed - above : 0u;
      uint32_t tm = 0u;
      if (above_m < target) tm = qv > 0ull ? (uint32_t)min((unsigned long long)L, (target - above_m + qv - 1ull) / qv) : L;
      const uint32_t take = min(L, max(tk, tm));
      uint32_t run = 0u;
      for (int w0 = 0; w0 < nw; w0 += 32) {
        const int w = w0 + lane;
        const uint32_t bits = w < nw ? mem[w] : 0u;
        const uint32_t c = __popc(bits);
        uint32_t pre = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, pre, o);
          if (lane >= o) pre += y;
        }
        uint32_t before = run + pre - c;  // undecided blocks in earlier words
        uint32_t keep = 0u, rest = bits;
        while (rest && before < take) {
          const uint32_t low = rest & (~rest + 1u);
          keep |= low;
          rest ^= low;
          ++before;
        }
        if (w < nw) kept[w] |= keep;
        run += __shfl_sync(0xffffffffu, pre, 31);
      }
      done = true;
    } else if (L <= (uint32_t)kCandCap) {
      // rank r of a candidate = candidates before it in (score desc, index asc) order;
      // keep the first `best` for the smallest best that completes both conditions.
      // The histogram is spent: it holds the candidates' order keys and masses, computed
      // once; candidates are in index order, so "index before" is "position before".
      uint32_t* ckey = cnt;
      unsigned long long* cmass = mass;
      for (uint32_t c = lane; c < L; c += 32) {
        const float v = sv[cand[c]];
        ckey[c] = order_bits(v);
        cmass[c] = mass_of(v, mx);
      }
      __syncwarp();
      uint32_t best = L;
      for (uint32_t c0 = 0; c0 < L; c0 += 32) {
        const uint32_t c = c0 + lane;
        uint32_t take = 0xffffffffu;
        if (c < L) {
          const uint32_t key = ckey[c];
          uint32_t rank = 0u;
          unsigned long long pre = 0ull;
          for (uint32_t dd = 0; dd < L; ++dd) {
            const uint32_t kd = ckey[dd];
            if (kd > key || (kd == key && dd < c)) {
              ++rank;
              pre += cmass[dd];
            }
          }
          if (above + rank + 1u >= kneed && above_m + pre + cmass[c] >= target) take = rank + 1u;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) take = min(take, __shfl_xor_sync(0xffffffffu, take, o));
        best = min(best, take);
      }
      for (uint32_t c0 = 0; c0 < L; c0 += 32) {
        const uint32_t c = c0 + lane;
        bool k = false;
        int ti = 0;
        if (c < L) {
          ti = cand[c];
          const uint32_t key = ckey[c];
          uint32_t rank = 0u;
          for (uint32_t dd = 0; dd < L; ++dd) {
            const uint32_t kd = ckey[dd];
            rank += (kd > key || (kd == key && dd < c)) ? 1u : 0u;
          }
          k = rank < best;
        }
        if (k) atomicOr(&kept[ti >> 5], 1u << (ti & 31));
      }
      done = true;
    } else {
      lo = vmin;  // narrow to the crossing bucket's own value range
      hi = vmax;
    }
    __syncwarp();
  }
  if (!done) {
    // not reached in practice (each level narrows the range 256-fold); rank the
    // undecided blocks against each other by scanning the row
    for (int t = lane; t < nb; t += 32) {
      if (!((mem[t >> 5] >> (t & 31)) & 1u)) continue;
      const uint32_t key = order_bits(sv[t]);
      uint32_t rank = 0u;
      unsigned long long pre = 0ull;
      for (int u = 0; u < nb; ++u) {
        if (!((mem[u >> 5] >> (u & 31)) & 1u)) continue;
        const uint32_t ku = order_bits(sv[u]);
        if (ku > key || (ku == key && u < t)) {
          ++rank;
          pre += mass_of(sv[u], mx);
        }
      }
      // kept iff the prefix before it still misses a condition
      if (above + rank < kneed || above_m + pre < target) atomicOr(&kept[t >> 5], 1u << (t & 31));
    }
    __syncwarp();
  }
  __syncwarp();
  return 0;
}

template <int R>
__global__ void __launch_bounds__(32 * R, 2) score_select_kernel(const float* __restrict__ qbar,
                                                              const float* __restrict__ kbar, int nb, int d,
                                                              float scale, int k_top, double tau,
                                                              int32_t* __restrict__ counts,
                                                              int32_t* __restrict__ idx) {
  constexpr int kThreads = 32 * R;
  extern __shared__ __align__(16) uint8_t smem[];
  const int h = blockIdx.y, i0 = blockIdx.x * R;
  const int nbs = (nb + 3) & ~3;
  float* qt = reinterpret_cast<float*>(smem);          // [d][R]
  float* S = qt + (size_t)d * R;                       // [R][nbs]
  uint8_t* uni = reinterpret_cast<uint8_t*>(S + (size_t)R * nbs);  // staging, then selection state
  float* kt = reinterpret_cast<float*>(uni);           // [2][kSsSlice][kSsKeys]
  const int tid = threadIdx.x;
  const float* A = qbar + (size_t)h * nb * d;
  const float* Bm = kbar + (size_t)h * nb * d;
  for (int e = tid; e < R * d; e += kThreads) {
    const int r = e / d, c = e - r * d;
    qt[c * R + r] = (i0 + r < nb) ? A[(size_t)(i0 + r) * d + c] : 0.f;
  }
  // ------------------------------------------------------------ score rows
  const int rg = tid >> 7;  // rows 4rg .. 4rg + 3
  const int kg = tid & 127; // keys 4kg .. 4kg + 3 of the tile
  constexpr int kPer = kSsKeys / kThreads;  // keys each thread stages per slice
  const int ns = d / kSsSlice;
  for (int k0 = 0; k0 < nb; k0 += kSsKeys) {
    float4 st[kPer][2];
    auto load = [&](int s) {
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int j = k0 + tid + u * kThreads;
        if (j < nb) {
          const float4* src = reinterpret_cast<const float4*>(Bm + (size_t)j * d + s * kSsSlice);
          st[u][0] = __ldg(src);
          st[u][1] = __ldg(src + 1);
        } else {
          st[u][0] = st[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    };
    auto store = [&](int buf) {
      float* dst = kt + (size_t)buf * kSsSlice * kSsKeys;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int jj = tid + u * kThreads;
        dst[0 * kSsKeys + jj] = st[u][0].x;
        dst[1 * kSsKeys + jj] = st[u][0].y;
        dst[2 * kSsKeys + jj] = st[u][0].z;
        dst[3 * kSsKeys + jj] = st[u][0].w;
        dst[4 * kSsKeys + jj] = st[u][1].x;
        dst[5 * kSsKeys + jj] = st[u][1].y;
        dst[6 * kSsKeys + jj] = st[u][1].z;
        dst[7 * kSsKeys + jj] = st[u][1].w;
      }
    };
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
    __syncthreads();  // qt written; the previous tile's readers of kt are done
    load(0);
    store(0);
    __syncthreads();
    for (int s = 0; s < ns; ++s) {
      const int buf = s & 1;
      if (s + 1 < ns) load(s + 1);
      const float* kb = kt + (size_t)buf * kSsSlice * kSsKeys;
#pragma unroll
      for (int dd = 0; dd < kSsSlice; ++dd) {
        const float4 a = *reinterpret_cast<const float4*>(qt + (size_t)(s * kSsSlice + dd) * R + 4 * rg);
        const float4 b = *reinterpret_cast<const float4*>(kb + dd * kSsKeys + 4 * kg);
        const float av[4] = {a.x, a.y, a.z, a.w};
        const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
      }
      if (s + 1 < ns) store(buf ^ 1);
      __syncthreads();
    }
    const int j0 = k0 + 4 * kg;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float* row = S + (size_t)(4 * rg + r) * nbs;
      if (j0 + 4 <= nb) {
        *reinterpret_cast<float4*>(row + j0) =
            make_float4(acc[r][0] * scale, acc[r][1] * scale, acc[r][2] * scale, acc[r][3] * scale);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (j0 + c < nb) row[j0 + c] = acc[r][c] * scale;
      }
    }
  }
  __syncthreads();  // score rows complete; the staging area becomes selection state
  // ------------------------------------------------------------- selection
  const int warp = tid >> 5, lane = tid & 31;
  const int i = i0 + warp;
  if (i >= nb) return;  // whole warp; nothing below synchronises across warps
  uint8_t* state = uni + (size_t)warp * sel_bytes(nb);
  const float* sv = S + (size_t)warp * nbs;
  select_row(sv, nb, k_top, tau, state);
  // ascending output from the kept bits
  const int nw = (nb + 31) / 32;
  const uint32_t* kept = reinterpret_cast<const uint32_t*>(state + kBins * 12 + kCandCap * 2) + nw;
  int32_t* out = idx + ((size_t)h * nb + i) * nb;
  uint32_t n = 0u;
  for (int t0 = 0; t0 < nb; t0 += 32) {
    const uint32_t bits = kept[t0 >> 5];
    if ((bits >> lane) & 1u) out[n + __popc(bits & ((1u << lane) - 1u))] = t0 + lane;
    n += __popc(bits);
  }
  if (lane == 0) counts[(size_t)h * nb + i] = (int32_t)n;
}

template <int R>
size_t score_select_smem(int nb, int d) {
  const size_t nbs = (size_t)((nb + 3) & ~3);
  const size_t stage = (size_t)2 * kSsSlice * kSsKeys * 4;
  return (size_t)d * R * 4 + (size_t)R * nbs * 4 + std::max(stage, (size_t)R * sel_bytes(nb));
}

}  // namespace

bool score_select_supported(int nb, int d) {
  return d % kSsSlice == 0 && d <= 256 && nb >= 1 && nb <= 4096 && score_select_smem<8>(nb, d) <= 232448;
}

cudaError_t score_select_launch(const float* qbar, const float* kbar, int Hh, int nb, int d, int k_top, double tau,
                                int32_t* counts, int32_t* idx, cudaStream_t st) {
  const float scale = 1.0f / sqrtf((float)d);
  cudaError_t e;
  const size_t s16 = score_select_smem<16>(nb, d);
  // 16-row CTAs while two of them fit on an SM, else 8-row CTAs (two or more per SM):
  // one CTA's selection then overlaps another's score rows
  if (2 * (s16 + 1024) <= 233472) {
    if ((e = cudaFuncSetAttribute(score_select_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s16)) !=
        cudaSuccess)
      return e;
    HookScope hs("score_select", st);
    score_select_kernel<16><<<dim3((nb + 15) / 16, Hh), 512, s16, st>>>(qbar, kbar, nb, d, scale, k_top, tau, counts,
                                                                         idx);
  } else {
    const size_t s8 = score_select_smem<8>(nb, d);
    if ((e = cudaFuncSetAttribute(score_select_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s8)) !=
        cudaSuccess)
      return e;
    HookScope hs("score_select", st);
    score_select_kernel<8><<<dim3((nb + 7) / 8, Hh), 256, s8, st>>>(qbar, kbar, nb, d, scale, k_top, tau, counts, idx);
  }
  return cudaGetLastError();
}

}  // namespace prism
