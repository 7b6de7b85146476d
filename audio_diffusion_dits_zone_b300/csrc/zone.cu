// Step 1 of the path: per-macro-zone block shape and the block-order permutation.
//
// "Prism: dynamic sparse attention for 2K joint video-audio generation training",
// section "Region-adapted block construction", paragraph 1: per macro-zone, the
// channel-wise variance of the video features (how fast, and along which axis,
// the content changes) and the audio-to-video cross-attention feature norm (how
// strongly audio drives the region) decide the block shape; axes of fast change or
// strong coupling are split more finely.
//
// Readings (the page gives no formula): v_a = mean over channels and over the
// zone's lines along axis a of the population variance along the line; u_a = the
// same for the A2V field; w = zone mean A2V / largest zone mean;
// S_a = v_a / sum v + w u_a / sum u; shape = argmin sum_a S_a log2 e_a (first on
// ties).  Block order: zones raster, tiles of the zone's shape in tile-raster order
// clipped at the zone edge, tokens raster inside a tile.
//
// Kernels (all HBM-bound or tiny):
//   zone_tma       (bf16 features, zones up to 3 x 9 in t x h) persistent CTAs of 8
//                  warps; each warp streams its own (zone, 64-channel) items as slabs of
//                  2 w columns: one 4D TMA box [t][h][w][64 channels] per slab into a
//                  four-stage shared-memory ring, so three slabs are in flight while one
//                  is reduced (lane = 2 channels on packed fp32 pairs, all line sums in
//                  registers, same arithmetic as zone_lines);
//   zone_lines     (zones up to 3 x 9 or 5 x 8 in t x h, even channel counts) one warp
//                  per (zone, 64 channels), lane = 2 channels, so every load is one
//                  128-byte run of a token row.  The warp streams the zone once,
//                  w outermost, t innermost, keeping every line sum in registers:
//                  per channel sum_lines (x - line mean)^2 = sum x^2 - sum_lines
//                  (line sum)^2 / L, with x taken relative to the zone's first token
//                  (a shift leaves every line variance unchanged and keeps the two
//                  terms small);
//   zone_partial   (any other zone) one CTA per (zone, channel chunk): the chunk is
//                  staged in shared memory and the two-pass line variances are
//                  summed for the three axes;
//   zone_finalize  one CTA per zone: fixed-order sum over chunks, A2V statistics;
//   zone_choose    one CTA: largest zone mean, per-zone scores, fp32 costs, argmin;
//   zone_perm      one thread per token: closed-form block-order position.
#include <algorithm>
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

constexpr int kZoneThreads = 256;
constexpr int kSmemBudget = 200 * 1024;

struct ZoneBox {
  int t0, h0, w0, Lt, Lh, Lw;
};

__device__ __forceinline__ ZoneBox zone_box(const ZoneGeom& g, int z) {
  ZoneBox b;
  const int zt = z / (g.nzh * g.nzw);
  const int rem = z - zt * g.nzh * g.nzw;
  const int zh = rem / g.nzw;
  const int zw = rem - zh * g.nzw;
  b.t0 = zt * g.zt;
  b.h0 = zh * g.zh;
  b.w0 = zw * g.zw;
  b.Lt = min(g.zt, g.T - b.t0);
  b.Lh = min(g.zh, g.H - b.h0);
  b.Lw = min(g.zw, g.W - b.w0);
  return b;
}

// Line geometry for axis a of a zone: number of lines, line length, first token
// of line `line` and the token stride along the line (local token p = (lt*Lh+lh)*Lw+lw).
__device__ __forceinline__ void line_of(const ZoneBox& b, int a, int line, int& p0, int& sp) {
  if (a == 0) {
    const int lh = line / b.Lw, lw = line - (line / b.Lw) * b.Lw;
    p0 = lh * b.Lw + lw;
    sp = b.Lh * b.Lw;
  } else if (a == 1) {
    const int lt = line / b.Lw, lw = line - (line / b.Lw) * b.Lw;
    p0 = lt * b.Lh * b.Lw + lw;
    sp = b.Lw;
  } else {
    const int lt = line / b.Lh, lh = line - (line / b.Lh) * b.Lh;
    p0 = (lt * b.Lh + lh) * b.Lw;
    sp = 1;
  }
}
__device__ __forceinline__ int nlines_of(const ZoneBox& b, int a) {
  return a == 0 ? b.Lh * b.Lw : (a == 1 ? b.Lt * b.Lw : b.Lt * b.Lh);
}
__device__ __forceinline__ int len_of(const ZoneBox& b, int a) { return a == 0 ? b.Lt : (a == 1 ? b.Lh : b.Lw); }

// Block-wide sums of three values; every thread receives the three totals.
// red must hold NW * 3 + 3 floats.  Fixed reduction order (deterministic).
template <int NW>
__device__ __forceinline__ void block_sum3(float (&acc)[3], float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    float v = acc[a];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp * 3 + a] = v;
  }
  __syncthreads();
  if (threadIdx.x < 3) {
    float s = 0.f;
    for (int w = 0; w < NW; ++w) s += red[w * 3 + threadIdx.x];
    red[NW * 3 + threadIdx.x] = s;
  }
  __syncthreads();
#pragma unroll
  for (int a = 0; a < 3; ++a) acc[a] = red[NW * 3 + a];
  __syncthreads();
}

// Sum over the chunk's channels and the zone's lines of sum_x (x - line mean)^2,
// for each axis.  part[(z * nchunks + chunk) * 3 + a].
template <typename T, int VW>
__global__ void __launch_bounds__(kZoneThreads) zone_partial_kernel(const T* __restrict__ feat, int64_t ld, int C,
                                                                    ZoneGeom g, int CH, float* __restrict__ part) {
  extern __shared__ __align__(16) float xs[];  // [tokens][CH] fp32
  __shared__ float red[(kZoneThreads / 32) * 3 + 3];
  const int z = blockIdx.x, chunk = blockIdx.y, nchunks = gridDim.y;
  const int c0 = chunk * CH;
  const ZoneBox b = zone_box(g, z);
  const int ntok = b.Lt * b.Lh * b.Lw;
  const int nch = min(CH, C - c0);

  if (VW > 1 && nch == CH) {
    const int vpr = CH / VW;  // vectors per token row
    for (int e = threadIdx.x; e < ntok * vpr; e += kZoneThreads) {
      const int p = e / vpr, q = e - (e / vpr) * vpr;
      const int lt = p / (b.Lh * b.Lw), rem = p - lt * b.Lh * b.Lw, lh = rem / b.Lw, lw = rem - lh * b.Lw;
      const int64_t n = ((int64_t)(b.t0 + lt) * g.H + (b.h0 + lh)) * g.W + (b.w0 + lw);
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(feat + n * ld + c0 + q * VW));
      float* dst = xs + p * CH + q * VW;
      if constexpr (sizeof(T) == 2) {
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(h2[k]);
          dst[2 * k] = f.x;
          dst[2 * k + 1] = f.y;
        }
      } else {
        const float* f = reinterpret_cast<const float*>(&raw);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = f[k];
      }
    }
  } else {
    for (int e = threadIdx.x; e < ntok * CH; e += kZoneThreads) {
      const int p = e / CH, c = e - (e / CH) * CH;
      const int lt = p / (b.Lh * b.Lw), rem = p - lt * b.Lh * b.Lw, lh = rem / b.Lw, lw = rem - lh * b.Lw;
      const int64_t n = ((int64_t)(b.t0 + lt) * g.H + (b.h0 + lh)) * g.W + (b.w0 + lw);
      xs[p * CH + c] = c < nch ? to_f32<T>(feat[n * ld + c0 + c]) : 0.f;
    }
  }
  __syncthreads();

  float acc[3] = {0.f, 0.f, 0.f};
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    const int L = len_of(b, a);
    if (L < 2) continue;
    const float inv_L = 1.f / (float)L;
    const int items = nlines_of(b, a) * CH;
    for (int e = threadIdx.x; e < items; e += kZoneThreads) {
      const int line = e / CH, c = e - (e / CH) * CH;
      int p0, sp;
      line_of(b, a, line, p0, sp);
      const float* x = xs + p0 * CH + c;
      float s = 0.f;
      for (int k = 0; k < L; ++k) s += x[k * sp * CH];
      const float mu = s * inv_L;
      float ss = 0.f;
      for (int k = 0; k < L; ++k) {
        const float dlt = x[k * sp * CH] - mu;
        ss = fmaf(dlt, dlt, ss);
      }
      acc[a] += ss;
    }
  }
  block_sum3<kZoneThreads / 32>(acc, red);
  if (threadIdx.x < 3) part[((size_t)z * nchunks + chunk) * 3 + threadIdx.x] = acc[threadIdx.x];
}

// Two consecutive channels of one token as fp32.
template <typename T>
__device__ __forceinline__ float2 load_pair(const T* p);
template <>
__device__ __forceinline__ float2 load_pair<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 load_pair<float>(const float* p) {
  return __ldg(reinterpret_cast<const float2*>(p));
}

constexpr int kLinesWarps = 8;
constexpr int kLinesChannels = 64;  // per warp

// part[(z * nchunks + chunk) * 3 + a] = sum over the chunk's channels and the zone's
// lines along axis a of sum_x (x - line mean)^2; chunk = 64 channels.
template <typename T, int MT, int MH>
__global__ void __launch_bounds__(kLinesWarps * 32) zone_lines_kernel(const T* __restrict__ feat, int64_t ld, int C,
                                                                      ZoneGeom g, int nchunks,
                                                                      float* __restrict__ part) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * kLinesWarps + warp;
  const int z = blockIdx.y;
  if (chunk >= nchunks) return;  // warp-uniform; no block-wide synchronisation below
  const ZoneBox b = zone_box(g, z);
  const int c = chunk * kLinesChannels + 2 * lane;
  const bool act = c < C;  // C is even: both channels of the pair exist
  const int64_t st = (int64_t)g.H * g.W * ld, sh = (int64_t)g.W * ld;
  const T* zp = feat + (((int64_t)b.t0 * g.H + b.h0) * g.W + b.w0) * ld + (act ? c : 0);
  const float2 x0 = load_pair<T>(zp);
  float wsum[MT][MH][2];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int h = 0; h < MH; ++h) wsum[t][h][0] = wsum[t][h][1] = 0.f;
  float sq[2] = {0.f, 0.f}, bt[2] = {0.f, 0.f}, bh[2] = {0.f, 0.f};
  for (int w = 0; w < b.Lw; ++w) {
    const T* pw = zp + (int64_t)w * ld;
    float hs[MT][2];
#pragma unroll
    for (int t = 0; t < MT; ++t) hs[t][0] = hs[t][1] = 0.f;
#pragma unroll
    for (int h = 0; h < MH; ++h) {
      if (h < b.Lh) {
        float ts[2] = {0.f, 0.f};
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          if (t < b.Lt) {
            float2 x = load_pair<T>(pw + h * sh + t * st);
            x.x -= x0.x;
            x.y -= x0.y;
            ts[0] += x.x;
            ts[1] += x.y;
            hs[t][0] += x.x;
            hs[t][1] += x.y;
            wsum[t][h][0] += x.x;
            wsum[t][h][1] += x.y;
            sq[0] = fmaf(x.x, x.x, sq[0]);
            sq[1] = fmaf(x.y, x.y, sq[1]);
          }
        }
        bt[0] = fmaf(ts[0], ts[0], bt[0]);  // t-line (h, w)
        bt[1] = fmaf(ts[1], ts[1], bt[1]);
      }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) {  // h-lines (t, w)
      bh[0] = fmaf(hs[t][0], hs[t][0], bh[0]);
      bh[1] = fmaf(hs[t][1], hs[t][1], bh[1]);
    }
  }
  float bw[2] = {0.f, 0.f};
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int h = 0; h < MH; ++h) {  // w-lines (t, h); unused slots hold 0
      bw[0] = fmaf(wsum[t][h][0], wsum[t][h][0], bw[0]);
      bw[1] = fmaf(wsum[t][h][1], wsum[t][h][1], bw[1]);
    }
  float ss[3] = {0.f, 0.f, 0.f};
  if (act) {
    const float* bl[3] = {bt, bh, bw};
    const int L[3] = {b.Lt, b.Lh, b.Lw};
#pragma unroll
    for (int a = 0; a < 3; ++a)
      if (L[a] > 1) {
        const float inv = 1.f / (float)L[a];
        ss[a] = fmaxf(sq[0] - bl[a][0] * inv, 0.f) + fmaxf(sq[1] - bl[a][1] * inv, 0.f);
      }
  }
#pragma unroll
  for (int a = 0; a < 3; ++a)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss[a] += __shfl_xor_sync(0xffffffffu, ss[a], o);
  if (lane < 3) part[((size_t)z * nchunks + chunk) * 3 + lane] = lane == 0 ? ss[0] : (lane == 1 ? ss[1] : ss[2]);
}

constexpr int kTmaWarps = 8;
constexpr int kSlabCh = 64;     // channels per slab: one 128-byte run of each token row, two per lane
constexpr int kWq = 4;          // w columns per slab (a quarter of a 16-wide zone)
constexpr int kTmaStages = 2;   // per warp: one slab in flight behind the one being reduced
constexpr int kTmaMT = 3, kTmaMH = 9;  // slab extent along t and h (zones up to 3 x 9 in t x h)
constexpr int kSlabBytes = kTmaMT * kTmaMH * kWq * kSlabCh * 2;  // 13,824 bytes

struct ZoneTmaSmem {
  uint8_t slab[kTmaWarps][kTmaStages][kSlabBytes];
  uint64_t full[kTmaWarps][kTmaStages];
};

// One slab [MT][MH][kWq][64 channels] bf16 of one (zone, 64 channels) item: accumulate,
// for this lane's channel pair, the shifted values v = x - x0 into the line sums along
// t (squared into bt per (h, w)), along h (squared into bh per (t, w)), along w (kept in
// wsum[t][h] across the item's slabs) and their squares (sq, one chain per t).
// CLIP: positions outside the zone (t >= Lt, h >= Lh, column >= wlim) count as 0.
template <int MT, int MH, bool CLIP>
__device__ __forceinline__ void zone_slab_sums(const uint8_t* slab, int lane, f2 nx0, int Lt, int Lh, int wlim,
                                               f2 (&wsum)[MT][MH], f2 (&sq)[MT], f2& bt, f2& bh) {
  const uint32_t* base = reinterpret_cast<const uint32_t*>(slab) + lane;
  const f2 zero{0ull};
#pragma unroll 1
  for (int w = 0; w < kWq; ++w) {
    f2 hs[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) hs[t] = zero;
#pragma unroll
    for (int h = 0; h < MH; ++h) {
      f2 ts = zero;
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const uint32_t raw = base[((t * MH + h) * kWq + w) * (kSlabCh / 2)];
        f2 v = f2_add(f2_make(__uint_as_float(raw << 16), __uint_as_float(raw & 0xffff0000u)), nx0);
        if (CLIP && !(t < Lt && h < Lh && w < wlim)) v = zero;
        ts = f2_add(ts, v);
        hs[t] = f2_add(hs[t], v);
        wsum[t][h] = f2_add(wsum[t][h], v);
        sq[t] = f2_fma(v, v, sq[t]);
      }
      bt = f2_fma(ts, ts, bt);
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) bh = f2_fma(hs[t], hs[t], bh);
  }
}

// part[(z * nchunks + chunk) * 3 + a] exactly as zone_lines_kernel (chunk = 64 channels),
// from slabs loaded with the 4D tensor map tm = feature viewed as [T][H][W][C] bf16 with
// box {64, kWq, MH, MT}.  Persistent CTAs of kTmaWarps warps; each warp streams its own
// items, up to nq slabs (kWq columns each) per item, through a kTmaStages-stage ring
// that its lane 0 refills (so the next slabs are in flight while this one is reduced).
// A zone cut short in w by the grid has only ceil(Lw / kWq) slabs (the ones wholly
// outside it are never loaded).  Slabs that lie inside the zone take the unpredicated
// path; the others (zones clipped in t or h, a last slab partly outside) mask the
// positions outside the zone, whose slab bytes are zero fill or a neighbour's tokens.
template <int MT, int MH>
__global__ void __launch_bounds__(kTmaWarps * 32, 1)
    zone_tma_kernel(const __grid_constant__ CUtensorMap tm, ZoneGeom g, int nchunks, int items, int nq,
                    float* __restrict__ part, uint32_t* status) {
  static_assert(MT * MH * kWq * kSlabCh * 2 <= kSlabBytes, "slab larger than its stage");
  extern __shared__ uint8_t smem_raw[];
  ZoneTmaSmem& sm = *reinterpret_cast<ZoneTmaSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    for (int s = 0; s < kTmaStages; ++s) mbar_init(smem_u32(&sm.full[warp][s]), 1);
    mbar_fence_init();
  }
  __syncwarp();
  // this warp's items: k = (blockIdx.x * kTmaWarps + warp) + n * stride, nq slabs each
  const int stride = gridDim.x * kTmaWarps;
  const int first = blockIdx.x * kTmaWarps + warp;
  const int nmine = first < items ? (items - first + stride - 1) / stride : 0;
  // the slabs of item n: the zone's w extent in kWq-column steps
  auto nq_of = [&](int n) {
    const ZoneBox b = zone_box(g, (first + n * stride) / nchunks);
    return min(nq, (b.Lw + kWq - 1) / kWq);
  };
  // a position in this warp's slab sequence: item n, slab q of its nqn
  struct Cursor {
    int n, q, nqn;
  };
  auto advance = [&](Cursor& c) {
    if (++c.q == c.nqn) {
      ++c.n;
      c.q = 0;
      c.nqn = c.n < nmine ? nq_of(c.n) : 0;
    }
  };
  auto issue = [&](const Cursor& c, int s) {  // the warp's slab number s -> stage s % kTmaStages
    const int k = first + c.n * stride;
    const int z = k / nchunks, chunk = k - z * nchunks;
    const ZoneBox b = zone_box(g, z);
    const uint32_t bar = smem_u32(&sm.full[warp][s % kTmaStages]);
    mbar_arrive_expect_tx(bar, (uint32_t)(MT * MH * kWq * kSlabCh * 2));
    tma_load_4d(smem_u32(sm.slab[warp][s % kTmaStages]), &tm, chunk * kSlabCh, b.w0 + c.q * kWq, b.h0, b.t0, bar);
  };
  Cursor pc{0, 0, nmine > 0 ? nq_of(0) : 0};  // lane 0: the next slab to load
  int issued = 0;                              // lane 0: slabs issued so far
  if (lane == 0) {
    tma_prefetch_desc(&tm);
    while (issued < kTmaStages && pc.n < nmine) {
      issue(pc, issued);
      ++issued;
      advance(pc);
    }
  }
  int abort = 0;
  const f2 zero{0ull};
  f2 wsum[MT][MH], sq[MT], bt = zero, bh = zero, nx0 = zero;
  Cursor cc{0, 0, nmine > 0 ? nq_of(0) : 0};  // the slab to reduce
  for (int s = 0; cc.n < nmine; ++s) {
    const int n = cc.n, q = cc.q;
    const int k = first + n * stride;
    const int z = k / nchunks, chunk = k - z * nchunks;
    const ZoneBox b = zone_box(g, z);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.full[warp][s % kTmaStages]),
                                                      (s / kTmaStages) & 1, &abort, status));
    if (!ok) break;
    const uint8_t* slab = sm.slab[warp][s % kTmaStages];
    if (q == 0) {  // new item: reset the sums; shift by the zone's first token
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        sq[t] = zero;
#pragma unroll
        for (int h = 0; h < MH; ++h) wsum[t][h] = zero;
      }
      bt = bh = zero;
      const uint32_t raw = reinterpret_cast<const uint32_t*>(slab)[lane];
      nx0 = f2_make(-__uint_as_float(raw << 16), -__uint_as_float(raw & 0xffff0000u));
    }
    const int wlim = b.Lw - q * kWq;  // columns of this slab inside the zone
    if (b.Lt == MT && b.Lh == MH && wlim >= kWq)
      zone_slab_sums<MT, MH, false>(slab, lane, nx0, MT, MH, kWq, wsum, sq, bt, bh);
    else
      zone_slab_sums<MT, MH, true>(slab, lane, nx0, b.Lt, b.Lh, wlim, wsum, sq, bt, bh);
    // every lane has read the stage: refill it with slab s + kTmaStages
    __syncwarp();
    if (lane == 0 && pc.n < nmine) {
      issue(pc, issued);
      ++issued;
      advance(pc);
    }
    if (q == cc.nqn - 1) {  // the item's last slab: one partial per (zone, 64 channels)
      f2 bw = zero;
#pragma unroll
      for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int h = 0; h < MH; ++h) bw = f2_fma(wsum[t][h], wsum[t][h], bw);
      f2 sqa = sq[0];
#pragma unroll
      for (int t = 1; t < MT; ++t) sqa = f2_add(sqa, sq[t]);
      float sqv[2], bl[3][2];
      f2_split(sqa, sqv[0], sqv[1]);
      f2_split(bt, bl[0][0], bl[0][1]);
      f2_split(bh, bl[1][0], bl[1][1]);
      f2_split(bw, bl[2][0], bl[2][1]);
      const int L[3] = {b.Lt, b.Lh, b.Lw};
      float ss[3] = {0.f, 0.f, 0.f};
#pragma unroll
      for (int a = 0; a < 3; ++a)
        if (L[a] > 1) {
          const float inv = 1.f / (float)L[a];
          ss[a] = fmaxf(sqv[0] - bl[a][0] * inv, 0.f) + fmaxf(sqv[1] - bl[a][1] * inv, 0.f);
        }
#pragma unroll
      for (int a = 0; a < 3; ++a)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss[a] += __shfl_xor_sync(0xffffffffu, ss[a], o);
      if (lane < 3) part[((size_t)z * nchunks + chunk) * 3 + lane] = lane == 0 ? ss[0] : (lane == 1 ? ss[1] : ss[2]);
    }
    advance(cc);
  }
  // a warp that gave up waits (bounded) for the copies it still has in flight: the
  // last slab issued into each stage completes that stage's phase (slab / stages) & 1
  if (abort && lane == 0)
    for (int s = issued - 1; s >= 0 && s >= issued - kTmaStages; --s)
      drain_wait(smem_u32(&sm.full[warp][s % kTmaStages]), (s / kTmaStages) & 1);
}

// stats[z * 8 + {0,1,2}] = v_a, {3,4,5} = u_a, 6 = zone mean of a2v.  The video term is
// the sum, in order c = 0 .. nparts - 1, of the partial sums part[z * zs + c * cs + a]
// (per-chunk partials of one call: zs = nparts * 3, cs = 3; partials of several
// channel slices gathered as [nparts][Z][3]: zs = 3, cs = Z * 3), over C channels.
__global__ void __launch_bounds__(kZoneThreads) zone_finalize_kernel(const float* __restrict__ part, int nparts,
                                                                     int zs, int cs, const float* __restrict__ a2v,
                                                                     ZoneGeom g, int C, float* __restrict__ stats) {
  extern __shared__ float as[];  // zone's a2v values
  __shared__ float red[(kZoneThreads / 32) * 3 + 3];
  const int z = blockIdx.x;
  const ZoneBox b = zone_box(g, z);
  const int ntok = b.Lt * b.Lh * b.Lw;
  for (int p = threadIdx.x; p < ntok; p += kZoneThreads) {
    const int lt = p / (b.Lh * b.Lw), rem = p - lt * b.Lh * b.Lw, lh = rem / b.Lw, lw = rem - lh * b.Lw;
    as[p] = a2v[((int64_t)(b.t0 + lt) * g.H + (b.h0 + lh)) * g.W + (b.w0 + lw)];
  }
  __syncthreads();
  float acc[3] = {0.f, 0.f, 0.f};
  for (int a = 0; a < 3; ++a) {
    const int L = len_of(b, a);
    if (L < 2) continue;
    const float inv_L = 1.f / (float)L;
    for (int line = threadIdx.x; line < nlines_of(b, a); line += kZoneThreads) {
      int p0, sp;
      line_of(b, a, line, p0, sp);
      float s = 0.f;
      for (int k = 0; k < L; ++k) s += as[p0 + k * sp];
      const float mu = s * inv_L;
      float ss = 0.f;
      for (int k = 0; k < L; ++k) {
        const float dlt = as[p0 + k * sp] - mu;
        ss = fmaf(dlt, dlt, ss);
      }
      acc[a] += ss;
    }
  }
  block_sum3<kZoneThreads / 32>(acc, red);
  float u[3] = {acc[0], acc[1], acc[2]};
  float m[3] = {0.f, 0.f, 0.f};
  for (int p = threadIdx.x; p < ntok; p += kZoneThreads) m[0] += as[p];
  block_sum3<kZoneThreads / 32>(m, red);
  if (threadIdx.x == 0) {
    const float inv_tok = 1.f / (float)ntok;
    for (int a = 0; a < 3; ++a) {
      float s = 0.f;
      for (int c = 0; c < nparts; ++c) s += part[(size_t)z * zs + (size_t)c * cs + a];
      stats[z * 8 + a] = s / ((float)C * (float)ntok);
      stats[z * 8 + 3 + a] = u[a] * inv_tok;
    }
    stats[z * 8 + 6] = m[0] * inv_tok;
    stats[z * 8 + 7] = 0.f;
  }
}

// out[z][a] = sum over chunks c (in order) of part[z][c][a].
__global__ void zone_sum_chunks_kernel(const float* __restrict__ part, int nchunks, int Z, float* __restrict__ out) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= Z * 3) return;
  const int z = t / 3, a = t - z * 3;
  float s = 0.f;
  for (int c = 0; c < nchunks; ++c) s += part[((size_t)z * nchunks + c) * 3 + a];
  out[t] = s;
}

__global__ void __launch_bounds__(1024) zone_choose_kernel(const float* __restrict__ stats, int Z, ShapeSet shapes,
                                                           int32_t* __restrict__ zone_shape) {
  __shared__ float red[32];
  float mx = 0.f;
  for (int z = threadIdx.x; z < Z; z += blockDim.x) mx = fmaxf(mx, stats[z * 8 + 6]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
    red[0] = m;
  }
  __syncthreads();
  const float amax = red[0];
  float lg[8][3];
  for (int s = 0; s < shapes.n; ++s)
    for (int a = 0; a < 3; ++a) lg[s][a] = log2f((float)shapes.e[s][a]);
  for (int z = threadIdx.x; z < Z; z += blockDim.x) {
    const float* st = stats + z * 8;
    const float vs = st[0] + st[1] + st[2];
    const float us = st[3] + st[4] + st[5];
    const float w = amax > 0.f ? st[6] / amax : 0.f;
    float S[3];
    for (int a = 0; a < 3; ++a) S[a] = (vs > 0.f ? st[a] / vs : 0.f) + w * (us > 0.f ? st[3 + a] / us : 0.f);
    int best = 0;
    float bc = 0.f;
    for (int s = 0; s < shapes.n; ++s) {
      const float c = S[0] * lg[s][0] + S[1] * lg[s][1] + S[2] * lg[s][2];
      if (s == 0 || c < bc) {
        bc = c;
        best = s;
      }
    }
    zone_shape[z] = best;
  }
}

__global__ void zone_perm_kernel(ZoneGeom g, const int32_t* __restrict__ zone_shape, ShapeSet shapes,
                                 int32_t* __restrict__ perm) {
  const int64_t N = (int64_t)g.T * g.H * g.W;
  for (int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; n < N; n += (int64_t)gridDim.x * blockDim.x) {
    const int w = (int)(n % g.W);
    const int h = (int)((n / g.W) % g.H);
    const int t = (int)(n / ((int64_t)g.W * g.H));
    const int zi_t = t / g.zt, zi_h = h / g.zh, zi_w = w / g.zw;
    const int z = (zi_t * g.nzh + zi_h) * g.nzw + zi_w;
    const int Lt = min(g.zt, g.T - zi_t * g.zt), Lh = min(g.zh, g.H - zi_h * g.zh), Lw = min(g.zw, g.W - zi_w * g.zw);
    // tokens of all zones before z in raster order (clipping is separable per axis)
    const int64_t zone_off = (int64_t)zi_t * g.zt * g.H * g.W + (int64_t)Lt * zi_h * g.zh * g.W +
                             (int64_t)Lt * Lh * zi_w * g.zw;
    const int s = zone_shape[z];
    const int et = shapes.e[s][0], eh = shapes.e[s][1], ew = shapes.e[s][2];
    const int lt = t - zi_t * g.zt, lh = h - zi_h * g.zh, lw = w - zi_w * g.zw;
    const int tt = lt / et, th = lh / eh, tw = lw / ew;
    const int Et = min(et, Lt - tt * et), Eh = min(eh, Lh - th * eh), Ew = min(ew, Lw - tw * ew);
    const int64_t tile_off = (int64_t)tt * et * Lh * Lw + (int64_t)Et * th * eh * Lw + (int64_t)Et * Eh * tw * ew;
    const int within = ((lt - tt * et) * Eh + (lh - th * eh)) * Ew + (lw - tw * ew);
    perm[zone_off + tile_off + within] = (int32_t)n;
  }
}

// Zone-chunked blocks: every zone's run of the block order cut into B-token blocks of
// its own (the last one short).  One CTA: the blocks of each zone (ceil(tokens / B)),
// their exclusive prefix over the zones in order (first[z]) and every block's length.
__global__ void __launch_bounds__(1024) zone_chunk_blocks_kernel(ZoneGeom g, int B, int32_t* __restrict__ first,
                                                                 int32_t* __restrict__ blen) {
  __shared__ int32_t wsum[32];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int z0 = 0; z0 < g.Z; z0 += blockDim.x) {
    const int z = z0 + threadIdx.x;
    int n = 0, nblk = 0;
    if (z < g.Z) {
      const ZoneBox b = zone_box(g, z);
      n = b.Lt * b.Lh * b.Lw;
      nblk = (n + B - 1) / B;
    }
    int incl = nblk;  // inclusive scan of the CTA's zones
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = carry;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    const int f = before + incl - nblk;
    if (z < g.Z) {
      first[z] = f;
      for (int m = 0; m < nblk; ++m) blen[f + m] = min(B, n - m * B);
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = before + incl;
    __syncthreads();
  }
}

__global__ void fill_i32_kernel(int32_t* __restrict__ p, int64_t n, int32_t v) {
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) p[e] = v;
}

// perm_padded[first[z] * B + position of the token in its zone] = raster token; the
// in-zone position is the consecutive-chunk layout's (zone_perm_kernel).
__global__ void zone_perm_chunked_kernel(ZoneGeom g, const int32_t* __restrict__ zone_shape, ShapeSet shapes, int B,
                                         const int32_t* __restrict__ first, int32_t* __restrict__ perm) {
  const int64_t N = (int64_t)g.T * g.H * g.W;
  for (int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; n < N; n += (int64_t)gridDim.x * blockDim.x) {
    const int w = (int)(n % g.W);
    const int h = (int)((n / g.W) % g.H);
    const int t = (int)(n / ((int64_t)g.W * g.H));
    const int zi_t = t / g.zt, zi_h = h / g.zh, zi_w = w / g.zw;
    const int z = (zi_t * g.nzh + zi_h) * g.nzw + zi_w;
    const int Lt = min(g.zt, g.T - zi_t * g.zt), Lh = min(g.zh, g.H - zi_h * g.zh), Lw = min(g.zw, g.W - zi_w * g.zw);
    const int s = zone_shape[z];
    const int et = shapes.e[s][0], eh = shapes.e[s][1], ew = shapes.e[s][2];
    const int lt = t - zi_t * g.zt, lh = h - zi_h * g.zh, lw = w - zi_w * g.zw;
    const int tt = lt / et, th = lh / eh, tw = lw / ew;
    const int Et = min(et, Lt - tt * et), Eh = min(eh, Lh - th * eh), Ew = min(ew, Lw - tw * ew);
    const int64_t tile_off = (int64_t)tt * et * Lh * Lw + (int64_t)Et * th * eh * Lw + (int64_t)Et * Eh * tw * ew;
    const int within = ((lt - tt * et) * Eh + (lh - th * eh)) * Ew + (lw - tw * ew);
    perm[(int64_t)first[z] * B + tile_off + within] = (int32_t)n;
  }
}

int chunk_channels(const ZoneGeom& g) {
  for (int ch = 64; ch >= 8; ch >>= 1)
    if ((size_t)g.max_tokens * ch * sizeof(float) <= (size_t)kSmemBudget) return ch;
  return 0;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// The streaming kernel applies: an instantiated zone size, an even channel count and
// row stride, and channel pairs aligned for one 4-byte (bf16) or 8-byte (f32) load.
// The TMA kernel applies: bf16, 16-byte aligned rows (ld % 8 == 0), whole 64-channel
// chunks, zones of at most 3 x 9 x 16 tokens.
bool tma_variant(const ZoneGeom& g, int C, int64_t ld, int dtype, const void* feat) {
  // the box spans kTmaMT x kTmaMH (t, h) tokens, so the grid must be at least that large
  return dtype == PRISM_BF16 && C % kSlabCh == 0 && ld % 8 == 0 && (reinterpret_cast<uintptr_t>(feat) & 15) == 0 &&
         g.T >= kTmaMT && g.H >= kTmaMH && g.W >= kWq && std::min(g.zt, g.T) <= kTmaMT && std::min(g.zh, g.H) <= kTmaMH;
}

int lines_variant(const ZoneGeom& g, int C, int64_t ld, int dtype, const void* feat) {
  const size_t al = dtype == PRISM_BF16 ? 4 : 8;
  if (C % 2 != 0 || ld % 2 != 0 || (reinterpret_cast<uintptr_t>(feat) % al) != 0) return 0;
  const int Lt = std::min(g.zt, g.T), Lh = std::min(g.zh, g.H);
  if (Lt <= 3 && Lh <= 9) return 1;
  if (Lt <= 5 && Lh <= 8) return 2;
  return 0;
}

size_t zone_ws_bytes(const ZoneGeom& g, int C, int /*dtype*/) {
  // both kernels write partials per 64-channel chunk (zone_partial: chunk <= 64)
  const int ch = chunk_channels(g);
  if (ch == 0) return 0;
  const int nchunks = std::max((C + ch - 1) / ch, (C + kLinesChannels - 1) / kLinesChannels);
  return align256((size_t)g.Z * nchunks * 3 * sizeof(float)) + align256((size_t)g.Z * 8 * sizeof(float));
}

namespace {

// Per-zone, per-axis partial sums of one call's feature channels, per channel chunk:
// part[z][chunk][a] = sum over the chunk's channels and the zone's lines along axis a
// of the squared deviations from the line mean.  *nchunks_out receives the chunks.
cudaError_t zone_partials_stage(const void* feat, int dtype, int64_t ld, int C, const ZoneGeom& g, float* part,
                                int* nchunks_out, cudaStream_t st, uint32_t* status) {
  const int ch = chunk_channels(g);
  const int variant = lines_variant(g, C, ld, dtype, feat);
  const bool by64 = variant || tma_variant(g, C, ld, dtype, feat);
  const int nchunks = by64 ? (C + kLinesChannels - 1) / kLinesChannels : (C + ch - 1) / ch;
  *nchunks_out = nchunks;
  const size_t smem = (size_t)g.max_tokens * ch * sizeof(float);
  const dim3 grid(g.Z, nchunks);
  cudaError_t e;
  if (tma_variant(g, C, ld, dtype, feat)) {
    // feature as [T][H][W][C] bf16; one box = 64 channels of kWq columns of a zone's
    // MT x MH (t, h) extent (clipped zones read zeros past the grid)
    CUtensorMap tm;
    const uint64_t dims[4] = {(uint64_t)C, (uint64_t)g.W, (uint64_t)g.H, (uint64_t)g.T};
    const uint64_t strides[3] = {(uint64_t)ld * 2, (uint64_t)g.W * ld * 2, (uint64_t)g.H * g.W * ld * 2};
    const uint32_t box[4] = {(uint32_t)kSlabCh, (uint32_t)kWq, (uint32_t)kTmaMH, (uint32_t)kTmaMT};
    if (!tensor_map_bf16(&tm, feat, 4, dims, strides, box)) return cudaErrorInvalidValue;
    const int items = g.Z * nchunks;
    const int nq = (std::min(g.zw, g.W) + kWq - 1) / kWq;
    int sms = 148;
    {
      int dev = 0;
      if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    const int grid = std::max(1, std::min(sms, (items + kTmaWarps - 1) / kTmaWarps));
    const size_t smem_t = sizeof(ZoneTmaSmem) + 128;
    auto kern = zone_tma_kernel<kTmaMT, kTmaMH>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_t)) != cudaSuccess)
      return e;
    HookScope hs("zone_tma", st);
    kern<<<grid, kTmaWarps * 32, smem_t, st>>>(tm, g, nchunks, items, nq, part, status);
  } else if (variant) {
    const dim3 lgrid((nchunks + kLinesWarps - 1) / kLinesWarps, g.Z);
    HookScope hs("zone_lines", st);
    if (dtype == PRISM_BF16) {
      if (variant == 1)
        zone_lines_kernel<__nv_bfloat16, 3, 9><<<lgrid, kLinesWarps * 32, 0, st>>>(
            static_cast<const __nv_bfloat16*>(feat), ld, C, g, nchunks, part);
      else
        zone_lines_kernel<__nv_bfloat16, 5, 8><<<lgrid, kLinesWarps * 32, 0, st>>>(
            static_cast<const __nv_bfloat16*>(feat), ld, C, g, nchunks, part);
    } else {
      if (variant == 1)
        zone_lines_kernel<float, 3, 9><<<lgrid, kLinesWarps * 32, 0, st>>>(static_cast<const float*>(feat), ld, C, g,
                                                                            nchunks, part);
      else
        zone_lines_kernel<float, 5, 8><<<lgrid, kLinesWarps * 32, 0, st>>>(static_cast<const float*>(feat), ld, C, g,
                                                                            nchunks, part);
    }
  } else if (dtype == PRISM_BF16) {
    const bool vec = (ld % 8 == 0) && (C % 8 == 0) && ((reinterpret_cast<uintptr_t>(feat) & 15) == 0);
    if (vec) {
      auto k = zone_partial_kernel<__nv_bfloat16, 8>;
      if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
      HookScope hs("zone_partial", st);
      k<<<grid, kZoneThreads, smem, st>>>(static_cast<const __nv_bfloat16*>(feat), ld, C, g, ch, part);
    } else {
      auto k = zone_partial_kernel<__nv_bfloat16, 1>;
      if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
      HookScope hs("zone_partial", st);
      k<<<grid, kZoneThreads, smem, st>>>(static_cast<const __nv_bfloat16*>(feat), ld, C, g, ch, part);
    }
  } else {
    const bool vec = (ld % 4 == 0) && (C % 4 == 0) && ((reinterpret_cast<uintptr_t>(feat) & 15) == 0);
    if (vec) {
      auto k = zone_partial_kernel<float, 4>;
      if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
      HookScope hs("zone_partial", st);
      k<<<grid, kZoneThreads, smem, st>>>(static_cast<const float*>(feat), ld, C, g, ch, part);
    } else {
      auto k = zone_partial_kernel<float, 1>;
      if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
      HookScope hs("zone_partial", st);
      k<<<grid, kZoneThreads, smem, st>>>(static_cast<const float*>(feat), ld, C, g, ch, part);
    }
  }
  return cudaGetLastError();
}

// stats, zone shapes and the permutation from partial sums part (strides zs, cs).
cudaError_t zone_choose_stage(const float* part, int nparts, int zs, int cs, int C, const float* a2v,
                              const ZoneGeom& g, const ShapeSet& shapes, float* stats, int32_t* zone_shape,
                              int32_t* perm, cudaStream_t st) {
  cudaError_t e;
  {
    HookScope hs("zone_finalize", st);
    zone_finalize_kernel<<<g.Z, kZoneThreads, (size_t)g.max_tokens * sizeof(float), st>>>(part, nparts, zs, cs, a2v,
                                                                                          g, C, stats);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    HookScope hs("zone_choose", st);
    zone_choose_kernel<<<1, 1024, 0, st>>>(stats, g.Z, shapes, zone_shape);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t N = (int64_t)g.T * g.H * g.W;
  const int blocks = (int)std::min<int64_t>((N + 255) / 256, 148 * 16);
  {
    HookScope hs("zone_perm", st);
    zone_perm_kernel<<<blocks, 256, 0, st>>>(g, zone_shape, shapes, perm);
  }
  return cudaGetLastError();
}

int ws_chunks_of(const ZoneGeom& g, int C) {
  const int ch = chunk_channels(g);
  return std::max((C + ch - 1) / ch, (C + kLinesChannels - 1) / kLinesChannels);
}

}  // namespace

cudaError_t zone_launch(const void* feat, int dtype, int64_t ld, int C, const float* a2v, const ZoneGeom& g,
                        const ShapeSet& shapes, int32_t* zone_shape, int32_t* perm, void* ws, cudaStream_t st,
                        uint32_t* status) {
  float* part = reinterpret_cast<float*>(ws);
  float* stats =
      reinterpret_cast<float*>(static_cast<char*>(ws) + align256((size_t)g.Z * ws_chunks_of(g, C) * 3 * 4));
  int nchunks = 0;
  cudaError_t e = zone_partials_stage(feat, dtype, ld, C, g, part, &nchunks, st, status);
  if (e != cudaSuccess) return e;
  return zone_choose_stage(part, nchunks, nchunks * 3, 3, C, a2v, g, shapes, stats, zone_shape, perm, st);
}

size_t zone_partials_ws_bytes(const ZoneGeom& g, int C) {
  return align256((size_t)g.Z * ws_chunks_of(g, C) * 3 * sizeof(float));
}

cudaError_t zone_partials_launch(const void* feat, int dtype, int64_t ld, int C, const ZoneGeom& g, float* out,
                                 void* ws, cudaStream_t st, uint32_t* status) {
  float* part = reinterpret_cast<float*>(ws);
  int nchunks = 0;
  cudaError_t e = zone_partials_stage(feat, dtype, ld, C, g, part, &nchunks, st, status);
  if (e != cudaSuccess) return e;
  HookScope hs("zone_sum_chunks", st);
  zone_sum_chunks_kernel<<<(g.Z * 3 + 255) / 256, 256, 0, st>>>(part, nchunks, g.Z, out);
  return cudaGetLastError();
}

void zone_chunked_size(const ZoneGeom& g, int B, int64_t* nb, int64_t* np) {
  int64_t blocks = 0;
  for (int zt = 0; zt < g.nzt; ++zt)
    for (int zh = 0; zh < g.nzh; ++zh)
      for (int zw = 0; zw < g.nzw; ++zw) {
        const int64_t n = (int64_t)std::min(g.zt, g.T - zt * g.zt) * std::min(g.zh, g.H - zh * g.zh) *
                          std::min(g.zw, g.W - zw * g.zw);
        blocks += (n + B - 1) / B;
      }
  *nb = blocks;
  *np = blocks * B;
}

cudaError_t zone_perm_chunked_launch(const int32_t* zone_shape, const ZoneGeom& g, const ShapeSet& shapes, int B,
                                     int32_t* perm, int32_t* blen, int64_t np, void* ws, cudaStream_t st) {
  int32_t* first = static_cast<int32_t*>(ws);
  {
    HookScope hs("zone_chunk_blocks", st);
    zone_chunk_blocks_kernel<<<1, 1024, 0, st>>>(g, B, first, blen);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    HookScope hs("fill_padding", st);
    fill_i32_kernel<<<(unsigned)std::min<int64_t>((np + 255) / 256, 148 * 16), 256, 0, st>>>(perm, np, -1);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t N = (int64_t)g.T * g.H * g.W;
  HookScope hs("zone_perm_chunked", st);
  zone_perm_chunked_kernel<<<(unsigned)std::min<int64_t>((N + 255) / 256, 148 * 16), 256, 0, st>>>(g, zone_shape,
                                                                                               shapes, B, first, perm);
  return cudaGetLastError();
}

size_t zone_from_partials_ws_bytes(const ZoneGeom& g) { return align256((size_t)g.Z * 8 * sizeof(float)); }

cudaError_t zone_from_partials_launch(const float* parts, int nparts, int C_total, const float* a2v,
                                      const ZoneGeom& g, const ShapeSet& shapes, int32_t* zone_shape, int32_t* perm,
                                      void* ws, cudaStream_t st) {
  return zone_choose_stage(parts, nparts, 3, g.Z * 3, C_total, a2v, g, shapes, static_cast<float*>(ws), zone_shape,
                           perm, st);
}

}  // namespace prism
