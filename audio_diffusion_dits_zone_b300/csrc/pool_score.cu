// Step 2 of the path: block-order gather, block-mean pooling of Q and K, and the
// block score matrix.
//
// "Prism: dynamic sparse attention for 2K joint video-audio generation training",
// section "Region-adapted block construction", paragraph 1: block-level features
// are what the selection looks at.  Reading: the block mean of Q and of K (true
// length for the short last block), score[h][i][j] = qbar[h][i] . kbar[h][j] / sqrt(d).
//
// pool_gather   one CTA per block: every thread owns 16-byte column vectors of the
//               token rows and walks the block's rows, so each warp reads 512
//               contiguous bytes per row (coalesced); it writes the block-order
//               copies and the fp32 column sums.  HBM-bound: reads Q, K (, V) once.
// scores        per head an [nb x d] x [d x nb] fp32 product on CUDA cores
//               (128 x 128 output tile per CTA, 8 x 8 per thread, the d axis staged
//               through shared memory 16 at a time, double-buffered).  fp32 keeps the
//               block order the selection depends on close to the exact one.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

constexpr int kPoolThreads = 256;

template <typename T, int VW>
struct Vec;
template <>
struct Vec<__nv_bfloat16, 8> {
  using raw = uint4;
  __device__ static void to_f32(const raw& r, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = __bfloat1622float2(h[k]);
      f[2 * k] = x.x;
      f[2 * k + 1] = x.y;
    }
  }
};
template <>
struct Vec<float, 4> {
  using raw = uint4;
  __device__ static void to_f32(const raw& r, float* f) {
    const float* x = reinterpret_cast<const float*>(&r);
#pragma unroll
    for (int k = 0; k < 4; ++k) f[k] = x[k];
  }
};
template <typename T>
struct Vec<T, 1> {
  using raw = T;
  __device__ static void to_f32(const raw& r, float* f) { f[0] = prism::to_f32<T>(r); }
};

template <typename T, int VW>
__global__ void __launch_bounds__(kPoolThreads)
    pool_gather_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, int64_t ld,
                       const int32_t* __restrict__ perm, int n_src, int N, int Hh, int d, int B, T* __restrict__ qb,
                       T* __restrict__ kb, T* __restrict__ vb, int64_t ldb, float* __restrict__ qbar,
                       float* __restrict__ kbar, int nb, uint32_t* status) {
  using R = typename Vec<T, VW>::raw;
  extern __shared__ int32_t rows[];  // source row of each block-order row (-1: padding)
  __shared__ int nvalid;
  const int b = blockIdx.x;
  const int r0 = b * B;
  const int len = min(B, N - r0);
  if (threadIdx.x == 0) nvalid = 0;
  __syncthreads();
  int mine = 0;
  for (int r = threadIdx.x; r < len; r += kPoolThreads) {
    int src = perm ? perm[r0 + r] : r0 + r;
    if (src < -1 || src >= n_src) {  // a corrupt permutation entry is read as padding and flagged
      flag_error(status, PRISM_DEV_BAD_INDEX);
      src = -1;
    }
    rows[r] = src;
    mine += src >= 0;
  }
  if (mine) atomicAdd(&nvalid, mine);
  __syncthreads();
  const int nvec = Hh * d / VW;
  const float inv_len = nvalid > 0 ? 1.f / (float)nvalid : 0.f;
  const R zero = {};
  for (int vi = threadIdx.x; vi < nvec; vi += kPoolThreads) {
    const int64_t col = (int64_t)vi * VW;
    float aq[VW], ak[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e) aq[e] = ak[e] = 0.f;
    int r = 0;
    for (; r + 4 <= len; r += 4) {
      R xq[4], xk[4], xv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int sr = rows[r + u];
        const int64_t src = (int64_t)max(sr, 0) * ld + col;
        xq[u] = sr >= 0 ? *reinterpret_cast<const R*>(q + src) : zero;
        xk[u] = sr >= 0 ? *reinterpret_cast<const R*>(k + src) : zero;
        if (vb) xv[u] = sr >= 0 ? *reinterpret_cast<const R*>(v + src) : zero;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t dst = (int64_t)(r0 + r + u) * ldb + col;
        if (qb) *reinterpret_cast<R*>(qb + dst) = xq[u];
        if (kb) *reinterpret_cast<R*>(kb + dst) = xk[u];
        if (vb) *reinterpret_cast<R*>(vb + dst) = xv[u];
        float f[VW];
        Vec<T, VW>::to_f32(xq[u], f);
#pragma unroll
        for (int e = 0; e < VW; ++e) aq[e] += f[e];
        Vec<T, VW>::to_f32(xk[u], f);
#pragma unroll
        for (int e = 0; e < VW; ++e) ak[e] += f[e];
      }
    }
    for (; r < len; ++r) {
      const int sr = rows[r];
      const int64_t src = (int64_t)max(sr, 0) * ld + col;
      const R xq = sr >= 0 ? *reinterpret_cast<const R*>(q + src) : zero;
      const R xk = sr >= 0 ? *reinterpret_cast<const R*>(k + src) : zero;
      const int64_t dst = (int64_t)(r0 + r) * ldb + col;
      if (qb) *reinterpret_cast<R*>(qb + dst) = xq;
      if (kb) *reinterpret_cast<R*>(kb + dst) = xk;
      if (vb) *reinterpret_cast<R*>(vb + dst) = sr >= 0 ? *reinterpret_cast<const R*>(v + src) : zero;
      float f[VW];
      Vec<T, VW>::to_f32(xq, f);
#pragma unroll
      for (int e = 0; e < VW; ++e) aq[e] += f[e];
      Vec<T, VW>::to_f32(xk, f);
#pragma unroll
      for (int e = 0; e < VW; ++e) ak[e] += f[e];
    }
    const int h = (int)(col / d), c = (int)(col - (int64_t)h * d);
    const size_t o = ((size_t)h * nb + b) * d + c;
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      if (qbar) qbar[o + e] = aq[e] * inv_len;
      if (kbar) kbar[o + e] = ak[e] * inv_len;
    }
  }
}

// scores: S = qbar kbar^T / sqrt(d) per head, fp32 on CUDA cores.  A CTA of 256
// threads owns a 128 x 128 tile of S; each thread an 8 x 8 register tile: rows
// 4ty .. 4ty + 3 and 64 + 4ty .. 64 + 4ty + 3, columns likewise from 4tx, so each
// channel step is four 16-byte shared loads for 64 FMAs.  k-slices of 16 are staged
// in shared memory, transposed (k-major), double-buffered through registers so the
// next slice's global loads overlap this slice's 8 x 8 x 16 FMAs, issued as packed
// pairs (fma.rn.f32x2: two independent round-to-nearest FMAs per instruction).  Every
// score is one FMA chain over the channels in ascending order, then the scale.
constexpr int kSTile = 128, kSK = 16, kSThreads = 256;

__global__ void __launch_bounds__(kSThreads, 2) scores_kernel(const float* __restrict__ qbar,
                                                           const float* __restrict__ kbar, int nb, int d,
                                                           float scale, float* __restrict__ S) {
  __shared__ __align__(16) float As[2][kSK][kSTile + 4];
  __shared__ __align__(16) float Bs[2][kSK][kSTile + 4];
  const int h = blockIdx.z;
  const int i0 = blockIdx.y * kSTile, j0 = blockIdx.x * kSTile;
  const float* A = qbar + (size_t)h * nb * d;
  const float* Bm = kbar + (size_t)h * nb * d;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  // loader: each thread brings 8 values of A and 8 of B per k-slice: rows lr, lr + 64;
  // columns lc .. lc + 3 (one float4 when d allows it)
  const int lr = threadIdx.x >> 2, lc = (threadIdx.x & 3) * 4;
  const bool vec = (d & 3) == 0;
  float4 ra[2], rb[2];
  auto load = [&](int k0) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int ri = i0 + lr + 64 * u, rj = j0 + lr + 64 * u;
      float a[4], b[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) a[e] = b[e] = 0.f;
      if (vec && k0 + lc + 3 < d) {
        if (ri < nb) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(A + (size_t)ri * d + k0 + lc));
          a[0] = x.x, a[1] = x.y, a[2] = x.z, a[3] = x.w;
        }
        if (rj < nb) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(Bm + (size_t)rj * d + k0 + lc));
          b[0] = x.x, b[1] = x.y, b[2] = x.z, b[3] = x.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = k0 + lc + e;
          if (c < d && ri < nb) a[e] = A[(size_t)ri * d + c];
          if (c < d && rj < nb) b[e] = Bm[(size_t)rj * d + c];
        }
      }
      ra[u] = make_float4(a[0], a[1], a[2], a[3]);
      rb[u] = make_float4(b[0], b[1], b[2], b[3]);
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = lr + 64 * u;
      As[buf][lc][r] = ra[u].x;
      As[buf][lc + 1][r] = ra[u].y;
      As[buf][lc + 2][r] = ra[u].z;
      As[buf][lc + 3][r] = ra[u].w;
      Bs[buf][lc][r] = rb[u].x;
      Bs[buf][lc + 1][r] = rb[u].y;
      Bs[buf][lc + 2][r] = rb[u].z;
      Bs[buf][lc + 3][r] = rb[u].w;
    }
  };
  f2 acc[8][4];  // columns (2w2, 2w2 + 1) of the 8 x 8 tile
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int w2 = 0; w2 < 4; ++w2) acc[u][w2] = f2_make(0.f, 0.f);
  const int nk = (d + kSK - 1) / kSK;
  load(0);
  store(0);
  __syncthreads();
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nk) load((kt + 1) * kSK);
#pragma unroll
    for (int c = 0; c < kSK; ++c) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][c][4 * ty]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][c][64 + 4 * ty]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][c][4 * tx]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][c][64 + 4 * tx]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const f2 b[4] = {f2_make(b0.x, b0.y), f2_make(b0.z, b0.w), f2_make(b1.x, b1.y), f2_make(b1.z, b1.w)};
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const f2 au = f2_make(a[u], a[u]);
#pragma unroll
        for (int w2 = 0; w2 < 4; ++w2) acc[u][w2] = f2_fma(au, b[w2], acc[u][w2]);
      }
    }
    if (kt + 1 < nk) store(buf ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int i = i0 + (u & 3) + 4 * ty + 64 * (u >> 2);
    if (i >= nb) continue;
    float* row = S + ((size_t)h * nb + i) * nb;
    float v[8];
#pragma unroll
    for (int w2 = 0; w2 < 4; ++w2) f2_split(acc[u][w2], v[2 * w2], v[2 * w2 + 1]);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int j = j0 + (w & 3) + 4 * tx + 64 * (w >> 2);
      if (j < nb) row[j] = v[w] * scale;
    }
  }
}

template <typename T, int VW>
cudaError_t launch_pool(const void* q, const void* k, const void* v, int64_t ld, const int32_t* perm, int n_src,
                        int N, int Hh, int d, int B, void* qb, void* kb, void* vb, int64_t ldb, float* qbar,
                        float* kbar, cudaStream_t st, uint32_t* status) {
  const int nb = (N + B - 1) / B;
  HookScope hs("pool_gather", st);
  pool_gather_kernel<T, VW><<<nb, kPoolThreads, (size_t)B * sizeof(int32_t), st>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), ld, perm, n_src, N, Hh, d, B,
      static_cast<T*>(qb), static_cast<T*>(kb), static_cast<T*>(vb), ldb, qbar, kbar, nb, status);
  return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

cudaError_t pool_launch(const void* q, const void* k, const void* v, int dtype, int64_t ld, const int32_t* perm,
                        int n_src, int N, int Hh, int d, int B, void* qb, void* kb, void* vb, int64_t ldb,
                        float* qbar, float* kbar, cudaStream_t st, uint32_t* status) {
  const bool ptr_ok = aligned16(q) && aligned16(k) && (!v || aligned16(v)) && (!qb || aligned16(qb)) &&
                      (!kb || aligned16(kb)) && (!vb || aligned16(vb));
  if (dtype == PRISM_BF16) {
    if (ptr_ok && d % 8 == 0 && ld % 8 == 0 && ldb % 8 == 0)
      return launch_pool<__nv_bfloat16, 8>(q, k, v, ld, perm, n_src, N, Hh, d, B, qb, kb, vb, ldb, qbar, kbar, st, status);
    return launch_pool<__nv_bfloat16, 1>(q, k, v, ld, perm, n_src, N, Hh, d, B, qb, kb, vb, ldb, qbar, kbar, st, status);
  }
  if (ptr_ok && d % 4 == 0 && ld % 4 == 0 && ldb % 4 == 0)
    return launch_pool<float, 4>(q, k, v, ld, perm, n_src, N, Hh, d, B, qb, kb, vb, ldb, qbar, kbar, st, status);
  return launch_pool<float, 1>(q, k, v, ld, perm, n_src, N, Hh, d, B, qb, kb, vb, ldb, qbar, kbar, st, status);
}

cudaError_t scores_launch(const float* qbar, const float* kbar, int Hh, int nb, int d, float* scores,
                          cudaStream_t st) {
  const dim3 grid((nb + kSTile - 1) / kSTile, (nb + kSTile - 1) / kSTile, Hh);
  HookScope hs("scores", st);
  scores_kernel<<<grid, kSThreads, 0, st>>>(qbar, kbar, nb, d, 1.0f / sqrtf((float)d), scores);
  return cudaGetLastError();
}

}  // namespace prism
