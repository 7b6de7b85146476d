// Block-sparse attention on CUDA cores, fp32 arithmetic: the path for fp32 inputs
// and for (d, B) outside the tensor-core kernels (d = 64 or B = 64).
//
// Prism Block Sparse Attention ("Prism: dynamic sparse attention for 2K joint
// video-audio generation training", section "Region-adapted block construction",
// paragraph 2): every query token of query block i attends to all tokens of the
// blocks in i's kept list, softmax scale 1/sqrt(d), no causal mask.  Backward:
// P = exp(S - lse), dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
// dS = P * (dP - D), dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d).
//
// Forward and dQ: one CTA per (query block, head), TPR threads per query row, each
// holding d / TPR channels; the kept key and value blocks are staged in shared
// memory in fp32 and walked with an online softmax.
// dK / dV: one CTA per (key block, head) walks the query blocks that kept it (the
// transposed lists), so no atomics are needed and results are deterministic.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// dK/dV CTAs own at most this many key rows (four fp32 row vectors per thread).
constexpr int kRowsPerCta = 64;

template <int TPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int o = 1; o < TPR; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T>
__device__ void stage_tile(float* dst, const T* src, int64_t ld, int h, int D, int row0, int len, int B) {
  for (int e = threadIdx.x; e < B * D; e += blockDim.x) {
    const int r = e / D, c = e - (e / D) * D;
    dst[e] = r < len ? to_f32<T>(src[(int64_t)(row0 + r) * ld + (int64_t)h * D + c]) : 0.f;
  }
}

template <typename T, int D, int TPR>
__global__ void bsa_fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                                    int64_t ld, int N, int B, const int32_t* __restrict__ counts,
                                    const int32_t* __restrict__ idx, int nb, const int32_t* __restrict__ blen,
                                    T* __restrict__ o, float* __restrict__ lse, uint32_t* status) {
  constexpr int DP = D / TPR;
  extern __shared__ float sm[];
  float* Ks = sm;
  float* Vs = sm + B * D;
  const int i = blockIdx.x, h = blockIdx.y;
  const int r = threadIdx.x / TPR, part = threadIdx.x % TPR;
  const int row = i * B + r;
  const bool valid = r < B && row < N && (!blen || r < blen[i]);  // padding rows are no queries
  const float sl2 = kLog2e * rsqrtf((float)D);
  float qv[DP], acc[DP];
#pragma unroll
  for (int c = 0; c < DP; ++c) {
    qv[c] = valid ? to_f32<T>(q[(int64_t)row * ld + (int64_t)h * D + part * DP + c]) * sl2 : 0.f;
    acc[c] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int hrow = h * nb + i;
  const int cnt = counts[hrow];
  const int32_t* lst = idx + (size_t)hrow * nb;
  for (int t = 0; t < cnt; ++t) {
    const int j = lst[t];
    if (j < 0 || j >= nb) {
      if (threadIdx.x == 0) flag_error(status, PRISM_DEV_BAD_INDEX);
      continue;
    }
    const int len = blen ? min(B, max(0, blen[j])) : min(B, N - j * B);
    __syncthreads();
    stage_tile<T>(Ks, k, ld, h, D, j * B, len, B);
    stage_tile<T>(Vs, v, ld, h, D, j * B, len, B);
    __syncthreads();
    for (int c = 0; c < len; ++c) {
      const float* kr = Ks + c * D + part * DP;
      float s = 0.f;
#pragma unroll
      for (int x = 0; x < DP; ++x) s = fmaf(qv[x], kr[x], s);
      s = group_sum<TPR>(s);
      const float mn = fmaxf(m, s);
      const float corr = exp2f(m - mn);
      const float p = exp2f(s - mn);
      l = l * corr + p;
      const float* vr = Vs + c * D + part * DP;
#pragma unroll
      for (int x = 0; x < DP; ++x) acc[x] = fmaf(p, vr[x], acc[x] * corr);
      m = mn;
    }
  }
  if (!valid) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int c = 0; c < DP; ++c) o[(int64_t)row * ld + (int64_t)h * D + part * DP + c] = from_f32<T>(acc[c] * inv);
  if (part == 0) lse[(size_t)h * N + row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

template <typename T, int D, int TPR>
__global__ void bsa_dq_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                                   const T* __restrict__ dO, const float* __restrict__ lse,
                                   const float* __restrict__ Drow, int64_t ld, int N, int B,
                                   const int32_t* __restrict__ counts, const int32_t* __restrict__ idx, int nb,
                                   const int32_t* __restrict__ blen, T* __restrict__ dq) {
  constexpr int DP = D / TPR;
  extern __shared__ float sm[];
  float* Ks = sm;
  float* Vs = sm + B * D;
  const int i = blockIdx.x, h = blockIdx.y;
  const int r = threadIdx.x / TPR, part = threadIdx.x % TPR;
  const int row = i * B + r;
  const bool valid = r < B && row < N && (!blen || r < blen[i]);  // padding rows are no queries
  const float scale = rsqrtf((float)D);
  float qv[DP], gv[DP], acc[DP];
#pragma unroll
  for (int c = 0; c < DP; ++c) {
    const int64_t off = (int64_t)row * ld + (int64_t)h * D + part * DP + c;
    qv[c] = valid ? to_f32<T>(q[off]) * scale : 0.f;
    gv[c] = valid ? to_f32<T>(dO[off]) : 0.f;
    acc[c] = 0.f;
  }
  const float L = valid ? lse[(size_t)h * N + row] : 0.f;
  const float Dr = valid ? Drow[(size_t)h * N + row] : 0.f;
  const int hrow = h * nb + i;
  const int cnt = counts[hrow];
  const int32_t* lst = idx + (size_t)hrow * nb;
  for (int t = 0; t < cnt; ++t) {
    const int j = lst[t];
    if (j < 0 || j >= nb) continue;
    const int len = blen ? min(B, max(0, blen[j])) : min(B, N - j * B);
    __syncthreads();
    stage_tile<T>(Ks, k, ld, h, D, j * B, len, B);
    stage_tile<T>(Vs, v, ld, h, D, j * B, len, B);
    __syncthreads();
    for (int c = 0; c < len; ++c) {
      const float* kr = Ks + c * D + part * DP;
      const float* vr = Vs + c * D + part * DP;
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int x = 0; x < DP; ++x) {
        s = fmaf(qv[x], kr[x], s);
        dp = fmaf(gv[x], vr[x], dp);
      }
      s = group_sum<TPR>(s);
      dp = group_sum<TPR>(dp);
      const float p = expf(s - L);
      const float ds = p * (dp - Dr);
#pragma unroll
      for (int x = 0; x < DP; ++x) acc[x] = fmaf(ds, kr[x], acc[x]);
    }
  }
  if (!valid) return;
#pragma unroll
  for (int c = 0; c < DP; ++c) dq[(int64_t)row * ld + (int64_t)h * D + part * DP + c] = from_f32<T>(acc[c] * scale);
}

template <typename T, int D, int TPR>
__global__ void bsa_dkdv_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                                     const T* __restrict__ dO, const float* __restrict__ lse,
                                     const float* __restrict__ Drow, int64_t ld, int N, int B,
                                     const int32_t* __restrict__ tcounts, const int32_t* __restrict__ tidx, int nb,
                                     const int32_t* __restrict__ blen, T* __restrict__ dk, T* __restrict__ dv) {
  constexpr int DP = D / TPR;
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Gs = sm + B * D;
  float* Ls = sm + 2 * B * D;
  float* Ds = Ls + B;
  // CTA x covers key rows [sub * kRowsPerCta, +kRowsPerCta) of key block j
  const int splits = B / kRowsPerCta;
  const int j = blockIdx.x / splits, sub = blockIdx.x - (blockIdx.x / splits) * splits, h = blockIdx.y;
  const int c = sub * kRowsPerCta + threadIdx.x / TPR, part = threadIdx.x % TPR;
  const int col = j * B + c;
  const bool valid = c < B && col < N && (!blen || c < blen[j]);  // padding rows are no keys
  const float scale = rsqrtf((float)D);
  float kv[DP], vv[DP], gk[DP], gvv[DP];
#pragma unroll
  for (int x = 0; x < DP; ++x) {
    const int64_t off = (int64_t)col * ld + (int64_t)h * D + part * DP + x;
    kv[x] = valid ? to_f32<T>(k[off]) * scale : 0.f;
    vv[x] = valid ? to_f32<T>(v[off]) : 0.f;
    gk[x] = 0.f;
    gvv[x] = 0.f;
  }
  const int hcol = h * nb + j;
  const int cnt = tcounts[hcol];
  const int32_t* lst = tidx + (size_t)hcol * nb;
  for (int t = 0; t < cnt; ++t) {
    const int i = lst[t];
    const int len = blen ? min(B, max(0, blen[i])) : min(B, N - i * B);
    __syncthreads();
    stage_tile<T>(Qs, q, ld, h, D, i * B, len, B);
    stage_tile<T>(Gs, dO, ld, h, D, i * B, len, B);
    for (int r = threadIdx.x; r < B; r += blockDim.x) {
      Ls[r] = r < len ? lse[(size_t)h * N + i * B + r] : 0.f;
      Ds[r] = r < len ? Drow[(size_t)h * N + i * B + r] : 0.f;
    }
    __syncthreads();
    for (int r = 0; r < len; ++r) {
      const float* qr = Qs + r * D + part * DP;
      const float* gr = Gs + r * D + part * DP;
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int x = 0; x < DP; ++x) {
        s = fmaf(kv[x], qr[x], s);
        dp = fmaf(vv[x], gr[x], dp);
      }
      s = group_sum<TPR>(s);
      dp = group_sum<TPR>(dp);
      const float p = expf(s - Ls[r]);
      const float ds = p * (dp - Ds[r]);
#pragma unroll
      for (int x = 0; x < DP; ++x) {
        gvv[x] = fmaf(p, gr[x], gvv[x]);
        gk[x] = fmaf(ds, qr[x], gk[x]);
      }
    }
  }
  if (!valid) return;
#pragma unroll
  for (int x = 0; x < DP; ++x) {
    const int64_t off = (int64_t)col * ld + (int64_t)h * D + part * DP + x;
    dk[off] = from_f32<T>(gk[x] * scale);
    dv[off] = from_f32<T>(gvv[x]);
  }
}

template <typename T, int D>
cudaError_t fwd_t(const void* q, const void* k, const void* v, int64_t ld, int N, int Hh, int B,
                  const int32_t* counts, const int32_t* idx, int nb, const int32_t* blen, void* o, float* lse,
                  cudaStream_t st, uint32_t* status) {
  constexpr int TPR = 2;
  auto kern = bsa_fwd_simt_kernel<T, D, TPR>;
  const size_t smem = (size_t)2 * B * D * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  HookScope hs("bsa_fwd_simt", st);
  kern<<<dim3(nb, Hh), B * TPR, smem, st>>>(static_cast<const T*>(q), static_cast<const T*>(k),
                                             static_cast<const T*>(v), ld, N, B, counts, idx, nb, blen,
                                             static_cast<T*>(o), lse, status);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_t(const void* q, const void* k, const void* v, const void* dO, const float* lse, int64_t ld, int N,
                  int Hh, int B, const int32_t* counts, const int32_t* idx, int nb, const int32_t* blen, void* dq,
                  void* dk, void* dv, const int32_t* tcounts, const int32_t* tidx, const float* Drow,
                  cudaStream_t st) {
  constexpr int TPR_Q = 2, TPR_K = 4;
  auto kq = bsa_dq_simt_kernel<T, D, TPR_Q>;
  auto kk = bsa_dkdv_simt_kernel<T, D, TPR_K>;
  const size_t smem_q = (size_t)2 * B * D * sizeof(float);
  const size_t smem_k = (size_t)(2 * B * D + 2 * B) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_k)) != cudaSuccess)
    return e;
  {
  HookScope hs("bsa_dq_simt", st);
  kq<<<dim3(nb, Hh), B * TPR_Q, smem_q, st>>>(static_cast<const T*>(q), static_cast<const T*>(k),
                                               static_cast<const T*>(v), static_cast<const T*>(dO), lse, Drow, ld,
                                               N, B, counts, idx, nb, blen, static_cast<T*>(dq));
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  HookScope hs("bsa_dkdv_simt", st);
  const int splits = B > kRowsPerCta ? B / kRowsPerCta : 1;
  kk<<<dim3(nb * splits, Hh), (B / splits) * TPR_K, smem_k, st>>>(static_cast<const T*>(q), static_cast<const T*>(k),
                                               static_cast<const T*>(v), static_cast<const T*>(dO), lse, Drow, ld,
                                               N, B, tcounts, tidx, nb, blen, static_cast<T*>(dk),
                                               static_cast<T*>(dv));
  return cudaGetLastError();
}

}  // namespace

cudaError_t bsa_fwd_simt_launch(const void* q, const void* k, const void* v, int dtype, int64_t ld, int N, int Hh,
                                int d, int B, const int32_t* counts, const int32_t* idx, int nb, const int32_t* blen,
                                void* o, float* lse, cudaStream_t st, uint32_t* status) {
  if (dtype == PRISM_BF16)
    return d == 64 ? fwd_t<__nv_bfloat16, 64>(q, k, v, ld, N, Hh, B, counts, idx, nb, blen, o, lse, st, status)
                   : fwd_t<__nv_bfloat16, 128>(q, k, v, ld, N, Hh, B, counts, idx, nb, blen, o, lse, st, status);
  return d == 64 ? fwd_t<float, 64>(q, k, v, ld, N, Hh, B, counts, idx, nb, blen, o, lse, st, status)
                 : fwd_t<float, 128>(q, k, v, ld, N, Hh, B, counts, idx, nb, blen, o, lse, st, status);
}

cudaError_t bsa_bwd_simt_launch(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                const float* lse, int dtype, int64_t ld, int N, int Hh, int d, int B,
                                const int32_t* counts, const int32_t* idx, int nb, const int32_t* blen, void* dq,
                                void* dk, void* dv, const int32_t* tcounts, const int32_t* tidx, float* Drow,
                                cudaStream_t st, uint32_t* /*status*/) {
  cudaError_t e = row_dot_launch(o, dO, dtype, ld, N, Hh, d, Drow, st);
  if (e != cudaSuccess) return e;
  if (dtype == PRISM_BF16)
    return d == 64 ? bwd_t<__nv_bfloat16, 64>(q, k, v, dO, lse, ld, N, Hh, B, counts, idx, nb, blen, dq, dk, dv,
                                              tcounts, tidx, Drow, st)
                   : bwd_t<__nv_bfloat16, 128>(q, k, v, dO, lse, ld, N, Hh, B, counts, idx, nb, blen, dq, dk, dv,
                                               tcounts, tidx, Drow, st);
  return d == 64 ? bwd_t<float, 64>(q, k, v, dO, lse, ld, N, Hh, B, counts, idx, nb, blen, dq, dk, dv, tcounts, tidx,
                                    Drow, st)
                 : bwd_t<float, 128>(q, k, v, dO, lse, ld, N, Hh, B, counts, idx, nb, blen, dq, dk, dv, tcounts,
                                     tidx, Drow, st);
}

}  // namespace prism
