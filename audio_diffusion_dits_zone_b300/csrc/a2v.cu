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
// The audio sequence is short (a few hundred tokens against tens of thousands of
// video tokens), so each head's audio keys and values fit in shared memory next to
// the video query tiles.  a2v_attn_kernel is persistent: one CTA per SM walks a
// contiguous range of (head, 128-row query tile) items, loading a head's K and V once
// (a full 128-row tile for tokens 0-127, a 32-row tile for tokens 128-159) and
// streaming the query tiles through a four-stage ring, deep enough to keep the DRAM
// stream of queries busy.  Per tile:
//   S_x = Q K_x^T for each audio block x (tcgen05, A and B from shared memory; the
//         last block only as wide as its keys, rounded up to 32);
//   softmax over all audio tokens at once: the whole S row (up to 160 tokens) in
//         registers after one TMEM round trip, which releases S to the next tile;
//         P = 2^((s - max) log2(e) / sqrt(d)) in bf16 into TMEM columns of its own;
//   O = sum_x P_x V_x (A = P from TMEM, only the key rows that exist);
//   |O / l|^2 per row in fp32 into sqn[h][n] (and O itself, if asked for), done
//         after the next tile's exponentials, so that P V runs behind them.
// TMEM: S_0 [0,128) S_1 [128,256) O [256,384) P_0 [384,448) P_1 [448,512).
// Warps: 0 TMA producer, 1 S issuer (TMEM owner), 2 P V issuer, 4-7 one query row
// per thread.  Longer audio sequences go to the general attention kernel in dense
// mode.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

constexpr int kA2vThreads = 256;
constexpr int kRows = 128;                 // query rows per tile = keys per audio block
constexpr int kHd = 128;                   // head dim
constexpr uint32_t kBox = 16384;           // 128 rows x 64 bf16, 128-byte swizzled
constexpr uint32_t kTileB = 2 * kBox;      // 128 x 128 bf16
constexpr int kMaxChunks = 5;              // audio tokens <= 160: a whole S row in registers
constexpr int kQStages = 4;                // video query tiles in flight per CTA
constexpr int kTailRows = 32;              // the second audio block holds <= 32 tokens
constexpr uint32_t kTailBox = kTailRows * 128;  // 32 rows x 64 bf16
constexpr uint32_t kTailB = 2 * kTailBox;
constexpr uint32_t kOCol = 256, kPCol = 384;
constexpr float kSl2 = 1.4426950408889634f * 0.08838834764831845f;  // log2(e) / sqrt(128)

struct A2vSmem {
  uint8_t k0[kTileB], v0[kTileB];   // audio block 0 (up to 128 tokens)
  uint8_t k1[kTailB], v1[kTailB];   // audio block 1 (tokens 128 .. 159)
  uint8_t q[kQStages][kTileB];
  uint64_t kv_full, kv_empty;
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t s_full, s_free, p_full, o_full, o_free, fin_s, fin_pv;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kA2vSmemBytes = sizeof(A2vSmem) + 1024;
static_assert(kA2vSmemBytes <= 232448, "shared memory budget");

// NCH = ceil(M / 32): 32-key chunks of an S row (the whole row lives in registers).
template <int NCH>
__global__ void __launch_bounds__(kA2vThreads, 1)
    a2v_attn_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmk1,
                    const __grid_constant__ CUtensorMap tmv1, __nv_bfloat16* __restrict__ o, int64_t ld,
                    float* __restrict__ sqn, int N, int M, int nbq, int nbk, int items, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  A2vSmem& sm = *reinterpret_cast<A2vSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int first = (int)((int64_t)items * blockIdx.x / gridDim.x);
  const int cnt = (int)((int64_t)items * (blockIdx.x + 1) / gridDim.x) - first;
  const int len_last = M - (nbk - 1) * kRows;  // keys in the last audio block, 1 .. 128
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.kv_full), 1);
    mbar_init(smem_u32(&sm.kv_empty), 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(smem_u32(&sm.q_full[s]), 1);
      mbar_init(smem_u32(&sm.q_empty[s]), 1);
    }
    mbar_init(smem_u32(&sm.s_full), 1);
    mbar_init(smem_u32(&sm.s_free), 4);
    mbar_init(smem_u32(&sm.p_full), 4);
    mbar_init(smem_u32(&sm.o_full), 1);
    mbar_init(smem_u32(&sm.o_free), 4);
    mbar_init(smem_u32(&sm.fin_s), 1);
    mbar_init(smem_u32(&sm.fin_pv), 1);
    sm.abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0 && cnt > 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      int cur = -1, epoch = -1, armed[kQStages] = {};
      for (int t = 0; t < cnt; ++t) {
        const int item = first + t, h = item / nbq, i = item - h * nbq;
        if (h != cur) {  // a new head: its audio K and V, once the last head's products are done
          if (epoch >= 0 && !mbar_wait(smem_u32(&sm.kv_empty), epoch & 1, abort, status)) break;
          ++epoch;
          cur = h;
          const uint32_t kvb = smem_u32(&sm.kv_full);
          mbar_arrive_expect_tx(kvb, 2u * kTileB + (nbk > 1 ? 2u * kTailB : 0u));
          tma_load_2d(smem_u32(sm.k0), &tmk, h * kHd, 0, kvb);
          tma_load_2d(smem_u32(sm.k0) + kBox, &tmk, h * kHd + 64, 0, kvb);
          tma_load_2d(smem_u32(sm.v0), &tmv, h * kHd, 0, kvb);
          tma_load_2d(smem_u32(sm.v0) + kBox, &tmv, h * kHd + 64, 0, kvb);
          if (nbk > 1) {  // 32-row boxes of the second block
            tma_load_2d(smem_u32(sm.k1), &tmk1, h * kHd, kRows, kvb);
            tma_load_2d(smem_u32(sm.k1) + kTailBox, &tmk1, h * kHd + 64, kRows, kvb);
            tma_load_2d(smem_u32(sm.v1), &tmv1, h * kHd, kRows, kvb);
            tma_load_2d(smem_u32(sm.v1) + kTailBox, &tmv1, h * kHd + 64, kRows, kvb);
          }
        }
        const int s = t % kQStages;
        if (t >= kQStages && !mbar_wait(smem_u32(&sm.q_empty[s]), ((t / kQStages) - 1) & 1, abort, status)) break;
        const uint32_t qb = smem_u32(&sm.q_full[s]);
        mbar_arrive_expect_tx(qb, kTileB);
        tma_load_2d(smem_u32(sm.q[s]), &tmq, h * kHd, i * kRows, qb);
        tma_load_2d(smem_u32(sm.q[s]) + kBox, &tmq, h * kHd + 64, i * kRows, qb);
        ++armed[s];
      }
      if (*abort) {  // wait (bounded) for the copies still in flight
        if (epoch >= 0) drain_wait(smem_u32(&sm.kv_full), epoch & 1);
        for (int s = 0; s < kQStages; ++s)
          if (armed[s]) drain_wait(smem_u32(&sm.q_full[s]), (armed[s] - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ S issuer
    // S(t) as soon as its query tile has landed and the softmax has read S(t-1)
    if (lane == 0 && cnt > 0) {
      const int n_last = (len_last + 31) & ~31;  // S width of the last block (multiple of 32)
      const uint32_t id_full = idesc_bf16_f32(kRows, kRows, false, false);
      const uint32_t id_last = idesc_bf16_f32(kRows, n_last, false, false);
      const uint64_t dq0 = smem_desc(smem_u32(sm.q[0]), 16, 1024, kSwizzle128B);
      const uint64_t dk0 = smem_desc(smem_u32(sm.k0), 16, 1024, kSwizzle128B);
      const uint64_t dk1 = smem_desc(smem_u32(sm.k1), 16, 1024, kSwizzle128B);
      int cur = -1, epoch = -1;
      bool ok = true;
      for (int t = 0; ok && t < cnt; ++t) {
        const int item = first + t, h = item / nbq, s = t % kQStages;
        if (h != cur) {
          ++epoch;
          cur = h;
          if (!(ok = mbar_wait(smem_u32(&sm.kv_full), epoch & 1, abort, status))) break;
        }
        if (!(ok = mbar_wait(smem_u32(&sm.q_full[s]), (t / kQStages) & 1, abort, status))) break;
        if (t > 0 && !(ok = mbar_wait(smem_u32(&sm.s_free), (t - 1) & 1, abort, status))) break;
        tc_fence_after();
        for (int x = 0; x < nbk; ++x) {
          const uint32_t id = x == nbk - 1 ? id_last : id_full;
          const uint64_t dkx = x == 0 ? dk0 : dk1;
          const uint32_t half = x == 0 ? kBox : kTailBox;  // bytes between the two 64-column halves
#pragma unroll
          for (int kk = 0; kk < kHd / 16; ++kk)
            mma_ss(tmem + x * kRows, desc_at(dq0, s * kTileB + (kk >> 2) * kBox + (kk & 3) * 32),
                   desc_at(dkx, (kk >> 2) * half + (kk & 3) * 32), id, kk > 0 ? 1u : 0u);
        }
        tc_commit(smem_u32(&sm.q_empty[s]));
        tc_commit(smem_u32(&sm.s_full));
      }
      tc_commit(smem_u32(&sm.fin_s));
      drain_wait(smem_u32(&sm.fin_s), 0);
    }
  } else if (warp == 2) {
    // ----------------------------------------------------------------- PV issuer
    // O(t) = sum_x P_x(t) V_x once P(t) is written and the softmax has read O(t-1)
    if (lane == 0 && cnt > 0) {
      const int k_last = (len_last + 15) >> 4;  // 16-key steps of the last block
      constexpr uint32_t id_pv = idesc_bf16_f32(kRows, kHd, false, true);
      const uint64_t dv0 = smem_desc(smem_u32(sm.v0), kBox, 1024, kSwizzle128B);
      const uint64_t dv1 = smem_desc(smem_u32(sm.v1), kTailBox, 1024, kSwizzle128B);
      bool ok = true;
      for (int t = 0; ok && t < cnt; ++t) {
        const int item = first + t, h = item / nbq;
        if (!(ok = mbar_wait(smem_u32(&sm.p_full), t & 1, abort, status))) break;
        if (t > 0 && !(ok = mbar_wait(smem_u32(&sm.o_free), (t - 1) & 1, abort, status))) break;
        tc_fence_after();
        for (int x = 0; x < nbk; ++x) {
          const int ksteps = x == nbk - 1 ? k_last : kRows / 16;
          const uint64_t dvx = x == 0 ? dv0 : dv1;
          for (int kk = 0; kk < ksteps; ++kk)
            mma_ts(tmem + kOCol, tmem + kPCol + x * 64 + kk * 8, desc_at(dvx, kk * 2048), id_pv,
                   (x > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&sm.o_full));
        // the head's last tile: K and V are free once these products are done (its S
        // products completed before the softmax could write this P)
        if (t + 1 == cnt || (first + t + 1) / nbq != h) tc_commit(smem_u32(&sm.kv_empty));
      }
      tc_commit(smem_u32(&sm.fin_pv));
      drain_wait(smem_u32(&sm.fin_pv), 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------- softmax rows
    // Per tile t: the whole S row in registers (one TMEM round trip), S released, P in
    // registers; then the epilogue of tile t-1 (whose P V ran meanwhile), then P(t)
    // into the P columns that P V(t-1) has finished reading.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    auto epilogue = [&](int tt, float l) -> bool {  // |O(tt) / l|^2 (and O) for this thread's row
      const bool ok2 = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.o_full), tt & 1, abort, status));
      if (!ok2) return false;
      tc_fence_after();
      const int item = first + tt, h = item / nbq, i = item - h * nbq;
      const int row = i * kRows + r;
      __nv_bfloat16* orow = o ? o + (int64_t)row * ld + (int64_t)h * kHd : nullptr;
      const float inv = 1.f / l;  // l >= 1: the row max contributes 2^0
      float ss = 0.f;
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {  // 64 columns per TMEM round trip
        uint32_t ra[32], rb[32];
        tmem_ld32(lane_base + kOCol + c2 * 64, ra);
        tmem_ld32(lane_base + kOCol + c2 * 64 + 32, rb);
        tmem_wait_ld();
        reg_fence(ra);
        reg_fence(rb);
        uint32_t pk[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const uint32_t* src = x < 16 ? ra : rb;
          const int e = (x & 15) * 2;
          const float a = __uint_as_float(src[e]) * inv, b = __uint_as_float(src[e + 1]) * inv;
          ss = fmaf(a, a, fmaf(b, b, ss));
          pk[x] = pack_bf16x2(a, b);
        }
        if (orow && row < N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c2 * 64);
#pragma unroll
          for (int x = 0; x < 8; ++x) dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.o_free));
      if (row < N) sqn[(size_t)h * N + row] = ss;
      return true;
    };
    bool ok = true;
    float l_prev = 1.f;
    for (int t = 0; t < cnt; ++t) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full), t & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      // chunk c holds audio tokens 32c .. 32c + 31: block c / 4, columns 32 (c % 4) ..
      uint32_t sr[NCH][32];
#pragma unroll
      for (int c = 0; c < NCH; ++c) tmem_ld32(lane_base + (c >> 2) * kRows + (c & 3) * 32, sr[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < NCH; ++c) reg_fence(sr[c]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.s_free));  // S(t + 1) may overwrite it now
      float m8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (c < NCH - 1 || 32 * c + e < M) m8[e & 7] = fmaxf(m8[e & 7], __uint_as_float(sr[c][e]));
      const float mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      const f2 scale2 = f2_make(kSl2, kSl2), shift2 = f2_make(-mx * kSl2, -mx * kSl2);
      f2 ls2 = f2_make(0.f, 0.f);
      uint32_t pk[NCH][16];
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float a0, a1;
          f2_split(f2_fma(f2_make(__uint_as_float(sr[c][2 * e]), __uint_as_float(sr[c][2 * e + 1])), scale2, shift2),
                   a0, a1);
          const float p0 = c < NCH - 1 || 32 * c + 2 * e < M ? fast_exp2(a0) : 0.f;
          const float p1 = c < NCH - 1 || 32 * c + 2 * e + 1 < M ? fast_exp2(a1) : 0.f;
          ls2 = f2_add(ls2, f2_make(p0, p1));
          pk[c][e] = pack_bf16x2(p0, p1);
        }
      float l0, l1;
      f2_split(ls2, l0, l1);
      // P V(t - 1) has run meanwhile: finish tile t - 1, which also frees the P columns
      if (t > 0 && !(ok = epilogue(t - 1, l_prev))) break;
      l_prev = l0 + l1;
#pragma unroll
      for (int c = 0; c < NCH; ++c) tmem_st16(lane_base + kPCol + (c >> 2) * 64 + (c & 3) * 16, pk[c]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_full));
    }
    if (ok && cnt > 0) epilogue(cnt - 1, l_prev);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

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

cudaError_t a2v_attn_launch(const void* qv, const void* ka, const void* va, int64_t ld_v, int64_t ld_a, int N,
                            int M, int Hh, void* o, float* sqn, cudaStream_t st, uint32_t* status) {
  const int nbq = (N + kRows - 1) / kRows, nbk = (M + kRows - 1) / kRows;
  if (M > 32 * kMaxChunks)  // longer audio: the general kernel, every key block, online softmax
    return attn_fwd_tc_launch(qv, ka, va, ld_v, ld_a, N, M, Hh, nullptr, nullptr, nbq, nbk, nullptr, nullptr, o, nullptr, sqn,
                              "a2v_attn", st, status);
  CUtensorMap mq, mk, mv, mk1, mv1;
  const uint64_t inner = (uint64_t)Hh * kHd;
  if (!tensor_map_2d_bf16(&mq, qv, inner, N, (uint64_t)ld_v * 2, 64, kRows) ||
      !tensor_map_2d_bf16(&mk, ka, inner, M, (uint64_t)ld_a * 2, 64, kRows) ||
      !tensor_map_2d_bf16(&mv, va, inner, M, (uint64_t)ld_a * 2, 64, kRows) ||
      !tensor_map_2d_bf16(&mk1, ka, inner, M, (uint64_t)ld_a * 2, 64, kTailRows) ||
      !tensor_map_2d_bf16(&mv1, va, inner, M, (uint64_t)ld_a * 2, 64, kTailRows))
    return cudaErrorInvalidValue;
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, __nv_bfloat16*, int64_t, float*,
               int, int, int, int, int, uint32_t*) = nullptr;
  switch ((M + 31) >> 5) {
    case 1: kern = a2v_attn_kernel<1>; break;
    case 2: kern = a2v_attn_kernel<2>; break;
    case 3: kern = a2v_attn_kernel<3>; break;
    case 4: kern = a2v_attn_kernel<4>; break;
    default: kern = a2v_attn_kernel<5>; break;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kA2vSmemBytes);
  if (e != cudaSuccess) return e;
  const int items = Hh * nbq;
  int sms = 148;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  const int grid = items < sms ? items : sms;
  HookScope hs("a2v_attn", st);
  kern<<<grid, kA2vThreads, kA2vSmemBytes, st>>>(mq, mk, mv, mk1, mv1, static_cast<__nv_bfloat16*>(o), ld_v, sqn,
                                                          N, M, nbq, nbk, items, status);
  return cudaGetLastError();
}

cudaError_t a2v_reduce_launch(const float* sqn, int N, int Hh, float* a2v, cudaStream_t st) {
  HookScope hs("a2v_reduce", st);
  a2v_reduce_kernel<<<(unsigned)((N + 255) / 256), 256, 0, st>>>(sqn, N, Hh, a2v);
  return cudaGetLastError();
}

}  // namespace prism
