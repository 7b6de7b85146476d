// Step 5 of the path on the tensor cores: gradients of Prism Block Sparse Attention
// for training, bf16, d = 128, 128-token blocks (sm_103a: TMA + tcgen05 + TMEM).
//
// "Prism: dynamic sparse attention for 2K joint video-audio generation training":
// training runs with Prism BSA on (section "Region-adapted block construction",
// paragraph 2; "Data preparation and training procedure").  With the kept lists
// held constant:  P = exp(S - lse), dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
// dS = P * (dP - D), dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d).
//
// Three kernels, no atomics (deterministic):
//   bwd_prep  L2[h][r] = lse * log2(e) (+inf past the last token, so padded query
//             rows get P = 0) and D[h][r], padded to whole blocks so the attention
//             kernels can bulk-copy 128 of them at a time;
//   dq        one CTA per (head, query block) walking its kept list:
//               S = Q K_j^T (TMEM), dP = dO V_j^T (TMEM), dS = P (dP - D) in bf16 into
//               a TMEM buffer of its own (double-buffered), dQ += dS K_j (A from TMEM);
//   dkdv      one CTA per (head, key block) walking the query blocks that kept it:
//               S^T = K_j Q_i^T, dP^T = V_j dO_i^T (TMEM),
//               P^T, dS^T in bf16 into those buffers, dV += P^T dO_i, dK += dS^T Q_i.
// Both attention kernels have one TMA producer warp, two MMA-issuing threads (one for
// the products that feed the softmax gradient, one for the accumulating products, so
// neither stream waits behind the other) and two warpgroups of softmax-gradient warps,
// each thread owning one TMEM lane (row) and half of the block's columns; each half is
// released as soon as it is written, so the products of one half overlap the
// arithmetic of the other.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstddef>

#include "common.cuh"
#include "internal.h"

namespace prism {
namespace {

constexpr int kB = 128;
constexpr int kD = 128;
constexpr uint32_t kHalf = 16384;
constexpr uint32_t kTile = 2 * kHalf;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSl2 = 1.4426950408889634f * 0.08838834764831845f;  // log2(e) / sqrt(128)
constexpr float kScale = 0.08838834764831845f;                      // 1 / sqrt(128)

// ------------------------------------------------------------------- prep
// 16 threads per (head, padded row), 8 channels (one 16-byte load of O and of dO) each.
// With dqacc != NULL it also clears the fused kernel's fp32 dQ accumulator
// ([Hh][npad][d]): each thread zeroes the 8 accumulator channels it owns.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dO,
                                                       const float* __restrict__ lse, int64_t ld, int N, int Hh,
                                                       int npad, float* __restrict__ L2, float* __restrict__ Dp,
                                                       float* __restrict__ dqacc, const int32_t* __restrict__ blen) {
  const int64_t gid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 4;
  const int sub = threadIdx.x & 15;
  if (gid >= (int64_t)Hh * npad) return;  // 16-lane groups are whole: the group exits together
  // rows fastest within a head, so consecutive groups read consecutive token rows
  const int h = (int)(gid / npad), r = (int)(gid - (int64_t)h * npad);
  if (dqacc) {
    float4* z = reinterpret_cast<float4*>(dqacc + ((int64_t)h * npad + r) * kD + sub * 8);
    z[0] = z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float s = 0.f;
  // padding rows of zone-chunked blocks are no queries: P = 0 there, like past the end
  const bool row_ok = r < N && (!blen || (r & (kB - 1)) < blen[r / kB]);
  if (row_ok) {
    const int64_t off = (int64_t)r * ld + (int64_t)h * kD + sub * 8;
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + off));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(dO + off));
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = __bfloat1622float2(a2[k]), y = __bfloat1622float2(b2[k]);
      s = fmaf(x.x, y.x, fmaf(x.y, y.y, s));
    }
  }
  const unsigned grp = 0xffffu << (threadIdx.x & 16);
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(grp, s, off);
  if (sub == 0) {
    const size_t at = (size_t)h * npad + r;
    Dp[at] = row_ok ? s : 0.f;
    L2[at] = row_ok ? lse[(size_t)h * N + r] * kLog2e : INFINITY;
  }
}

// --------------------------------------------------------------------- dQ
// Warps: 0 TMA producer, 1 issuer of S and dP (TMEM owner), 10 issuer of dQ,
// 2-5 softmax gradient of key columns 0-63 of every block, 6-9 of columns 64-127
// (a thread owns one query row of one half).
constexpr int kDqThreads = 352;

constexpr int kDqKStages = 3, kDqVStages = 2;
struct DqSmem {
  uint8_t q[kTile];
  uint8_t dO[kTile];
  uint8_t k[kDqKStages][kTile];
  uint8_t v[kDqVStages][kTile];
  uint64_t q_full;
  uint64_t k_full[kDqKStages], k_empty[kDqKStages];  // K_t: read by S(t) and dQ(t)
  uint64_t v_full[kDqVStages], v_empty[kDqVStages];  // V_t: read by dP(t) only
  uint64_t s_full, dp_full, dp_free;  // dp_free: S(t) and dP(t) are in the softmax's registers
  uint64_t ds_full[2][2];  // [dS buffer][key half]
  uint64_t dq_done[2];     // dQ(t) has read dS buffer t & 1
  uint64_t a_issued;       // the S / dP issuer has enqueued block t + 1's products
  uint64_t acc_done, in_done;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kDqSmemBytes = sizeof(DqSmem) + 1024;
static_assert(kDqSmemBytes <= 232448, "shared memory budget");

// TMEM: S [0,128) dS0 [128,192) dS1 [192,256) dP [256,384) dQ [384,512).
// Two issuing threads:
//   warp 1   dP(t+1) and S(t+1) as soon as both halves have loaded S(t) and dP(t) into
//            registers (S and dP are single-buffered), so the next block's inputs are
//            computed while block t's gradient is formed, whatever the dQ products do;
//   warp 10  dQ(t) += dS(t) K_t in two K = 64 steps, one per key half, as soon as that
//            half's warpgroup has written it;
// dS(t) (bf16 pairs) goes into dS buffer t & 1, which the softmax overwrites only after
// dQ(t - 2), its last reader, has completed.
__global__ void __launch_bounds__(kDqThreads, 1)
    bsa_dq_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                     const float* __restrict__ L2, const float* __restrict__ Dp, int npad,
                     __nv_bfloat16* __restrict__ dq, int64_t ld, int N, const int32_t* __restrict__ counts,
                     const int32_t* __restrict__ idx, int nb, const int32_t* __restrict__ blen,
                     const int32_t* __restrict__ order, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  DqSmem& sm = *reinterpret_cast<DqSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = order ? order[blockIdx.x] : (int)blockIdx.x;
  if (item < 0 || item >= (int)gridDim.x) {
    if (threadIdx.x == 0) flag_error(status, PRISM_DEV_BAD_INDEX);
    return;
  }
  const int h = item / nb, i = item - h * nb;
  int cnt = counts[item];
  if (cnt < 0 || cnt > nb) cnt = cnt < 0 ? 0 : nb;
  const int32_t* lst = idx + (size_t)item * nb;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    for (int s = 0; s < kDqKStages; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), 1);
      mbar_init(smem_u32(&sm.k_empty[s]), 1);
    }
    for (int s = 0; s < kDqVStages; ++s) {
      mbar_init(smem_u32(&sm.v_full[s]), 1);
      mbar_init(smem_u32(&sm.v_empty[s]), 1);
    }
    mbar_init(smem_u32(&sm.s_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&sm.ds_full[s][0]), 4);
      mbar_init(smem_u32(&sm.ds_full[s][1]), 4);
    }
    mbar_init(smem_u32(&sm.dp_full), 1);
    mbar_init(smem_u32(&sm.dp_free), 8);
    mbar_init(smem_u32(&sm.dq_done[0]), 1);
    mbar_init(smem_u32(&sm.dq_done[1]), 1);
    mbar_init(smem_u32(&sm.a_issued), 1);
    mbar_init(smem_u32(&sm.acc_done), 1);
    mbar_init(smem_u32(&sm.in_done), 1);
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
    if (lane == 0 && cnt > 0) {
      const uint32_t qb = smem_u32(&sm.q_full);
      mbar_arrive_expect_tx(qb, 2 * kTile);
      tma_load_2d(smem_u32(sm.q), &tmq, h * kD, i * kB, qb);
      tma_load_2d(smem_u32(sm.q) + kHalf, &tmq, h * kD + 64, i * kB, qb);
      tma_load_2d(smem_u32(sm.dO), &tmdo, h * kD, i * kB, qb);
      tma_load_2d(smem_u32(sm.dO) + kHalf, &tmdo, h * kD + 64, i * kB, qb);
      // K and V in separate rings: V_t is free once dP(t) has completed, K_t only once
      // dQ(t) has, so V can run further ahead than K
      int karmed[kDqKStages] = {0, 0, 0}, varmed[kDqVStages] = {0, 0};
      for (int it = 0; it < cnt; ++it) {
        const int ks = it % kDqKStages, vs = it % kDqVStages;
        int j = lst[it];
        if (j < 0 || j >= nb) j = 0;
        if (it >= kDqVStages && !mbar_wait(smem_u32(&sm.v_empty[vs]), ((it / kDqVStages) - 1) & 1, abort, status)) break;
        const uint32_t vbar = smem_u32(&sm.v_full[vs]);
        mbar_arrive_expect_tx(vbar, kTile);
        tma_load_2d(smem_u32(sm.v[vs]), &tmv, h * kD, j * kB, vbar);
        tma_load_2d(smem_u32(sm.v[vs]) + kHalf, &tmv, h * kD + 64, j * kB, vbar);
        ++varmed[vs];
        if (it >= kDqKStages && !mbar_wait(smem_u32(&sm.k_empty[ks]), ((it / kDqKStages) - 1) & 1, abort, status)) break;
        const uint32_t kbar = smem_u32(&sm.k_full[ks]);
        mbar_arrive_expect_tx(kbar, kTile);
        tma_load_2d(smem_u32(sm.k[ks]), &tmk, h * kD, j * kB, kbar);
        tma_load_2d(smem_u32(sm.k[ks]) + kHalf, &tmk, h * kD + 64, j * kB, kbar);
        ++karmed[ks];
      }
      if (*abort) {
        drain_wait(qb, 0);
        for (int s = 0; s < kDqKStages; ++s)
          if (karmed[s]) drain_wait(smem_u32(&sm.k_full[s]), (karmed[s] - 1) & 1);
        for (int s = 0; s < kDqVStages; ++s)
          if (varmed[s]) drain_wait(smem_u32(&sm.v_full[s]), (varmed[s] - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------- issuer of S and dP
    if (lane == 0 && cnt > 0) {
      constexpr uint32_t id_ss = idesc_bf16_f32(kB, kB, false, false);
      const uint64_t dq_q = smem_desc(smem_u32(sm.q), 16, 1024, kSwizzle128B);
      const uint64_t dq_do = smem_desc(smem_u32(sm.dO), 16, 1024, kSwizzle128B);
      const uint64_t dk0 = smem_desc(smem_u32(sm.k[0]), 16, 1024, kSwizzle128B);
      const uint64_t dv0 = smem_desc(smem_u32(sm.v[0]), 16, 1024, kSwizzle128B);
      auto koff = [](int kk) -> uint32_t { return (kk >> 2) * kHalf + (kk & 3) * 32; };
      auto issue_dp = [&](int t) {  // dP(t) = dO V_t^T; V_t's stage is free once it completes
        const int vs = t % kDqVStages;
        const uint64_t dv = desc_at(dv0, vs * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tmem + 256, desc_at(dq_do, koff(kk)), desc_at(dv, koff(kk)), id_ss, kk > 0);
        tc_commit(smem_u32(&sm.dp_full));
        tc_commit(smem_u32(&sm.v_empty[vs]));
      };
      auto issue_s = [&](int t) {  // S(t) = Q K_t^T
        const uint64_t dk = desc_at(dk0, (t % kDqKStages) * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tmem, desc_at(dq_q, koff(kk)), desc_at(dk, koff(kk)), id_ss, kk > 0);
        tc_commit(smem_u32(&sm.s_full));
      };
      bool ok = mbar_wait(smem_u32(&sm.q_full), 0, abort, status) &&
                mbar_wait(smem_u32(&sm.v_full[0]), 0, abort, status) &&
                mbar_wait(smem_u32(&sm.k_full[0]), 0, abort, status);
      if (ok) {
        tc_fence_after();
        issue_dp(0);
        issue_s(0);
      }
      for (int it = 0; ok && it + 1 < cnt; ++it) {
        const int t = it + 1;
        if (!(ok = mbar_wait(smem_u32(&sm.dp_free), it & 1, abort, status))) break;
        if (!(ok = mbar_wait(smem_u32(&sm.v_full[t % kDqVStages]), (t / kDqVStages) & 1, abort, status))) break;
        tc_fence_after();
        issue_dp(t);
        if (!(ok = mbar_wait(smem_u32(&sm.k_full[t % kDqKStages]), (t / kDqKStages) & 1, abort, status))) break;
        tc_fence_after();
        issue_s(t);
        mbar_arrive(smem_u32(&sm.a_issued));  // dQ(t - 1) may follow them into the tensor pipe
      }
      tc_commit(smem_u32(&sm.in_done));
      drain_wait(smem_u32(&sm.in_done), 0);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ issuer of dQ
    if (lane == 0 && cnt > 0) {
      constexpr uint32_t id_ts = idesc_bf16_f32(kB, kD, false, true);
      const uint64_t dkmn0 = smem_desc(smem_u32(sm.k[0]), kHalf, 1024, kSwizzle128B);
      bool ok = true;
      for (int it = 0; ok && it < cnt; ++it) {
        const int b = it & 1, ks = it % kDqKStages;
        const uint64_t dkt = desc_at(dkmn0, ks * kTile);
        // the next block's S and dP go first: the softmax waits on them, nothing waits on dQ
        if (it + 1 < cnt && !(ok = mbar_wait(smem_u32(&sm.a_issued), it & 1, abort, status))) break;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if (!(ok = mbar_wait(smem_u32(&sm.ds_full[b][half]), (it >> 1) & 1, abort, status))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + 384, tmem + 128 + b * 64 + half * 32 + kk * 8, desc_at(dkt, (half * 4 + kk) * 2048), id_ts,
                   (it > 0 || half > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.k_empty[ks]));
        tc_commit(smem_u32(&sm.dq_done[b]));
      }
      // every dQ product has completed once this barrier flips; every S and dP product
      // completed before the softmax could write the last block's dS
      tc_commit(smem_u32(&sm.acc_done));
      drain_wait(smem_u32(&sm.acc_done), 0);
    }
  } else {
    const int half = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int c0 = half * 64;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const int row = i * kB + r;
    const float l2 = L2[(size_t)h * npad + row];
    const float dr = Dp[(size_t)h * npad + row];
    const f2 scale2 = f2_make(kSl2, kSl2), neg_l2 = f2_make(-l2, -l2), neg_dr = f2_make(-dr, -dr);
    bool ok = true;
    int j_next = cnt > 0 ? lst[0] : 0;  // block indices are read one block ahead
    for (int it = 0; it < cnt; ++it) {
      const int b = it & 1;
      const int j = j_next;
      if (it + 1 < cnt) j_next = lst[it + 1];
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full), it & 1, abort, status) &&
                                       mbar_wait(smem_u32(&sm.dp_full), it & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      const int len = (j >= 0 && j < nb) ? (blen ? min(kB, max(0, blen[j])) : min(kB, N - j * kB)) : 0;
      uint32_t s0[32], s1[32], d0[32], d1[32];
      tmem_ld32(lane_base + c0, s0);
      tmem_ld32(lane_base + c0 + 32, s1);
      tmem_ld32(lane_base + 256 + c0, d0);
      tmem_ld32(lane_base + 256 + c0 + 32, d1);
      tmem_wait_ld();
      reg_fence(s0);
      reg_fence(s1);
      reg_fence(d0);
      reg_fence(d1);
      // S and dP are in registers: the next block's products may overwrite them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.dp_free));
      if (len < c0 + 64) {  // short or skipped key block (warp-uniform): masked keys get P = 0
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          if (c0 + x >= len) s0[x] = __float_as_uint(-INFINITY);
          if (c0 + 32 + x >= len) s1[x] = __float_as_uint(-INFINITY);
        }
      }
      // dS buffer b was last read by dQ(it - 2): long done unless the tensor pipe is far
      // behind (a completed phase is seen by the non-blocking test at once)
      if (it >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.dq_done[b]), ((it >> 1) - 1) & 1, abort, status));
        if (!ok) break;
        tc_fence_after();
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const uint32_t* sr = cc ? s1 : s0;
        const uint32_t* pr = cc ? d1 : d0;
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          float a0, a1;
          f2_split(f2_fma(f2_make(__uint_as_float(sr[2 * x]), __uint_as_float(sr[2 * x + 1])), scale2, neg_l2), a0, a1);
          const f2 p = f2_make(fast_exp2(a0), fast_exp2(a1));
          const f2 g = f2_add(f2_make(__uint_as_float(pr[2 * x]), __uint_as_float(pr[2 * x + 1])), neg_dr);
          pk[x] = f2_pack_bf16(f2_mul(p, g));  // dS = P (dP - D)
        }
        tmem_st16(lane_base + 128 + b * 64 + half * 32 + cc * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.ds_full[b][half]));
    }
    __nv_bfloat16* out = dq + (int64_t)row * ld + (int64_t)h * kD + c0;
    if (ok && cnt > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.acc_done), 0, abort, status));
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t rr[32];
          tmem_load_row32(lane_base + 384 + c0 + c2 * 32, rr);
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x)
            pk[x] = pack_bf16x2(__uint_as_float(rr[2 * x]) * kScale, __uint_as_float(rr[2 * x + 1]) * kScale);
          if (row < N) {
            uint4* dst = reinterpret_cast<uint4*>(out + c2 * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x) dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
          }
        }
      }
    } else if (cnt == 0 && row < N) {
      uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
      for (int x = 0; x < 8; ++x) dst[x] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------- dK dV
// Warps: 0 TMA producer, 1 issuer of S^T and dP^T (TMEM owner), 10 issuer of dV and
// dK, 2-5 softmax gradient of query columns 0-63 of every query block, 6-9 of
// columns 64-127; a thread owns one key row (its TMEM lane) of one half.
constexpr int kDkdvThreads = 352;

struct QdoStage {
  uint8_t q[kTile];
  uint8_t dO[kTile];
};
struct DkdvSmem {
  uint8_t k[kTile];
  uint8_t v[kTile];
  QdoStage st[2];
  float l2[2][kB];  // lse * log2(e) of the stage's query rows
  float dr[2][kB];  // D of the stage's query rows
  uint64_t kv_full;
  uint64_t qdo_full[2], qdo_empty[2];
  uint64_t s_full[2], dp_full[2];  // [query half]: S^T, dP^T of that half computed
  uint64_t p_full[2], ds_full[2];  // [query half]: P^T, dS^T of that half written
  uint64_t v_done[2], k_done[2];   // [query half]: dV has read P^T / dK has read dS^T
  uint64_t acc_done, in_done;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kDkdvSmemBytes = sizeof(DkdvSmem) + 1024;
static_assert(kDkdvSmemBytes <= 232448, "shared memory budget");
static_assert(sizeof(QdoStage) % 1024 == 0, "stages keep 1024-byte alignment for the swizzled tiles");

// TMEM: S^T_a [0,64) S^T_b [64,128) dP^T_a [128,192) dP^T_b [192,256) dV [256,384)
// dK [384,512); half a = query rows 0-63 of the query block, half b = rows 64-127.
// Per query half x and pair t:  S^T_x = K Q_x^T and dP^T_x = V dO_x^T (N = 64);
// the half's warpgroup writes P^T_x (bf16) over the first 32 columns of S^T_x and
// dS^T_x over the first 32 of dP^T_x; dV += P^T_x dO_x and dK += dS^T_x Q_x (K = 64).
// Two issuing threads: warp 10 issues dV of a half as soon as its P^T is written and
// dK as soon as its dS^T is; warp 1 issues the next pair's S^T_x once that dV has
// completed and dP^T_x once that dK has.  So a half's S^T -> P^T -> dV chain does not
// wait for its dS^T, and the halves alternate in the tensor pipe: one half's products
// run while the other half's softmax gradient is computed.
__global__ void __launch_bounds__(kDkdvThreads, 1)
    bsa_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                       const float* __restrict__ L2, const float* __restrict__ Dp, int npad,
                       __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int64_t ld, int N,
                       const int32_t* __restrict__ tcounts, const int32_t* __restrict__ tidx, int nb,
                       const int32_t* __restrict__ blen, const int32_t* __restrict__ order, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  DkdvSmem& sm = *reinterpret_cast<DkdvSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = order ? order[blockIdx.x] : (int)blockIdx.x;
  if (item < 0 || item >= (int)gridDim.x) {
    if (threadIdx.x == 0) flag_error(status, PRISM_DEV_BAD_INDEX);
    return;
  }
  const int h = item / nb, j = item - h * nb;
  const int cnt = tcounts[item];
  const int32_t* lst = tidx + (size_t)item * nb;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.kv_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&sm.qdo_full[s]), 1);
      mbar_init(smem_u32(&sm.qdo_empty[s]), 1);
      mbar_init(smem_u32(&sm.s_full[s]), 1);
      mbar_init(smem_u32(&sm.dp_full[s]), 1);
      mbar_init(smem_u32(&sm.p_full[s]), 4);
      mbar_init(smem_u32(&sm.ds_full[s]), 4);
      mbar_init(smem_u32(&sm.v_done[s]), 1);
      mbar_init(smem_u32(&sm.k_done[s]), 1);
    }
    mbar_init(smem_u32(&sm.acc_done), 1);
    mbar_init(smem_u32(&sm.in_done), 1);
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
    if (lane == 0 && cnt > 0) {
      const uint32_t kvb = smem_u32(&sm.kv_full);
      mbar_arrive_expect_tx(kvb, 2 * kTile);
      tma_load_2d(smem_u32(sm.k), &tmk, h * kD, j * kB, kvb);
      tma_load_2d(smem_u32(sm.k) + kHalf, &tmk, h * kD + 64, j * kB, kvb);
      tma_load_2d(smem_u32(sm.v), &tmv, h * kD, j * kB, kvb);
      tma_load_2d(smem_u32(sm.v) + kHalf, &tmv, h * kD + 64, j * kB, kvb);
      int armed[2] = {0, 0};
      for (int it = 0; it < cnt; ++it) {
        const int s = it & 1;
        if (it >= 2 && !mbar_wait(smem_u32(&sm.qdo_empty[s]), ((it >> 1) - 1) & 1, abort, status)) break;
        const int i = lst[it];
        QdoStage& g = sm.st[s];
        const uint32_t bar = smem_u32(&sm.qdo_full[s]);
        mbar_arrive_expect_tx(bar, 2 * kTile + 2 * kB * 4);
        tma_load_2d(smem_u32(g.q), &tmq, h * kD, i * kB, bar);
        tma_load_2d(smem_u32(g.q) + kHalf, &tmq, h * kD + 64, i * kB, bar);
        tma_load_2d(smem_u32(g.dO), &tmdo, h * kD, i * kB, bar);
        tma_load_2d(smem_u32(g.dO) + kHalf, &tmdo, h * kD + 64, i * kB, bar);
        bulk_load(smem_u32(sm.l2[s]), L2 + (size_t)h * npad + (size_t)i * kB, kB * 4, bar);
        bulk_load(smem_u32(sm.dr[s]), Dp + (size_t)h * npad + (size_t)i * kB, kB * 4, bar);
        ++armed[s];
      }
      if (*abort) {
        drain_wait(kvb, 0);
        for (int s = 0; s < 2; ++s)
          if (armed[s]) drain_wait(smem_u32(&sm.qdo_full[s]), (armed[s] - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ issuer of S^T and dP^T
    if (lane == 0 && cnt > 0) {
      constexpr uint32_t id_h = idesc_bf16_f32(kB, 64, false, false);  // M = 128 keys, N = 64 queries
      const uint64_t dk_k = smem_desc(smem_u32(sm.k), 16, 1024, kSwizzle128B);
      const uint64_t dk_v = smem_desc(smem_u32(sm.v), 16, 1024, kSwizzle128B);
      const uint64_t dq0 = smem_desc(smem_u32(sm.st[0].q), 16, 1024, kSwizzle128B);
      const uint64_t ddo0 = smem_desc(smem_u32(sm.st[0].dO), 16, 1024, kSwizzle128B);
      auto koff = [](int kk) -> uint32_t { return (kk >> 2) * kHalf + (kk & 3) * 32; };
      bool ok = mbar_wait(smem_u32(&sm.kv_full), 0, abort, status);
      for (int it = 0; ok && it < cnt; ++it) {
        const int s = it & 1;
        if (!(ok = mbar_wait(smem_u32(&sm.qdo_full[s]), (it >> 1) & 1, abort, status))) break;
        const uint32_t so = s * (uint32_t)sizeof(QdoStage);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          // the half's rows of the Q / dO tiles start 64 rows (8 KB) into each box
          const uint64_t dq = desc_at(dq0, so + half * 8192), ddo = desc_at(ddo0, so + half * 8192);
          // S^T_x overwrites the P^T_x that the previous pair's dV read
          if (it > 0 && !(ok = mbar_wait(smem_u32(&sm.v_done[half]), (it - 1) & 1, abort, status))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + half * 64, desc_at(dk_k, koff(kk)), desc_at(dq, koff(kk)), id_h, kk > 0);
          tc_commit(smem_u32(&sm.s_full[half]));
          // dP^T_x overwrites the dS^T_x that the previous pair's dK read
          if (it > 0 && !(ok = mbar_wait(smem_u32(&sm.k_done[half]), (it - 1) & 1, abort, status))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + 128 + half * 64, desc_at(dk_v, koff(kk)), desc_at(ddo, koff(kk)), id_h, kk > 0);
          tc_commit(smem_u32(&sm.dp_full[half]));
        }
      }
      tc_commit(smem_u32(&sm.in_done));
      drain_wait(smem_u32(&sm.in_done), 0);
    }
  } else if (warp == 10) {
    // -------------------------------------------------- issuer of dV and dK
    if (lane == 0 && cnt > 0) {
      constexpr uint32_t id_ts = idesc_bf16_f32(kB, kD, false, true);
      const uint64_t dqmn0 = smem_desc(smem_u32(sm.st[0].q), kHalf, 1024, kSwizzle128B);
      const uint64_t ddomn0 = smem_desc(smem_u32(sm.st[0].dO), kHalf, 1024, kSwizzle128B);
      bool ok = true;
      for (int it = 0; ok && it < cnt; ++it) {
        const int s = it & 1;
        const uint32_t so = s * (uint32_t)sizeof(QdoStage);
        const uint64_t dqmn = desc_at(dqmn0, so), ddomn = desc_at(ddomn0, so);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if (!(ok = mbar_wait(smem_u32(&sm.p_full[half]), it & 1, abort, status))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // dV += P^T_x dO_x
            mma_ts(tmem + 256, tmem + half * 64 + kk * 8, desc_at(ddomn, (half * 4 + kk) * 2048), id_ts,
                   (it > 0 || half > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&sm.v_done[half]));
          if (!(ok = mbar_wait(smem_u32(&sm.ds_full[half]), it & 1, abort, status))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // dK += dS^T_x Q_x
            mma_ts(tmem + 384, tmem + 128 + half * 64 + kk * 8, desc_at(dqmn, (half * 4 + kk) * 2048), id_ts,
                   (it > 0 || half > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&sm.k_done[half]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.qdo_empty[s]));
      }
      // every dV / dK product has completed once this barrier flips; every S^T and dP^T
      // product completed before the softmax could write the last pair's P^T, dS^T
      tc_commit(smem_u32(&sm.acc_done));
      drain_wait(smem_u32(&sm.acc_done), 0);
    }
  } else {
    const int half = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int c = quarter * 32 + lane;  // key row of block j = TMEM lane
    const int q0 = half * 64;           // this thread's query columns q0 .. q0 + 63
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const bool key_ok = blen ? c < blen[j] : j * kB + c < N;
    const f2 scale2 = f2_make(kSl2, kSl2);
    bool ok = true;
    for (int it = 0; it < cnt; ++it) {
      const int s = it & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.qdo_full[s]), (it >> 1) & 1, abort, status) &&
                                       mbar_wait(smem_u32(&sm.s_full[half]), it & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      const float4* l2v = reinterpret_cast<const float4*>(sm.l2[s] + q0);
      const float4* drv = reinterpret_cast<const float4*>(sm.dr[s] + q0);
      f2 p[32];  // P^T of this key row and the half's 64 query columns, fp32 pairs
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {  // 32 query columns at a time
        uint32_t sr[32];
        tmem_load_row32(lane_base + q0 + cc * 32, sr);
        uint32_t pp[16];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {  // 4 query columns per vector load of the row statistics
          const float4 L = l2v[cc * 8 + q4];
#pragma unroll
          for (int u = 0; u < 2; ++u) {  // two query columns per packed pair
            const int e = 4 * q4 + 2 * u;
            const f2 nl = u ? f2_make(-L.z, -L.w) : f2_make(-L.x, -L.y);
            float a0, a1;
            f2_split(f2_fma(f2_make(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), scale2, nl), a0, a1);
            p[cc * 16 + 2 * q4 + u] = key_ok ? f2_make(fast_exp2(a0), fast_exp2(a1)) : f2_make(0.f, 0.f);
            pp[2 * q4 + u] = f2_pack_bf16(p[cc * 16 + 2 * q4 + u]);
          }
        }
        // P^T_x over the first 32 columns of S^T_x (this chunk's columns were read above;
        // the writes land in columns already read)
        tmem_st16(lane_base + q0 + cc * 16, pp);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_full[half]));
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.dp_full[half]), it & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t pr[32];
        tmem_load_row32(lane_base + 128 + q0 + cc * 32, pr);
        uint32_t dd[16];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 Dv = drv[cc * 8 + q4];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = 4 * q4 + 2 * u;
            const f2 nd = u ? f2_make(-Dv.z, -Dv.w) : f2_make(-Dv.x, -Dv.y);
            dd[2 * q4 + u] = f2_pack_bf16(
                f2_mul(p[cc * 16 + 2 * q4 + u], f2_add(f2_make(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1])), nd)));
          }
        }
        // dS^T_x over the first 32 columns of dP^T_x
        tmem_st16(lane_base + 128 + q0 + cc * 16, dd);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.ds_full[half]));
    }
    const int col = j * kB + c;
    __nv_bfloat16* dk_row = dk + (int64_t)col * ld + (int64_t)h * kD + q0;
    __nv_bfloat16* dv_row = dv + (int64_t)col * ld + (int64_t)h * kD + q0;
    if (ok && cnt > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.acc_done), 0, abort, status));
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int which = 0; which < 2; ++which) {  // dV, then dK (scaled by 1/sqrt(d))
          __nv_bfloat16* out = which ? dk_row : dv_row;
          const float sc = which ? kScale : 1.f;
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t rr[32];
            tmem_load_row32(lane_base + 256 + which * 128 + q0 + c2 * 32, rr);
            uint32_t pk[16];
#pragma unroll
            for (int x = 0; x < 16; ++x)
              pk[x] = pack_bf16x2(__uint_as_float(rr[2 * x]) * sc, __uint_as_float(rr[2 * x + 1]) * sc);
            if (col < N) {
              uint4* dst = reinterpret_cast<uint4*>(out + c2 * 32);
#pragma unroll
              for (int x = 0; x < 4; ++x)
                dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
            }
          }
        }
      }
    } else if (cnt == 0 && col < N) {
      uint4* a = reinterpret_cast<uint4*>(dk_row);
      uint4* b = reinterpret_cast<uint4*>(dv_row);
#pragma unroll
      for (int x = 0; x < 8; ++x) a[x] = b[x] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------- fused dK, dV, dQ
// One CTA per (head, key block j) walking the query blocks that kept j, like dkdv,
// that also forms dQ.  Per kept query block i:
//   S^T = K_j Q_i^T, dP^T = V_j dO_i^T                (TMEM, M = 128 keys, N = 128 queries)
//   P^T, dS^T (bf16, per query half x of 64 queries, written by that half's warps)
//   dV += P^T_x dO_x, dK += dS^T_x Q_x               (A from TMEM, K = 64 per half)
//   dQ_i^T = K_j^T dS^T                               (M = 128 channels, N = 128 queries,
//                                                      K = 128 keys; both operands
//                                                      MN-major in shared memory: K_j's
//                                                      tile as loaded, dS^T as written
//                                                      by the softmax warps)
// and adds dQ_i into an fp32 accumulator in global memory ([Hh][npad][d]: the head a
// wave of CTAs works on is one contiguous range) with 16-byte reductions issued
// straight from registers.  Five tile products per kept pair
// instead of the seven of the split kernels (whose dq kernel recomputes S and dP), all
// 128 x 128 x 128 (full-width products read 64 KB of operands per 512 tensor cycles,
// which shared memory sustains; products split into 64-query halves would read 1.5x as
// much per FLOP).  The reduce-adds make dQ's summation order, and so its last bits,
// depend on scheduling.
//
// Warps: 0 TMA producer, 1 issuer of S^T and dP^T (TMEM owner), 2 issuer of dV, dK
// and dQ^T, 3 idle; 4-7 softmax gradient of query rows 0-63 (half a) of every query
// block, 8-11 of rows 64-127 (half b), a thread per key row (its TMEM lane); 12-15
// the dQ drain, a thread per channel (TMEM lane of dQ^T).
constexpr int kFusedThreads = 512;

struct FusedSmem {
  uint8_t k[kTile];
  uint8_t v[kTile];
  QdoStage st[2];
  // dS^T (128 key rows x 128 queries bf16): [query half][128 rows x 128 bytes], each
  // half in the 128-byte-swizzled layout of a loaded tile; the B operand of dQ^T
  uint8_t ds[2][kHalf];
  float l2[2][kB];  // lse * log2(e) of the stage's query rows
  float dr[2][kB];  // D of the stage's query rows
  uint64_t kv_full;
  uint64_t qdo_full[2], qdo_empty[2];
  uint64_t s_full, dp_full;        // S^T, dP^T computed
  uint64_t p_full[2], ds_full[2];  // [query half]: P^T, dS^T written
  uint64_t pair_done;              // dV and dK of the pair have read P^T and dS^T
  uint64_t dq_full;                // dQ^T computed (the dS^T tile read)
  uint64_t dq_free;                // dQ^T loaded by the drain (TMEM columns free)
  uint64_t acc_done, in_done;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kFusedSmemBytes = sizeof(FusedSmem);
static_assert(kFusedSmemBytes <= 232448, "shared memory budget");
static_assert(offsetof(FusedSmem, ds) % 1024 == 0, "swizzled tiles need 1024-byte alignment");

// TMEM: S^T [0,128) (query q in column q), dP^T [128,256), dV [256,384), dK [384,512).
// Query half x (columns 64x .. 64x + 63 of S^T) writes P^T_x (bf16) over the first 32 of
// its own columns and dS^T_x over the last 32; dQ^T is computed into the dP^T columns
// once both halves have loaded them.  Issuer 1: S^T once dV and dK of the previous pair
// have completed; dP^T once the drain has loaded the previous dQ^T.  Issuer 2: dV_a,
// dV_b as the halves' P^T are written, dK_a, dK_b as their dS^T are, then dQ^T.
__global__ void __launch_bounds__(kFusedThreads, 1)
    bsa_bwd_fused_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                         float* __restrict__ dqacc, const float* __restrict__ L2,
                         const float* __restrict__ Dp, int npad, __nv_bfloat16* __restrict__ dk,
                         __nv_bfloat16* __restrict__ dv, int64_t ld, int N, const int32_t* __restrict__ tcounts,
                         const int32_t* __restrict__ tidx, int nb, const int32_t* __restrict__ blen,
                         const int32_t* __restrict__ order, uint32_t* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the swizzled tiles need it; never seen, but checked
    if (threadIdx.x == 0) flag_error(status, PRISM_DEV_TMEM);
    return;
  }
  FusedSmem& sm = *reinterpret_cast<FusedSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = order ? order[blockIdx.x] : (int)blockIdx.x;
  if (item < 0 || item >= (int)gridDim.x) {
    if (threadIdx.x == 0) flag_error(status, PRISM_DEV_BAD_INDEX);
    return;
  }
  const int h = item / nb, j = item - h * nb;
  int cnt = tcounts[item];
  if (cnt < 0 || cnt > nb) cnt = cnt < 0 ? 0 : nb;
  const int32_t* lst = tidx + (size_t)item * nb;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.kv_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&sm.qdo_full[s]), 1);
      mbar_init(smem_u32(&sm.qdo_empty[s]), 1);
      mbar_init(smem_u32(&sm.p_full[s]), 4);
      mbar_init(smem_u32(&sm.ds_full[s]), 4);
    }
    mbar_init(smem_u32(&sm.s_full), 1);
    mbar_init(smem_u32(&sm.dp_full), 1);
    mbar_init(smem_u32(&sm.pair_done), 1);
    mbar_init(smem_u32(&sm.dq_full), 1);
    mbar_init(smem_u32(&sm.dq_free), 4);
    mbar_init(smem_u32(&sm.acc_done), 1);
    mbar_init(smem_u32(&sm.in_done), 1);
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
    // ---------------------------------------------------------------- producer
    if (lane == 0 && cnt > 0) {
      const uint32_t kvb = smem_u32(&sm.kv_full);
      mbar_arrive_expect_tx(kvb, 2 * kTile);
      tma_load_2d(smem_u32(sm.k), &tmk, h * kD, j * kB, kvb);
      tma_load_2d(smem_u32(sm.k) + kHalf, &tmk, h * kD + 64, j * kB, kvb);
      tma_load_2d(smem_u32(sm.v), &tmv, h * kD, j * kB, kvb);
      tma_load_2d(smem_u32(sm.v) + kHalf, &tmv, h * kD + 64, j * kB, kvb);
      int armed[2] = {0, 0};
      for (int it = 0; it < cnt; ++it) {
        const int s = it & 1;
        if (it >= 2 && !mbar_wait(smem_u32(&sm.qdo_empty[s]), ((it >> 1) - 1) & 1, abort, status)) break;
        int i = lst[it];
        if (i < 0 || i >= nb) i = 0;  // lists come from the library's own transpose: never taken
        QdoStage& g = sm.st[s];
        const uint32_t bar = smem_u32(&sm.qdo_full[s]);
        mbar_arrive_expect_tx(bar, 2 * kTile + 2 * kB * 4);
        tma_load_2d(smem_u32(g.q), &tmq, h * kD, i * kB, bar);
        tma_load_2d(smem_u32(g.q) + kHalf, &tmq, h * kD + 64, i * kB, bar);
        tma_load_2d(smem_u32(g.dO), &tmdo, h * kD, i * kB, bar);
        tma_load_2d(smem_u32(g.dO) + kHalf, &tmdo, h * kD + 64, i * kB, bar);
        bulk_load(smem_u32(sm.l2[s]), L2 + (size_t)h * npad + (size_t)i * kB, kB * 4, bar);
        bulk_load(smem_u32(sm.dr[s]), Dp + (size_t)h * npad + (size_t)i * kB, kB * 4, bar);
        ++armed[s];
      }
      if (*abort) {
        drain_wait(kvb, 0);
        for (int s = 0; s < 2; ++s)
          if (armed[s]) drain_wait(smem_u32(&sm.qdo_full[s]), (armed[s] - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ issuer of S^T and dP^T
    if (lane == 0 && cnt > 0) {
      constexpr uint32_t id_ss = idesc_bf16_f32(kB, kB, false, false);  // M = 128 keys, N = 128 queries
      const uint64_t dk_k = smem_desc(smem_u32(sm.k), 16, 1024, kSwizzle128B);
      const uint64_t dk_v = smem_desc(smem_u32(sm.v), 16, 1024, kSwizzle128B);
      const uint64_t dq0 = smem_desc(smem_u32(sm.st[0].q), 16, 1024, kSwizzle128B);
      const uint64_t ddo0 = smem_desc(smem_u32(sm.st[0].dO), 16, 1024, kSwizzle128B);
      auto koff = [](int kk) -> uint32_t { return (kk >> 2) * kHalf + (kk & 3) * 32; };
      bool ok = mbar_wait(smem_u32(&sm.kv_full), 0, abort, status);
      for (int it = 0; ok && it < cnt; ++it) {
        const int s = it & 1;
        const uint32_t so = s * (uint32_t)sizeof(QdoStage);
        if (!(ok = mbar_wait(smem_u32(&sm.qdo_full[s]), (it >> 1) & 1, abort, status))) break;
        // S^T overwrites the P^T / dS^T that the previous pair's dV / dK read
        if (it > 0 && !(ok = mbar_wait(smem_u32(&sm.pair_done), (it - 1) & 1, abort, status))) break;
        tc_fence_after();
        const uint64_t dq = desc_at(dq0, so), ddo = desc_at(ddo0, so);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tmem, desc_at(dk_k, koff(kk)), desc_at(dq, koff(kk)), id_ss, kk > 0);
        tc_commit(smem_u32(&sm.s_full));
        // dP^T overwrites the dQ^T of the previous pair once the drain has loaded it
        if (it > 0 && !(ok = mbar_wait(smem_u32(&sm.dq_free), (it - 1) & 1, abort, status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + 128, desc_at(dk_v, koff(kk)), desc_at(ddo, koff(kk)), id_ss, kk > 0);
        tc_commit(smem_u32(&sm.dp_full));
      }
      tc_commit(smem_u32(&sm.in_done));
      drain_wait(smem_u32(&sm.in_done), 0);
    }
  } else if (warp == 2) {
    // -------------------------------------------- issuer of dV, dK and dQ^T
    if (lane == 0 && cnt > 0) {
      constexpr uint32_t id_ts = idesc_bf16_f32(kB, kD, false, true);
      constexpr uint32_t id_dq = idesc_bf16_f32(kD, kB, true, true);  // M = 128 channels, N = 128 queries
      const uint64_t dqmn0 = smem_desc(smem_u32(sm.st[0].q), kHalf, 1024, kSwizzle128B);
      const uint64_t ddomn0 = smem_desc(smem_u32(sm.st[0].dO), kHalf, 1024, kSwizzle128B);
      // K_j read as K_j^T: M = channels (two 64-wide atoms kHalf apart), K = keys
      const uint64_t dkt = smem_desc(smem_u32(sm.k), kHalf, 1024, kSwizzle128B);
      // dS^T: N = queries (two 64-wide atoms, the halves' tiles kHalf apart), K = keys
      const uint64_t dds = smem_desc(smem_u32(sm.ds[0]), kHalf, 1024, kSwizzle128B);
      bool ok = true;
      for (int it = 0; ok && it < cnt; ++it) {
        const int s = it & 1;
        const uint32_t so = s * (uint32_t)sizeof(QdoStage);
        const uint64_t dqmn = desc_at(dqmn0, so), ddomn = desc_at(ddomn0, so);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!(ok = mbar_wait(smem_u32(&sm.p_full[x]), it & 1, abort, status))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // dV += P^T_x dO_x
            mma_ts(tmem + 256, tmem + x * 64 + kk * 8, desc_at(ddomn, (x * 4 + kk) * 2048), id_ts,
                   (it > 0 || x > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!(ok = mbar_wait(smem_u32(&sm.ds_full[x]), it & 1, abort, status))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // dK += dS^T_x Q_x
            mma_ts(tmem + 384, tmem + x * 64 + 32 + kk * 8, desc_at(dqmn, (x * 4 + kk) * 2048), id_ts,
                   (it > 0 || x > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.pair_done));
        tc_commit(smem_u32(&sm.qdo_empty[s]));  // dK_b was the last reader of Q_i, dO_i
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // dQ^T = K_j^T dS^T
          mma_ss(tmem + 128, desc_at(dkt, kk * 2048), desc_at(dds, kk * 2048), id_dq, kk > 0);
        tc_commit(smem_u32(&sm.dq_full));
      }
      // every product has completed once this barrier flips
      tc_commit(smem_u32(&sm.acc_done));
      drain_wait(smem_u32(&sm.acc_done), 0);
    }
  } else if (warp >= 4 && warp < 12) {
    // ----------------------------------------------------- softmax gradient
    const int x = (warp - 4) >> 2;      // query half
    const int quarter = warp & 3;
    const int c = quarter * 32 + lane;  // key row of block j = TMEM lane
    const int q0 = x * 64;              // this thread's query columns q0 .. q0 + 63
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    // rows past the last token (zero-filled) or padding of zone-chunked blocks give nothing
    const bool key_ok = blen ? c < blen[j] : j * kB + c < N;
    const uint32_t dsrow = smem_u32(sm.ds[x]) + c * 128;
    const uint32_t sw = c & 7;
    const f2 scale2 = f2_make(kSl2, kSl2);
    bool ok = true;
    for (int it = 0; it < cnt; ++it) {
      const int s = it & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.qdo_full[s]), (it >> 1) & 1, abort, status) &&
                                       mbar_wait(smem_u32(&sm.s_full), it & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      const float4* l2v = reinterpret_cast<const float4*>(sm.l2[s] + q0);
      const float4* drv = reinterpret_cast<const float4*>(sm.dr[s] + q0);
      f2 p[32];  // P^T of this key row and the half's 64 query columns, fp32 pairs
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {  // 16 query columns at a time
        uint32_t sr[16];
        tmem_ld16(lane_base + q0 + cc * 16, sr);
        tmem_wait_ld();
        reg_fence16(sr);
        uint32_t pp[8];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 L = l2v[cc * 4 + q4];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = 4 * q4 + 2 * u;
            const f2 nl = u ? f2_make(-L.z, -L.w) : f2_make(-L.x, -L.y);
            float a0, a1;
            f2_split(f2_fma(f2_make(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), scale2, nl), a0, a1);
            const f2 pv = key_ok ? f2_make(fast_exp2(a0), fast_exp2(a1)) : f2_make(0.f, 0.f);
            p[cc * 8 + 2 * q4 + u] = pv;
            pp[2 * q4 + u] = f2_pack_bf16(pv);
          }
        }
        // P^T_x over columns q0 + 8cc .. of S^T (this half's columns, already loaded)
        tmem_st8(lane_base + q0 + cc * 8, pp);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_full[x]));
      // dS^T_x overwrites the shared tile that the previous pair's dQ^T read
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.dp_full), it & 1, abort, status) &&
                                       (it == 0 || mbar_wait(smem_u32(&sm.dq_full), (it - 1) & 1, abort, status)));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t pr[16];
        tmem_ld16(lane_base + 128 + q0 + cc * 16, pr);
        tmem_wait_ld();
        reg_fence16(pr);
        uint32_t dd[8];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 Dv = drv[cc * 4 + q4];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = 4 * q4 + 2 * u;
            const f2 nd = u ? f2_make(-Dv.z, -Dv.w) : f2_make(-Dv.x, -Dv.y);
            dd[2 * q4 + u] = f2_pack_bf16(
                f2_mul(p[cc * 8 + 2 * q4 + u], f2_add(f2_make(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1])), nd)));
          }
        }
        // dS^T_x over columns q0 + 32 + 8cc .. of S^T (A of dK) and into row c of the
        // half's shared dS^T tile (B of dQ^T): 16-byte chunk k of the row at k ^ (c & 7)
        tmem_st8(lane_base + q0 + 32 + cc * 8, dd);
        st_shared_v4(dsrow + ((((uint32_t)(2 * cc)) ^ sw) << 4), dd[0], dd[1], dd[2], dd[3]);
        st_shared_v4(dsrow + ((((uint32_t)(2 * cc + 1)) ^ sw) << 4), dd[4], dd[5], dd[6], dd[7]);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.ds_full[x]));
    }
    const int col = j * kB + c;
    __nv_bfloat16* dk_row = dk + (int64_t)col * ld + (int64_t)h * kD + q0;
    __nv_bfloat16* dv_row = dv + (int64_t)col * ld + (int64_t)h * kD + q0;
    if (ok && cnt > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.acc_done), 0, abort, status));
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int which = 0; which < 2; ++which) {  // dV, then dK (scaled by 1/sqrt(d))
          __nv_bfloat16* out = which ? dk_row : dv_row;
          const float sc = which ? kScale : 1.f;
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t rr[32];
            tmem_load_row32(lane_base + 256 + which * 128 + q0 + c2 * 32, rr);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * sc, __uint_as_float(rr[2 * e + 1]) * sc);
            if (col < N) {
              uint4* dst = reinterpret_cast<uint4*>(out + c2 * 32);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
            }
          }
        }
      }
    } else if (cnt == 0 && col < N) {
      uint4* a = reinterpret_cast<uint4*>(dk_row);
      uint4* b = reinterpret_cast<uint4*>(dv_row);
#pragma unroll
      for (int e = 0; e < 8; ++e) a[e] = b[e] = make_uint4(0u, 0u, 0u, 0u);
    }
  } else if (warp >= 12) {
    // -------------------------------------------------------------- dQ drain
    // Thread = channel dch (TMEM lane of dQ^T).  Per pair: load the 128 query columns
    // in two 64-column rounds (the columns are freed once both are loaded), and per 4
    // queries transpose 4 x 4 values inside each quad of lanes (after it, lane 4g + k
    // holds query 4s + k of channels 4g .. 4g + 3) and add them to the accumulator
    // with 16-byte reductions: one warp instruction covers 4 query rows x 128 bytes.
    const int quarter = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const int k = lane & 3, g = lane >> 2;
    float* acc_h = dqacc + (int64_t)h * nb * kB * kD;  // this head's [npad][d]
    bool ok = true;
    for (int it = 0; ok && it < cnt; ++it) {
      int i = lst[it];
      if (i < 0 || i >= nb) i = 0;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.dq_full), it & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t r[64];
        tmem_ld32(lane_base + 128 + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld32(lane_base + 128 + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_wait_ld();
        reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        if (half == 1) {  // all 128 columns read: dP^T of the next pair may overwrite them
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm.dq_free));
        }
        float* base = acc_h + (int64_t)(i * kB + half * 64 + k) * kD + quarter * 32 + 4 * g;
#pragma unroll
        for (int s4 = 0; s4 < 16; ++s4) {
          float v0 = __uint_as_float(r[4 * s4]), v1 = __uint_as_float(r[4 * s4 + 1]);
          float v2 = __uint_as_float(r[4 * s4 + 2]), v3 = __uint_as_float(r[4 * s4 + 3]);
          // swap the off-diagonal 2 x 2 blocks with lane k ^ 2, then transpose inside them with k ^ 1
          {
            const bool hi = k & 2;
            const float a = __shfl_xor_sync(0xffffffffu, hi ? v0 : v2, 2);
            const float b = __shfl_xor_sync(0xffffffffu, hi ? v1 : v3, 2);
            if (hi) v0 = a, v1 = b;
            else v2 = a, v3 = b;
          }
          {
            const bool odd = k & 1;
            const float a = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
            const float b = __shfl_xor_sync(0xffffffffu, odd ? v2 : v3, 1);
            if (odd) v0 = a, v2 = b;
            else v1 = a, v3 = b;
          }
          red_add_v4(base + (int64_t)(4 * s4) * kD, v0, v1, v2, v3);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dq[r][h][c] = bf16(acc[h][r][c] / sqrt(d)): one thread per 8 channels of a (head, token)
// row, threads in accumulator order (contiguous reads; each row of 256 bytes written whole).
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc, int Hh, int N, int npad,
                                                         __nv_bfloat16* __restrict__ dq, int64_t ld) {
  const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= (int64_t)Hh * N * (kD / 8)) return;
  const int cv = (int)(v & (kD / 8 - 1));
  const int64_t hr = v / (kD / 8);
  const int h = (int)(hr / N);
  const int64_t r = hr - (int64_t)h * N;
  const float4* src = reinterpret_cast<const float4*>(acc + ((int64_t)h * npad + r) * kD + (int64_t)cv * 8);
  const float4 a = __ldcs(src), b = __ldcs(src + 1);
  uint4 o;
  o.x = pack_bf16x2(a.x * kScale, a.y * kScale);
  o.y = pack_bf16x2(a.z * kScale, a.w * kScale);
  o.z = pack_bf16x2(b.x * kScale, b.y * kScale);
  o.w = pack_bf16x2(b.z * kScale, b.w * kScale);
  *reinterpret_cast<uint4*>(dq + r * ld + (int64_t)h * kD + (int64_t)cv * 8) = o;
}

}  // namespace

size_t bwd_tc_rowstats_bytes(int Hh, int nb) { return (size_t)2 * Hh * nb * kB * sizeof(float); }
size_t bwd_tc_dqacc_bytes(int Hh, int nb) { return (size_t)nb * kB * Hh * kD * sizeof(float); }

cudaError_t bsa_bwd_tc_launch(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, int64_t ld, int N, int Hh, const int32_t* counts,
                              const int32_t* idx, int nb, void* dq, void* dk, void* dv, const int32_t* tcounts,
                              const int32_t* tidx, const int32_t* blen, const int32_t* qorder,
                              const int32_t* korder, float* rowstats, float* dqacc, cudaStream_t st,
                              uint32_t* status) {
  const int npad = nb * kB;
  float* L2 = rowstats;
  float* Dp = rowstats + (size_t)Hh * npad;
  const int64_t threads = (int64_t)Hh * npad * 16;
  {
    HookScope hs("bwd_prep", st);
    bwd_prep_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), lse, ld, N, Hh, npad, L2, Dp,
        dqacc, blen);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv, mdo;
  const uint64_t inner = (uint64_t)Hh * kD, row_bytes = (uint64_t)ld * 2;
  if (!tensor_map_2d_bf16(&mq, q, inner, N, row_bytes, 64, kB) ||
      !tensor_map_2d_bf16(&mk, k, inner, N, row_bytes, 64, kB) ||
      !tensor_map_2d_bf16(&mv, v, inner, N, row_bytes, 64, kB) ||
      !tensor_map_2d_bf16(&mdo, dO, inner, N, row_bytes, 64, kB))
    return cudaErrorInvalidValue;
  if (dqacc) {
    // fused: one kernel for dK, dV and the fp32 dQ accumulator, then the conversion
    if ((e = cudaFuncSetAttribute(bsa_bwd_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kFusedSmemBytes)) != cudaSuccess)
      return e;
    {
      HookScope hs("bsa_bwd_tc", st);
      bsa_bwd_fused_kernel<<<(unsigned)Hh * nb, kFusedThreads, kFusedSmemBytes, st>>>(
          mq, mk, mv, mdo, dqacc, L2, Dp, npad, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), ld,
          N, tcounts, tidx, nb, blen, korder, status);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t vecs = (int64_t)N * Hh * (kD / 8);
    HookScope hs("dq_convert", st);
    dq_convert_kernel<<<(unsigned)((vecs + 255) / 256), 256, 0, st>>>(dqacc, Hh, N, npad,
                                                                      static_cast<__nv_bfloat16*>(dq), ld);
    return cudaGetLastError();
  }
  // split: dQ recomputes S and dP per query block; dK / dV per key block
  if ((e = cudaFuncSetAttribute(bsa_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kDqSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(bsa_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kDkdvSmemBytes)) != cudaSuccess)
    return e;
  {
    HookScope hs("bsa_dq_tc", st);
    bsa_dq_tc_kernel<<<(unsigned)Hh * nb, kDqThreads, kDqSmemBytes, st>>>(
        mq, mk, mv, mdo, L2, Dp, npad, static_cast<__nv_bfloat16*>(dq), ld, N, counts, idx, nb, blen, qorder, status);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  HookScope hs("bsa_dkdv_tc", st);
  bsa_dkdv_tc_kernel<<<(unsigned)Hh * nb, kDkdvThreads, kDkdvSmemBytes, st>>>(
      mq, mk, mv, mdo, L2, Dp, npad, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), ld, N,
      tcounts, tidx, nb, blen, korder, status);
  return cudaGetLastError();
}

}  // namespace prism
