// Step 4 of the path on the tensor cores: Prism Block Sparse Attention forward,
// bf16 inputs, d = 128, 128-token blocks (sm_103a: TMA + tcgen05 + TMEM).
//
// "Prism: dynamic sparse attention for 2K joint video-audio generation training",
// section "Region-adapted block construction", paragraph 2: attention runs only on
// the blocks the hybrid selection kept for each query block.  For every query
// token r of query block i and every token c of the kept blocks:
//   O[r] = sum_c softmax_c(Q[r].K[c] / sqrt(d)) V[c],  lse[r] = log sum_c exp(Q[r].K[c] / sqrt(d)).
//
// One CTA per (head, query block), 8 warps with fixed roles:
//   warp 0      TMA producer of K tiles (3-stage ring), walking the kept list;
//   warp 6      TMA producer of the Q tile and of V tiles (3-stage ring);
//   warp 1      TMEM owner and S issuer (one thread):
//                 S_b = Q K_j^T   (A, B from shared memory, K-major, 128B swizzle)
//   warp 7      PV issuer (one thread):
//                 O  += P_b V_j   (A = P from TMEM, B = V from shared memory, MN-major)
//               S has three TMEM buffers: the S issuer runs up to three blocks
//               ahead and overwrites buffer j % 3 only after PV(j-3), its last reader,
//               has completed; the two issuers keep the tensor pipe supplied while the
//               other waits; P (bf16) overwrites the S buffer it came from;
//   warps 2-5   softmax: one thread per query row (its TMEM lane); online softmax in
//               the log2 domain with ex2.approx; the O accumulator in TMEM is
//               rescaled only when the running row max grows by more than 2^8
//               (otherwise P is taken against the stale max, which bounds P by 256).
// TMEM columns: S0 [0,128), S1 [128,256), S2 [256,384), O [384,512).
// The same kernel serves a key sequence of another length (the audio keys of the A2V
// cross-attention): no lists means every key block in order, and the outputs O and lse
// are optional while |O row|^2 (fp32, before rounding) can be written instead.
// The kept lists give block coordinates directly (tokens are already in block
// order), so gathering a key block is one TMA box coordinate.  Every wait is
// bounded; on a timeout the CTA drains its copies and MMAs, frees TMEM and exits
// with PRISM_DEV_TIMEOUT in the status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace prism {

// ------------------------------------------------------------- tensor maps
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

bool tensor_map_2d_bf16(void* map_out, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                        uint32_t box_inner, uint32_t box_outer) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(static_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool tensor_map_2d_f32_sw128(void* map_out, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                             uint32_t box_inner, uint32_t box_outer) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(static_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool tensor_map_bf16(void* map_out, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                     const uint32_t* box) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int k = 0; k < rank; ++k) {
    d[k] = dims[k];
    bx[k] = box[k];
    es[k] = 1;
    if (k + 1 < rank) st[k] = strides_bytes[k];
  }
  const CUresult r = g_encode(static_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                              const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

constexpr int kBM = 128;   // query rows per tile
constexpr int kBN = 128;   // key rows per tile
constexpr int kD = 128;    // head dim
constexpr int kStages = 3;
constexpr int kSBuf = 3;                   // S buffers in TMEM
constexpr uint32_t kOCol = 384;            // O accumulator columns [384, 512)
constexpr uint32_t kHalf = 16384;          // one 128-row x 64-col bf16 box (128B swizzled)
constexpr uint32_t kTile = 2 * kHalf;      // a 128 x 128 bf16 tile
constexpr int kThreads = 256;  // 8 warps
constexpr float kSl2 = 1.4426950408889634f * 0.08838834764831845f;  // log2(e) / sqrt(128)
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

struct FwdSmem {
  uint8_t q[kTile];
  uint8_t k[kStages][kTile];
  uint8_t v[kStages][kTile];
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[kSBuf], p_full[kSBuf];
  uint64_t o_bar[2];           // PV(t) done, t even / odd
  uint64_t pv_done[kSBuf];     // PV(t) done, t mod 3 (the S issuer may then overwrite buffer t mod 3)
  uint64_t mma_done, s_done;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kFwdSmemBytes = sizeof(FwdSmem) + 1024;
static_assert(kFwdSmemBytes <= 232448, "shared memory budget");

// Key block of step `it`: the kept list's entry, or `it` itself when there is no list
// (dense: every key block in order).
__device__ __forceinline__ int block_of(const int32_t* lst, int it, int nbk, bool& ok) {
  const int j = lst ? lst[it] : it;
  ok = (j >= 0 && j < nbk);
  return ok ? j : 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    bsa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, __nv_bfloat16* __restrict__ o,
                      float* __restrict__ lse, float* __restrict__ sqn, int64_t ld, int N, int Nk,
                      const int32_t* __restrict__ counts, const int32_t* __restrict__ idx, int nbq,
                      int nbk, const int32_t* __restrict__ blen, const int32_t* __restrict__ order,
                      uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = order ? order[blockIdx.x] : (int)blockIdx.x;  // head * nbq + query block
  if (item < 0 || item >= (int)gridDim.x) {
    if (threadIdx.x == 0) flag_error(status, PRISM_DEV_BAD_INDEX);
    return;
  }
  const int h = item / nbq, i = item - h * nbq;
  int cnt = counts ? counts[item] : nbk;  // no lists: every key block
  if (cnt < 0 || cnt > nbk) {
    if (threadIdx.x == 0) flag_error(status, PRISM_DEV_BAD_INDEX);
    cnt = cnt < 0 ? 0 : nbk;
  }
  const int32_t* lst = counts ? idx + (size_t)item * nbk : nullptr;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), 1);
      mbar_init(smem_u32(&sm.k_empty[s]), 1);
      mbar_init(smem_u32(&sm.v_full[s]), 1);
      mbar_init(smem_u32(&sm.v_empty[s]), 1);
    }
    for (int b = 0; b < kSBuf; ++b) {
      mbar_init(smem_u32(&sm.s_full[b]), 1);
      mbar_init(smem_u32(&sm.p_full[b]), 4);
    }
    mbar_init(smem_u32(&sm.o_bar[0]), 1);
    mbar_init(smem_u32(&sm.o_bar[1]), 1);
    for (int b = 0; b < kSBuf; ++b) mbar_init(smem_u32(&sm.pv_done[b]), 1);
    mbar_init(smem_u32(&sm.mma_done), 1);
    mbar_init(smem_u32(&sm.s_done), 1);
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
    // ---------------------------------------------------------------- K producer
    if (lane == 0 && cnt > 0) {
      tma_prefetch_desc(&tmk);
      int armed[kStages] = {0, 0, 0};
      for (int it = 0; it < cnt; ++it) {
        const int st = it % kStages;
        if (it >= kStages && !mbar_wait(smem_u32(&sm.k_empty[st]), ((it / kStages) - 1) & 1, abort, status)) break;
        bool ok;
        const int j = block_of(lst, it, nbk, ok);
        const uint32_t bar = smem_u32(&sm.k_full[st]);
        mbar_arrive_expect_tx(bar, kTile);
        tma_load_2d(smem_u32(sm.k[st]), &tmk, h * kD, j * kBN, bar);
        tma_load_2d(smem_u32(sm.k[st]) + kHalf, &tmk, h * kD + 64, j * kBN, bar);
        ++armed[st];
      }
      if (*abort)
        for (int s = 0; s < kStages; ++s)
          if (armed[s]) drain_wait(smem_u32(&sm.k_full[s]), (armed[s] - 1) & 1);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ Q / V producer
    if (lane == 0 && cnt > 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmv);
      const uint32_t qbar = smem_u32(&sm.q_full);
      mbar_arrive_expect_tx(qbar, kTile);
      tma_load_2d(smem_u32(sm.q), &tmq, h * kD, i * kBM, qbar);
      tma_load_2d(smem_u32(sm.q) + kHalf, &tmq, h * kD + 64, i * kBM, qbar);
      int armed[kStages] = {0, 0, 0};
      for (int it = 0; it < cnt; ++it) {
        const int st = it % kStages;
        if (it >= kStages && !mbar_wait(smem_u32(&sm.v_empty[st]), ((it / kStages) - 1) & 1, abort, status)) break;
        bool ok;
        const int j = block_of(lst, it, nbk, ok);
        const uint32_t bar = smem_u32(&sm.v_full[st]);
        mbar_arrive_expect_tx(bar, kTile);
        tma_load_2d(smem_u32(sm.v[st]), &tmv, h * kD, j * kBN, bar);
        tma_load_2d(smem_u32(sm.v[st]) + kHalf, &tmv, h * kD + 64, j * kBN, bar);
        ++armed[st];
      }
      if (*abort) {
        drain_wait(qbar, 0);
        for (int s = 0; s < kStages; ++s)
          if (armed[s]) drain_wait(smem_u32(&sm.v_full[s]), (armed[s] - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- S issuer
    // S(j) = Q K_j^T into TMEM buffer j % 3, as soon as K_j has landed and PV(j - 3),
    // the last reader of that buffer, has completed.
    if (lane == 0 && cnt > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, false, false);
      const uint64_t dq0 = smem_desc(smem_u32(sm.q), 16, 1024, kSwizzle128B);
      const uint64_t dk0 = smem_desc(smem_u32(sm.k[0]), 16, 1024, kSwizzle128B);
      bool ok = mbar_wait(smem_u32(&sm.q_full), 0, abort, status);
      for (int j = 0; ok && j < cnt; ++j) {
        const int st = j % kStages, b = j % kSBuf;
        if (j >= kSBuf && !(ok = mbar_wait(smem_u32(&sm.pv_done[b]), ((j / kSBuf) - 1) & 1, abort, status))) break;
        if (!(ok = mbar_wait(smem_u32(&sm.k_full[st]), (j / kStages) & 1, abort, status))) break;
        tc_fence_after();
        const uint64_t dk = desc_at(dk0, st * kTile);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          mma_ss(tmem + b * 128, desc_at(dq0, off), desc_at(dk, off), idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(smem_u32(&sm.k_empty[st]));
        tc_commit(smem_u32(&sm.s_full[b]));
      }
      tc_commit(smem_u32(&sm.s_done));
      drain_wait(smem_u32(&sm.s_done), 0);
    }
  } else if (warp == 7) {
    // --------------------------------------------------------------- PV issuer
    // O += P(t) V_t as soon as the softmax has written P(t); a second issuing thread,
    // so these products never queue behind the issue of an S product.
    if (lane == 0 && cnt > 0) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, kD, false, true);
      const uint64_t dv0 = smem_desc(smem_u32(sm.v[0]), kHalf, 1024, kSwizzle128B);
      bool ok = true;
      for (int t = 0; ok && t < cnt; ++t) {
        const int b = t % kSBuf, st = t % kStages;
        if (!(ok = mbar_wait(smem_u32(&sm.p_full[b]), (t / kSBuf) & 1, abort, status))) break;
        if (!(ok = mbar_wait(smem_u32(&sm.v_full[st]), (t / kStages) & 1, abort, status))) break;
        tc_fence_after();
        const uint64_t dv = desc_at(dv0, st * kTile);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(tmem + kOCol, tmem + b * 128 + kk * 8, desc_at(dv, kk * 2048), idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
        tc_commit(smem_u32(&sm.v_empty[st]));
        tc_commit(smem_u32(&sm.o_bar[t & 1]));
        tc_commit(smem_u32(&sm.pv_done[b]));
      }
      // every PV has completed once this barrier flips; every S product completed
      // before the softmax could write the P of the last block
      tc_commit(smem_u32(&sm.mma_done));
      drain_wait(smem_u32(&sm.mma_done), 0);
    }
  } else {
    // ------------------------------------------------------------- softmax rows
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    int j_next = cnt > 0 ? (lst ? lst[0] : 0) : 0;  // block indices are read one block ahead
    for (int it = 0; it < cnt; ++it) {
      const int b = it % kSBuf;
      const int j_raw = j_next;
      if (it + 1 < cnt) j_next = lst ? lst[it + 1] : it + 1;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full[b]), (it / kSBuf) & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      const bool jok = j_raw >= 0 && j_raw < nbk;
      const int j = jok ? j_raw : 0;
      // keys of block j: the first blen[j] rows (zone-chunked blocks), else the B-token
      // chunk, the last one short
      const int len = jok ? (blen ? min(kBN, max(0, blen[j])) : min(kBN, Nk - j * kBN)) : 0;
      if (!jok && r == 0) flag_error(status, PRISM_DEV_BAD_INDEX);
      // the whole S row: four loads in flight, one wait
      float s[128];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(lane_base + b * 128, r0);
        tmem_ld32(lane_base + b * 128 + 32, r1);
        tmem_ld32(lane_base + b * 128 + 64, r2);
        tmem_ld32(lane_base + b * 128 + 96, r3);
        tmem_wait_ld();
        reg_fence(r0);
        reg_fence(r1);
        reg_fence(r2);
        reg_fence(r3);
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          s[x] = __uint_as_float(r0[x]);
          s[32 + x] = __uint_as_float(r1[x]);
          s[64 + x] = __uint_as_float(r2[x]);
          s[96 + x] = __uint_as_float(r3[x]);
        }
      }
      if (len < kBN) {  // short or skipped block (warp-uniform): masked keys never count
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = c < len ? s[c] : -INFINITY;
      }
      // row max: eight chains of three-input maxima
      float m8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) m8[k] = s[k];
#pragma unroll
      for (int c = 8; c < 128; c += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = max3(m8[k], s[c + k], s[c + 8 + k]);
      const float mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      const float m_new = fmaxf(m_used, mx * kSl2);
      if (m_new > m_used + kRescaleLog2) {
        const float alpha = fast_exp2(m_used - m_new);
        if (it > 0) {
          // PV(it - 1) done; PV(it - 3) (same barrier, previous phase) completed before S(it)
          ok = __all_sync(0xffffffffu,
                          mbar_wait(smem_u32(&sm.o_bar[(it - 1) & 1]), ((it - 1) >> 1) & 1, abort, status));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t rr[32];
            tmem_load_row32(lane_base + kOCol + c4 * 32, rr);
#pragma unroll
            for (int x = 0; x < 32; ++x) rr[x] = __float_as_uint(__uint_as_float(rr[x]) * alpha);
            tmem_st32(lane_base + kOCol + c4 * 32, rr);
          }
        }
        l *= alpha;
        m_used = m_new;
      }
      // no live key yet (only skipped blocks so far): P = 0 (warp-uniform)
      const float neg_m = m_used > -INFINITY ? -m_used : -INFINITY;
      const f2 scale2 = f2_make(kSl2, kSl2), shift2 = f2_make(neg_m, neg_m);
      f2 ls2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const int c = half * 64 + 2 * x;
          float a0, a1;
          f2_split(f2_fma(f2_make(s[c], s[c + 1]), scale2, shift2), a0, a1);  // s * log2(e)/sqrt(d) - m
          const float p0 = fast_exp2(a0);
          const float p1 = fast_exp2(a1);
          ls2[x & 1] = f2_add(ls2[x & 1], f2_make(p0, p1));
          pk[x] = pack_bf16x2(p0, p1);
        }
        tmem_st32(lane_base + b * 128 + half * 32, pk);
      }
      float l0, l1, l2_, l3;
      f2_split(ls2[0], l0, l1);
      f2_split(ls2[1], l2_, l3);
      const float lsum = (l0 + l1) + (l2_ + l3);
      tmem_wait_st();
      l += lsum;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_full[b]));
    }
    // ---------------------------------------------------------------- epilogue
    // O (if asked for), lse (if asked for) and |O row|^2 in fp32 before rounding (if asked for)
    const int row = i * kBM + r;
    __nv_bfloat16* orow = o ? o + (int64_t)row * ld + (int64_t)h * kD : nullptr;
    if (ok && cnt > 0) {
      // every MMA of the CTA has completed once mma_done flips (it completes once)
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.mma_done), 0, abort, status));
      if (ok) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float ss = 0.f;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t rr[32];
          tmem_load_row32(lane_base + kOCol + c4 * 32, rr);
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const float a = __uint_as_float(rr[2 * x]) * inv, b2 = __uint_as_float(rr[2 * x + 1]) * inv;
            ss = fmaf(a, a, fmaf(b2, b2, ss));
            pk[x] = pack_bf16x2(a, b2);
          }
          if (orow && row < N) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c4 * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x) dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
          }
        }
        if (row < N) {
          if (lse) lse[(size_t)h * N + row] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
          if (sqn) sqn[(size_t)h * N + row] = ss;
        }
      }
    } else if (cnt == 0 && row < N) {
      if (orow) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int x = 0; x < 16; ++x) dst[x] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (lse) lse[(size_t)h * N + row] = -INFINITY;
      if (sqn) sqn[(size_t)h * N + row] = 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------ layout self-test
// One 128 x 128 x 128 tile: S = A B^T (both K-major, from shared memory) and
// O = bf16(S) B (A from TMEM, B MN-major).  `variant` 1 swaps the two byte
// offsets of the MN-major descriptor; every address stays inside the 96 KB
// staging buffer either way.
__global__ void __launch_bounds__(128, 1) umma_selftest_kernel(const __grid_constant__ CUtensorMap tma,
                                                               const __grid_constant__ CUtensorMap tmb,
                                                               float* __restrict__ out_s, float* __restrict__ out_o,
                                                               int variant, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a = base;
  uint8_t* bt = base + kTile;
  __shared__ uint64_t bar_ld, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar_ld), 1);
    mbar_init(smem_u32(&bar_mma), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(smem_u32(&bar_ld), 2 * kTile);
    tma_load_2d(smem_u32(a), &tma, 0, 0, smem_u32(&bar_ld));
    tma_load_2d(smem_u32(a) + kHalf, &tma, 64, 0, smem_u32(&bar_ld));
    tma_load_2d(smem_u32(bt), &tmb, 0, 0, smem_u32(&bar_ld));
    tma_load_2d(smem_u32(bt) + kHalf, &tmb, 64, 0, smem_u32(&bar_ld));
  }
  bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_ld), 0, &abort_flag, status));
  __syncthreads();
  if (threadIdx.x == 0 && ok) {
    tc_fence_after();
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
      mma_ss(tmem, smem_desc(smem_u32(a) + off, 16, 1024, kSwizzle128B),
             smem_desc(smem_u32(bt) + off, 16, 1024, kSwizzle128B), idesc_bf16_f32(128, 128, false, false),
             kk > 0 ? 1u : 0u);
    }
    tc_commit(smem_u32(&bar_mma));
  }
  ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_mma), 0, &abort_flag, status));
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  const int r = warp * 32 + lane;
  if (ok) {
    tc_fence_after();
    for (int c4 = 0; c4 < 4; ++c4) {
      uint32_t rr[32];
      tmem_load_row32(lane_base + c4 * 32, rr);
      for (int x = 0; x < 32; ++x) out_s[r * 128 + c4 * 32 + x] = __uint_as_float(rr[x]);
      uint32_t pk[16];
      for (int x = 0; x < 16; ++x) pk[x] = pack_bf16x2(__uint_as_float(rr[2 * x]), __uint_as_float(rr[2 * x + 1]));
      uint32_t st32[32];
      for (int x = 0; x < 32; ++x) st32[x] = 0;
      // columns c4*16 .. c4*16+15 of the packed P
      for (int x = 0; x < 16; ++x) st32[x] = pk[x];
      asm volatile(
          "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
          "%14, %15, %16};" ::"r"(lane_base + c4 * 16),
          "r"(st32[0]), "r"(st32[1]), "r"(st32[2]), "r"(st32[3]), "r"(st32[4]), "r"(st32[5]), "r"(st32[6]),
          "r"(st32[7]), "r"(st32[8]), "r"(st32[9]), "r"(st32[10]), "r"(st32[11]), "r"(st32[12]), "r"(st32[13]),
          "r"(st32[14]), "r"(st32[15])
          : "memory");
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && ok) {
    tc_fence_after();
    const uint32_t lbo = variant == 0 ? kHalf : 1024u, sbo = variant == 0 ? 1024u : kHalf;
    for (int kk = 0; kk < 8; ++kk)
      mma_ts(tmem + 128, tmem + kk * 8, smem_desc(smem_u32(bt) + kk * 2048, lbo, sbo, kSwizzle128B),
             idesc_bf16_f32(128, 128, false, true), kk > 0 ? 1u : 0u);
    tc_commit(smem_u32(&bar_mma));
  }
  ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_mma), 1, &abort_flag, status));
  if (ok) {
    tc_fence_after();
    for (int c4 = 0; c4 < 4; ++c4) {
      uint32_t rr[32];
      tmem_load_row32(lane_base + 128 + c4 * 32, rr);
      for (int x = 0; x < 32; ++x) out_o[r * 128 + c4 * 32 + x] = __uint_as_float(rr[x]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Failure-path check: one CTA waits on an mbarrier that nothing ever arrives on, so
// the bounded wait runs out after `limit_ns`, flags PRISM_DEV_TIMEOUT and the kernel
// returns; it then writes `marker` so the host can see that it exited normally.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, uint32_t* status, int* marker) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const bool ok = mbar_wait_limit(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
  __syncthreads();
  if (threadIdx.x == 0) *marker = ok ? 1 : 2;
}

}  // namespace

cudaError_t wait_timeout_selftest_launch(uint64_t limit_ns, int* marker, cudaStream_t st, uint32_t* status) {
  wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(limit_ns, status, marker);
  return cudaGetLastError();
}

cudaError_t bsa_fwd_tc_launch(const void* q, const void* k, const void* v, int64_t ld, int N, int Hh,
                              const int32_t* counts, const int32_t* idx, int nb, const int32_t* blen,
                              const int32_t* order, void* o, float* lse, cudaStream_t st, uint32_t* status) {
  return attn_fwd_tc_launch(q, k, v, ld, ld, N, N, Hh, counts, idx, nb, nb, blen, order, o, lse, nullptr, "bsa_fwd_tc",
                            st, status);
}

cudaError_t attn_fwd_tc_launch(const void* q, const void* k, const void* v, int64_t ld, int64_t ld_kv, int N,
                               int Nk, int Hh, const int32_t* counts, const int32_t* idx, int nbq, int nbk,
                               const int32_t* blen, const int32_t* order, void* o, float* lse, float* sqn,
                               const char* name, cudaStream_t st, uint32_t* status) {
  CUtensorMap mq, mk, mv;
  const uint64_t inner = (uint64_t)Hh * kD;
  if (!tensor_map_2d_bf16(&mq, q, inner, N, (uint64_t)ld * 2, 64, kBM) ||
      !tensor_map_2d_bf16(&mk, k, inner, Nk, (uint64_t)ld_kv * 2, 64, kBN) ||
      !tensor_map_2d_bf16(&mv, v, inner, Nk, (uint64_t)ld_kv * 2, 64, kBN))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(bsa_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kFwdSmemBytes);
  if (e != cudaSuccess) return e;
  HookScope hs(name, st);
  bsa_fwd_tc_kernel<<<(unsigned)Hh * nbq, kThreads, kFwdSmemBytes, st>>>(
      mq, mk, mv, static_cast<__nv_bfloat16*>(o), lse, sqn, ld, N, Nk, counts, idx, nbq, nbk, blen, order, status);
  return cudaGetLastError();
}

cudaError_t umma_selftest_launch(const void* a, const void* b, float* out_s, float* out_o, int variant,
                                 cudaStream_t st, uint32_t* status) {
  CUtensorMap ma, mb;
  if (!tensor_map_2d_bf16(&ma, a, 128, 128, 256, 64, 128) || !tensor_map_2d_bf16(&mb, b, 128, 128, 256, 64, 128))
    return cudaErrorInvalidValue;
  const int smem = 3 * kTile + 1024;
  cudaError_t e = cudaFuncSetAttribute(umma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  umma_selftest_kernel<<<1, 128, smem, st>>>(ma, mb, out_s, out_o, variant, status);
  return cudaGetLastError();
}

}  // namespace prism
