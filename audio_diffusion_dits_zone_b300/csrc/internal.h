// Host-side launchers shared between the C-ABI shim (prism_api.cu) and the kernel
// files.  Arguments are validated by the shim before any launcher runs.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace prism {

// Record `msg` as the calling thread's last error (prism_last_error) and return `code`.
int report_error(int code, const char* msg);

// Launch observer (prism_set_launch_hook): called right before (phase 0) and right
// after (phase 1) a kernel is enqueued on `st`.
void launch_hook(const char* kernel, cudaStream_t st, int phase);
struct HookScope {
  const char* name;
  cudaStream_t st;
  HookScope(const char* n, cudaStream_t s) : name(n), st(s) { launch_hook(name, st, 0); }
  ~HookScope() { launch_hook(name, st, 1); }
};

struct ZoneGeom {
  int T, H, W;      // token grid
  int zt, zh, zw;   // zone extents
  int nzt, nzh, nzw;
  int Z;            // zones
  int max_tokens;   // tokens of the largest zone
};

struct ShapeSet {
  int n;
  int e[8][3];
};

// zone.cu
size_t zone_ws_bytes(const ZoneGeom& g, int C, int dtype);
cudaError_t zone_launch(const void* feat, int dtype, int64_t ld, int C, const float* a2v, const ZoneGeom& g,
                        const ShapeSet& shapes, int32_t* zone_shape, int32_t* perm, void* ws, cudaStream_t st,
                        uint32_t* status);

// The zone step in two halves, for channels split over several calls (one per rank):
// per-zone, per-axis partial sums of one call's channels ([Z][3]), and the shapes and
// permutation from partial sums gathered as [nparts][Z][3] (summed in part order).
size_t zone_partials_ws_bytes(const ZoneGeom& g, int C);
cudaError_t zone_partials_launch(const void* feat, int dtype, int64_t ld, int C, const ZoneGeom& g, float* out,
                                 void* ws, cudaStream_t st, uint32_t* status);
size_t zone_from_partials_ws_bytes(const ZoneGeom& g);
cudaError_t zone_from_partials_launch(const float* parts, int nparts, int C_total, const float* a2v,
                                      const ZoneGeom& g, const ShapeSet& shapes, int32_t* zone_shape, int32_t* perm,
                                      void* ws, cudaStream_t st);

// Zone-chunked blocks (each zone cut into B-token blocks of its own): block count nb
// and padded length np = nb * B; the padded permutation (-1 at padding) and the block
// lengths from the zone shapes; ws holds Z int32.
void zone_chunked_size(const ZoneGeom& g, int B, int64_t* nb, int64_t* np);
cudaError_t zone_perm_chunked_launch(const int32_t* zone_shape, const ZoneGeom& g, const ShapeSet& shapes, int B,
                                     int32_t* perm, int32_t* blen, int64_t np, void* ws, cudaStream_t st);

// pool_score.cu
// Block order of N positions from n_src source rows; perm entries -1 are padding (zero
// rows in the copies, not counted in the block means).
cudaError_t pool_launch(const void* q, const void* k, const void* v, int dtype, int64_t ld, const int32_t* perm,
                        int n_src, int N, int Hh, int d, int B, void* qb, void* kb, void* vb, int64_t ldb,
                        float* qbar, float* kbar, cudaStream_t st, uint32_t* status);
cudaError_t scores_launch(const float* qbar, const float* kbar, int Hh, int nb, int d, float* scores,
                          cudaStream_t st);

// select.cu
cudaError_t select_launch(const float* scores, int Hh, int nb, int k_top, double tau, int32_t* counts,
                          int32_t* idx, cudaStream_t st);

// score_select.cu: scores and selection in one kernel (no score matrix in memory).
bool score_select_supported(int nb, int d);
cudaError_t score_select_launch(const float* qbar, const float* kbar, int Hh, int nb, int d, int k_top, double tau,
                                int32_t* counts, int32_t* idx, cudaStream_t st);

// bsa_simt.cu (CUDA-core attention for f32 inputs and shapes outside the tensor-core path)
cudaError_t bsa_fwd_simt_launch(const void* q, const void* k, const void* v, int dtype, int64_t ld, int N, int Hh,
                                int d, int B, const int32_t* counts, const int32_t* idx, int nb, const int32_t* blen,
                                void* o, float* lse, cudaStream_t st, uint32_t* status);
cudaError_t bsa_bwd_simt_launch(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                const float* lse, int dtype, int64_t ld, int N, int Hh, int d, int B,
                                const int32_t* counts, const int32_t* idx, int nb, const int32_t* blen, void* dq,
                                void* dk, void* dv, const int32_t* tcounts, const int32_t* tidx, float* Drow,
                                cudaStream_t st, uint32_t* status);

// bsa_lists.cu (transposed kept lists and the backward row statistic)
size_t lists_ws_bytes(int Hh, int nb);
// Launch order of the attention kernels' CTAs: per head, rows by list length, longest
// first (stable).  order [Hh * nb] receives h * nb + row.  Needs (nb + 1) * 4 bytes of
// shared memory, at most kOrderSmemMax.
constexpr size_t kOrderSmemMax = 48 * 1024;
bool order_rows_supported(int nb);
cudaError_t order_rows_launch(const int32_t* counts, int Hh, int nb, int32_t* order, const char* name,
                              cudaStream_t st);
cudaError_t transpose_lists_launch(const int32_t* counts, const int32_t* idx, int Hh, int nb, void* ws,
                                   int32_t** tcounts, int32_t** tidx, cudaStream_t st, uint32_t* status);
cudaError_t row_dot_launch(const void* o, const void* dO, int dtype, int64_t ld, int N, int Hh, int d, float* Drow,
                           cudaStream_t st);

// bsa_tc_fwd.cu / bsa_tc_bwd.cu (tcgen05 tensor-core path: bf16, d = 128, B = 128)
// blen (nullable): tokens of each block (zone-chunked blocks); NULL = B-token chunks, the
// last one short.
cudaError_t bsa_fwd_tc_launch(const void* q, const void* k, const void* v, int64_t ld, int N, int Hh,
                              const int32_t* counts, const int32_t* idx, int nb, const int32_t* blen,
                              const int32_t* order, void* o, float* lse, cudaStream_t st, uint32_t* status);
// The same kernel with a key sequence of its own (Nk tokens in nbk blocks, row stride
// ld_kv) and optional outputs: o, lse and sqn ([Hh][N] fp32, the squared L2 norm of each
// normalised output row) may each be NULL.  counts == NULL visits every key block.
// order (nullable, from order_rows_launch): CTA b processes item order[b]; NULL = item b.
// The items are independent, so the order changes the schedule, not the results.
cudaError_t attn_fwd_tc_launch(const void* q, const void* k, const void* v, int64_t ld, int64_t ld_kv, int N,
                               int Nk, int Hh, const int32_t* counts, const int32_t* idx, int nbq, int nbk,
                               const int32_t* blen, const int32_t* order, void* o, float* lse, float* sqn,
                               const char* name, cudaStream_t st, uint32_t* status);
// The cross-attention of the A2V field (a2v.cu): sqn[h][n] = |O[n][h]|^2, O optional.
cudaError_t a2v_attn_launch(const void* qv, const void* ka, const void* va, int64_t ld_v, int64_t ld_a, int N,
                            int M, int Hh, void* o, float* sqn, cudaStream_t st, uint32_t* status);
// a2v[n] = sqrt(sum_h sqn[h][n]).
cudaError_t a2v_reduce_launch(const float* sqn, int N, int Hh, float* a2v, cudaStream_t st);
size_t bwd_tc_rowstats_bytes(int Hh, int nb);
// fp32 dQ accumulator of the fused backward: [Hh][nb * 128][128]
size_t bwd_tc_dqacc_bytes(int Hh, int nb);
// dqacc != NULL: the fused kernel (dK, dV and dQ in one pass over the transposed lists,
// dQ reduce-added into dqacc, then converted); dqacc == NULL: the split kernels (dQ per
// query block, recomputing S and dP; dK and dV per key block).  qorder / korder
// (nullable): launch orders of the query-block (dQ) and key-block (dK/dV, fused) CTAs.
cudaError_t bsa_bwd_tc_launch(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, int64_t ld, int N, int Hh, const int32_t* counts,
                              const int32_t* idx, int nb, void* dq, void* dk, void* dv, const int32_t* tcounts,
                              const int32_t* tidx, const int32_t* blen, const int32_t* qorder,
                              const int32_t* korder, float* rowstats, float* dqacc, cudaStream_t st,
                              uint32_t* status);

// pab.cu: per-head mean squared difference of two [N][Hh][d] tensors (row stride ld);
// part holds Hh * attn_mse_chunks(N, Hh) fp32 partial sums.
int attn_mse_chunks(int N, int Hh);
cudaError_t attn_mse_launch(const void* a, const void* b, int dtype, int64_t ld, int N, int Hh, int d, float* mse,
                            float* part, cudaStream_t st);

// Driver entry point for tensor-map encoding (resolved once through the runtime).
bool tensor_map_2d_bf16(void* map_out, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                        uint32_t box_inner, uint32_t box_outer);
// fp32 2D tensor map with 128-byte swizzle (box_inner * 4 <= 128 bytes).
bool tensor_map_2d_f32_sw128(void* map_out, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                             uint32_t box_inner, uint32_t box_outer);
// bf16 tensor map of rank 1..5, no swizzle: dims innermost first, strides_bytes[k] =
// byte stride of dimension k + 1.
bool tensor_map_bf16(void* map_out, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                     const uint32_t* box);

}  // namespace prism
