// C ABI of libprism.so (declared in include/prism.h): argument checks, workspace
// sizing, dispatch to the kernel launchers, and the device status word.
//
// Nothing here allocates device memory: scratch space is the caller's workspace.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "internal.h"

namespace prism {
cudaError_t umma_selftest_launch(const void* a, const void* b, float* out_s, float* out_o, int variant,
                                 cudaStream_t st, uint32_t* status);
cudaError_t wait_timeout_selftest_launch(uint64_t limit_ns, int* marker, cudaStream_t st, uint32_t* status);
}

namespace {

__device__ uint32_t g_status_word;

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};

// Count the kernels a successful call enqueued.
int launched(int n) {
  g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed);
  return PRISM_OK;
}

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return PRISM_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PRISM_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device address of the status word of the current device, resolved once per device.
uint32_t* status_ptr() {
  static std::mutex mu;
  static uint32_t* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

constexpr size_t kMinWs = 256;

size_t ws_round(size_t x) { return x < kMinWs ? kMinWs : ((x + 255) & ~(size_t)255); }

// Common workspace protocol: ws == NULL -> report the size; else check it.
bool ws_query(void* ws, size_t* ws_bytes, size_t need, int* rc) {
  if (!ws_bytes) {
    *rc = fail(PRISM_EINVAL, "ws_bytes must not be NULL");
    return true;
  }
  if (!ws) {
    *ws_bytes = need;
    *rc = ok();
    return true;
  }
  if (*ws_bytes < need) {
    *rc = fail(PRISM_EINVAL, "workspace of %zu bytes is smaller than the %zu required", *ws_bytes, need);
    return true;
  }
  if (reinterpret_cast<uintptr_t>(ws) & 255) {
    *rc = fail(PRISM_EINVAL, "workspace must be 256-byte aligned");
    return true;
  }
  return false;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int check_attention_args(const void* q, const void* k, const void* v, int32_t dtype, int64_t ld, int32_t N,
                         int32_t Hh, int32_t d, int32_t B, const int32_t* counts, const int32_t* idx, int32_t nb) {
  if (dtype != PRISM_F32 && dtype != PRISM_BF16) return fail(PRISM_EINVAL, "dtype must be PRISM_F32 or PRISM_BF16");
  if (N < 1 || Hh < 1) return fail(PRISM_EINVAL, "N and Hh must be >= 1 (got %d, %d)", N, Hh);
  if (d != 64 && d != 128) return fail(PRISM_EUNSUPPORTED, "head dim %d not built (64 or 128)", d);
  if (B != 64 && B != 128) return fail(PRISM_EUNSUPPORTED, "block size %d not built (64 or 128)", B);
  if (nb != cdiv(N, B)) return fail(PRISM_EINVAL, "nb = %d but ceil(N / B) = %lld", nb, (long long)cdiv(N, B));
  if (ld < (int64_t)Hh * d) return fail(PRISM_EINVAL, "ld = %lld < Hh * d = %d", (long long)ld, Hh * d);
  if (!q || !k || !v || !counts || !idx) return fail(PRISM_EINVAL, "NULL input pointer");
  if ((int64_t)Hh * nb * nb > ((int64_t)1 << 40)) return fail(PRISM_EINVAL, "Hh * nb * nb too large");
  return PRISM_OK;
}

// The tensor-core backward runs the split kernels (dQ per query block, recomputing S
// and dP; dK and dV per key block: seven tile products per kept pair, deterministic)
// unless PRISM_BWD_FUSED=1 is set in the environment when the library is first used:
// then the fused kernel (five products per pair, dQ reduce-added in fp32), which was
// measured no faster on B300 and is kept to compare the two designs.  Both compute
// the full gradients.
bool fused_backward() {
  static const bool fused = [] {
    const char* v = std::getenv("PRISM_BWD_FUSED");
    return v && v[0] == '1';
  }();
  return fused;
}

bool use_tc(int32_t dtype, int32_t d, int32_t B, int64_t ld, std::initializer_list<const void*> ptrs) {
  if (dtype != PRISM_BF16 || d != 128 || B != 128 || ld % 8 != 0) return false;
  for (const void* p : ptrs)
    if (!aligned16(p)) return false;
  return true;
}

}  // namespace

namespace prism {
int report_error(int code, const char* msg) { return fail(code, "%s", msg); }

namespace {
std::atomic<prism_launch_hook_fn> g_hook{nullptr};
std::atomic<void*> g_hook_user{nullptr};
}  // namespace

void launch_hook(const char* kernel, cudaStream_t st, int phase) {
  prism_launch_hook_fn f = g_hook.load(std::memory_order_acquire);
  if (f) f(kernel, st, phase, g_hook_user.load(std::memory_order_relaxed));
}
}  // namespace prism

extern "C" {

}  // extern "C"

namespace {

// Grid, zone extents and (optionally) shape set of the zone calls; PRISM_OK or an error.
int zone_geometry(int32_t T, int32_t H, int32_t W, int32_t zt, int32_t zh, int32_t zw, prism::ZoneGeom* g) {
  if (T < 1 || H < 1 || W < 1) return fail(PRISM_EINVAL, "grid must be positive");
  if ((int64_t)T * H * W > INT32_MAX) return fail(PRISM_EINVAL, "too many tokens");
  if (zt < 1 || zh < 1 || zw < 1) return fail(PRISM_EINVAL, "zone extents must be >= 1");
  *g = prism::ZoneGeom{};
  g->T = T, g->H = H, g->W = W, g->zt = zt, g->zh = zh, g->zw = zw;
  g->nzt = (int)cdiv(T, zt), g->nzh = (int)cdiv(H, zh), g->nzw = (int)cdiv(W, zw);
  g->Z = g->nzt * g->nzh * g->nzw;
  g->max_tokens = std::min(zt, T) * std::min(zh, H) * std::min(zw, W);
  if ((int64_t)g->max_tokens * 8 * 4 > 200 * 1024)
    return fail(PRISM_EUNSUPPORTED, "zones of %d tokens exceed the shared-memory staging limit (6400)",
                g->max_tokens);
  return PRISM_OK;
}

int shape_set(const int32_t* shapes, int32_t n_shapes, prism::ShapeSet* ss) {
  if (n_shapes < 1 || n_shapes > 8 || !shapes) return fail(PRISM_EINVAL, "need 1..8 shapes (host array)");
  *ss = prism::ShapeSet{};
  ss->n = n_shapes;
  for (int s = 0; s < n_shapes; ++s)
    for (int a = 0; a < 3; ++a) {
      ss->e[s][a] = shapes[3 * s + a];
      if (ss->e[s][a] < 1) return fail(PRISM_EINVAL, "shape extents must be >= 1");
    }
  return PRISM_OK;
}

int feature_args(int32_t feat_dtype, int64_t feat_ld, int32_t C) {
  if (feat_dtype != PRISM_F32 && feat_dtype != PRISM_BF16) return fail(PRISM_EINVAL, "feat_dtype invalid");
  if (C < 1 || feat_ld < C) return fail(PRISM_EINVAL, "need 1 <= C <= feat_ld");
  return PRISM_OK;
}

}  // namespace

extern "C" {

int prism_zone_shapes(const void* feat, int32_t feat_dtype, int64_t feat_ld, int32_t C, const float* a2v, int32_t T,
                      int32_t H, int32_t W, int32_t zt, int32_t zh, int32_t zw, const int32_t* shapes,
                      int32_t n_shapes, int32_t* zone_shape, int32_t* perm, void* ws, size_t* ws_bytes,
                      void* stream) {
  prism::ZoneGeom g;
  prism::ShapeSet ss;
  int rc;
  if ((rc = feature_args(feat_dtype, feat_ld, C)) != PRISM_OK) return rc;
  if ((rc = shape_set(shapes, n_shapes, &ss)) != PRISM_OK) return rc;
  if ((rc = zone_geometry(T, H, W, zt, zh, zw, &g)) != PRISM_OK) return rc;
  if (ws_query(ws, ws_bytes, ws_round(prism::zone_ws_bytes(g, C, feat_dtype)), &rc)) return rc;
  if (!feat || !a2v || !zone_shape || !perm) return fail(PRISM_EINVAL, "NULL pointer");
  cudaError_t e = prism::zone_launch(feat, feat_dtype, feat_ld, C, a2v, g, ss, zone_shape, perm, ws,
                                     static_cast<cudaStream_t>(stream), status_ptr());
  return e == cudaSuccess ? (launched(4), ok()) : cuda_fail(e, "prism_zone_shapes");
}

int prism_zone_partials(const void* feat, int32_t feat_dtype, int64_t feat_ld, int32_t C, int32_t T, int32_t H,
                        int32_t W, int32_t zt, int32_t zh, int32_t zw, float* partials, void* ws, size_t* ws_bytes,
                        void* stream) {
  prism::ZoneGeom g;
  int rc;
  if ((rc = feature_args(feat_dtype, feat_ld, C)) != PRISM_OK) return rc;
  if ((rc = zone_geometry(T, H, W, zt, zh, zw, &g)) != PRISM_OK) return rc;
  if (ws_query(ws, ws_bytes, ws_round(prism::zone_partials_ws_bytes(g, C)), &rc)) return rc;
  if (!feat || !partials) return fail(PRISM_EINVAL, "NULL pointer");
  cudaError_t e = prism::zone_partials_launch(feat, feat_dtype, feat_ld, C, g, partials, ws,
                                              static_cast<cudaStream_t>(stream), status_ptr());
  return e == cudaSuccess ? (launched(2), ok()) : cuda_fail(e, "prism_zone_partials");
}

int prism_zone_shapes_from_partials(const float* partials, int32_t n_parts, int32_t C_total, const float* a2v,
                                    int32_t T, int32_t H, int32_t W, int32_t zt, int32_t zh, int32_t zw,
                                    const int32_t* shapes, int32_t n_shapes, int32_t* zone_shape, int32_t* perm,
                                    void* ws, size_t* ws_bytes, void* stream) {
  prism::ZoneGeom g;
  prism::ShapeSet ss;
  int rc;
  if (n_parts < 1 || n_parts > 4096) return fail(PRISM_EINVAL, "n_parts must be in [1, 4096]");
  if (C_total < 1) return fail(PRISM_EINVAL, "C_total must be >= 1");
  if ((rc = shape_set(shapes, n_shapes, &ss)) != PRISM_OK) return rc;
  if ((rc = zone_geometry(T, H, W, zt, zh, zw, &g)) != PRISM_OK) return rc;
  if (ws_query(ws, ws_bytes, ws_round(prism::zone_from_partials_ws_bytes(g)), &rc)) return rc;
  if (!partials || !a2v || !zone_shape || !perm) return fail(PRISM_EINVAL, "NULL pointer");
  cudaError_t e = prism::zone_from_partials_launch(partials, n_parts, C_total, a2v, g, ss, zone_shape, perm, ws,
                                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? (launched(3), ok()) : cuda_fail(e, "prism_zone_shapes_from_partials");
}

int prism_zone_chunked_size(int32_t T, int32_t H, int32_t W, int32_t zt, int32_t zh, int32_t zw, int32_t B,
                            int32_t* nb, int64_t* np) {
  prism::ZoneGeom g;
  int rc;
  if ((rc = zone_geometry(T, H, W, zt, zh, zw, &g)) != PRISM_OK) return rc;
  if (B < 1) return fail(PRISM_EINVAL, "B must be >= 1");
  if (!nb || !np) return fail(PRISM_EINVAL, "NULL pointer");
  int64_t n = 0, p = 0;
  prism::zone_chunked_size(g, B, &n, &p);
  if (n > INT32_MAX || p > INT32_MAX) return fail(PRISM_EINVAL, "too many blocks");
  *nb = (int32_t)n;
  *np = p;
  return ok();
}

int prism_zone_perm_chunked(const int32_t* zone_shape, int32_t T, int32_t H, int32_t W, int32_t zt, int32_t zh,
                            int32_t zw, const int32_t* shapes, int32_t n_shapes, int32_t B, int32_t* perm_padded,
                            int32_t* blen, void* ws, size_t* ws_bytes, void* stream) {
  prism::ZoneGeom g;
  prism::ShapeSet ss;
  int rc;
  if ((rc = shape_set(shapes, n_shapes, &ss)) != PRISM_OK) return rc;
  if ((rc = zone_geometry(T, H, W, zt, zh, zw, &g)) != PRISM_OK) return rc;
  if (B < 1) return fail(PRISM_EINVAL, "B must be >= 1");
  int64_t nb = 0, np = 0;
  prism::zone_chunked_size(g, B, &nb, &np);
  if (np > INT32_MAX) return fail(PRISM_EINVAL, "too many blocks");
  if (ws_query(ws, ws_bytes, ws_round((size_t)g.Z * sizeof(int32_t)), &rc)) return rc;
  if (!zone_shape || !perm_padded || !blen) return fail(PRISM_EINVAL, "NULL pointer");
  cudaError_t e = prism::zone_perm_chunked_launch(zone_shape, g, ss, B, perm_padded, blen, np, ws,
                                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? (launched(3), ok()) : cuda_fail(e, "prism_zone_perm_chunked");
}

namespace {
int pool_score_impl(const void* q, const void* k, const void* v, int32_t dtype, int64_t ld, const int32_t* perm,
                    int32_t n_src, int32_t N, int32_t Hh, int32_t d, int32_t B, void* q_blk, void* k_blk, void* v_blk,
                    int64_t ld_blk, float* qbar, float* kbar, float* scores, void* stream, const char* name) {
  if (dtype != PRISM_F32 && dtype != PRISM_BF16) return fail(PRISM_EINVAL, "dtype invalid");
  if (N < 1 || n_src < 1 || Hh < 1 || d < 1 || B < 1) return fail(PRISM_EINVAL, "sizes must be >= 1");
  if (d > 256) return fail(PRISM_EUNSUPPORTED, "d > 256");
  if (!q || !k) return fail(PRISM_EINVAL, "q and k must not be NULL");
  if (ld < (int64_t)Hh * d) return fail(PRISM_EINVAL, "ld < Hh * d");
  const bool copies = q_blk || k_blk || v_blk;
  if (!perm && copies) return fail(PRISM_EINVAL, "block-order copies need perm");
  if (copies && ld_blk < (int64_t)Hh * d) return fail(PRISM_EINVAL, "ld_blk < Hh * d");
  if (v_blk && !v) return fail(PRISM_EINVAL, "v_blk needs v");
  if (scores && (!qbar || !kbar)) return fail(PRISM_EINVAL, "scores need the qbar and kbar buffers");
  const int nb = (int)cdiv(N, B);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (qbar || kbar || copies)
    e = prism::pool_launch(q, k, v, dtype, ld, perm, n_src, N, Hh, d, B, q_blk, k_blk, v_blk, copies ? ld_blk : ld,
                           qbar, kbar, st, status_ptr());
  if (e == cudaSuccess && scores) e = prism::scores_launch(qbar, kbar, Hh, nb, d, scores, st);
  if (e != cudaSuccess) return cuda_fail(e, name);
  launched((qbar || kbar || copies ? 1 : 0) + (scores ? 1 : 0));
  return ok();
}
}  // namespace

int prism_pool_score(const void* q, const void* k, const void* v, int32_t dtype, int64_t ld, const int32_t* perm,
                     int32_t N, int32_t Hh, int32_t d, int32_t B, void* q_blk, void* k_blk, void* v_blk,
                     int64_t ld_blk, float* qbar, float* kbar, float* scores, void* stream) {
  return pool_score_impl(q, k, v, dtype, ld, perm, N, N, Hh, d, B, q_blk, k_blk, v_blk, ld_blk, qbar, kbar, scores,
                         stream, "prism_pool_score");
}

int prism_pool_score_chunked(const void* q, const void* k, const void* v, int32_t dtype, int64_t ld, int32_t n_src,
                             const int32_t* perm_padded, int32_t np, int32_t Hh, int32_t d, int32_t B, void* q_blk,
                             void* k_blk, void* v_blk, int64_t ld_blk, float* qbar, float* kbar, float* scores,
                             void* stream) {
  if (!perm_padded) return fail(PRISM_EINVAL, "perm_padded must not be NULL");
  if (np % B != 0) return fail(PRISM_EINVAL, "np = %d is not a multiple of B = %d", np, B);
  return pool_score_impl(q, k, v, dtype, ld, perm_padded, n_src, np, Hh, d, B, q_blk, k_blk, v_blk, ld_blk, qbar,
                         kbar, scores, stream, "prism_pool_score_chunked");
}

int prism_select(const float* scores, int32_t Hh, int32_t nb, double sparsity, double cdf_tau, int32_t* counts,
                 int32_t* idx, void* stream) {
  if (!scores || !counts || !idx) return fail(PRISM_EINVAL, "NULL pointer");
  if (Hh < 1 || nb < 1) return fail(PRISM_EINVAL, "Hh and nb must be >= 1");
  if (nb > 4096) return fail(PRISM_EUNSUPPORTED, "nb = %d > 4096", nb);
  if (!(sparsity >= 0.0 && sparsity < 1.0)) return fail(PRISM_EINVAL, "sparsity must be in [0, 1)");
  if (!(cdf_tau >= 0.0 && cdf_tau <= 1.0)) return fail(PRISM_EINVAL, "cdf_tau must be in [0, 1]");
  const double kk = std::ceil((1.0 - sparsity) * nb - 1e-9);
  const int k_top = (int)std::min<double>(nb, std::max<double>(1.0, kk));
  cudaError_t e = prism::select_launch(scores, Hh, nb, k_top, cdf_tau, counts, idx,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? (launched(1), ok()) : cuda_fail(e, "prism_select");
}

int prism_score_select(const float* qbar, const float* kbar, int32_t Hh, int32_t nb, int32_t d, double sparsity,
                       double cdf_tau, int32_t* counts, int32_t* idx, void* stream) {
  if (!qbar || !kbar || !counts || !idx) return fail(PRISM_EINVAL, "NULL pointer");
  if (Hh < 1 || nb < 1 || d < 1) return fail(PRISM_EINVAL, "Hh, nb and d must be >= 1");
  if (!(sparsity >= 0.0 && sparsity < 1.0)) return fail(PRISM_EINVAL, "sparsity must be in [0, 1)");
  if (!(cdf_tau >= 0.0 && cdf_tau <= 1.0)) return fail(PRISM_EINVAL, "cdf_tau must be in [0, 1]");
  if (!prism::score_select_supported(nb, d))
    return fail(PRISM_EUNSUPPORTED, "prism_score_select needs d a multiple of 8, d <= 256, nb <= 4096 (got d = %d, "
                                    "nb = %d); use prism_pool_score scores + prism_select", d, nb);
  if (!aligned16(qbar) || !aligned16(kbar)) return fail(PRISM_EINVAL, "qbar and kbar must be 16-byte aligned");
  const double kk = std::ceil((1.0 - sparsity) * nb - 1e-9);
  const int k_top = (int)std::min<double>(nb, std::max<double>(1.0, kk));
  cudaError_t e = prism::score_select_launch(qbar, kbar, Hh, nb, d, k_top, cdf_tau, counts, idx,
                                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? (launched(1), ok()) : cuda_fail(e, "prism_score_select");
}

int prism_bsa_fwd(const void* q_blk, const void* k_blk, const void* v_blk, int32_t dtype, int64_t ld, int32_t N,
                  int32_t Hh, int32_t d, int32_t B, const int32_t* counts, const int32_t* idx, int32_t nb,
                  const int32_t* blen, void* o_blk, float* lse, void* ws, size_t* ws_bytes, void* stream) {
  int rc = check_attention_args(q_blk, k_blk, v_blk, dtype, ld, N, Hh, d, B, counts, idx, nb);
  if (rc != PRISM_OK) return rc;
  // workspace (tensor-core path): the CTAs' launch order, longest lists first per head
  const bool tc = use_tc(dtype, d, B, ld, {q_blk, k_blk, v_blk, o_blk});
  const bool ordered = tc && prism::order_rows_supported(nb);
  if (ws_query(ws, ws_bytes, ws_round(ordered ? (size_t)Hh * nb * sizeof(int32_t) : 0), &rc)) return rc;
  if (!o_blk || !lse) return fail(PRISM_EINVAL, "NULL output pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  int32_t* order = ordered ? static_cast<int32_t*>(ws) : nullptr;
  if (ordered) e = prism::order_rows_launch(counts, Hh, nb, order, "order_rows", st);
  if (e == cudaSuccess) {
    if (tc)
      e = prism::bsa_fwd_tc_launch(q_blk, k_blk, v_blk, ld, N, Hh, counts, idx, nb, blen, order, o_blk, lse, st,
                                   status_ptr());
    else
      e = prism::bsa_fwd_simt_launch(q_blk, k_blk, v_blk, dtype, ld, N, Hh, d, B, counts, idx, nb, blen, o_blk, lse,
                                     st, status_ptr());
  }
  return e == cudaSuccess ? (launched(ordered ? 2 : 1), ok()) : cuda_fail(e, "prism_bsa_fwd");
}

int prism_a2v_norm(const void* qv, const void* ka, const void* va, int32_t dtype, int64_t ld_v, int64_t ld_a,
                   int32_t N, int32_t M, int32_t Hh, int32_t d, void* o, float* a2v, void* ws, size_t* ws_bytes,
                   void* stream) {
  if (dtype != PRISM_BF16 || d != 128) return fail(PRISM_EUNSUPPORTED, "prism_a2v_norm is built for bf16, d = 128");
  if (N < 1 || M < 1 || Hh < 1) return fail(PRISM_EINVAL, "N, M and Hh must be >= 1 (got %d, %d, %d)", N, M, Hh);
  if (ld_v < (int64_t)Hh * d || ld_a < (int64_t)Hh * d)
    return fail(PRISM_EINVAL, "row strides %lld, %lld < Hh * d = %d", (long long)ld_v, (long long)ld_a, Hh * d);
  if (ld_v % 8 != 0 || ld_a % 8 != 0) return fail(PRISM_EINVAL, "row strides must be multiples of 8 elements");
  int rc;
  if (ws_query(ws, ws_bytes, ws_round((size_t)Hh * N * sizeof(float)), &rc)) return rc;
  if (!qv || !ka || !va || !a2v) return fail(PRISM_EINVAL, "NULL pointer");
  if (!aligned16(qv) || !aligned16(ka) || !aligned16(va) || (o && !aligned16(o)))
    return fail(PRISM_EINVAL, "qv, ka, va and o must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* sqn = static_cast<float*>(ws);
  cudaError_t e = prism::a2v_attn_launch(qv, ka, va, ld_v, ld_a, N, M, Hh, o, sqn, st, status_ptr());
  if (e == cudaSuccess) e = prism::a2v_reduce_launch(sqn, N, Hh, a2v, st);
  return e == cudaSuccess ? (launched(2), ok()) : cuda_fail(e, "prism_a2v_norm");
}

int prism_bsa_bwd(const void* q_blk, const void* k_blk, const void* v_blk, const void* o_blk, const void* do_blk,
                  const float* lse, int32_t dtype, int64_t ld, int32_t N, int32_t Hh, int32_t d, int32_t B,
                  const int32_t* counts, const int32_t* idx, int32_t nb, const int32_t* blen, void* dq, void* dk,
                  void* dv, void* ws, size_t* ws_bytes, void* stream) {
  int rc = check_attention_args(q_blk, k_blk, v_blk, dtype, ld, N, Hh, d, B, counts, idx, nb);
  if (rc != PRISM_OK) return rc;
  // workspace: transposed lists | row statistics | (tensor-core path) launch orders of
  // the query-block and key-block CTAs | (fused tensor-core path) fp32 dQ accumulator
  auto r256 = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t lists = r256(prism::lists_ws_bytes(Hh, nb));
  const bool tc = use_tc(dtype, d, B, ld, {q_blk, k_blk, v_blk, o_blk, do_blk, dq, dk, dv});
  const bool fused = tc && fused_backward();
  const bool ordered = tc && prism::order_rows_supported(nb);
  const size_t rows = r256(tc ? prism::bwd_tc_rowstats_bytes(Hh, nb) : (size_t)Hh * N * sizeof(float));
  const size_t ord = ordered ? 2 * r256((size_t)Hh * nb * sizeof(int32_t)) : 0;
  const size_t acc = fused ? prism::bwd_tc_dqacc_bytes(Hh, nb) : 0;
  if (ws_query(ws, ws_bytes, ws_round(lists + rows + ord + acc), &rc)) return rc;
  if (!o_blk || !do_blk || !lse || !dq || !dk || !dv) return fail(PRISM_EINVAL, "NULL pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* tcounts = nullptr;
  int32_t* tidx = nullptr;
  float* rowstats = reinterpret_cast<float*>(static_cast<char*>(ws) + lists);
  int32_t* qorder = ordered ? reinterpret_cast<int32_t*>(static_cast<char*>(ws) + lists + rows) : nullptr;
  int32_t* korder = ordered ? qorder + ord / (2 * sizeof(int32_t)) : nullptr;
  float* dqacc = fused ? reinterpret_cast<float*>(static_cast<char*>(ws) + lists + rows + ord) : nullptr;
  cudaError_t e = prism::transpose_lists_launch(counts, idx, Hh, nb, ws, &tcounts, &tidx, st, status_ptr());
  if (e == cudaSuccess && ordered && !fused) e = prism::order_rows_launch(counts, Hh, nb, qorder, "order_rows_q", st);
  if (e == cudaSuccess && ordered) e = prism::order_rows_launch(tcounts, Hh, nb, korder, "order_rows_k", st);
  if (e == cudaSuccess) {
    if (tc)
      e = prism::bsa_bwd_tc_launch(q_blk, k_blk, v_blk, o_blk, do_blk, lse, ld, N, Hh, counts, idx, nb, dq, dk, dv,
                                   tcounts, tidx, blen, fused ? nullptr : qorder, korder, rowstats, dqacc, st,
                                   status_ptr());
    else
      e = prism::bsa_bwd_simt_launch(q_blk, k_blk, v_blk, o_blk, do_blk, lse, dtype, ld, N, Hh, d, B, counts, idx,
                                     nb, blen, dq, dk, dv, tcounts, tidx, rowstats, st, status_ptr());
  }
  return e == cudaSuccess ? (launched(5 + (ordered ? (fused ? 1 : 2) : 0)), ok()) : cuda_fail(e, "prism_bsa_bwd");
}

int prism_attn_mse(const void* a, const void* b, int32_t dtype, int64_t ld, int32_t N, int32_t Hh, int32_t d,
                   float* mse, void* ws, size_t* ws_bytes, void* stream) {
  if (dtype != PRISM_F32 && dtype != PRISM_BF16) return fail(PRISM_EINVAL, "dtype must be PRISM_F32 or PRISM_BF16");
  if (N < 1 || Hh < 1 || d < 1) return fail(PRISM_EINVAL, "N, Hh and d must be >= 1");
  if (ld < (int64_t)Hh * d) return fail(PRISM_EINVAL, "ld = %lld < Hh * d = %d", (long long)ld, Hh * d);
  int rc;
  if (ws_query(ws, ws_bytes, ws_round((size_t)Hh * prism::attn_mse_chunks(N, Hh) * sizeof(float)), &rc)) return rc;
  if (!a || !b || !mse) return fail(PRISM_EINVAL, "NULL pointer");
  cudaError_t e = prism::attn_mse_launch(a, b, dtype, ld, N, Hh, d, mse, static_cast<float*>(ws),
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? (launched(2), ok()) : cuda_fail(e, "prism_attn_mse");
}

int prism_status_check(void* stream, uint32_t* word) {
  uint32_t* p = status_ptr();
  if (!p) return fail(PRISM_ECUDA, "no CUDA device");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t w = 0;
  cudaError_t e = cudaMemcpyAsync(&w, p, sizeof(w), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "prism_status_check");
  if (word) *word = w;
  if (w & PRISM_DEV_TIMEOUT) return fail(PRISM_ETIMEOUT, "a bounded device wait gave up (status 0x%x)", w);
  if (w & PRISM_DEV_BAD_INDEX) return fail(PRISM_EINDEX, "an out-of-range block index was skipped (status 0x%x)", w);
  if (w) return fail(PRISM_ECUDA, "device status 0x%x", w);
  return ok();
}

const char* prism_last_error(void) { return g_last_error.c_str(); }

uint64_t prism_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void prism_set_launch_hook(prism_launch_hook_fn fn, void* user) {
  prism::g_hook_user.store(user, std::memory_order_relaxed);
  prism::g_hook.store(fn, std::memory_order_release);
}

const char* prism_build_info(void) {
  return "libprism 0.1 | sm_103a | bsa_fwd: tcgen05+TMA for bf16 d=128 B=128, CUDA cores otherwise | "
         "bsa_bwd: tcgen05+TMA for bf16 d=128 B=128, CUDA cores otherwise | select: nb <= 4096 | zone: <= 6400 tokens per zone";
}

int prism_selftest_umma(const void* a, const void* b, float* out_s, float* out_o, int32_t variant, void* stream) {
  if (!a || !b || !out_s || !out_o || !aligned16(a) || !aligned16(b)) return fail(PRISM_EINVAL, "bad pointer");
  cudaError_t e = prism::umma_selftest_launch(a, b, out_s, out_o, variant ? 1 : 0, static_cast<cudaStream_t>(stream),
                                              status_ptr());
  return e == cudaSuccess ? ok() : cuda_fail(e, "prism_selftest_umma");
}

int prism_selftest_wait_timeout(int64_t limit_ns, int32_t* marker, void* stream) {
  if (!marker) return fail(PRISM_EINVAL, "marker must not be NULL");
  if (limit_ns < 1000 || limit_ns > 1000000000) return fail(PRISM_EINVAL, "limit_ns must be in [1 us, 1 s]");
  cudaError_t e = prism::wait_timeout_selftest_launch((uint64_t)limit_ns, marker, static_cast<cudaStream_t>(stream),
                                                      status_ptr());
  return e == cudaSuccess ? ok() : cuda_fail(e, "prism_selftest_wait_timeout");
}

}  // extern "C"
