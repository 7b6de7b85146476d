/*
 * prism.h -- C ABI of libprism.so: Prism-style dynamic block-sparse self-attention
 * over 3D (t, h, w) video-latent tokens, for NVIDIA B300 (sm_103a).
 *
 * Source of the method: "Prism: dynamic sparse attention for 2K joint video-audio
 * generation training" (trawling.dev/post/2299), section "Region-adapted block
 * construction".  Paragraph 1: tokens are grouped into spatio-temporal macro-zones;
 * per zone, the channel-wise variance of the video features and the feature norm
 * of the audio-to-video cross-attention set the zone's block shape, splitting more
 * finely along axes of fast video change or strong audio-video coupling.
 * Paragraph 2: a hybrid block selection makes each query's sparsity dynamic;
 * Prism Block Sparse Attention (BSA) runs on the selected blocks; the settings use
 * sparsity 0.75 / 0.80 / 0.85 / 0.93 and a CDF threshold of 0.20.
 * The page gives no formulas; every reading taken where it is silent is stated at
 * the call it concerns.
 *
 * Conventions shared by every call
 *   - All array arguments are CUDA device pointers owned by the caller unless a
 *     comment says "host".  The library never frees, keeps or allocates them, and
 *     allocates no device memory of its own: scratch space comes from the caller's
 *     workspace `ws` (query its size by passing ws = NULL; *ws_bytes receives it).
 *   - Every call enqueues its kernels on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and returns without synchronising.  Buffers must stay valid
 *     until the stream has executed the work.
 *   - Token grid (T, H, W), N = T*H*W tokens.  "Raster order": token n = (t*H + h)*W + w.
 *     "Block order": the order given by `perm` (see prism_zone_shapes); block b is
 *     the B consecutive block-order tokens [b*B, min((b+1)*B, N)), nb = ceil(N/B);
 *     only the last block can be short.
 *   - Per-head tensors are [N][Hh][d] row-major with a token row stride `ld`
 *     (elements, >= Hh*d, multiple of 8): element (n, h, c) is at n*ld + h*d + c.
 *     A group of heads of a larger tensor is addressed by offsetting the pointer by
 *     h0*d elements and keeping ld.  Pointers to bf16 data must be 16-byte aligned.
 *   - Status: 0 = PRISM_OK; other values as below.  On an error nothing is enqueued
 *     and prism_last_error() describes it.  Device-side conditions (a bounded wait
 *     that gave up, an out-of-range block index that was skipped) are recorded in a
 *     device status word read by prism_status_check().
 */
#ifndef PRISM_H
#define PRISM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  PRISM_OK = 0,
  PRISM_EINVAL = 1,        /* bad size, pointer, alignment or argument value        */
  PRISM_EUNSUPPORTED = 2,  /* valid request outside what this build implements      */
  PRISM_ECUDA = 3,         /* a CUDA runtime call or kernel launch failed           */
  PRISM_ETIMEOUT = 4,      /* (status word) a bounded device wait gave up           */
  PRISM_EINDEX = 5         /* (status word) an out-of-range block index was skipped */
};

enum { PRISM_F32 = 0, PRISM_BF16 = 1 };

/* Bits of the device status word returned by prism_status_check(). */
enum { PRISM_DEV_TIMEOUT = 1u, PRISM_DEV_BAD_INDEX = 2u, PRISM_DEV_TMEM = 4u };

/*
 * prism_zone_shapes -- step 1: per-macro-zone block shape and the block-order
 * permutation (Prism page, "Region-adapted block construction", paragraph 1).
 *
 * Readings where the page is silent:
 *   zones of extent (zt, zh, zw) tile the grid from the origin; the last zone on
 *   an axis is clipped; zones are numbered in raster order of (zone_t, zone_h, zone_w).
 *   v_a(z) = mean over channels and over the zone's lines along axis a of the
 *            population variance of the feature along the line (0 for length 1);
 *   u_a(z) = mean over the zone's lines along axis a of the population variance of
 *            the A2V norm field; abar(z) = zone mean of the field;
 *   w(z)   = abar(z) / max_z abar (0 if that max is 0);
 *   S_a    = v_a / sum_b v_b + w * u_a / sum_b u_b  (0/0 := 0);
 *   shape  = argmin over the shape set of sum_a S_a * log2(e_a), first index on ties
 *            (costs compared in fp32).
 *   Block order: zones in raster order; inside a zone, tiles of the chosen shape in
 *   tile-raster order, clipped at the zone edge; inside a tile, tokens in raster order.
 *
 * feat       [N][feat_ld] raster order, `feat_dtype` PRISM_F32 or PRISM_BF16; the
 *            first C channels of each row are the video feature (e.g. V, all heads).
 * a2v        [N] fp32 raster order: A2V cross-attention feature-norm field.
 * shapes     HOST [n_shapes][3] int32 (e_t, e_h, e_w), each >= 1; 1 <= n_shapes <= 8.
 * zone_shape out [Z] int32, Z = ceil(T/zt)*ceil(H/zh)*ceil(W/zw): chosen shape index.
 * perm       out [N] int32: perm[r] = raster index of the token at block-order position r.
 * ws         workspace of *ws_bytes bytes (NULL = size query).  Alignment 256 bytes.
 */
int prism_zone_shapes(const void* feat, int32_t feat_dtype, int64_t feat_ld, int32_t C,
                      const float* a2v, int32_t T, int32_t H, int32_t W,
                      int32_t zt, int32_t zh, int32_t zw,
                      const int32_t* shapes, int32_t n_shapes,
                      int32_t* zone_shape, int32_t* perm,
                      void* ws, size_t* ws_bytes, void* stream);

/*
 * The zone step split over channels, for a layer whose heads (hence V's channels) are
 * spread over several GPUs (the Prism page, "Data preparation and training procedure",
 * paragraph 3, trains with FSDP and sequence parallelism; a head-sharded layer is the
 * form in which attention itself splits): every rank calls prism_zone_partials on its own channels,
 * the ranks gather the [Z][3] results (e.g. torch.distributed.all_gather), and every
 * rank calls prism_zone_shapes_from_partials on the gathered [n_parts][Z][3] array.
 * The partial sums are additive over channels (the definition of v_a above is a mean
 * over channels of per-channel sums), so the result is prism_zone_shapes' up to the
 * fp32 summation order; every rank that passes the same gathered array gets the same
 * shapes and permutation, because the parts are summed in index order.
 *
 * prism_zone_partials -- partials[z][a] = sum over this call's C channels c and over the
 *   zone's lines l along axis a of sum_{k in l} (F[k][c] - mean_l F[.][c])^2  (fp32).
 *   feat, feat_dtype, feat_ld, C, grid and zone extents as in prism_zone_shapes.
 *   partials  out [Z][3] fp32 device array.  ws: workspace (NULL = size query).
 *
 * prism_zone_shapes_from_partials -- zone shapes and permutation from n_parts partial
 *   arrays [n_parts][Z][3] (device, summed in order p = 0 .. n_parts - 1) of C_total
 *   channels in all, and the A2V field a2v [N]; v_a(z) = sum / (C_total * tokens of z).
 *   Shapes, zone_shape and perm as in prism_zone_shapes.  1 <= n_parts <= 4096.
 */
int prism_zone_partials(const void* feat, int32_t feat_dtype, int64_t feat_ld, int32_t C,
                        int32_t T, int32_t H, int32_t W, int32_t zt, int32_t zh, int32_t zw,
                        float* partials, void* ws, size_t* ws_bytes, void* stream);
int prism_zone_shapes_from_partials(const float* partials, int32_t n_parts, int32_t C_total,
                                    const float* a2v, int32_t T, int32_t H, int32_t W,
                                    int32_t zt, int32_t zh, int32_t zw,
                                    const int32_t* shapes, int32_t n_shapes,
                                    int32_t* zone_shape, int32_t* perm,
                                    void* ws, size_t* ws_bytes, void* stream);

/*
 * Zone-chunked blocks -- the other reading of the block construction (Prism page,
 * "Region-adapted block construction", paragraph 1: blocks are built per macro-zone):
 * instead of cutting the whole block order into consecutive B-token blocks (a block
 * may then span the end of one zone and the start of the next), every zone's run of
 * the block order is cut into B-token blocks of its own, the last one short, so that
 * no block holds tokens of two zones.  Same token order as prism_zone_shapes' perm.
 * The blocks are laid out in a padded block order: each zone's run is followed by
 * padding up to a multiple of B, so block b is positions [b*B, (b+1)*B) and holds
 * blen[b] tokens at its start.  The other calls take this layout with N = np and
 * nb = np / B: prism_pool_score reads perm entries -1 as padding, and the attention
 * calls take blen.
 *
 * prism_zone_chunked_size -- host only: nb (blocks) and np = nb * B for the grid,
 *   zone extents and B.
 * prism_zone_perm_chunked -- from zone_shape (prism_zone_shapes' output):
 *   perm_padded out [np] int32: raster token at each padded position, -1 at padding;
 *   blen out [nb] int32: tokens of each block (1 .. B).
 *   ws: workspace (NULL = size query): one int32 per zone.
 */
int prism_zone_chunked_size(int32_t T, int32_t H, int32_t W, int32_t zt, int32_t zh, int32_t zw,
                            int32_t B, int32_t* nb, int64_t* np);
int prism_zone_perm_chunked(const int32_t* zone_shape, int32_t T, int32_t H, int32_t W,
                            int32_t zt, int32_t zh, int32_t zw,
                            const int32_t* shapes, int32_t n_shapes, int32_t B,
                            int32_t* perm_padded, int32_t* blen,
                            void* ws, size_t* ws_bytes, void* stream);

/*
 * prism_zone_shapes_noalloc -- the same computation and outputs as
 * prism_zone_shapes, for callers that cannot give the library device memory (their
 * device memory belongs to another allocator, or they run in a hook that must not
 * allocate).  The page has no counterpart of this call; it only changes where the
 * scratch lives.  There is no workspace argument: the scratch is a fixed 1 MiB
 * device array inside the library (held by every GPU that loads it until exit),
 * enough for e.g. 700 zones x 5,120 feature channels.  Grids that need more return
 * PRISM_EUNSUPPORTED with a message; use prism_zone_shapes with a workspace then.
 * The first call on a device looks up the array's device address (make that first
 * call before any stream capture).  All calls on a device share the array: calls
 * that overlap on the GPU race and must be ordered by the caller.  Allocates nothing.
 */
/*
 * prism_pool_score_chunked -- prism_pool_score for zone-chunked blocks: q, k, v are the
 * n_src raster rows; perm_padded [np] (prism_zone_perm_chunked) gives the block order
 * with -1 at padding positions, whose rows of the copies are written as zeros and are
 * not counted in the block means (each mean is over the block's blen tokens).
 * np must be a multiple of B; the other arguments as prism_pool_score with N = np.
 */
int prism_pool_score_chunked(const void* q, const void* k, const void* v, int32_t dtype, int64_t ld,
                             int32_t n_src, const int32_t* perm_padded, int32_t np, int32_t Hh,
                             int32_t d, int32_t B, void* q_blk, void* k_blk, void* v_blk,
                             int64_t ld_blk, float* qbar, float* kbar, float* scores, void* stream);

int prism_zone_shapes_noalloc(const void* feat, int32_t feat_dtype, int64_t feat_ld, int32_t C,
                              const float* a2v, int32_t T, int32_t H, int32_t W,
                              int32_t zt, int32_t zh, int32_t zw,
                              const int32_t* shapes, int32_t n_shapes,
                              int32_t* zone_shape, int32_t* perm, void* stream);

/*
 * prism_pool_score -- step 2: block-mean pooling of Q and K and block scores.
 * The page names "block-level features"; the reading is the block mean (true
 * length for the short last block) and the score qbar . kbar / sqrt(d).
 *
 * q, k, v    [N][Hh][d] with row stride ld, in raster order if perm != NULL (then
 *            the block-order copies below are written), else already in block order.
 * dtype      PRISM_F32 or PRISM_BF16 for q, k, v and the copies.
 * perm       [N] int32 from prism_zone_shapes, or NULL.
 * q_blk, k_blk, v_blk  out [N][Hh][d], row stride ld_blk: block-order copies
 *            (row r = input row perm[r]); each may be NULL to skip it; must all be
 *            NULL when perm is NULL.  v may be NULL when v_blk is NULL.
 * qbar, kbar out [Hh][nb][d] fp32 block means (either may be NULL).
 * scores     out [Hh][nb][nb] fp32: scores[h][i][j] = qbar[h][i] . kbar[h][j] / sqrt(d);
 *            may be NULL; when given, qbar and kbar must be given too.
 * Limits: d <= 256, B >= 1.
 */
int prism_pool_score(const void* q, const void* k, const void* v, int32_t dtype, int64_t ld,
                     const int32_t* perm, int32_t N, int32_t Hh, int32_t d, int32_t B,
                     void* q_blk, void* k_blk, void* v_blk, int64_t ld_blk,
                     float* qbar, float* kbar, float* scores, void* stream);

/*
 * prism_select -- step 3: hybrid block selection (Prism page, "Region-adapted
 * block construction", paragraph 2).  Reading: per (head h, query block i), with
 * blocks ordered by score descending (equal scores: smaller index first),
 *   k = min(nb, max(1, ceil((1 - sparsity) * nb - 1e-9)))   (top-(1-s) fraction),
 *   m = the shortest prefix whose softmax mass (softmax over the row) reaches cdf_tau,
 * and the kept set is the union, i.e. the first max(k, m) blocks of that order.
 *
 * scores  [Hh][nb][nb] fp32.   sparsity in [0, 1); cdf_tau in [0, 1].
 * counts  out [Hh][nb] int32: number of kept blocks.
 * idx     out [Hh][nb][nb] int32: idx[h][i][0:counts[h][i]] = kept blocks, ascending;
 *         the rest of each row is left untouched.
 * Limits: 1 <= nb <= 4096.
 */
int prism_select(const float* scores, int32_t Hh, int32_t nb, double sparsity, double cdf_tau,
                 int32_t* counts, int32_t* idx, void* stream);

/*
 * prism_score_select -- steps 2 (scores) and 3 (selection) in one call, from the block
 * means of prism_pool_score, without the [Hh][nb][nb] score matrix: each kernel block
 * keeps its score rows on chip and selects from them.  Same readings, arithmetic and
 * result as prism_pool_score's scores followed by prism_select (Prism page,
 * "Region-adapted block construction", paragraph 2): scores qbar . kbar / sqrt(d)
 * summed in fp32 over channels in ascending order, the kept set the first max(k, m)
 * blocks of the (score desc, index asc) order; the lists equal theirs bit for bit.
 *
 * qbar, kbar  [Hh][nb][d] fp32, 16-byte aligned.   sparsity in [0, 1); cdf_tau in [0, 1].
 * counts, idx as prism_select (idx row stride nb; entries past counts left untouched).
 * Limits: d a multiple of 8, d <= 256; nb <= 4096.  No workspace.
 */
int prism_score_select(const float* qbar, const float* kbar, int32_t Hh, int32_t nb, int32_t d,
                       double sparsity, double cdf_tau, int32_t* counts, int32_t* idx, void* stream);

/*
 * prism_bsa_fwd -- step 4: block-sparse attention forward (Prism BSA, same page,
 * paragraph 2).  For every head h and query block i, each query token r attends to
 * all tokens c of the blocks idx[h][i][0:counts[h][i]]:
 *   O[r] = sum_c softmax_c(Q[r].K[c] / sqrt(d)) V[c],  lse[h][r] = log sum_c exp(Q[r].K[c] / sqrt(d)).
 * No causal mask.  A query block with an empty list gets O = 0 and lse = -inf.
 *
 * q_blk, k_blk, v_blk  [N][Hh][d] block order, row stride ld, dtype PRISM_BF16
 *         (tensor-core path for d = 128, B = 128; CUDA-core path otherwise) or
 *         PRISM_F32 (CUDA-core path).
 * counts  [Hh][nb] int32;  idx [Hh][nb][nb] int32 (row stride nb), nb = ceil(N/B).
 *         Entries outside [0, nb) are skipped and flagged PRISM_DEV_BAD_INDEX.
 * blen    NULL (blocks are the B-token chunks of the block order, the last one short),
 *         or [nb] int32 for zone-chunked blocks in the padded block order
 *         (prism_zone_perm_chunked; N = nb * B): block b holds its first blen[b] rows;
 *         the other rows are padding, neither queries nor keys (their O and lse rows
 *         are unspecified).
 * o_blk   out [N][Hh][d], row stride ld, same dtype as the inputs.
 * lse     out [Hh][N] fp32 (natural log).
 * ws      workspace (NULL = size query): on the tensor-core path, the order in which the
 *         query blocks' CTAs are launched (Hh * nb int32): within each head, longest
 *         kept list first; the order changes the schedule, never the results.
 * Limits: d in {64, 128}; B in {64, 128}; the tensor-core path needs d = B = 128.
 */
int prism_bsa_fwd(const void* q_blk, const void* k_blk, const void* v_blk, int32_t dtype,
                  int64_t ld, int32_t N, int32_t Hh, int32_t d, int32_t B,
                  const int32_t* counts, const int32_t* idx, int32_t nb, const int32_t* blen,
                  void* o_blk, float* lse, void* ws, size_t* ws_bytes, void* stream);

/*
 * prism_a2v_norm -- the A2V field that prism_zone_shapes takes: the audio-to-video
 * cross-attention and its per-token feature norm ("Prism: dynamic sparse attention
 * for 2K joint video-audio generation training", section "Region-adapted block
 * construction", paragraph 1: each macro-zone uses the feature norm of the
 * audio-to-video cross-attention, a measure of how strongly the audio drives that
 * region).  Reading of that passage: for every video token n and head h,
 *   O[n][h] = sum_m softmax_m(Qv[n][h] . Ka[m][h] / sqrt(d)) Va[m][h],
 *   a2v[n]  = sqrt(sum_h |O[n][h]|^2)   (L2 norm of the Hh * d output feature).
 *
 * qv      [N][Hh][d] video queries, row stride ld_v (raster order).
 * ka, va  [M][Hh][d] audio keys and values, row stride ld_a.
 *         dtype PRISM_BF16 and d = 128 only (the tensor-core attention kernel);
 *         row strides multiples of 8 elements; pointers 16-byte aligned.
 * o       out [N][Hh][d] bf16, row stride ld_v, or NULL (not written).
 * a2v     out [N] fp32.
 * ws      workspace (NULL = size query): Hh * N fp32 squared norms.
 * Errors: PRISM_EUNSUPPORTED for another dtype or d; PRISM_EINVAL for sizes, strides,
 * alignment or NULL inputs.  Launches two kernels on `stream`.
 */
int prism_a2v_norm(const void* qv, const void* ka, const void* va, int32_t dtype,
                   int64_t ld_v, int64_t ld_a, int32_t N, int32_t M, int32_t Hh, int32_t d,
                   void* o, float* a2v, void* ws, size_t* ws_bytes, void* stream);

/*
 * prism_bsa_bwd -- step 5: gradients of block-sparse attention for training (the
 * page trains with Prism BSA switched on).  With the same kept lists as the
 * forward, treated as constants (no gradient through selection):
 *   P = exp(Q K^T / sqrt(d) - lse), dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
 *   dS = P * (dP - D), dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d).
 *
 * q_blk .. do_blk  [N][Hh][d] block order, row stride ld, dtype as in the forward.
 * lse     [Hh][N] fp32 from prism_bsa_fwd.
 * blen    as prism_bsa_fwd (padding rows get zero gradients; their dO rows are ignored).
 * dq, dk, dv  out [N][Hh][d], row stride ld, same dtype.
 * ws      workspace (NULL = size query): transposed lists, row statistics and, on the
 *         tensor-core path, the launch orders of the query-block and key-block CTAs
 *         (longest list first within each head).  With PRISM_BWD_FUSED=1 in the
 *         environment the tensor-core path also holds an fp32 dQ accumulator.
 * Limits as prism_bsa_fwd.
 */
int prism_bsa_bwd(const void* q_blk, const void* k_blk, const void* v_blk,
                  const void* o_blk, const void* do_blk, const float* lse, int32_t dtype,
                  int64_t ld, int32_t N, int32_t Hh, int32_t d, int32_t B,
                  const int32_t* counts, const int32_t* idx, int32_t nb, const int32_t* blen,
                  void* dq, void* dk, void* dv, void* ws, size_t* ws_bytes, void* stream);

/*
 * prism_attn_mse -- per-head mean squared difference of two attention outputs:
 *   mse[h] = (1 / (N d)) sum_{n, c} (a[n][h][c] - b[n][h][c])^2.
 * The measure that decides how far attention outputs may be broadcast to later
 * diffusion steps ("Real-time video generation with pyramid attention broadcast",
 * method: the MSE between consecutive steps' attention outputs; their difference is
 * small through the middle of the schedule, so outputs computed there are reused).
 *
 * a, b    [N][Hh][d] with row stride ld, dtype PRISM_BF16 or PRISM_F32 (both the same).
 * mse     out [Hh] fp32 (summed in fp64 in a fixed order: the same inputs give the
 *         same bits).
 * ws      workspace (NULL = size query): per-head partial sums.
 */
int prism_attn_mse(const void* a, const void* b, int32_t dtype, int64_t ld, int32_t N, int32_t Hh,
                   int32_t d, float* mse, void* ws, size_t* ws_bytes, void* stream);

/*
 * prism_status_check -- synchronise `stream`, return PRISM_OK if the device status
 * word is clear, else PRISM_ETIMEOUT or PRISM_EINDEX (the first set condition), and
 * clear the word.  *word (may be NULL) receives the raw PRISM_DEV_* bits.
 */
int prism_status_check(void* stream, uint32_t* word);

/* Message for the last non-OK status returned on this host thread ("" if none). */
const char* prism_last_error(void);

/* Number of kernels the library has enqueued since it was loaded (all devices and
 * threads): a counter for measuring how many launches a step makes. */
uint64_t prism_launch_count(void);

/* Launch observer for profiling: when set, fn(kernel_name, stream, phase, user) is
 * called on the calling host thread right before (phase 0) and right after (phase 1)
 * each of the library's kernels is enqueued on `stream`, so a caller can record
 * CUDA events around every kernel.  NULL removes it.  Changing it while other
 * threads are inside library calls is not synchronised with those calls. */
typedef void (*prism_launch_hook_fn)(const char* kernel, void* stream, int32_t phase, void* user);
void prism_set_launch_hook(prism_launch_hook_fn fn, void* user);

/* Build description: version, target architecture, compile-time limits. */
const char* prism_build_info(void);

/*
 * Diagnostics: prism_selftest_umma runs one 128 x 128 x 128 tile through the same
 * tensor-core operand layouts the attention kernels use: out_s = A B^T (A, B from
 * shared memory, K-major, 128-byte swizzle) and out_o = bf16(out_s) B (A operand
 * from tensor memory, B read MN-major).  a, b: [128][128] bf16 row-major device
 * arrays (16-byte aligned); out_s, out_o: [128][128] fp32.  `variant` 0 is the
 * layout the kernels use; 1 swaps the two byte offsets of the MN-major descriptor.
 */
int prism_selftest_umma(const void* a, const void* b, float* out_s, float* out_o, int32_t variant, void* stream);

/*
 * Diagnostics: prism_selftest_wait_timeout launches one CTA that waits on an
 * mbarrier nothing arrives on, with the same bounded wait the attention kernels
 * use but a limit of limit_ns (1 us .. 1 s).  The wait gives up, the kernel sets
 * PRISM_DEV_TIMEOUT in the status word and writes 2 to *marker (device int32) on
 * its way out, so prism_status_check then returns PRISM_ETIMEOUT and the context
 * stays usable.  Used to test the failure path without faulting or hanging a GPU.
 */
int prism_selftest_wait_timeout(int64_t limit_ns, int32_t* marker, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PRISM_H */
