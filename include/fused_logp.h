/*
 * fused_logp.h: C ABI of the GB300 selected-token log-probability library
 * (libfused_logp.so, sm_103a).
 *
 * The operation (RL-Kernel issue #241 "TP-aware deterministic logprob",
 * Background and Goal): for BF16 logits x[N, V] and int64 targets y[N],
 *     LSE_t  = log sum_v exp(x[t, v])           (FP32 accumulation)
 *     logp_t = x[t, y_t] - LSE_t
 * and its gradient (RL-Kernel PR #495 "zero-workspace fused backward",
 * Summary item 2) for an upstream gradient g[N]:
 *     dlogits[t, v] = g_t * (onehot(y_t)[v] - exp(x[t, v] - LSE_t))
 * written straight to BF16 with no FP32 [N, V] workspace.
 *
 * A row is ACTIVE when 0 <= y_t < V and y_t != ignore_index.  Inactive rows
 * get logp = 0 and an all-zero gradient row (PR #495, Behavior changes:
 * out-of-range targets); their LSE is still computed.
 *
 * Vocabulary tiles.  Each row is cut into FLP_NUM_TILES = 16 fixed tiles of
 * width W = flp_tile_width(V) = 8 * ceil(V / 128) columns (the last ones
 * clipped or empty).  Every tile is reduced by the same fixed tree whatever N,
 * the row's position in the batch, or the shard that holds it; the 16 tile
 * partials are then merged in tile-index order.  This is the tile-level merge
 * of RL-Kernel PR #314 ("Deterministic config option", the tensor-parallel
 * section: fixed tiles reduced as the same shape on any rank, then one fixed
 * merge order), which makes results bitwise independent of N, of the row's
 * position and of the shard split.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers of one CUDA device, owned and allocated by
 *     the caller.  The library allocates nothing (no workspace, PR #495
 *     Summary item 2).  BF16 buffers are passed as void pointers to
 *     IEEE bfloat16 data.  Row-major with a row stride (ld) in elements.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *     and run on the device that holds `logits` (or the first device pointer);
 *     the caller's current device is restored before returning (the device
 *     guard of PR #495's review thread).
 *   - All extents and index arithmetic are int64 (PR #495 review: the
 *     int32 loop overflow near INT_MAX).
 *   - n == 0 returns FLP_OK without touching the device (PR #495 Tests:
 *     empty input).
 *   - Errors are reported by the return code, before any launch, with a
 *     thread-local message from flp_last_error().  Nothing traps on the GPU.
 *   - Results are deterministic: repeated calls give identical bits.
 */
#ifndef FUSED_LOGP_H
#define FUSED_LOGP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum flp_status {
    FLP_OK = 0,
    FLP_EINVAL = 1,        /* null pointer, bad extent or stride, host pointer,
                              pointers on different devices, bad overlap */
    FLP_EUNSUPPORTED = 2,  /* shard bounds off the tile grid */
    FLP_ECUDA = 3          /* a CUDA runtime call or the launch failed */
} flp_status;

/* Same type as cudaStream_t, declared without CUDA headers. */
typedef struct CUstream_st* flp_stream_t;

#define FLP_NUM_TILES 16

/* Logit dtypes of the _ex entry points (the gradient is written in the same
 * dtype).  PR #495 Tests name FP32/BF16/FP16 logits. */
#define FLP_DTYPE_BF16 0
#define FLP_DTYPE_F16 1
#define FLP_DTYPE_F32 2

/* Message of the last failing call on this thread ("" after success). */
const char* flp_last_error(void);

/* Library version string. */
const char* flp_version(void);

/* Tile width W for a vocabulary of v columns: 8 * ceil(v / 128); 0 if v < 1. */
int64_t flp_tile_width(int64_t v);

/*
 * Forward.  For t in [0, n):
 *   lse[t]  = M + log S, with (M, S) the index-order merge of the 16 tile
 *             partials (m_k, s_k), m_k = max over tile k, s_k = sum over tile
 *             k of exp(x - m_k), all FP32; the final log and add are carried
 *             in FP64 and rounded once to FP32.
 *   logp[t] = x[t, y_t] - lse (rounded once from FP64) if the row is active,
 *             else 0.
 *   logits   [n, ld] BF16, ld >= v >= 1 (columns >= v are never read)
 *   targets  [n] int64
 *   logp     [n] FP32 out
 *   lse      [n] FP32 out (keep it for the backward)
 *   lse_lo   [n] FP32 out, or NULL: the FP32 rounding residual of the LSE
 *            (LSE - lse, |lse_lo| <= half an ulp of lse).  Passing it to the
 *            backward removes the FP32 quantisation of the LSE from the
 *            gradient (an addition of this library; the pages store FP32 only).
 * Any alignment and any ld are accepted.  16-byte aligned rows with ld % 8 == 0
 * (and v < 2^31) stream through per-warp bulk-copy (TMA) rings in shared
 * memory; other layouts take a scalar-load path with the same arithmetic
 * (same bits).
 * Errors: FLP_EINVAL for n < 0, v < 1, ld < v, a null or host pointer.
 */
flp_status fused_logp_forward(const void* logits, int64_t n, int64_t v, int64_t ld,
                              const int64_t* targets, int64_t ignore_index,
                              float* logp, float* lse, float* lse_lo, flp_stream_t stream);

/*
 * Backward.  dlogits[t, c] for c in [0, v):
 *   active row:   g_t * (onehot(y_t)[c] - exp(x[t, c] - lse[t])), rounded
 *                 to nearest-even BF16 once, from an FP32 computation whose
 *                 exponent argument is carried with its rounding error;
 *   inactive row: +0.
 *   logits   [n, ld] BF16
 *   targets  [n] int64, lse [n] FP32 (from fused_logp_forward), grad [n] FP32
 *   lse_lo   [n] FP32 from fused_logp_forward, or NULL (then taken as 0)
 *   dlogits  [n, ld_out] BF16 out, ld_out >= v; columns >= v are untouched.
 * Gradient values below 2^-126 in magnitude flush to zero.
 * dlogits may alias logits exactly (same pointer and ld == ld_out: the
 * gradient then overwrites the logits in place); any other overlap is
 * FLP_EINVAL.  Elementwise, so batch-invariant by construction.
 */
flp_status fused_logp_backward(const void* logits, int64_t n, int64_t v, int64_t ld,
                               const int64_t* targets, int64_t ignore_index,
                               const float* lse, const float* lse_lo, const float* grad,
                               void* dlogits, int64_t ld_out, flp_stream_t stream);

/*
 * Vocab-shard partials (issue #241 PR 3 and PR 6 bullets; PR #314
 * ReductionSpec).  A shard holds global columns [vocab_start, vocab_start +
 * real_width) of a v_total-column vocabulary in its own buffer
 * shard_logits[n, ld_shard] (ld_shard >= real_width; columns >= real_width
 * are padding, masked to -inf, never read).  For each global tile k the shard
 * covers, writes part_max[t, k] and part_sum[t, k] (FP32, [n, 16] row-major),
 * bitwise equal to the forward's own tile partials.  For each row whose
 * target falls inside the shard, writes sel[t] = x[t, y_t] (the single-owner
 * copy of the selected logit); other rows' sel is left untouched.
 * The shard bounds must lie on the tile grid: vocab_start % W == 0, and
 * real_width % W == 0 unless the shard ends at v_total; otherwise
 * FLP_EUNSUPPORTED (the capability gate of issue #241 PR 6).
 * Columns of part_max/part_sum for tiles outside the shard are untouched.
 */
flp_status logp_shard_partials(const void* shard_logits, int64_t n, int64_t ld_shard,
                               int64_t vocab_start, int64_t real_width, int64_t v_total,
                               const int64_t* targets, float* part_max, float* part_sum,
                               float* sel, flp_stream_t stream);

/*
 * Merge (issue #241 PR 3 bullets: M = max m_l, S = sum s_l exp(m_l - M),
 * LSE = M + log S in fixed index order).  Folds the tile partials [n, 16]
 * of tiles 0 .. ceil(v_total / W) - 1 in index order with the same arithmetic
 * as the forward, then writes lse[t] and logp[t] = sel[t] - lse (active rows)
 * or 0.  Together with logp_shard_partials over shards that cover
 * [0, v_total), the results are bitwise equal to fused_logp_forward.
 * sel is read only for active rows.  lse_lo (nullable) as in the forward.
 */
flp_status logp_merge_partials(const float* part_max, const float* part_sum,
                               const float* sel, const int64_t* targets,
                               int64_t ignore_index, int64_t n, int64_t v_total,
                               float* logp, float* lse, float* lse_lo, flp_stream_t stream);

/*
 * Generalised forms (the calls above are these with FLP_DTYPE_BF16, no mask
 * and inv_temperature = 1).
 *   dtype           FLP_DTYPE_BF16 / FLP_DTYPE_F16 / FLP_DTYPE_F32: the dtype of
 *                   logits, shard_logits and dlogits.
 *   active_mask     [n] uint8 or NULL: a row is active only if its byte is
 *                   nonzero (and its target is in [0, v) and not ignore_index)
 *                   (PR #314, MaskMode explicit_active_mask).
 *   inv_temperature s = 1/T > 0, finite: the logits are scaled by s before the
 *                   log-softmax, as in rollout logprobs at a temperature (PR
 *                   #495, provider experiment at T = 1.0 and 0.7):
 *                   LSE = log sum exp(s x), logp = s x_y - LSE, and the
 *                   gradient with respect to the unscaled logits is
 *                   s g (onehot - exp(s x - LSE)).
 * Shard partials hold m = max x (unscaled) and sum exp(s (x - m)); a merge
 * must use the same inv_temperature as the partials.  Any other value of
 * dtype or inv_temperature is FLP_EINVAL.
 */
flp_status fused_logp_forward_ex(const void* logits, int dtype, int64_t n, int64_t v, int64_t ld,
                                 const int64_t* targets, int64_t ignore_index,
                                 const uint8_t* active_mask, float inv_temperature, float* logp,
                                 float* lse, float* lse_lo, flp_stream_t stream);
flp_status fused_logp_backward_ex(const void* logits, int dtype, int64_t n, int64_t v, int64_t ld,
                                  const int64_t* targets, int64_t ignore_index,
                                  const uint8_t* active_mask, float inv_temperature,
                                  const float* lse, const float* lse_lo, const float* grad,
                                  void* dlogits, int64_t ld_out, flp_stream_t stream);
flp_status logp_shard_partials_ex(const void* shard_logits, int dtype, int64_t n, int64_t ld_shard,
                                  int64_t vocab_start, int64_t real_width, int64_t v_total,
                                  float inv_temperature, const int64_t* targets, float* part_max,
                                  float* part_sum, float* sel, flp_stream_t stream);
flp_status logp_merge_partials_ex(const float* part_max, const float* part_sum, const float* sel,
                                  const int64_t* targets, int64_t ignore_index,
                                  const uint8_t* active_mask, int64_t n, int64_t v_total,
                                  float inv_temperature, float* logp, float* lse, float* lse_lo,
                                  flp_stream_t stream);

/*
 * Backward of one vocabulary shard (PR #314 "Deterministic config option":
 * the vocab-parallel logprob op is an autograd function over the local shard,
 * whose backward each rank runs on its own columns with the merged LSE; the
 * method's backward, PR #495 Summary item 2).  The shard holds global columns
 * [vocab_start, vocab_start + real_width) of a v_total-column vocabulary in
 * shard_logits[n, ld_shard].  For c in [0, real_width):
 *   dshard[t, c] = s g_t (onehot(y_t)[vocab_start + c] - exp(s x[t, c] - LSE_t))
 * with lse (+ lse_lo) the merged, global values.  A row is active by its
 * global target (0 <= y_t < v_total, not ignore_index, mask byte nonzero);
 * the one-hot term appears only in the shard that holds y_t.  Inactive rows
 * get +0.  Elementwise, with the unsharded backward's arithmetic: the shards'
 * outputs side by side are bitwise the unsharded dlogits, for any split (the
 * bounds need not lie on the tile grid).  dshard may alias shard_logits
 * exactly (in place); other overlap is FLP_EINVAL.  Other arguments and
 * errors as for fused_logp_backward_ex; FLP_EINVAL if the shard is not inside
 * [0, v_total).
 */
flp_status logp_shard_backward(const void* shard_logits, int64_t n, int64_t ld_shard, int64_t vocab_start,
                               int64_t real_width, int64_t v_total, const int64_t* targets,
                               int64_t ignore_index, const float* lse, const float* lse_lo,
                               const float* grad, void* dshard, int64_t ld_out, flp_stream_t stream);
flp_status logp_shard_backward_ex(const void* shard_logits, int dtype, int64_t n, int64_t ld_shard,
                                  int64_t vocab_start, int64_t real_width, int64_t v_total,
                                  const int64_t* targets, int64_t ignore_index, const uint8_t* active_mask,
                                  float inv_temperature, const float* lse, const float* lse_lo,
                                  const float* grad, void* dshard, int64_t ld_out, flp_stream_t stream);

/*
 * Merge of partials gathered from the ranks of a vocabulary-parallel group
 * (issue #241 PR 3 bullets: per-shard (max, sumexp) partials, the collective
 * only transports them, one merge in fixed index order; PR 6: each rank emits
 * (max, sumexp, selected_logit); PR #314 Tensor Parallel section: the tile
 * partials are all-gathered and every rank runs the same merge).
 *   gathered     device FP32; rank r's block starts at gathered + r *
 *                rank_stride and holds, in this order, its tile maxima
 *                [n, 16], tile sums [n, 16] and selected logits [n] (33 n
 *                floats), as logp_shard_partials_ex writes them into
 *                part_max = block, part_sum = block + 16 n, sel = block + 32 n.
 *                An all-gather of each rank's block is the whole exchange.
 *   rank_stride  floats between consecutive ranks' blocks (>= 33 n when
 *                world > 1; ignored when world == 1)
 *   world        ranks, 1 ..16
 *   vocab_starts, real_widths  HOST arrays [world]: rank r's shard is
 *                [vocab_starts[r], vocab_starts[r] + real_widths[r]); each on
 *                the tile grid (as logp_shard_partials requires), together
 *                covering every tile of [0, v_total) exactly once, else
 *                FLP_EUNSUPPORTED (off the grid) or FLP_EINVAL (gap, overlap).
 * Tile k's partial is read from the rank holding it; row t's selected logit
 * from the rank holding column y_t.  Other bytes of the blocks are never
 * read.  Then as logp_merge_partials_ex: the result is bitwise equal to
 * fused_logp_forward_ex on the unsharded logits, for any world and split.
 */
flp_status logp_merge_gathered_partials_ex(const float* gathered, int64_t rank_stride, int64_t world,
                                           const int64_t* vocab_starts, const int64_t* real_widths,
                                           const int64_t* targets, int64_t ignore_index,
                                           const uint8_t* active_mask, int64_t n, int64_t v_total,
                                           float inv_temperature, float* logp, float* lse, float* lse_lo,
                                           flp_stream_t stream);

/*
 * Fused LM head + logp (linear_logp, named in RL-Kernel PR #495 Summary; the
 * pages give no formula or design).  The logits z = H W^T of BF16 hidden
 * states and BF16 LM-head weight rows are formed on the tensor cores and
 * reduced where they are formed; they never reach memory.  Then, as for
 * fused_logp_forward_ex on logits s z:
 *   lse[t]  = log sum_j exp(s z[t, j]),  logp[t] = s z[t, y_t] - lse[t]
 * (0 for inactive rows), lse_lo[t] the FP32 rounding residual of the LSE.
 *   hidden    [n, ld_h] BF16 device, row-major; the first d columns are used
 *   weight    [v, ld_w] BF16 device, row-major (one row per vocabulary entry)
 *   targets   [n] int64; ignore_index and active_mask as for the forward
 *   inv_temperature  s = 1/T (> 0, finite)
 *   workspace device scratch of at least fused_linear_logp_workspace_size
 *             bytes (16-byte aligned), owned by the caller; contents on
 *             return are unspecified.  Layout: FP32 tile maxima [n,
 *             ceil(v/256)], tile sums [n, ceil(v/256)], selected logits [n].
 *   logp, lse [n] FP32 out; lse_lo [n] FP32 out or NULL
 * Accumulation: FP32 on the tensor cores (BF16 products exact), 128 x 256
 * tiles, K in increasing order; each row's result is independent of n, of
 * its position in the batch and of the grid (deterministic, batch-invariant).
 * Requirements: hidden and weight 16-byte aligned, ld_h and ld_w multiples
 * of 8 (16-byte row strides for the tensor-map copies), n, v, d < 2^31;
 * otherwise FLP_EUNSUPPORTED.  FLP_EINVAL for negative sizes, ld < d, a null
 * or small workspace, pointers on different devices.  n == 0 is a no-op.
 * Asynchronous on `stream`; the library allocates nothing.
 */
flp_status fused_linear_logp_workspace_size(int64_t n, int64_t v, int64_t* bytes);
flp_status fused_linear_logp_forward(const void* hidden, int64_t n, int64_t d, int64_t ld_h,
                                     const void* weight, int64_t v, int64_t ld_w, const int64_t* targets,
                                     int64_t ignore_index, const uint8_t* active_mask, float inv_temperature,
                                     void* workspace, int64_t workspace_bytes, float* logp, float* lse,
                                     float* lse_lo, flp_stream_t stream);

/*
 * Vocabulary-sharded fused LM head on one GPU (issue #241 PR 3 and PR 6: a
 * shard emits (max, sumexp) partials of the tiles it holds plus the selected
 * logit it owns; one fixed-order merge; PR #314 Tensor Parallel section: the
 * tile grid makes every shard count give the same bits).  The weight rows of
 * a vocabulary-parallel LM head are split into shards; shard l holds global
 * columns [vocab_start, vocab_start + real_width) as its own [real_width,
 * ld_w] BF16 buffer.
 *   fused_linear_logp_shard_partials writes that shard's tile partials into
 *     `workspace` (the layout of fused_linear_logp_forward's workspace for n
 *     rows and v_total columns: FP32 [n, ceil(v_total/256)] maxima and sums,
 *     [n] selected logits) and the selected logit of every row whose target
 *     is in the shard.  vocab_start must be a multiple of 256 (the tile
 *     grid), else FLP_EUNSUPPORTED; [vocab_start, vocab_start + real_width)
 *     must lie in [0, v_total).
 *   fused_linear_logp_merge merges, in tile order, the partials of all tiles
 *     of [0, v_total) into logp, lse (and lse_lo), as the forward does.
 * The shards must together cover [0, v_total) (the merge reads every tile's
 * partial).  With that, the result is bitwise equal to
 * fused_linear_logp_forward on the unsharded weight, for any shard count.
 * All calls asynchronous on `stream`; the library allocates nothing.
 */
flp_status fused_linear_logp_shard_partials(const void* hidden, int64_t n, int64_t d, int64_t ld_h,
                                            const void* weight_shard, int64_t real_width, int64_t ld_w,
                                            int64_t vocab_start, int64_t v_total, const int64_t* targets,
                                            float inv_temperature, void* workspace, int64_t workspace_bytes,
                                            flp_stream_t stream);
flp_status fused_linear_logp_merge(const void* workspace, int64_t workspace_bytes, int64_t n, int64_t v_total,
                                   const int64_t* targets, int64_t ignore_index, const uint8_t* active_mask,
                                   float inv_temperature, float* logp, float* lse, float* lse_lo,
                                   flp_stream_t stream);

/*
 * Backward of the fused LM head (no counterpart in the pages beyond the name
 * linear_logp; the method's backward, PR #495 Summary item 2, taken through
 * the contraction): for the loss sum_t grad[t] logp[t],
 *   dZ[t, j] = s grad[t] (onehot(y_t)[j] - exp(s z[t, j] - LSE_t)),
 *   dhidden = dZ W   [n, d],   dweight = dZ^T H   [v, d],
 * with dZ recomputed on the tensor cores from hidden and weight and the
 * forward's lse (+ lse_lo) and written in BF16 (as the method writes dlogits)
 * one chunk of 4096 rows at a time into the workspace, never as an [n, v]
 * tensor.  The two products run on this library's own tensor-core kernels,
 * reading dZ, W and H where they lie (FP32 accumulation): dhidden in
 * S = ceil(ceil(v / 64) / 512) fixed splits of the vocabulary added in split
 * order, dweight added chunk after chunk in row order.  No atomics:
 * deterministic.
 *   hidden, weight, targets, ignore_index, active_mask, inv_temperature: as
 *             for fused_linear_logp_forward (the same call's arguments)
 *   lse       [n] FP32, lse_lo [n] FP32 or NULL: the forward's outputs
 *   grad      [n] FP32 d loss / d logp (0 for inactive rows by definition)
 *   workspace device scratch of fused_linear_logp_backward_workspace_size
 *             bytes (256-byte aligned), caller-owned: dZ [4096, ceil(v/8)*8]
 *             BF16 and, when S > 1, the splits' partial dhidden
 *             [S, 4096, d] FP32
 *   dhidden   [n, ld_dh] FP32 out
 *   dweight   [v, ld_dw] FP32: overwritten with dZ^T H when
 *             accumulate_dweight == 0 (all zero when n == 0), or with
 *             dweight + dZ^T H when it is nonzero (gradient accumulation over
 *             micro-batches; unchanged when n == 0).  With n == 0 only dweight
 *             is touched and the workspace may be NULL.
 * Each element of dhidden is a tensor-core dot product over the vocabulary
 * with split points fixed by v, whatever else the chunk holds, so a row's
 * dhidden does not depend on n or on its position.
 * Requirements and errors as for the forward, plus ld_dh, ld_dw >= d.
 * Asynchronous on `stream`; the library allocates nothing.
 */
flp_status fused_linear_logp_backward_workspace_size(int64_t d, int64_t v, int64_t* bytes);
flp_status fused_linear_logp_backward(const void* hidden, int64_t n, int64_t d, int64_t ld_h, const void* weight,
                                      int64_t v, int64_t ld_w, const int64_t* targets, int64_t ignore_index,
                                      const uint8_t* active_mask, float inv_temperature, const float* lse,
                                      const float* lse_lo, const float* grad, void* workspace,
                                      int64_t workspace_bytes, float* dhidden, int64_t ld_dh, float* dweight,
                                      int64_t ld_dw, int accumulate_dweight, flp_stream_t stream);

/*
 * Backward of one vocabulary shard of the fused LM head (the shard layout of
 * fused_linear_logp_shard_partials; lse and lse_lo are the merged, global
 * values): dZ for the shard's columns, its rows of dweight, and its term of
 * dhidden = sum over shards of dZ_shard W_shard.
 *   dhidden           [n, ld_dh] FP32: overwritten with this shard's term,
 *                     or added to when accumulate_dhidden is nonzero (call
 *                     the shards in a fixed order, the first without it)
 *   dweight_shard     [real_width, ld_dw] FP32 (overwritten, or added to with
 *                     accumulate_dweight)
 *   workspace         fused_linear_logp_backward_workspace_size(d, real_width)
 * vocab_start must be a multiple of 256, else FLP_EUNSUPPORTED.  The
 * summed dhidden is deterministic for a fixed shard layout; it is not bitwise
 * equal to the unsharded backward's (the sum over the vocabulary is split).
 * Other arguments and errors as for fused_linear_logp_backward.
 */
flp_status fused_linear_logp_shard_backward(const void* hidden, int64_t n, int64_t d, int64_t ld_h,
                                            const void* weight_shard, int64_t real_width, int64_t ld_w,
                                            int64_t vocab_start, int64_t v_total, const int64_t* targets,
                                            int64_t ignore_index, const uint8_t* active_mask, float inv_temperature,
                                            const float* lse, const float* lse_lo, const float* grad,
                                            void* workspace, int64_t workspace_bytes, float* dhidden,
                                            int64_t ld_dh, int accumulate_dhidden, float* dweight_shard,
                                            int64_t ld_dw, int accumulate_dweight, flp_stream_t stream);

/*
 * Fused LM head + logp with no allocation and no workspace argument.  The
 * pages have no counterpart: this is a convenience of this library.
 *
 * Some callers cannot allocate device memory at all: a plugin that a host
 * application hands only its input and output buffers, code running under an
 * application-wide memory pool that owns all device memory and forbids direct
 * cudaMalloc calls, or a tight loop where a cudaMalloc/cudaFree pair would
 * synchronise the device.  For them this entry point computes exactly what
 * fused_linear_logp_forward computes (same arguments minus the workspace;
 * identical bits) and takes its scratch from a fixed 16 MiB array in the
 * library's static device memory.  It calls no allocator.
 *   Limit: the scratch needed, fused_linear_logp_workspace_size(n, v), must
 *   be at most 16 MiB (16777216 bytes): up to 3527 rows per call at
 *   v = 151936.  Larger calls return FLP_EUNSUPPORTED with a message naming
 *   the sizes; split the rows, or use fused_linear_logp_forward.
 *   Memory: every GPU that loads the library holds the 16 MiB until the
 *   process exits.
 *   First call per device: looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make
 *   that first call before any stream capture.  The cached address belongs
 *   to the device's context: after cudaDeviceReset it is stale, so do not
 *   call this entry point again in a process that has reset the device.
 *   Sharing: all calls in the process use the same array.  Calls whose work
 *   can overlap on a GPU (different streams, or different host threads
 *   without ordering) race on it and give wrong results; order them, e.g. on
 *   one stream.  The array keeps the previous call's contents, and nothing in
 *   it needs to start at zero: every element a call reads was written
 *   earlier in that same call.
 * Errors: as fused_linear_logp_forward, plus FLP_EUNSUPPORTED above the limit.
 */
flp_status fused_linear_logp_forward_noalloc(const void* hidden, int64_t n, int64_t d, int64_t ld_h,
                                             const void* weight, int64_t v, int64_t ld_w,
                                             const int64_t* targets, int64_t ignore_index,
                                             const uint8_t* active_mask, float inv_temperature, float* logp,
                                             float* lse, float* lse_lo, flp_stream_t stream);

/*
 * The fused LM head across several processes, one vocabulary slice of the
 * weight per rank (the tensor-parallel output layer; the exchange is the
 * tile-partial all-gather of issue #241 PR 3 / PR #314 Tensor Parallel,
 * transport only, then the same fixed-order merge on every rank).
 *
 * fused_linear_logp_merge_gathered: every rank ran
 * fused_linear_logp_shard_partials on its slice into its own workspace (the
 * slices on the 256-column tile grid, covering every tile once); `gathered`
 * holds the world workspaces one after another, rank r's at gathered +
 * r * rank_stride (floats; rank_stride >= (2 ceil(v_total / 256) + 1) n, e.g.
 * the workspace's size / 4).  vocab_starts / real_widths are host arrays of
 * world entries (at most 16).  Tile k is read from the rank that holds it
 * and row t's selected logit from the rank that holds its target's tile:
 * logp, lse (and lse_lo) are those of fused_linear_logp_merge over one
 * workspace that all slices wrote, bit for bit.
 * Errors: FLP_EINVAL for bad extents, a stride below one block, a slice
 * outside the vocabulary, a tile held by no rank or by two;
 * FLP_EUNSUPPORTED for a slice off the tile grid.
 *
 * flp_sum_blocks: out[r, c] = ((b_0 + b_1) + b_2) + ... over world FP32
 * blocks [rows, cols] (row pitch cols) at blocks + k * block_stride, one
 * rounding per addition in block order -- the sum that the one-GPU sharded
 * LM-head backward forms when each later shard adds its term of dhidden, so
 * the ranks' all-gathered terms summed here give its dhidden bit for bit.
 * out has row pitch ld_out and must not overlap the blocks.
 */
flp_status fused_linear_logp_merge_gathered(const float* gathered, int64_t rank_stride, int world,
                                            const int64_t* vocab_starts, const int64_t* real_widths, int64_t n,
                                            int64_t v_total, const int64_t* targets, int64_t ignore_index,
                                            const uint8_t* active_mask, float inv_temperature, float* logp,
                                            float* lse, float* lse_lo, flp_stream_t stream);
flp_status flp_sum_blocks(const float* blocks, int64_t block_stride, int world, int64_t rows, int64_t cols,
                          float* out, int64_t ld_out, flp_stream_t stream);

/*
 * GRPO loss on the logp path (issue #241 PR 5: ratio, clip, KL, advantage,
 * a declared normaliser and a fixed summation order; the pages name these
 * terms, the formulas below are the standard clipped-surrogate form).
 * Per active token t (active_mask byte nonzero, or all when NULL):
 *   r = exp(logp - old_logp),
 *   pg = max(-A r, -A clip(r, 1 - eps_lo, 1 + eps_hi)),
 *   kl = exp(ref - logp) - (ref - logp) - 1 (only if ref_logp != NULL),
 *   l = pg + beta kl.
 * mode FLP_GRPO_TOKEN_MEAN:          loss = sum_t l / D (D = active tokens)
 *      FLP_GRPO_SEQ_MEAN_TOKEN_MEAN: loss = mean over non-empty sequences of
 *                                    the sequence's mean l
 *      FLP_GRPO_SEQ_MEAN_TOKEN_SUM:  loss = mean over non-empty sequences of
 *                                    the sequence's summed l
 * Sequences are [cu_seqlens[s], cu_seqlens[s+1]) for s < num_seqs (int64 on
 * the device; bounds are clamped to [0, n]); with cu_seqlens == NULL the whole
 * batch is one sequence.  normalizer > 0 replaces D (token mean) or the
 * sequence count, e.g. by a count global to all micro-batches.
 *   loss       [1] FP32 out
 *   grad       [n] FP32 out: d loss / d logp (the unclipped term's -A r when
 *              it is the max, ties included, else 0; plus beta (1 - e^(ref -
 *              logp)); times the token's normaliser weight; 0 when inactive)
 *              -- the upstream gradient for fused_logp_backward.
 *   token_loss [n] FP32 out or NULL: l per token (0 when inactive).
 *   workspace  device scratch of logp_grpo_loss_workspace_size(n, num_seqs)
 *              bytes (16-byte aligned), caller-owned, no initial contents
 *              needed: 32 bytes for a count and the fold's ticket, 9.5 KB
 *              for the token pass's per-CTA sums, 16 KB of counts, and with
 *              sequences 8 bytes per sequence and 4 per 16 tokens; rounded
 *              up to 256 bytes.  One workspace serves one call at a time.
 * Tokens outside every sequence (before cu_seqlens[0] or from
 * cu_seqlens[num_seqs] on) are inactive: l = 0, grad 0.  cu_seqlens must be
 * non-decreasing; for one that is not, the result is unspecified, but every
 * access stays inside the arrays.
 * Kernels: when a weight depends on the mask (any normaliser but the
 * caller's uniform one), a count of the mask's active tokens per 16-token
 * word and per range, then per sequence its active count, the number of
 * non-empty sequences and the active tokens; then one token pass that
 * writes each final gradient once and folds the loss.  Integer counts are
 * exact.  Deterministic: the batch is cut into fixed 256-token chunks (one
 * warp each) whatever the sequence lengths; sums are plain FP32 within a
 * chunk and compensated two-float sums in FP32 from there on, folded per
 * warp over its contiguous chunks, per CTA in warp order and over the CTAs
 * in order, a shape fixed by n; the result does not depend on timing.  A
 * gradient is dl/dlogp times its weight, rounded once: 1 / den, or for the
 * sequence mean of token means the product of the correctly rounded 1 / den
 * and 1 / n_s.  With logp == old_logp the ratio is exactly 1 and grad = -A
 * times the weight (the KL = 0 identity of PR 5).
 * Errors: FLP_EINVAL for a bad mode, eps_lo outside [0, 1), a negative or
 * non-finite eps_hi, beta or normalizer, a sequence mode without sequences,
 * or num_seqs >= 2^31 - 1.
 */
#define FLP_GRPO_TOKEN_MEAN 0
#define FLP_GRPO_SEQ_MEAN_TOKEN_MEAN 1
#define FLP_GRPO_SEQ_MEAN_TOKEN_SUM 2
flp_status logp_grpo_loss_workspace_size(int64_t n, int64_t num_seqs, int64_t* bytes);
flp_status logp_grpo_loss(const float* logp, const float* old_logp, const float* ref_logp,
                          const float* advantages, const uint8_t* active_mask,
                          const int64_t* cu_seqlens, int64_t num_seqs, int64_t n, int mode,
                          float eps_lo, float eps_hi, float beta, float normalizer, void* workspace,
                          int64_t workspace_bytes, float* loss, float* grad, float* token_loss,
                          flp_stream_t stream);

/*
 * The GRPO loss in two parts, for a batch whose layout (active_mask,
 * cu_seqlens, n, num_seqs, mode, normalizer) is known before its logp: the
 * normaliser weights depend on the layout only (issue #241 PR 5's declared
 * normaliser), so they can be counted once, e.g. on a second stream while
 * the logp forward runs, or once for several optimisation epochs over the
 * same batch.
 *
 * logp_grpo_loss_counts runs the counting kernels of logp_grpo_loss (the
 * mask's counts, each sequence's active count, the number of non-empty
 * sequences) into `workspace` and records a tag of the layout: the mask and
 * cu_seqlens pointers, n, num_seqs, mode and normalizer.  Arguments as for
 * logp_grpo_loss; nothing else is read or written.
 *
 * logp_grpo_loss_counted is logp_grpo_loss with the counting left out: it
 * runs the token pass on counts that an earlier logp_grpo_loss_counts (or
 * logp_grpo_loss) call left in the same workspace, which must have completed
 * on the device first (same stream, or an event).  Results are bitwise those
 * of logp_grpo_loss.  The layout arguments must be the ones the counts were
 * taken for and the mask and cu_seqlens contents unchanged since: the token
 * pass compares the recorded tag with the call's, and on a mismatch writes
 * NaN for the loss and for the gradient of every token inside a sequence (the
 * contents themselves are not compared).  Calls may repeat on the same
 * counts.  When the weight is the caller's (a normalizer with the token mean
 * or the sequence mean of token sums) nothing is counted and the call is
 * logp_grpo_loss, which replaces the counts and the tag in the workspace
 * (a later counted call for the earlier layout then gets NaN: count again).
 * Errors: as logp_grpo_loss.
 */
flp_status logp_grpo_loss_counts(const uint8_t* active_mask, const int64_t* cu_seqlens, int64_t num_seqs,
                                 int64_t n, int mode, float normalizer, void* workspace, int64_t workspace_bytes,
                                 flp_stream_t stream);
flp_status logp_grpo_loss_counted(const float* logp, const float* old_logp, const float* ref_logp,
                                  const float* advantages, const uint8_t* active_mask,
                                  const int64_t* cu_seqlens, int64_t num_seqs, int64_t n, int mode,
                                  float eps_lo, float eps_hi, float beta, float normalizer, void* workspace,
                                  int64_t workspace_bytes, float* loss, float* grad, float* token_loss,
                                  flp_stream_t stream);

/*
 * Health of the device side (no counterpart in the pages: a guard of this
 * library's own waits).  The bulk-copy forward waits on its own copies with a
 * bounded wait (about 2 s); if one runs out, the kernel records it in a
 * sticky device word, stops issuing copies, drains the ones in flight and
 * returns, so the context stays usable.  flp_device_error synchronises with
 * `device`, returns that word in *code (0 = no wait ran out) and clears it.
 */
flp_status flp_device_error(int device, int* code);

/*
 * Self-test of the bounded wait: launches one thread on `device` that waits on
 * a barrier nothing arrives on, with a limit of limit_cycles SM cycles
 * (at most 1e8), synchronises, and sets *timed_out = 1 if the wait gave up
 * (it must).  Also sets the sticky word read by flp_device_error.
 */
flp_status flp_selftest_wait_timeout(int device, int64_t limit_cycles, int* timed_out);

/*
 * Self-test of the exp2 bias correction (no counterpart in the pages).  The
 * forward sums terms 2^a from the special-function unit's ex2.approx, whose
 * results are low by a nearly constant ~5e-8 relative; each tile sum is
 * scaled by (1 + c) to remove it.  This measures the mean relative error of
 * ex2.approx over 2^20 arguments in [-24, 0) on `device` (synchronising) and
 * returns it with the compiled-in c, so a test can check that c still
 * matches the hardware (mean_rel_err ~ -c).
 */
flp_status flp_selftest_ex2_bias(int device, double* mean_rel_err, double* compensation);

#ifdef __cplusplus
}
#endif

#endif /* FUSED_LOGP_H */
