/*
 * attn.h -- C ABI of the GB300 (sm_103a) tiled online-softmax attention library.
 *
 * Exact scaled-dot-product attention over [B, H, N, d] tensors:
 *
 *   O = softmax(scale * Q K^T) V
 *
 * ("FlashAttention hardware-aware analysis" (huaweicloud), section one, part 2,
 * and the PyTorch scaled_dot_product_attention call of section five, part 1,
 * whose [Batch, Heads, Seq_Len, Head_Dim] layout and is_causal flag this ABI
 * keeps.)  The forward pass streams K/V tiles through the online-softmax
 * recurrence (running row max m and row sum l, partial output rescaled by
 * exp(m_old - m_new); huaweicloud page, section two; "Understanding online
 * softmax in Flash Attention from scratch", section 3.1), defers the 1/l
 * normalisation to the end, and saves the per-row logsumexp.  The backward
 * pass recomputes P tile by tile from that logsumexp ("Understanding
 * FlashAttention, Part 2", section 2.4; huaweicloud page, section four,
 * part 1: recomputation) and never stores an N x N matrix.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are dense, row-major [B][H][N][d] with d fastest ("contiguous"),
 *    in the 16-bit type given by `dt`.  lse is float32 [B][H][N].
 *  - All pointers are DEVICE pointers on the current CUDA device unless stated.
 *    Every base pointer must be 16-byte aligned.  The caller owns all memory;
 *    the library allocates nothing on the device and keeps no state between
 *    calls.
 *  - d must be 64, 128 or 256 (64 and 128 are the head dimensions the huaweicloud
 *    page's section five, part 2 recommends; 256 is listed with them in its part
 *    1); attn_fwd_fp8 takes 128 only.  Anything else returns ATTN_ERR_UNSUPPORTED.
 *    N >= 1 may be any value (ragged last tiles are masked, never padded in
 *    memory).  B, H >= 1 and B*H*N*d < 2^31.
 *  - causal != 0 keeps key j for query i iff j <= i (the lower triangle,
 *    huaweicloud page, section five, part 3); tiles wholly above the
 *    diagonal are skipped, not masked.
 *  - scale multiplies Q K^T; pass 1/sqrt(d) for standard attention.  It must
 *    be finite and positive.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Argument errors are returned before anything is
 *    launched.  A launch failure returns ATTN_ERR_CUDA.
 *  - dev_status (nullable) is a device int the caller zeroes; a kernel whose
 *    bounded wait on an mbarrier expires (a hardware or library fault, never
 *    a normal outcome) stores ATTN_ERR_TIMEOUT there, abandons its tile and
 *    exits cleanly.  Read it after synchronising the stream.  (The d = 256
 *    backward kernels also store ATTN_ERR_CUDA there, and do nothing, if
 *    their dynamic shared memory does not start within 768 bytes of a
 *    1024-byte boundary; it starts on one on current drivers.)
 *  - On any error the output buffers' contents are unspecified.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, bad scale, ws too small */
    ATTN_ERR_UNSUPPORTED = 2,   /* d not supported by the call, unknown dtype, device is not sm_103 */
    ATTN_ERR_CUDA = 3,          /* a CUDA runtime/driver call or a launch failed */
    ATTN_ERR_TIMEOUT = 4        /* (device-side only) a bounded wait expired */
} attn_status;

typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1 } attn_dtype;

/*
 * attn_fwd -- forward pass.
 *   q, k, v : [B][H][N][d] inputs (read only).
 *   o       : [B][H][N][d] output, O = softmax(scale*QK^T) V rounded to dt.
 *   lse     : [B][H][N] float32 output, natural-log logsumexp of the scaled
 *             scores of each row, lse_i = m_i + ln l_i (the saved statistics
 *             of "Understanding FlashAttention, Part 2", section 2.2).
 *   o and lse must not overlap the inputs.
 *   d may be 64, 128 or 256 (at 256 each CTA owns one 128-row query tile).
 * At d = 128 without a causal mask, rows of at least 48 key tiles of 128 run on CTA
 * pairs: two CTAs on neighbouring SMs share each product (tcgen05 cta_group::2) and each
 * keeps three score tiles in flight; everything else runs one CTA per two query tiles.
 * Both give the same bytes.  The environment variable ATTN_FWD_CTA_PAIR=1 or =0, read on
 * every call, forces the pair or the one-CTA kernel.  At d = 64 with an even number of
 * 128-row query tiles, ATTN_FWD_PERSIST=1 (read on every call) runs a persistent grid
 * instead, whose CTAs take further work units from the hardware scheduler (cluster launch
 * control); the same bytes, faster only for short rows of many heads, so not the default.
 */
ATTN_API attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                     int *dev_status, void *stream);

/*
 * attn_fwd_rect -- attn_fwd with Nq queries against Nk keys (cross-attention, or a
 * block of new queries attending to earlier positions as well).
 *   q, o    : [B][H][Nq][d];  k, v : [B][H][Nk][d];  lse : [B][H][Nq].
 *   causal  : the lower triangle of the huaweicloud page's section five, part 3,
 *             aligned to the last key: query i sees key j iff j <= i + (Nk - Nq),
 *             so the queries are the last Nq of Nk positions.  Needs Nk >= Nq
 *             (else ATTN_ERR_INVALID_ARG); Nq = Nk is attn_fwd.
 * Everything else (d in {64, 128, 256}, dtypes, scale, errors) is as for attn_fwd;
 * the size limit applies to B*H*max(Nq, Nk)*d.
 */
ATTN_API attn_status attn_fwd_rect(const void *q, const void *k, const void *v, void *o, float *lse,
                          int B, int H, int Nq, int Nk, int d, attn_dtype dt, int causal, float scale,
                          int *dev_status, void *stream);

/*
 * attn_fwd_varlen / attn_bwd_varlen -- a batch of B sequences of different lengths packed
 * along the token axis (no padding): q, o, dout, dq are [Tq][H][d], k, v, dk, dv
 * [Tk][H][d], lse [H][Tq] float32.  cu_q and cu_k are DEVICE int32 arrays of B + 1
 * token offsets (cu[0] = 0, non-decreasing, cu[B] <= T): sequence b owns query tokens
 * cu_q[b] .. cu_q[b+1]-1 and key tokens cu_k[b] .. cu_k[b+1]-1, and each sequence and
 * head is the attention of its own rows (causal as in attn_fwd_rect: aligned to the
 * sequence's last key).  max_q, max_k bound the lengths (they size the grid); lengths
 * are clamped to them and to [0, T], so a malformed table cannot make the kernels
 * write outside the buffers, but its results are unspecified.  A sequence with no key,
 * or causal with fewer keys than queries, gets O = 0, lse = -inf and zero gradients.
 * The backward workspace is attn_bwd_workspace_bytes(B, H, max_q, d).  d in {64, 128, 256}.
 * Everything else is as for attn_fwd / attn_bwd.
 */
ATTN_API attn_status attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                            const int *cu_q, const int *cu_k, int B, int H, int max_q, int max_k,
                            int Tq, int Tk, int d, attn_dtype dt, int causal, float scale,
                            int *dev_status, void *stream);
ATTN_API attn_status attn_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                            const void *dout, const float *lse, void *dq, void *dk, void *dv,
                            void *workspace, size_t workspace_bytes, const int *cu_q, const int *cu_k,
                            int B, int H, int max_q, int max_k, int Tq, int Tk, int d, attn_dtype dt,
                            int causal, float scale, int *dev_status, void *stream);

/*
 * attn_fwd_dropout / attn_bwd_dropout -- attn_fwd / attn_bwd with dropout on the
 * attention probabilities (the recomputing backward of "Understanding
 * FlashAttention, Part 2", section 2.4, also covers dropout).  The pages fix no
 * random-number semantics; this library's are:
 *   t = round(256 * p_drop), p_drop finite in [0, 1) with t <= 255 (else
 *   ATTN_ERR_INVALID_ARG); the drop probability is t / 256.
 *   Element (bh, i, j) (bh = b*H + h, query i, key j) reads byte j mod 16 of
 *   Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3",
 *   SC 2011) at counter (j / 16, i, bh, 0) with key (seed low 32 bits, seed high
 *   32 bits), bytes taken little-endian from the four output words in order; it is
 *   kept iff that byte >= t.
 *   O = (P o Z) V with Z = keep * 256 / (256 - t); lse is the logsumexp of the
 *   scores, as without dropout.  The backward must get the same p_drop and seed:
 *   dV = (P o Z)^T dO, dS = P o (Z o dP - D), D_i = rowsum(dO_i o O_i).
 * d in {64, 128, 256}; square shapes (rectangular ones and packed batches: the
 * entry points below).
 * Everything else is as for attn_fwd / attn_bwd.
 * p_drop = 0 runs the plain kernels.
 */
ATTN_API attn_status attn_fwd_dropout(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                             float p_drop, uint64_t seed, int *dev_status, void *stream);
ATTN_API attn_status attn_bwd_dropout(const void *q, const void *k, const void *v, const void *o,
                             const void *dout, const float *lse, void *dq, void *dk, void *dv,
                             void *workspace, size_t workspace_bytes,
                             int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                             float p_drop, uint64_t seed, int *dev_status, void *stream);

/*
 * attn_fwd_dropout_bits / attn_bwd_dropout_bits -- attn_fwd_dropout / attn_bwd_dropout
 * with the keep decisions drawn once: the forward also stores every decision it draws
 * into keep_bits, and the backward reads them there instead of drawing them again (the
 * same decisions, so the results equal the drawing path's: O and lse byte for byte, dK
 * and dV byte for byte, dQ up to the order of the drawing path's float32 additions).
 * With the decisions stored, drawing them twice costs nothing, so the backward runs the
 * two deterministic kernels of attn_bwd (which read the bits), not the fused pass: the
 * same speed on GB300, and the same dQ bytes on every call.
 *   keep_bits      : device buffer of at least attn_dropout_bits_bytes(B, H, N, N) bytes,
 *                    16-byte aligned, owned by the caller; written by the forward, read
 *                    by the backward (which needs the forward's q, k, v, p and seed).
 *                    Bit b of 32-bit word ((bh * ceil(N/128) + j) * 4 + w) * Npad + i
 *                    (Npad = N rounded up to 128, bh = b * H + h) is the decision for
 *                    query i and key 128 j + 32 w + b; words of key tiles a causal query
 *                    tile never visits, and of rows past N, are not written.
 *   p_drop         : as for attn_fwd_dropout, but at least 1/512 (round(256 p) >= 1);
 *                    the backward takes no seed.
 *   d in {64, 128} (d = 256: ATTN_ERR_UNSUPPORTED).  Everything else is as for
 *   attn_fwd_dropout / attn_bwd_dropout.
 * attn_dropout_bits_bytes -- B*H*ceil(Nk/128)*4*Npad(Nq)*4 bytes (N^2/8 per head for
 *   Nq = Nk = N); 0 for invalid sizes.
 */
ATTN_API size_t attn_dropout_bits_bytes(int B, int H, int Nq, int Nk);
ATTN_API attn_status attn_fwd_dropout_bits(const void *q, const void *k, const void *v, void *o, float *lse,
                                  void *keep_bits, size_t keep_bits_bytes,
                                  int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                                  float p_drop, uint64_t seed, int *dev_status, void *stream);
ATTN_API attn_status attn_bwd_dropout_bits(const void *q, const void *k, const void *v, const void *o,
                                  const void *dout, const float *lse, const void *keep_bits,
                                  size_t keep_bits_bytes, void *dq, void *dk, void *dv,
                                  void *workspace, size_t workspace_bytes,
                                  int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                                  float p_drop, int *dev_status, void *stream);

/*
 * attn_fwd_rect_dropout / attn_bwd_rect_dropout -- attn_fwd_rect / attn_bwd_rect (Nq
 * queries against Nk keys, causal aligned to the last key) with attn_fwd_dropout's
 * dropout; element (bh, i, j) is query i and key j of the rectangular problem.
 * d in {64, 128, 256}; everything else is as for attn_fwd_rect / attn_bwd_rect.
 */
ATTN_API attn_status attn_fwd_rect_dropout(const void *q, const void *k, const void *v, void *o, float *lse,
                                  int B, int H, int Nq, int Nk, int d, attn_dtype dt, int causal,
                                  float scale, float p_drop, uint64_t seed, int *dev_status, void *stream);
ATTN_API attn_status attn_bwd_rect_dropout(const void *q, const void *k, const void *v, const void *o,
                                  const void *dout, const float *lse, void *dq, void *dk, void *dv,
                                  void *workspace, size_t workspace_bytes, int B, int H, int Nq, int Nk,
                                  int d, attn_dtype dt, int causal, float scale, float p_drop,
                                  uint64_t seed, int *dev_status, void *stream);

/*
 * attn_fwd_varlen_dropout / attn_bwd_varlen_dropout -- attn_fwd_varlen / attn_bwd_varlen
 * with attn_fwd_dropout's dropout.  The mask of a packed batch is that of the padded
 * batch: element (b, h, i, j) -- sequence b, head h, query i and key j counted from the
 * sequence's first token -- reads Philox at counter (j / 16, i, b*H + h, 0).  The
 * backward must get the same p_drop and seed.  d in {64, 128, 256}; everything else is
 * as for attn_fwd_varlen / attn_bwd_varlen and attn_fwd_dropout.
 */
ATTN_API attn_status attn_fwd_varlen_dropout(const void *q, const void *k, const void *v, void *o, float *lse,
                                    const int *cu_q, const int *cu_k, int B, int H, int max_q, int max_k,
                                    int Tq, int Tk, int d, attn_dtype dt, int causal, float scale,
                                    float p_drop, uint64_t seed, int *dev_status, void *stream);
ATTN_API attn_status attn_bwd_varlen_dropout(const void *q, const void *k, const void *v, const void *o,
                                    const void *dout, const float *lse, void *dq, void *dk, void *dv,
                                    void *workspace, size_t workspace_bytes, const int *cu_q,
                                    const int *cu_k, int B, int H, int max_q, int max_k, int Tq, int Tk,
                                    int d, attn_dtype dt, int causal, float scale, float p_drop,
                                    uint64_t seed, int *dev_status, void *stream);

/*
 * attn_fwd_splitkv -- the forward pass for shapes with too few query tiles to fill
 * the GPU (few heads, long sequences): every pair of 128-row query tiles has its key
 * tiles cut into n_splits contiguous ranges, each processed by its own CTA, which
 * writes its range's normalised partial output and logsumexp; a merge kernel then
 * combines the ranges with the two-block merge rule of "FlashAttention
 * hardware-aware analysis" (huaweicloud), section two:
 *   M = max_s lse_s,  O = sum_s e^(lse_s - M) O_s / sum_s e^(lse_s - M),
 *   lse = M + ln sum_s e^(lse_s - M).
 * Results equal attn_fwd's up to rounding (the partials are kept in float32).
 *   n_splits  : 1..64; a pair with fewer visible key tiles than n_splits uses as
 *               many ranges as it has tiles.  (At d = 256 the unit is one query
 *               tile instead of a pair.)
 *   workspace : device scratch of attn_fwd_splitkv_workspace_bytes(B, H, N, d,
 *               n_splits) = n_splits*B*H*N*(d+1)*4 bytes, 16-byte aligned, owned by
 *               the caller, clobbered.  It must not overlap any other argument.
 * Everything else (layouts, d in {64, 128, 256}, causal, scale, errors) is as for
 * attn_fwd.
 */
ATTN_API size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int N, int d, int n_splits);
ATTN_API attn_status attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                             void *workspace, size_t workspace_bytes,
                             int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                             int n_splits, int *dev_status, void *stream);

/*
 * attn_fwd_splitkv_rect -- attn_fwd_splitkv for attn_fwd_rect's shapes: Nq queries
 * against Nk keys, q, o [B][H][Nq][d], k, v [B][H][Nk][d], lse [B][H][Nq], causal
 * aligned to the last key (Nk >= Nq).  Meant for few queries over a long key sequence
 * (decoding a block of new tokens after a long prefix), where the query tiles alone
 * leave most of the GPU idle.  The workspace is attn_fwd_splitkv_workspace_bytes(B, H,
 * Nq, d, n_splits).  Everything else is as for attn_fwd_splitkv / attn_fwd_rect.
 */
ATTN_API attn_status attn_fwd_splitkv_rect(const void *q, const void *k, const void *v, void *o, float *lse,
                                  void *workspace, size_t workspace_bytes,
                                  int B, int H, int Nq, int Nk, int d, attn_dtype dt, int causal,
                                  float scale, int n_splits, int *dev_status, void *stream);

/*
 * attn_fwd_varlen_splitkv -- attn_fwd_varlen with split-KV: each sequence's query tiles
 * have their visible key tiles cut into n_splits ranges (1..64), each range's CTA writes
 * a float32 partial output and logsumexp, and the merge kernel combines them (the rule
 * of attn_fwd_splitkv).  For batches of few sequences and heads with long keys (decoding
 * several sequences of different lengths).  Rows of a degenerate sequence get O = 0,
 * lse = -inf as in attn_fwd_varlen; tokens outside cu_q[0] .. cu_q[B] are not written.
 *   workspace : device scratch of attn_fwd_varlen_splitkv_workspace_bytes(H, Tq, d,
 *               n_splits) = n_splits*Tq*H*(d+1)*4 bytes, 16-byte aligned, owned by the
 *               caller, clobbered; it must not overlap any other argument.
 * d in {64, 128, 256}; everything else is as for attn_fwd_varlen.
 */
ATTN_API size_t attn_fwd_varlen_splitkv_workspace_bytes(int H, int Tq, int d, int n_splits);
ATTN_API attn_status attn_fwd_varlen_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                                    void *workspace, size_t workspace_bytes, const int *cu_q,
                                    const int *cu_k, int B, int H, int max_q, int max_k, int Tq, int Tk,
                                    int d, attn_dtype dt, int causal, float scale, int n_splits,
                                    int *dev_status, void *stream);

/*
 * attn_fwd_fp8 -- forward pass on FP8 inputs with per-block scale factors (the FP8
 * support with block-wise scaling of "FlashAttention hardware-aware analysis"
 * (huaweicloud), section four, part 3).
 *   q8, k8, v8 : [B][H][N][d] E4M3 bytes (1 sign, 4 exponent bits with bias 7, 3
 *                mantissa bits; no infinities, S.1111.111 is NaN; largest 448),
 *                16-byte aligned.
 *   q_scale, k_scale, v_scale : float32 [B][H][ceil(N/128)], 4-byte aligned: the
 *                scale of each block of 128 consecutive rows of one head.  The value
 *                an input stands for is X[b,h,n,:] = e4m3(X8[b,h,n,:]) *
 *                x_scale[b,h,n/128].  Scales must be finite and > 0 (else the output
 *                is unspecified; nothing faults).
 *   o, lse     : as for attn_fwd, with o in the 16-bit type out_dt: the attention of
 *                the dequantised Q, K, V and its natural-log logsumexp.
 * d must be 128 (else ATTN_ERR_UNSUPPORTED).  Both products run on the tensor cores'
 * 8-bit path: S = Q8 K8^T exactly (times the two block scales and `scale`), and P V
 * with P rounded to E4M3 after V's block scale is folded into it.  Accuracy: the
 * logsumexp as attn_fwd's; each output element differs from the exact attention of the
 * dequantised inputs by at most 2^-4 times the attention of |V| (the E4M3 rounding of
 * P), plus 2^-8 |O| (rounding to out_dt), plus the flush of probabilities below 2^-12
 * of the row's largest term.  Other conventions (causal, scale, dev_status, errors,
 * overlap rules) are as for attn_fwd.
 */
ATTN_API attn_status attn_fwd_fp8(const void *q8, const void *k8, const void *v8, const float *q_scale,
                         const float *k_scale, const float *v_scale, void *o, float *lse,
                         int B, int H, int N, int d, attn_dtype out_dt, int causal, float scale,
                         int *dev_status, void *stream);

/*
 * attn_bwd_workspace_bytes -- size of the device workspace attn_bwd and its variants
 * need: two float32 values per row (D_i = rowsum(dO_i * O_i), and the logsumexp in base
 * 2) and, for d in {64, 128}, the float32 dQ accumulator of the fused pass (d values per
 * row), rows padded to whole 128-row tiles: (2 + d) * B*H*ceil(N/128)*128 * 4 bytes
 * (d = 256: 2 * B*H*ceil(N/128)*128 * 4 bytes).  Returns 0 for invalid sizes.
 *
 * attn_bwd_deterministic_workspace_bytes -- the two per-row values only:
 * 2 * B*H*ceil(N/128)*128 * 4 bytes (attn_bwd_deterministic and the stage entry points
 * attn_bwd_prepare / attn_bwd_dkdv / attn_bwd_dq).
 */
ATTN_API size_t attn_bwd_workspace_bytes(int B, int H, int N, int d);
ATTN_API size_t attn_bwd_deterministic_workspace_bytes(int B, int H, int N, int d);

/*
 * attn_bwd -- backward pass: gradients of a loss L given dout = dL/dO.
 *   q, k, v, o, dout : [B][H][N][d] (o is the output of attn_fwd on q, k, v).
 *   lse              : [B][H][N] float32 from the same attn_fwd call.
 *   dq, dk, dv       : [B][H][N][d] outputs in dt:
 *                        dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
 *                        dQ = scale dS K,  dK = scale dS^T Q,
 *                      with D_i = rowsum(dO_i * O_i) and P recomputed from lse
 *                      ("Understanding FlashAttention, Part 2", section 2.4,
 *                      Figs 16-20).
 *   workspace        : device scratch of at least attn_bwd_workspace_bytes();
 *                      16-byte aligned; contents need not be initialised and
 *                      are clobbered.  The caller owns it.
 *   Outputs must not overlap inputs or each other.
 *   d in {64, 128}: two kernels, dK and dV over 128-key tiles and dQ over 128-query tiles
 *   (the second recomputes S and dP in its own tile order: seven N x N x d products per
 *   tile pair, no atomics, the same bytes on every call), launched as one grid.  With
 *   dropout drawn in the backward (attn_bwd_dropout and its variants other than
 *   attn_bwd_dropout_bits) the fused pass of attn_bwd_dkdvdq runs instead: one pass over each key tile's query tiles gives dK, dV and that tile's
 *   share of dQ from the same recomputed tiles (five products, the keep bits drawn once
 *   instead of twice), dQ summed over the key tiles in the workspace's float32
 *   accumulator by atomic reductions and then rounded to dt; the order of those
 *   additions varies, so that dQ may differ in its last bit between identical calls.
 *   Without dropout the two-kernel form measured faster on GB300 and is used.
 *   d = 256: the gradients come from three kernels (dV and dK, one 128-key tile per CTA
 *   each, and dQ, one 128-query tile per CTA), each streaming its operands in
 *   128-column halves: deterministic, the same gradients in more passes.
 */
ATTN_API attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o,
                     const void *dout, const float *lse, void *dq, void *dk, void *dv,
                     void *workspace, size_t workspace_bytes,
                     int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                     int *dev_status, void *stream);

/*
 * attn_bwd_deterministic -- the backward with a guarantee that its results are the same
 * bytes on every call, whatever path attn_bwd takes: dK and dV from one kernel over key
 * tiles, dQ from one over query tiles, no atomics.  Workspace:
 * attn_bwd_deterministic_workspace_bytes().  Everything else is as for attn_bwd.
 */
ATTN_API attn_status attn_bwd_deterministic(const void *q, const void *k, const void *v, const void *o,
                                   const void *dout, const float *lse, void *dq, void *dk, void *dv,
                                   void *workspace, size_t workspace_bytes,
                                   int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                                   int *dev_status, void *stream);

/*
 * The fused backward (d in {64, 128}) as two stages, run in order on one stream after
 * attn_bwd_prepare with a workspace of attn_bwd_workspace_bytes() (which then also
 * clears the dQ accumulator).  attn_bwd runs them for its dropout variants; they are
 * exported so that a caller can run or time the five-product pass without dropout too.
 *
 * attn_bwd_dkdvdq    -- dK and dV, and each key tile's share of dQ added to the
 *                       workspace's float32 accumulator; one 128-key tile per CTA.
 * attn_bwd_dq_finish -- dQ = scale * accumulator, rounded to dt.
 * Argument meanings, layouts and errors are those of attn_bwd; d = 256 returns
 * ATTN_ERR_UNSUPPORTED.
 */
ATTN_API attn_status attn_bwd_dkdvdq(const void *q, const void *k, const void *v, const void *dout,
                            void *workspace, size_t workspace_bytes, void *dk, void *dv,
                            int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                            int *dev_status, void *stream);
ATTN_API attn_status attn_bwd_dq_finish(const void *workspace, size_t workspace_bytes, void *dq,
                               int B, int H, int N, int d, attn_dtype dt, float scale, void *stream);

/*
 * attn_bwd_rect -- attn_bwd for attn_fwd_rect's shapes: q, o, dout, dq [B][H][Nq][d],
 * k, v, dk, dv [B][H][Nk][d], lse [B][H][Nq]; the workspace is
 * attn_bwd_workspace_bytes(B, H, Nq, d).  Causal masking and Nk >= Nq as in
 * attn_fwd_rect; d in {64, 128, 256}.  Everything else is as for attn_bwd.
 */
ATTN_API attn_status attn_bwd_rect(const void *q, const void *k, const void *v, const void *o,
                          const void *dout, const float *lse, void *dq, void *dk, void *dv,
                          void *workspace, size_t workspace_bytes,
                          int B, int H, int Nq, int Nk, int d, attn_dtype dt, int causal, float scale,
                          int *dev_status, void *stream);

/*
 * The three stages attn_bwd_deterministic runs, in order, on one stream.  They are
 * exported so that a caller can time them one by one or run the two independent
 * gradient stages on two streams once the preparation has finished.  Argument
 * meanings, layouts and errors are those of attn_bwd_deterministic (workspace of at
 * least attn_bwd_deterministic_workspace_bytes()).
 *
 * attn_bwd_prepare -- fills the workspace: D_i = rowsum(dO_i * O_i) (the
 *   softmax-Jacobian row term of "Understanding FlashAttention, Part 2",
 *   section 2.4, Fig 18) and the logsumexp in base 2, for every row; rows of
 *   the last partial 128-row tile get D = 0 and an infinite logsumexp.  When
 *   d is 64 or 128 and workspace_bytes >= attn_bwd_workspace_bytes(), it also
 *   clears the fused backward's dQ accumulator (the first of attn_bwd's stages).
 * attn_bwd_dkdv -- dK and dV, one 128-key tile per CTA (reads the workspace; at
 *   d = 256 two launches, dV then dK).  At d = 128 the environment variable
 *   ATTN_BWD_CTA_PAIR=1, read on every call, runs it on CTA pairs instead (two key
 *   tiles per pair of neighbouring SMs sharing each product, tcgen05 cta_group::2): the
 *   same bytes, measured slower on this GPU, so not the default.
 * attn_bwd_dq   -- dQ, one 128-query tile per CTA (reads the workspace).
 */
ATTN_API attn_status attn_bwd_prepare(const void *o, const void *dout, const float *lse,
                             void *workspace, size_t workspace_bytes,
                             int B, int H, int N, int d, attn_dtype dt, void *stream);
ATTN_API attn_status attn_bwd_dkdv(const void *q, const void *k, const void *v, const void *dout,
                          const void *workspace, size_t workspace_bytes, void *dk, void *dv,
                          int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                          int *dev_status, void *stream);
ATTN_API attn_status attn_bwd_dq(const void *q, const void *k, const void *v, const void *dout,
                        const void *workspace, size_t workspace_bytes, void *dq,
                        int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                        int *dev_status, void *stream);

/*
 * attn_bwd_noalloc -- attn_bwd for callers that cannot allocate device memory.
 * (The pages have no counterpart to this entry point; it exists for
 * integration, not for the method.)
 *
 * Some callers have no way to hand attn_bwd its workspace: a plugin whose host
 * framework owns every byte of device memory through its own allocator, an
 * engine that fixes its memory budget once at start-up, or a foreign-function
 * caller that reaches the GPU only through this C ABI and has no CUDA runtime
 * of its own to call cudaMalloc with.  This entry point takes the workspace
 * from a fixed array of ATTN_NOALLOC_SCRATCH_BYTES (8 MiB) in the library's own
 * device image instead; every GPU that loads the library holds that array
 * until the process exits.  The caller still passes every input and output.
 *
 *  - Arguments and layouts are those of attn_bwd without the workspace pair.  It
 *    runs the kernels of attn_bwd_deterministic, which need the smaller workspace,
 *    so its results equal attn_bwd_deterministic's byte for byte.
 *  - Limit: the workspace attn_bwd_deterministic would need,
 *    attn_bwd_deterministic_workspace_bytes(B, H, N, d) = 8 * B*H*ceil(N/128)*128
 *    bytes, must fit in the array, i.e. B*H*ceil(N/128)*128 <= 1048576 rows (for
 *    example 128 heads of N = 8192).  Larger sizes return ATTN_ERR_INVALID_ARG
 *    before anything is launched.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.  Every call
 *    looks up the array's device address on the current device
 *    (cudaGetSymbolAddress, a lookup that allocates nothing), so the address is
 *    right for whichever device is current and stays right after a
 *    cudaDeviceReset.  The first call on a device may load the library's device
 *    code; make it before any stream capture.
 *  - Every call shares the one array and it keeps the last call's contents;
 *    nothing needs clearing because the preparation stage rewrites every value
 *    the gradient stages read.  Calls that overlap on the GPU (on different
 *    streams, or from different host threads without ordering) race on the
 *    array and produce wrong gradients: order them.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
ATTN_API attn_status attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                             const void *dout, const float *lse, void *dq, void *dk, void *dv,
                             int B, int H, int N, int d, attn_dtype dt, int causal, float scale,
                             int *dev_status, void *stream);

/* attn_status_string -- a static, human-readable name for a status code. */
ATTN_API const char *attn_status_string(attn_status s);

/*
 * attn_selftest_bounded_wait -- exercises the library's bounded mbarrier wait
 * on the device: one tiny kernel waits on a barrier that nothing completes,
 * gives up after `limit_ns` nanoseconds (clamped to [1 us, 1 s]) and stores
 * ATTN_ERR_TIMEOUT into *dev_status (device int, must be non-null).  It
 * checks the failure-reporting path without faulting or hanging the GPU.
 */
ATTN_API attn_status attn_selftest_bounded_wait(int *dev_status, uint64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
