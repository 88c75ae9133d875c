/*
 * ds4a.h - C ABI of the GB300 fused multi-query attention forward used by the
 * DeepSeek V4 Flash layers of the ds4 engine.
 *
 * Sources of the operation (page titles and sections):
 *  [P1] "How DeepSeek V4 Flash Model Inference Works on Apple Silicon with
 *       Metal Backend": "KV-Cache Management on Metal Device Buffers" (K/V rows
 *       padded to a multiple of 32), "FlashAttention Kernel Architecture" (pad,
 *       block-scan and fused attention kernels; Q.K, softmax and V weighting in
 *       one dispatch), "Mask Handling and Block Skipping" (one status byte per
 *       block, fully masked blocks skipped), "Memory Layout and Zero-Copy Buffer
 *       Access" (raw byte buffers with host-computed byte strides).
 *  [P2] "DwarfStar 4 (DS4) - DeepSeek V4 Flash Inference Engine": "Fixed Model
 *       Shape" (64 query heads, 1 K/V head, head dim 512, 128-token sliding
 *       window), "Layer Compression" (raw-only layers, ratio-4 layers with a
 *       top-512 index list, ratio-128 layers), "GPU Backend Architecture"
 *       (raw / mixed / indexed mixed heads and prefill attention ops), "KV Cache
 *       Design" (raw ring rows, compressed rows pooled every 4 or 128 tokens),
 *       "Whole-Model Graph Execution" (2048-token prefill chunks, one-token
 *       decode).
 *
 * What every attention call computes, for each query token t at position
 * p = q_pos0 + t and each head h < 64:
 *
 *     o[t][h] = sum_j softmax_j( scale * q[t][h] . k_j + bias_j ) * v_j
 *
 * over the rows j the token may see:
 *   - raw row i (position raw_pos0 + i) when p - window + 1 <= raw_pos0 + i <= p;
 *   - structural mode: compressed row c when (c + 1) * ratio <= p + 1
 *     (its pooled span c*ratio .. (c+1)*ratio-1 has ended);
 *   - indexed mode: compressed row idx[t][k] for every list entry >= 0 (each
 *     entry counts once per occurrence);
 *   - dense-mask mode: every real row of the padded logical sequence whose
 *     mask entry is not -inf; the entry is bias_j (natural-log units).
 * bias_j = 0 outside dense-mask mode.  A token with no visible row gets o = 0
 * and lse = -inf.  lse[t][h] = log(sum_j exp(scale*q.k_j + bias_j)).
 *
 * Logical sequence (block numbering, dense masks):
 *     [ raw rows, padded to a multiple of 32 | compressed rows, padded to 32 ]
 * Pad rows are never visible.  Block b covers logical rows 32b .. 32b+31.
 *
 * Conventions shared by all calls
 *   - Head count H = 64 and head dim D = 512 are fixed.  Every tensor is fp16
 *     (IEEE binary16) unless stated.  All arithmetic after the fp16 loads is
 *     fp32; outputs are rounded to fp16 to nearest-even.
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  The
 *     library keeps no reference after the call returns and allocates no
 *     device memory.
 *   - A row of K or V is 512 contiguous fp16 (1024 bytes).  Row strides are in
 *     BYTES, must be >= 1024 and multiples of 16; base pointers must be
 *     16-byte aligned.  Q and O are [T][64][512]: heads contiguous (1024 bytes
 *     apart), token stride in bytes (>= 65536, multiple of 16).
 *   - K and V may alias (k == v), as in an engine that stores one KV row.
 *     When they alias in every segment that has rows, every row is read once
 *     and serves both Q.K and the V weighting (fp16 rows in prefill and
 *     decode; E4M3 rows and ds4a_attn_indexed read K and V as two arrays even
 *     when they alias, and so do calls where only one segment aliases).
 *   - Rows that a token cannot see must still hold finite values (pad rows
 *     written by ds4a_pad_kv are +0.0): an invisible row gets weight 0, and
 *     0 * inf or 0 * nan would poison the sum.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream).  Bad
 *     arguments are reported synchronously, before anything is launched.  A
 *     failed launch returns DS4A_ERR_CUDA.  Kernels never trap: every device
 *     wait is bounded, and a wait that runs out records an error word read by
 *     ds4a_device_status().
 *   - The calls hold no mutable host state and are safe to issue from several
 *     host threads on different streams.
 */
#ifndef DS4A_H
#define DS4A_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DS4A_HEADS 64
#define DS4A_HEAD_DIM 512
#define DS4A_BLOCK_ROWS 32
#define DS4A_ROW_BYTES 1024

/* A CUDA stream handle (cudaStream_t / CUstream). */
typedef struct CUstream_st *ds4a_stream_t;

typedef enum {
  DS4A_OK = 0,
  DS4A_ERR_INVALID_ARG = 1, /* an argument breaks the contract; nothing launched */
  DS4A_ERR_UNSUPPORTED = 2, /* valid request the library does not serve (e.g. no sm_103a device) */
  DS4A_ERR_WORKSPACE = 3,   /* workspace missing or smaller than ds4a_attn_decode_workspace_size() */
  DS4A_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (launch, tensor-map encode, ...) */
  DS4A_ERR_TIMEOUT = 5      /* a bounded device wait ran out (reported by ds4a_device_status) */
} ds4a_status;

/* Static message for a status code; never NULL. */
const char *ds4a_status_string(int status);

/* The CUDA call and error code behind the latest DS4A_ERR_CUDA returned on the
 * calling thread (e.g. "kernel launch: error 1 invalid argument"); "" when
 * there was none.  The string belongs to the library and stays valid until the
 * thread's next failing call. */
const char *ds4a_last_cuda_error(void);

/* Library version string, "ds4a 0.2 sm_103a".  The minor number changes
 * whenever a layout callers can see changes: 0.2 is the first version whose
 * decode workspace holds fp16 normalised partials with the merge weight
 * W_s = 2^(m_s - M) l_s (0.1 held fp32 unnormalised sums). */
const char *ds4a_version(void);

/*
 * Query geometry.  All positions are absolute token positions ([P2] "KV Cache
 * Design": raw rows are kept in logical order; compressed rows are numbered
 * from the start of the sequence).
 *   T        query tokens in this call (>= 0); token t is at q_pos0 + t.
 *   q_pos0   position of token 0 (>= 0).
 *   n_raw    raw rows passed (>= 0); raw row i is at position raw_pos0 + i.
 *   raw_pos0 position of raw row 0 (>= 0).
 *   n_comp   compressed rows passed (>= 0; 0 = none).
 *   ratio    pooling ratio of the compressed rows (>= 1 when n_comp > 0; the
 *            model uses 4 and 128).
 *   window   sliding-window length in positions, self included (>= 1; the
 *            model uses 128).
 *   scale    softmax scale applied to q.k (the model uses 1/sqrt(512)).
 */
typedef struct {
  int32_t T, q_pos0;
  int32_t n_raw, raw_pos0;
  int32_t n_comp, ratio;
  int32_t window;
  float scale;
} ds4a_layout;

/*
 * Operands of one attention call (device pointers, byte strides).
 *   q      fp16 [T][64][512]; token stride q_tok_stride.
 *   k_raw, v_raw   fp16 [n_raw][512]; row stride raw_row_stride.  May be NULL
 *          when n_raw == 0.
 *   k_comp, v_comp fp16 [n_comp][512]; row stride comp_row_stride.  May be NULL
 *          when n_comp == 0.
 *   o      fp16 [T][64][512] output; token stride o_tok_stride.  Must not
 *          overlap any input.
 *   lse    fp32 [T][64] output (natural log), or NULL.
 */
typedef struct {
  const void *q;
  int64_t q_tok_stride;
  const void *k_raw, *v_raw;
  int64_t raw_row_stride;
  const void *k_comp, *v_comp;
  int64_t comp_row_stride;
  void *o;
  int64_t o_tok_stride;
  float *lse;
} ds4a_tensors;

/*
 * ds4a_pad_kv - [P1] "KV-Cache Management on Metal Device Buffers" and
 * "FlashAttention Kernel Architecture" (the pad kernel): writes
 *     dst[i] = src[i]  for i <  n_rows,
 *     dst[i] = +0.0    for n_rows <= i < ceil(n_rows / 32) * 32,
 * row by row (512 fp16 per row).  dst must hold ceil(n_rows/32)*32 rows at
 * dst_row_stride.  In-place use (dst == src, equal strides) only writes the
 * zero tail.  Other overlaps are invalid.  n_rows == 0 is a no-op.
 */
ds4a_status ds4a_pad_kv(const void *src, int64_t src_row_stride, int32_t n_rows,
                        void *dst, int64_t dst_row_stride, ds4a_stream_t stream);

/*
 * ds4a_quantize_kv_fp8 - [P2] "GPU Backend Architecture" (DS4-specific FP8 KV
 * quantization) and "Whole-Model Graph Execution" (K/V rows are quantised to
 * FP8 before they are stored).  The pages do not define the format; this
 * library's reading: E4M3 codes (bias 7, no infinities, largest finite 448)
 * with one fp32 scale per row, scale = absmax/448 and
 * code = E4M3(x * (448/absmax)) (fp32 quotients and product, round to nearest
 * even, saturating); an all-zero row gets scale 0.  A row's value is
 * decode(code) * scale.  Exact (bit-for-bit) for the given rows.
 *   src         fp16 [n_rows][512], row stride src_row_stride bytes (>= 1024,
 *               multiple of 16), 16-byte aligned.
 *   dst_codes   uint8 [n_rows][512] out, row stride dst_row_stride bytes
 *               (>= 512, multiple of 16), 16-byte aligned.
 *   scales      fp32 [n_rows] out.
 */
ds4a_status ds4a_quantize_kv_fp8(const void *src, int64_t src_row_stride, int32_t n_rows, void *dst_codes,
                                 int64_t dst_row_stride, float *scales, ds4a_stream_t stream);

/* Number of 32-row blocks of the padded logical sequence of L
 * (ceil(n_raw/32) + ceil(n_comp/32)), or -1 if L is NULL. */
int32_t ds4a_block_count(const ds4a_layout *L);

/*
 * ds4a_block_mask - [P1] "Mask Handling and Block Skipping" (the block-scan
 * kernel): one status byte per (q-tile of q_tile consecutive tokens, 32-row
 * block of the logical sequence), row-major [ceil(T/q_tile)][block_count]:
 *     0 = no (token, row) pair of the tile and block is visible (skippable),
 *     2 = every pair is visible with zero bias,
 *     1 = otherwise.
 * dense_mask == NULL: the structural rule (window + pooled compressed rows).
 * Otherwise dense_mask is fp16 [T][block_count*32] at mask_row_stride bytes
 * (>= block_count*64, multiple of 16); a pair is visible iff its entry is not
 * -inf and the row is real; "zero bias" means the entry is +0.0 or -0.0.
 * q_tile >= 1.  The result is exact (integer work).
 */
ds4a_status ds4a_block_mask(const ds4a_layout *L, const void *dense_mask, int64_t mask_row_stride,
                            int32_t q_tile, uint8_t *status, ds4a_stream_t stream);

/*
 * ds4a_attn_prefill - [P1] "FlashAttention Kernel Architecture" (the fused
 * attention kernel) with [P2] "GPU Backend Architecture" (raw heads, mixed
 * heads, flash attention prefill) and "Whole-Model Graph Execution"
 * (2048-token prefill chunks).  One pass per query token over its visible
 * rows; the output is normalised in the same kernel.
 *   dense_mask / mask_row_stride: NULL for the structural rule, else as in
 *          ds4a_block_mask (the mask replaces the structural rule).
 *   status / q_tile: optional block-status bytes as written by
 *          ds4a_block_mask for the same layout, mask and q_tile.  With a
 *          dense mask, blocks marked 0 are skipped and mask entries of blocks
 *          marked 2 are not read.  Without a mask the kernel derives the same
 *          skips from the layout (it never reads a row of a block marked 0), so
 *          status is not needed and, if given, must agree with the layout.
 * Any T >= 0 is accepted.
 */
ds4a_status ds4a_attn_prefill(const ds4a_layout *L, const ds4a_tensors *X,
                              const void *dense_mask, int64_t mask_row_stride,
                              const uint8_t *status, int32_t q_tile, ds4a_stream_t stream);

/*
 * ds4a_attn_decode - the same result as ds4a_attn_prefill for few query
 * tokens and many rows ([P2] "Whole-Model Graph Execution": decode processes
 * single tokens): each token's visible rows are split into n_splits ranges
 * processed by different SMs, and a second kernel merges the partial results
 * by their log-sum-exp.  Structural rule only (no dense mask).
 *   n_splits   ranges per token, >= 1, or <= 0 for the library's choice
 *              (ds4a_attn_decode_default_splits).
 *   workspace  device scratch of at least ds4a_attn_decode_workspace_size()
 *              bytes, 256-byte aligned, owned by the caller; it need not be
 *              initialised.  Every (m, l) pair is written by the call; the
 *              o_part slot of a split with no visible row is not, and the
 *              merge drops whatever that slot holds (bytes of an earlier
 *              call, or anything) by selecting on the split's zero weight.
 *              Two calls in flight at the same time must not share a
 *              workspace.
 */
int32_t ds4a_attn_decode_default_splits(const ds4a_layout *L);
size_t ds4a_attn_decode_workspace_size(const ds4a_layout *L, int32_t n_splits);
ds4a_status ds4a_attn_decode(const ds4a_layout *L, const ds4a_tensors *X, int32_t n_splits,
                             void *workspace, size_t workspace_bytes, ds4a_stream_t stream);

/*
 * ds4a_attn_decode_partials / ds4a_attn_decode_merge - the two halves of
 * ds4a_attn_decode, for callers that merge partial results themselves (for
 * instance across devices that each hold part of the compressed rows).
 * Workspace layout, with I = T * n_splits items (item = t * n_splits + s):
 *   fp16 o_part[I][64][512]    the split's own attention output
 *                              sum_j p_j v_j / l, rounded to fp16
 *   float2 ml[I][64]           (m, l): p_j = 2^(log2(e) * (scale q.k_j + bias_j) - m),
 *                              l = sum_j p_j; m = -inf and l = 0 for a split with
 *                              no visible row (its o_part slot is then not
 *                              written and may hold stale bytes; the merge
 *                              never uses it, since its weight is 0)
 * The merge computes o = sum_s W_s o_s / L with W_s = 2^(m_s - M) l_s,
 * L = sum_s W_s, M = max_s m_s, and lse = (M + log2 L) * ln 2.  decode_partials ignores X->o
 * and X->lse; decode_merge reads only the workspace and writes X->o / X->lse
 * (X->q and the K/V pointers are not used and may be NULL).
 */
ds4a_status ds4a_attn_decode_partials(const ds4a_layout *L, const ds4a_tensors *X, int32_t n_splits,
                                      void *workspace, size_t workspace_bytes, ds4a_stream_t stream);
ds4a_status ds4a_attn_decode_merge(const ds4a_layout *L, const ds4a_tensors *X, int32_t n_splits,
                                   const void *workspace, size_t workspace_bytes, ds4a_stream_t stream);

/*
 * ds4a_attn_decode_fp8 - ds4a_attn_decode with the compressed rows stored as
 * FP8 ([P2] "GPU Backend Architecture": DS4-specific FP8 KV quantization;
 * "Whole-Model Graph Execution": K/V rows quantised to FP8 before they are
 * stored), the format of ds4a_quantize_kv_fp8: E4M3 codes and one fp32 scale
 * per row.  The result is the attention over the rows' values
 * decode(code) * scale, within the usual fp16/fp32 tolerance; the compressed
 * rows cost half the bytes of fp16 rows.  Raw rows, Q and O are fp16 as in
 * ds4a_attn_decode.
 *   X->k_comp, X->v_comp  uint8 [n_comp][512] E4M3 codes at X->comp_row_stride
 *                         bytes (>= 512, multiple of 16), 16-byte aligned.
 *   k_comp_scale, v_comp_scale  fp32 [n_comp] row scales.
 *   n_splits, workspace   as for ds4a_attn_decode (same workspace size).
 * Equivalent to ds4a_attn_decode_fp8kv with fp16 raw rows (below).
 */
ds4a_status ds4a_attn_decode_fp8(const ds4a_layout *L, const ds4a_tensors *X, const float *k_comp_scale,
                                 const float *v_comp_scale, int32_t n_splits, void *workspace,
                                 size_t workspace_bytes, ds4a_stream_t stream);

/*
 * ds4a_attn_decode_fp8kv / ds4a_attn_prefill_fp8kv - decode (split-KV, as
 * ds4a_attn_decode) and structural prefill (as ds4a_attn_prefill without a
 * mask) over E4M3 rows, the raw rows included when their scales are given
 * ([P2] "Whole-Model Graph Execution": K/V rows are quantised to FP8 before
 * they are stored, raw rows as well as compressed ones; "GPU Backend
 * Architecture": DS4-specific FP8 KV quantization).  The format is that of
 * ds4a_quantize_kv_fp8; a row's value is decode(code) * scale and the result
 * is the attention over those values, within the usual fp16/fp32 tolerance.
 *   S->k_comp, S->v_comp  fp32 [n_comp] scales of the E4M3 compressed rows
 *                         X->k_comp / X->v_comp (uint8 [n_comp][512] at
 *                         X->comp_row_stride bytes: >= 512, multiple of 16).
 *   S->k_raw, S->v_raw    fp32 [n_raw] scales of E4M3 raw rows (X->k_raw /
 *                         X->v_raw then uint8 [n_raw][512] at X->raw_row_stride
 *                         bytes, >= 512, multiple of 16), or both NULL: the raw
 *                         rows are fp16 as in ds4a_attn_decode.
 *   n_splits, workspace   (decode) as for ds4a_attn_decode, same workspace size.
 * K and V are read as two arrays even when their pointers are equal.
 */
typedef struct {
  const float *k_raw, *v_raw;
  const float *k_comp, *v_comp;
} ds4a_fp8_scales;

ds4a_status ds4a_attn_decode_fp8kv(const ds4a_layout *L, const ds4a_tensors *X, const ds4a_fp8_scales *S,
                                   int32_t n_splits, void *workspace, size_t workspace_bytes, ds4a_stream_t stream);
ds4a_status ds4a_attn_prefill_fp8kv(const ds4a_layout *L, const ds4a_tensors *X, const ds4a_fp8_scales *S,
                                    ds4a_stream_t stream);

/*
 * ds4a_attn_prefill_fp8kv_ws - ds4a_attn_prefill_fp8kv with a workspace, same
 * operands and result.  When the raw rows are E4M3 (S->k_raw given), the call
 * has no compressed rows, window <= 128 and T >= 2, each raw row that some
 * query sees is decoded once into an fp16 row of the workspace, its values
 * decode(code) * scale rounded once to fp16, and the prefill runs over those
 * rows as ds4a_attn_prefill does (pairs of consecutive queries over one
 * 128-row tile).  Other calls ignore the workspace and run as
 * ds4a_attn_prefill_fp8kv.
 *   workspace  device memory, 256-byte aligned, at least
 *              ds4a_attn_prefill_fp8kv_workspace_size(L) bytes (may be NULL
 *              when that is 0); overwritten; must not overlap the operands.
 * Returns DS4A_ERR_WORKSPACE when the workspace is missing, short or
 * misaligned.
 */
size_t ds4a_attn_prefill_fp8kv_workspace_size(const ds4a_layout *L);
ds4a_status ds4a_attn_prefill_fp8kv_ws(const ds4a_layout *L, const ds4a_tensors *X, const ds4a_fp8_scales *S,
                                       void *workspace, size_t workspace_bytes, ds4a_stream_t stream);

/*
 * ds4a_attn_decode_batch - one decode step for n_seq independent sequences in
 * one launch (the pages' "serving many requests in parallel", page 4): each
 * sequence has one query token, its own position and row counts, and its own
 * K/V rows.  Sequence b's results equal ds4a_attn_decode on its own layout.
 *   shape      ratio, window and scale shared by the batch (other fields are
 *              ignored).
 *   seq_geom   device int32 [n_seq][4], 16-byte aligned: per sequence
 *              (q_pos, n_raw, raw_pos0, n_comp) with the meaning of the
 *              ds4a_layout fields; the row counts are clamped to raw_rows and
 *              comp_rows.  Read on the device (not validated on the host).
 *   X          batch tensors: sequence b's K/V row i at base + b*seq_stride +
 *              i*row_stride (bytes); Q and O fp16 [n_seq][64][512] at their
 *              sequence strides; lse fp32 [n_seq][64] or NULL.
 *   n_splits   row ranges per sequence (<= 0: the library's choice);
 *              workspace as in ds4a_attn_decode, of at least
 *              ds4a_attn_decode_batch_workspace_size() bytes.
 */
typedef struct {
  const void *q;       /* fp16 [n_seq][64][512] */
  int64_t q_seq_stride;
  const void *k_raw, *v_raw;
  int64_t raw_row_stride, raw_seq_stride;
  int32_t raw_rows;    /* rows each sequence's raw K/V tensors hold */
  const void *k_comp, *v_comp;
  int64_t comp_row_stride, comp_seq_stride;
  int32_t comp_rows;
  void *o;             /* fp16 [n_seq][64][512] */
  int64_t o_seq_stride;
  float *lse;
} ds4a_batch_tensors;

int32_t ds4a_attn_decode_batch_default_splits(int32_t n_seq, const ds4a_layout *shape, int32_t raw_rows,
                                              int32_t comp_rows);
size_t ds4a_attn_decode_batch_workspace_size(int32_t n_seq, int32_t n_splits);
ds4a_status ds4a_attn_decode_batch(int32_t n_seq, const ds4a_layout *shape, const int32_t *seq_geom,
                                   const ds4a_batch_tensors *X, int32_t n_splits, void *workspace,
                                   size_t workspace_bytes, ds4a_stream_t stream);

/*
 * ds4a_attn_decode_noalloc - ds4a_attn_decode for callers that cannot
 * allocate device memory: code living inside a host framework whose memory
 * pool owns the device, or a serving loop that forbids allocations once it is
 * running, has no way to hand this library a workspace.  The pages have no
 * counterpart of this call; it exists for those callers.
 *   The split-KV partials go to an 8 MiB array inside the library (a
 *   file-scope device array that every device loading the library holds until
 *   the process exits), so T * n_splits * 66048 bytes must fit in 8 MiB
 *   (T * n_splits <= 127).  n_splits <= 0 picks the usual split count, capped to
 *   fit; a T or n_splits that cannot fit returns DS4A_ERR_WORKSPACE before any
 *   launch.  Nothing is allocated: no cudaMalloc, no cudaFree.
 *   The array needs no clearing.  A call writes every (m, l) pair it reads;
 *   the o_part slot of a split with no visible row keeps whatever an earlier
 *   call left there, and the merge drops it by selecting on that split's zero
 *   weight.  All calls share the one array, so calls whose kernels overlap on
 *   the GPU (different streams, or different host threads) race on it and
 *   must be serialised by the caller.
 *   The first call of the library on a device (any entry point) looks up the
 *   array's device address; make that first call before any stream capture.
 */
ds4a_status ds4a_attn_decode_noalloc(const ds4a_layout *L, const ds4a_tensors *X, int32_t n_splits,
                                     ds4a_stream_t stream);

/*
 * ds4a_attn_indexed - [P2] "Layer Compression" (ratio-4 layers: an indexer
 * selects the top-512 compressed rows) and "GPU Backend Architecture"
 * (indexed mixed heads): each token sees its raw window rows plus the
 * compressed rows its own index list names.
 *   idx        int32 [T][top_k] at idx_row_stride bytes (>= 4*top_k, multiple
 *              of 16).  Entries < 0 are empty slots; entries >= n_comp are
 *              treated as empty.  Order does not matter.  The entries are not
 *              checked against the causal rule: the caller's indexer owns that.
 *   top_k      list length, 1 .. 4096 (the model uses 512).
 */
ds4a_status ds4a_attn_indexed(const ds4a_layout *L, const ds4a_tensors *X,
                              const int32_t *idx, int64_t idx_row_stride, int32_t top_k,
                              ds4a_stream_t stream);

/*
 * ds4a_attn_indexed_fp8kv - ds4a_attn_indexed over E4M3 rows: the compressed
 * rows the lists name are E4M3 codes with per-row scales (required), the raw
 * rows too when their scales are given ([P2] "Layer Compression": top-512
 * lists on the ratio-4 layers; "Whole-Model Graph Execution": K/V rows are
 * quantised to FP8 before they are stored).  Operands as for
 * ds4a_attn_prefill_fp8kv (X->k_comp / X->v_comp uint8 [n_comp][512] codes,
 * S->k_comp / S->v_comp their fp32 scales; S->k_raw / S->v_raw both given or
 * both NULL), lists as for ds4a_attn_indexed.  A listed row's value is
 * decode(code) * scale of that row.
 */
ds4a_status ds4a_attn_indexed_fp8kv(const ds4a_layout *L, const ds4a_tensors *X, const ds4a_fp8_scales *S,
                                   const int32_t *idx, int64_t idx_row_stride, int32_t top_k, ds4a_stream_t stream);

/*
 * ds4a_indexer_scores - [P2] "Layer Compression" (on ratio-4 layers a learned
 * indexer selects the top-512 compressed rows for each query) and "GPU
 * Backend Architecture" (indexer scoring among the GPU ops).  The pages give
 * no score formula; this library's reading is
 *     s[t][c] = sum_h w[t][h] * f(scale * q[t][h][:] . k[c][:]),
 * with f = max(0, x) when relu != 0 and the identity otherwise, for every
 * compressed row c whose pooled span has ended, (c+1)*ratio <= q_pos0+t+1;
 * every other row of the token gets -inf.  One head, w = 1 and relu = 0 is the
 * plain dot product.  fp16 inputs, fp32 accumulation (tensor cores).
 *   L             T, q_pos0, n_comp and ratio are used (the layer's attention
 *                 layout); T = 0 or n_comp = 0 does nothing.
 *   q_idx         fp16 [T][n_heads][head_dim], heads contiguous, token stride
 *                 q_tok_stride bytes (multiple of 16, >= 2*n_heads*head_dim).
 *   n_heads       1, 2, 4, 8, 16, 32, 64 or 128.   head_dim: 64, 128 or 256.
 *   k_idx         fp16 [n_comp][head_dim], row stride k_row_stride bytes
 *                 (multiple of 16, >= 2*head_dim): the indexer's own
 *                 compressed rows ([P2] "KV Cache Design": index_comp_kv),
 *                 not the attention's.
 *   head_weights  fp32 [T][n_heads], contiguous.
 *   scale         finite.
 *   scores        fp32 [T][n_comp] out, row stride score_row_stride bytes
 *                 (multiple of 16, >= 4*n_comp).
 * Device pointers owned by the caller, 16-byte aligned (head_weights 4-byte).
 */
ds4a_status ds4a_indexer_scores(const ds4a_layout *L, const void *q_idx, int64_t q_tok_stride, int32_t n_heads,
                                int32_t head_dim, const void *k_idx, int64_t k_row_stride,
                                const float *head_weights, float scale, int32_t relu, float *scores,
                                int64_t score_row_stride, ds4a_stream_t stream);

/*
 * ds4a_indexer_topk - the selection half of the indexer ([P2] "Layer
 * Compression": the top-512 compressed rows; "GPU Backend Architecture":
 * indexer top-k).  For each token, the top_k candidate rows (as above) with
 * the largest scores; equal scores go to the lower row; a NaN score counts as
 * -inf.  The chosen rows are written in ascending order, then -1 when a token
 * has fewer than top_k candidates: the index lists ds4a_attn_indexed takes.
 * The result is exact (integer work) for the scores given.
 *   scores   fp32 [T][>= n_comp] at score_row_stride bytes (multiple of 4,
 *            >= 4*n_comp); only the candidates of each token are read.
 *   top_k    1 .. 4096.
 *   idx      int32 [T][top_k] out at idx_row_stride bytes (multiple of 16,
 *            >= 4*top_k).
 */
ds4a_status ds4a_indexer_topk(const ds4a_layout *L, const float *scores, int64_t score_row_stride, int32_t top_k,
                              int32_t *idx, int64_t idx_row_stride, ds4a_stream_t stream);

/*
 * ds4a_compress_append - the compressor ([P2] "Layer Compression": a rolling
 * K/V and score state, a pooled row appended at each ratio boundary; "KV Cache
 * Design": attn_state_kv / attn_state_score; "GPU Backend Architecture":
 * compressor update, prefill and replay).  One call covers all three: it
 * appends n_new positions (one token in decode, a chunk in prefill, stored
 * rows after a restore) to a state that holds the n_state positions of the
 * span in progress.  The pages give no pooling formula; this library's
 * reading: each position brings a row kv[i] and a score row s[i] of the same
 * width, and a completed span of `ratio` positions becomes one row
 *     row[d] = sum_i exp(s[i][d] - m[d]) * kv[i][d] / sum_i exp(s[i][d] - m[d]),
 * m[d] = max_i s[i][d], a softmax over the span taken per dimension.  With
 * N = n_state + n_new, the call writes n_out = N / ratio pooled rows (span 0
 * starts with the state's rows) and leaves the last N % ratio positions, in
 * order, in the state's rows 0 .. (N % ratio) - 1.  The learned initial states
 * of ratio-4 layers are not modelled: a fresh state has n_state = 0.
 * fp32 loads and arithmetic; pooled rows are rounded to fp16.
 *   width        elements per row, a multiple of 4, 4 .. 65536.
 *   ratio        span length, 1 .. 65536.   n_state: 0 .. ratio - 1.
 *   kv, score    fp32 [n_new][width] at new_row_stride bytes; scores finite.
 *   state_kv, state_score
 *                fp32 [ratio - 1][width] at state_row_stride bytes, read and
 *                updated in place (unused, may be NULL, when ratio == 1).
 *   out          fp16 [n_out][width] at out_row_stride bytes: the pooled rows,
 *                for instance the next free rows of the compressed K or V
 *                rows.  May be NULL when n_out == 0.
 * Strides are at least one row and multiples of 16 bytes (of 8 bytes for the
 * output); pointers are device pointers owned by the caller, 16-byte aligned.  kv and score may be the
 * same rows; otherwise no two of the ranges (new rows, the two state tensors,
 * the output) may overlap (DS4A_ERR_INVALID_ARG).  n_new == 0 does nothing.
 * ds4a_compress_rows returns n_out for the arguments (-1 if they are invalid).
 */
int32_t ds4a_compress_rows(int32_t n_state, int32_t n_new, int32_t ratio);
ds4a_status ds4a_compress_append(int32_t width, int32_t ratio, int32_t n_state, const float *kv, const float *score,
                                 int64_t new_row_stride, int32_t n_new, float *state_kv, float *state_score,
                                 int64_t state_row_stride, void *out, int64_t out_row_stride, ds4a_stream_t stream);

/*
 * ds4a_device_status - synchronises `stream`, then reports the device error
 * word the kernels set when a bounded wait runs out (DS4A_ERR_TIMEOUT) or
 * DS4A_OK.  clear != 0 resets the word.  A CUDA error from the
 * synchronisation is DS4A_ERR_CUDA.
 */
ds4a_status ds4a_device_status(ds4a_stream_t stream, int clear);

/*
 * ds4a_device_error_word - like ds4a_device_status, but returns the raw error
 * word in *word (0 = no error).  For a wait that ran out the word is
 * 0x01000000 | site, where site names the barrier that was waited on.
 * Attention kernel: 1 Q buffer free, 2 K/V stage free, 3 Q loaded, 4 S buffer
 * free, 5 K/V stage loaded, 6 P written, 7 O read, 8 S computed, 9 P consumed,
 * 10 O complete, 11 draining copies, 12 self test.  Raw-prefill pair kernel:
 * 0x20 ring slot free, 0x21 ring slot loaded, 0x22 S buffer free, 0x23 S
 * computed, 0x24 P written, 0x26 O buffer drained, 0x27 O block complete,
 * 0x28 draining copies, 0x29 extra-row scores ready, 0x2A extra-row buffer or
 * Q box free, 0x2B row statistics ready, 0x2C row statistics read.  Indexer
 * scores: 0x40 q free, 0x41 k stage free, 0x42 q loaded, 0x43 accumulator
 * free, 0x44 k stage loaded, 0x45 accumulator complete, 0x46 draining.
 * clear != 0 resets the word.
 */
ds4a_status ds4a_device_error_word(ds4a_stream_t stream, uint32_t *word, int clear);

/*
 * ds4a_selftest_wait_timeout - diagnostic: launches one CTA that waits on a
 * barrier nothing ever completes, with the given bound (nanoseconds, 1e3 ..
 * 1e10).  The wait runs out, the kernel records DS4A_ERR_TIMEOUT in the
 * device error word and returns normally.  Used by the tests to show that a
 * stuck wait ends as a status, not a hang.
 */
ds4a_status ds4a_selftest_wait_timeout(uint64_t timeout_ns, ds4a_stream_t stream);

/*
 * ds4a_graph_begin / ds4a_graph_end / ds4a_graph_launch / ds4a_graph_destroy -
 * record the ds4a calls a thread makes on one stream and replay them as one
 * CUDA graph (a serving step issued as one launch instead of each call's host
 * work: argument checks, tensor maps, one launch per kernel; the counterpart
 * of the engine's one command-buffer chain per layer, [P2] "Whole-Model Graph
 * Execution").  Runtime plumbing: it computes nothing itself.
 *   ds4a_graph_begin(stream)   starts the recording.  stream must be a created
 *                              stream (NULL, the legacy default stream, is
 *                              rejected).  The first call on a device loads
 *                              every kernel of the library first: a kernel's
 *                              first launch loads its code, which a recording
 *                              does not allow.
 *   ds4a calls on stream       checked as usual; a call that returns an error
 *                              records nothing.  Their kernels are recorded,
 *                              not run.  Calls that read results back to the
 *                              host (ds4a_device_status, ds4a_device_error_word)
 *                              cannot be recorded.
 *   ds4a_graph_end(stream, &g) ends the recording (always) and instantiates
 *                              it into *g; DS4A_ERR_CUDA and *g = NULL when a
 *                              recorded launch failed.
 *   ds4a_graph_launch(g, s)    runs the recorded kernels on stream s with the
 *                              arguments they were recorded with: the same
 *                              buffers, sizes and layouts, whatever those
 *                              buffers hold then.  A recorded call's workspace
 *                              is reused by every launch, so launches that
 *                              share one must not overlap (one stream, or
 *                              events between streams).
 *   ds4a_graph_destroy(g)      frees the graph (NULL: no-op); launches already
 *                              issued complete, none may be issued after.
 */
typedef struct ds4a_graph_s *ds4a_graph;
ds4a_status ds4a_graph_begin(ds4a_stream_t stream);
ds4a_status ds4a_graph_end(ds4a_stream_t stream, ds4a_graph *graph);
ds4a_status ds4a_graph_launch(ds4a_graph graph, ds4a_stream_t stream);
void ds4a_graph_destroy(ds4a_graph graph);

#ifdef __cplusplus
}
#endif

#endif /* DS4A_H */
