// Launchers shared between the kernel translation units and the C ABI.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "attn_params.h"
#include "indexer_params.h"

namespace ds4a {

struct GeomScalars {
  int T, q_pos0, n_raw, raw_pos0, n_comp, ratio, window;
};

// attn.cu
cudaError_t prepare_attn_kernel();
cudaError_t launch_attn(const AttnParams &p, int grid, cudaStream_t s);

// attn_pair.cu: pairs of consecutive tokens over raw rows (structural rule,
// no compressed rows, window <= 128).
struct PairParams {
  CUtensorMap tm_q2;          // 3-D {512, 64, T}, box {64, 64, 2}: both tokens of a pair, 128-byte swizzle
  CUtensorMap tm_k, tm_v;     // 2-D {512, n_raw}, box {64, 128}, 128-byte swizzle
  int T, q_pos0, n_raw, raw_pos0, window;
  float scale_log2;
  const uint8_t *k_raw, *v_raw;  // the row below a pair's tile is read directly
  long long raw_row_stride;      // bytes
  __half *o;
  long long o_tok_stride;        // elements
  int o_v8;                      // o and its token stride are 32-byte aligned: 32-byte stores
  float *lse;
  unsigned long long timeout_ns;
  unsigned int *err;
};
cudaError_t prepare_pair_kernel();
cudaError_t launch_pair(const PairParams &p, int grid, cudaStream_t s);

// aux.cu
cudaError_t launch_pad(const void *src, long long src_stride, int n_rows, void *dst, long long dst_stride,
                       int first_row, cudaStream_t s);
cudaError_t launch_block_mask_struct(const GeomScalars &g, int q_tile, uint8_t *status, cudaStream_t s);
cudaError_t launch_block_mask_dense(const GeomScalars &g, const __half *mask, long long mask_stride, int q_tile,
                                    uint8_t *status, cudaStream_t s);
cudaError_t launch_combine(const __half *ws_o, const float2 *ws_ml, int n_splits, int T, __half *o,
                           long long o_tok_stride, float *lse, cudaStream_t s);
cudaError_t launch_selftest_wait(unsigned long long timeout_ns, unsigned int *err, cudaStream_t s);
cudaError_t launch_widen_e4m3_rows(const void *k_codes, const void *v_codes, const float *k_scale,
                                   const float *v_scale, long long stride, int n_rows, __half *k_out, __half *v_out,
                                   cudaStream_t s);
cudaError_t preload_aux_kernels();
cudaError_t launch_quantize_fp8(const void *src, long long src_stride, int n_rows, void *dst, long long dst_stride,
                                float *scales, cudaStream_t s);

// indexer.cu
constexpr int kTopkMaxCachedKeys = 32768;  // candidate keys a top-k CTA keeps in shared memory
cudaError_t launch_indexer_topk(const TopkParams &p, int dyn_smem, cudaStream_t s);
cudaError_t launch_indexer_scores(const ScoreParams &p, int n_heads, int grid, cudaStream_t s);
cudaError_t preload_indexer_kernels();

// compressor.cu
// One append of n_new rows to a compressor state holding n_state rows
// (strides in elements).  n_out = (n_state + n_new) / ratio pooled rows are
// written; tail = (n_state + n_new) % ratio rows remain in the state.
struct CompressParams {
  const float *kv, *score;
  long long new_stride;
  float *state_kv, *state_score;
  long long state_stride;
  __half *out;
  long long out_stride;
  int width, ratio, n_state, n_new, n_out, tail;
  int splits;  // warps that share one span: 1, 2, 4 or 8
  int slots;   // row slots per warp: 1, 2 or 4 (a chunk is 128 / slots dimensions)
  int chunks;  // ceil(width / (128 / slots))
};
void compress_shape(int ratio, int *splits, int *slots);
cudaError_t launch_compress(const CompressParams &p, cudaStream_t s);
cudaError_t preload_compressor_kernels();

}  // namespace ds4a
