// Constants, shared-memory bookkeeping and launch parameters of the fused
// attention kernel.  Included by the kernel's translation unit and by the host
// code that fills the parameters.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

namespace ds4a {

constexpr int kH = 64;
constexpr int kD = 512;
constexpr int kTile = 128;
// Warps 0-7: softmax + epilogue.  Warp w reads TMEM lane quarter (w % 4) and
// owns heads 32*(w / 4) .. +31 of those rows.  Warps 8-14: loaders (Q and
// every K/V stage: TMA tiles, or 16-byte cp.async gathers of index-listed
// rows).  Warp 15: TMEM allocator and MMA issuer.  Sixteen warps hold as many
// registers per thread (128) as thirteen, since one SM sub-partition holds
// four warps either way; the three extra loader warps raise the gather rate of
// indexed attention (334 -> 313 us for 2048 tokens) and, through one
// converter thread per row, the E4M3 decode (93.5 -> 83.5 us at 262,144 rows).
constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kLoaderWarp0 = 8;
constexpr int kLoaderWarps = 7;
constexpr int kLoaderThreads = 32 * kLoaderWarps;
constexpr int kMmaWarp = kLoaderWarp0 + kLoaderWarps;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kStages = 4;
constexpr uint32_t kQBytes = 65536;     // 8 boxes of [64 heads][64 dims] fp16
constexpr uint32_t kQBoxBytes = 8192;
constexpr uint32_t kBoxBytes = 16384;   // [128 rows][64 dims] fp16
constexpr uint32_t kStageBytes = 32768; // two boxes: 128 dims of a 128-row tile
constexpr uint32_t kPBytes = 16384;     // P^T [128 rows][64 heads] fp16
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kQBytes;
constexpr uint32_t kOffP = kOffKV + kStages * kStageBytes;
constexpr uint32_t kOffMisc = kOffP + kPBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 256;        // S^T buffers at columns 256 and 320
constexpr float kTau = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum Mode : int { MODE_STRUCT = 0, MODE_INDEXED = 1, MODE_MASK = 2 };

// Wait-site ids recorded with a timeout.
enum : unsigned int {
  SITE_Q_EMPTY = 1, SITE_KV_EMPTY, SITE_Q_FULL, SITE_S_EMPTY, SITE_KV_FULL, SITE_P_FULL, SITE_O_EMPTY,
  SITE_S_FULL, SITE_P_EMPTY, SITE_O_FULL, SITE_DRAIN, SITE_SELFTEST
};

struct Misc {
  alignas(16) float red[4][kH];   // per-warp partial max / sum of each head
  alignas(16) float m_use[kH];    // reference max used for P (log2 units)
  alignas(16) float alpha[kH];    // rescale factor of the previous reference
  alignas(16) float inv_l[kH];
  alignas(16) int idx_s[2][128];  // compressed rows of the gathered tiles, by tile parity
  alignas(8) uint64_t q_full, q_empty;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t code_full[kStages];    // E4M3 codes of a part landed (upper half of the stage)
  uint64_t s_full[2], s_empty[2];
  uint64_t o_full[4];              // O^T block m (dims 128m ..) final for the item
  uint64_t p_full, p_empty, o_empty, mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int resc_flag[2];
};
static_assert(offsetof(Misc, red) % 16 == 0 && offsetof(Misc, m_use) % 16 == 0 &&
                  offsetof(Misc, q_full) % 8 == 0,
              "shared-memory bookkeeping must stay aligned");

constexpr uint32_t kSmemBytes = kOffMisc + ((sizeof(Misc) + 127) / 128) * 128 + 1024;

struct AttnParams {
  CUtensorMap tm_q;        // 4-D {64, 64 heads, T, 8 dim blocks}, box {64, 64, 1, 8}
  CUtensorMap tm_k[2];     // [raw, comp] 3-D {64, rows, 8 dim blocks}, box {64, tile rows, 2}
                           // (batched decode: 3-D {512, rows, sequences}, box {64, 128, 1})
  CUtensorMap tm_v[2];
  CUtensorMap tm_kg, tm_vg;  // compressed rows, box {64, 1} (gather4)
  CUtensorMap tm_o;        // 3-D {512, 64, T}, box {128, 64, 1}, no swizzle (epilogue stores)
  CUtensorMap tm_k8[2], tm_v8[2];  // E4M3 rows [raw, comp]: bytes {512, rows}, box {128, 128}, no swizzle
  int T, q_pos0, n_raw, raw_pos0, n_comp, ratio, window;
  float scale_log2;
  int mode;
  int n_splits;            // row ranges per token
  int partial;             // 1: per-split outputs and (m, l) to the workspace
  int top_k;
  const void *k_comp, *v_comp;  // compressed rows (read directly by the gather warps)
  const float *k_scale[2], *v_scale[2];  // per-row scales of E4M3 rows [raw, comp]
  long long comp_row_stride;    // bytes
  const int32_t *idx;
  long long idx_stride;    // elements
  const __half *mask;
  long long mask_stride;   // elements
  const uint8_t *status;
  int q_tile, n_blocks, nbr;  // nbr = raw blocks (ceil(n_raw / 32))
  int comp_fp8;            // 1: compressed rows are E4M3 codes with per-row scales (k_scale[1], v_scale[1])
  int raw_fp8;             // 1: raw rows are E4M3 codes too (k_scale[0], v_scale[0])
  int alias_kv;            // 1: K and V are the same rows in every segment (each part loaded once)
  int kv_pair;             // 1: 64-row tiles, each stage holds the K and the V part of one 128-dim slice
  int tile_rows;           // rows per tile: 128, or 64 with kv_pair
  const int4 *batch_geom;  // batched decode: per sequence (q_pos, n_raw, raw_pos0, n_comp); "token" t = sequence t
  __half *o;
  long long o_tok_stride;  // elements
  float *lse;
  __half *ws_o;            // [T * n_splits][64][512]: the split's o = sum_j p_j v_j / l, fp16
  float2 *ws_ml;           // [T * n_splits][64] (m in log2 units, l)
  unsigned long long timeout_ns;
  unsigned int *err;       // device error word
  const uint8_t *q_ptr;    // Q [T][64][512] fp16 (copied with cp.async when TMA is left to K/V)
  long long q_tok_bytes;
};

}  // namespace ds4a
