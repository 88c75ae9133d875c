// Small kernels around the fused attention: K/V padding, block status,
// split-KV merge and the bounded-wait self test.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ds4a {

// ------------------------------------------------------------------ pad
// "How DeepSeek V4 Flash Model Inference Works on Apple Silicon with Metal
// Backend", sections "KV-Cache Management on Metal Device Buffers" and
// "FlashAttention Kernel Architecture" (the pad kernel): rows are copied and
// the block is completed with +0.0 rows up to a multiple of 32.  Each thread
// moves 16-byte chunks (64 per 1024-byte row), grid-stride, coalesced.

__global__ void pad_kernel(const uint8_t *__restrict__ src, long long src_stride, int n_rows,
                           uint8_t *__restrict__ dst, long long dst_stride, int first_row, int n_out) {
  const long long n_chunks = (long long)(n_out - first_row) * 64;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_chunks;
       i += (long long)gridDim.x * blockDim.x) {
    const int row = first_row + (int)(i >> 6);
    const int c = (int)(i & 63);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < n_rows) v = __ldg(reinterpret_cast<const uint4 *>(src + row * src_stride) + c);
    reinterpret_cast<uint4 *>(dst + row * dst_stride)[c] = v;
  }
}

cudaError_t launch_pad(const void *src, long long src_stride, int n_rows, void *dst, long long dst_stride,
                       int first_row, cudaStream_t s) {
  const int n_out = (n_rows + 31) / 32 * 32;
  const long long n_chunks = (long long)(n_out - first_row) * 64;
  if (n_chunks <= 0) return cudaSuccess;
  long long blocks = (n_chunks + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  pad_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const uint8_t *>(src), src_stride, n_rows,
                                         static_cast<uint8_t *>(dst), dst_stride, first_row, n_out);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ block status
// Same page, section "Mask Handling and Block Skipping": one byte per (q-tile,
// 32-row block): 0 = no visible pair, 2 = every pair visible with zero bias,
// 1 = otherwise.  Blocks number [raw rows padded to 32 | compressed rows padded
// to 32]; pad rows are never visible.

// Structural rule by interval arithmetic.  A raw row at position x is seen by
// positions x .. x+window-1; compressed row c by positions >= (c+1)*ratio - 1.
// The q-tile covers positions P0 .. P1.
__global__ void block_mask_struct_kernel(GeomScalars g, int q_tile, int n_qt, int nbr, int nbc,
                                         uint8_t *__restrict__ status) {
  const int n_blocks = nbr + nbc;
  const long long total = (long long)n_qt * n_blocks;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i / n_blocks);
    const int k = (int)(i - (long long)b * n_blocks);
    const long long P0 = (long long)g.q_pos0 + (long long)b * q_tile;
    const long long t_end = min((long long)g.T, (long long)(b + 1) * q_tile);
    const long long P1 = (long long)g.q_pos0 + t_end - 1;
    bool some, every;
    if (k < nbr) {
      const long long lo = 32LL * k, hi = min(32LL * k + 31, (long long)g.n_raw - 1);
      const long long x0 = g.raw_pos0 + lo, x1 = g.raw_pos0 + hi;
      some = x0 <= P1 && x1 + g.window - 1 >= P0;
      every = (hi - lo == 31) && x1 <= P0 && x0 + g.window - 1 >= P1;
    } else {
      const long long kc = k - nbr;
      const long long lo = 32LL * kc, hi = min(32LL * kc + 31, (long long)g.n_comp - 1);
      some = (lo + 1) * g.ratio - 1 <= P1;
      every = (hi - lo == 31) && (hi + 1) * g.ratio - 1 <= P0;
    }
    status[i] = every ? 2 : (some ? 1 : 0);
  }
}

// Dense mask: one warp per (q-tile, block); lane = row of the block.
__global__ void block_mask_dense_kernel(GeomScalars g, const __half *__restrict__ mask, long long mask_stride,
                                        int q_tile, int n_qt, int nbr, int nbc, uint8_t *__restrict__ status) {
  const int n_blocks = nbr + nbc;
  const long long total = (long long)n_qt * n_blocks;
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long i = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5); i < total; i += warps) {
    const int b = (int)(i / n_blocks);
    const int k = (int)(i - (long long)b * n_blocks);
    const bool real = k < nbr ? (32 * k + lane < g.n_raw) : (32 * (k - nbr) + lane < g.n_comp);
    const int col = 32 * k + lane;
    const int t0 = b * q_tile, t1 = min(g.T, (b + 1) * q_tile);
    bool any_vis = false, all_zero = real;
    if (real) {
      for (int t = t0; t < t1; ++t) {
        const __half hv = mask[(long long)t * mask_stride + col];
        const float m = __half2float(hv);
        const bool vis = m != -INFINITY;
        any_vis = any_vis || vis;
        all_zero = all_zero && vis && m == 0.f;
      }
    }
    const bool some = __any_sync(0xffffffffu, any_vis);
    const bool every = __all_sync(0xffffffffu, all_zero);
    if (lane == 0) status[i] = every ? 2 : (some ? 1 : 0);
  }
}

static int grid_for(long long work, int per_block) {
  long long b = (work + per_block - 1) / per_block;
  if (b < 1) b = 1;
  if (b > 152 * 8) b = 152 * 8;
  return (int)b;
}

cudaError_t launch_block_mask_struct(const GeomScalars &g, int q_tile, uint8_t *status, cudaStream_t s) {
  const int n_qt = (g.T + q_tile - 1) / q_tile;
  const int nbr = (g.n_raw + 31) / 32, nbc = (g.n_comp + 31) / 32;
  const long long total = (long long)n_qt * (nbr + nbc);
  if (total == 0) return cudaSuccess;
  block_mask_struct_kernel<<<grid_for(total, 256), 256, 0, s>>>(g, q_tile, n_qt, nbr, nbc, status);
  return cudaGetLastError();
}

cudaError_t launch_block_mask_dense(const GeomScalars &g, const __half *mask, long long mask_stride, int q_tile,
                                    uint8_t *status, cudaStream_t s) {
  const int n_qt = (g.T + q_tile - 1) / q_tile;
  const int nbr = (g.n_raw + 31) / 32, nbc = (g.n_comp + 31) / 32;
  const long long total = (long long)n_qt * (nbr + nbc);
  if (total == 0) return cudaSuccess;
  block_mask_dense_kernel<<<grid_for(total, 8), 256, 0, s>>>(g, mask, mask_stride, q_tile, n_qt, nbr, nbc,
                                                             status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ split merge
// Each split s of a token left its own normalised o_s (fp16) with its
// reference max m_s (log2 units) and row sum l_s.  With M = max_s m_s and the
// split weights W_s = 2^(m_s - M) l_s:
//   o = sum_s W_s o_s / L,  L = sum_s W_s,  lse = (M + log2 L) ln 2.
// One block per (token, head, half of the dims), 256 threads, one dim each.
// The split weights are computed once into shared memory; the partials are
// then streamed with eight independent loads in flight per thread.

constexpr int kCombineThreads = 256;
constexpr int kCombineMaxSplits = 4096;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float *red) {
  for (int o = 16; o > 0; o >>= 1) {
    const float x = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, x) : v + x;
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = l < kCombineThreads / 32 ? red[l] : (is_max ? -INFINITY : 0.f);
  for (int o = 4; o > 0; o >>= 1) {
    const float x = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, x) : v + x;
  }
  return __shfl_sync(0xffffffffu, v, 0);
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const __half *__restrict__ ws_o,
                                                                  const float2 *__restrict__ ws_ml, int n_splits,
                                                                  __half *__restrict__ o, long long o_tok_stride,
                                                                  float *__restrict__ lse) {
  __shared__ float w_s[kCombineMaxSplits];
  __shared__ float red[kCombineThreads / 32];
  grid_dependency_wait();  // the partials come from the previous kernel
  grid_launch_dependents();
  const int half = blockIdx.x, h = blockIdx.y, t = blockIdx.z;
  const long long base = (long long)t * n_splits;
  float mx = -INFINITY;
  for (int s = threadIdx.x; s < n_splits; s += kCombineThreads) mx = fmaxf(mx, ws_ml[(base + s) * 64 + h].x);
  const float M = block_reduce(mx, true, red);
  float lsum = 0.f;
  for (int s = threadIdx.x; s < n_splits; s += kCombineThreads) {
    const float2 ml = ws_ml[(base + s) * 64 + h];
    const float wgt = (ml.x == -INFINITY || M == -INFINITY) ? 0.f : exp2f(ml.x - M) * ml.y;
    w_s[s] = wgt;
    lsum += wgt;
  }
  const float L = block_reduce(lsum, false, red);  // also orders the w_s writes before the reads below
  const int d = 256 * half + threadIdx.x;
  const __half *src = ws_o + (base * 64 + h) * 512 + d;
  const long long step = 64LL * 512;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  int s = 0;
  // A split without visible rows left its o_part slot unwritten (stale bytes,
  // possibly NaN): its weight is 0 and the branch never reads the slot.
  for (; s + 8 <= n_splits; s += 8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float wgt = w_s[s + i];  // same for every thread: no divergence
      if (wgt != 0.f) acc[i] += wgt * __half2float(__ldg(src + (long long)(s + i) * step));
    }
  }
  for (; s < n_splits; ++s) {
    const float wgt = w_s[s];
    if (wgt != 0.f) acc[0] += wgt * __half2float(__ldg(src + (long long)s * step));
  }
  const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
  o[(long long)t * o_tok_stride + h * 512 + d] = __float2half_rn(L > 0.f ? sum / L : 0.f);
  if (lse != nullptr && half == 0 && threadIdx.x == 0)
    lse[(long long)t * 64 + h] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

// Many splits (a long decode): one block per (token, head, 64-dim chunk), 512
// blocks per token.  Thread (warp w, lane l) owns dims 8 (l & 7) .. +7 of the
// chunk (one 16-byte load per split) for the splits g, g + 32, g + 64, ... with
// g = 4 w + (l >> 3).  The loads of the first 256 splits are issued before the
// split weights are known, together with the (m, l) pairs, so that up to 256
// splits cost one round of memory latency; the per-thread sums are then added
// across the lanes of a dim group (shuffles) and across warps (shared memory).
constexpr int kWideChunks = 8;      // 64-dim chunks per head
constexpr int kWideMinSplits = 17;  // below this the one-dim-per-thread merge is as fast
constexpr int kWideGroups = kCombineThreads / 8;  // split groups: 8 threads of 16 bytes cover a chunk
constexpr int kWideLoads = 8;                     // loads in registers per thread and round
constexpr int kWideRound = kWideGroups * kWideLoads;

__device__ __forceinline__ void add_weighted(float (&acc)[8], const uint4 &v, float wgt) {
  const __half2 *h2 = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(h2[e]);
    // A split without visible rows left its o_part slot unwritten (stale bytes,
    // possibly NaN): its weight is 0 and the select (never a multiply, which
    // would turn 0 * NaN into NaN) drops it.
    acc[2 * e] += wgt != 0.f ? wgt * f.x : 0.f;
    acc[2 * e + 1] += wgt != 0.f ? wgt * f.y : 0.f;
  }
}

__global__ void __launch_bounds__(kCombineThreads) combine_wide_kernel(const __half *__restrict__ ws_o,
                                                                       const float2 *__restrict__ ws_ml,
                                                                       int n_splits, __half *__restrict__ o,
                                                                       long long o_tok_stride,
                                                                       float *__restrict__ lse) {
  __shared__ float w_s[kCombineMaxSplits];
  __shared__ float red[kCombineThreads / 32];
  __shared__ float part[kCombineThreads / 32][64];
  grid_dependency_wait();  // the partials come from the previous kernel
  grid_launch_dependents();
  const int chunk = blockIdx.x, h = blockIdx.y, t = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = 4 * warp + (lane >> 3), c8 = lane & 7;
  const long long base = (long long)t * n_splits;
  const __half *src = ws_o + (base * 64 + h) * 512 + 64 * chunk + 8 * c8;
  const long long step = 64LL * 512;
  uint4 x[kWideLoads];
#pragma unroll
  for (int k = 0; k < kWideLoads; ++k) {
    const int s = g + kWideGroups * k;
    x[k] = s < n_splits ? __ldg(reinterpret_cast<const uint4 *>(src + s * step)) : make_uint4(0u, 0u, 0u, 0u);
  }
  const float2 ml0 = tid < n_splits ? ws_ml[(base + tid) * 64 + h] : make_float2(-INFINITY, 0.f);
  float mx = ml0.x;
  for (int s = tid + kCombineThreads; s < n_splits; s += kCombineThreads)
    mx = fmaxf(mx, ws_ml[(base + s) * 64 + h].x);
  const float M = block_reduce(mx, true, red);
  float lsum = 0.f;
  if (tid < n_splits) {
    const float wgt = (ml0.x == -INFINITY || M == -INFINITY) ? 0.f : exp2f(ml0.x - M) * ml0.y;
    w_s[tid] = wgt;
    lsum = wgt;
  }
  for (int s = tid + kCombineThreads; s < n_splits; s += kCombineThreads) {
    const float2 ml = ws_ml[(base + s) * 64 + h];
    const float wgt = (ml.x == -INFINITY || M == -INFINITY) ? 0.f : exp2f(ml.x - M) * ml.y;
    w_s[s] = wgt;
    lsum += wgt;
  }
  const float L = block_reduce(lsum, false, red);  // also orders the w_s writes before the reads below
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
  for (int k = 0; k < kWideLoads; ++k) {
    const int s = g + kWideGroups * k;
    if (s < n_splits) add_weighted(acc, x[k], w_s[s]);
  }
  for (int r = kWideRound; r < n_splits; r += kWideRound) {
#pragma unroll
    for (int k = 0; k < kWideLoads; ++k) {
      const int s = r + g + kWideGroups * k;
      x[k] = s < n_splits ? __ldg(reinterpret_cast<const uint4 *>(src + s * step)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < kWideLoads; ++k) {
      const int s = r + g + kWideGroups * k;
      if (s < n_splits) add_weighted(acc, x[k], w_s[s]);
    }
  }
  // the four split groups of a warp hold the same dims in lanes l, l ^ 8, l ^ 16, l ^ 24
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 8);
    acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
  }
  if (lane < 8) {
#pragma unroll
    for (int e = 0; e < 8; ++e) part[warp][8 * c8 + e] = acc[e];
  }
  __syncthreads();
  if (tid < 32) {
    float2 sum = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kCombineThreads / 32; ++w) {
      sum.x += part[w][2 * tid];
      sum.y += part[w][2 * tid + 1];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    *reinterpret_cast<__half2 *>(o + (long long)t * o_tok_stride + h * 512 + 64 * chunk + 2 * tid) =
        __floats2half2_rn(sum.x * inv, sum.y * inv);
  }
  if (lse != nullptr && chunk == 0 && tid == 0)
    lse[(long long)t * 64 + h] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

// Few splits (a short decode): one block per (token, head), warp w owning dims
// 64w .. 64w+63 (a half2 per lane).  Each warp reads the (m, l) pairs (one per
// lane) and every partial value of its dims at once, and reduces with shuffles:
// one round of memory latency, no shared memory and no block barrier.
constexpr int kSmallMaxSplits = 8;

__global__ void __launch_bounds__(kCombineThreads) combine_small_kernel(const __half *__restrict__ ws_o,
                                                                        const float2 *__restrict__ ws_ml,
                                                                        int n_splits, __half *__restrict__ o,
                                                                        long long o_tok_stride,
                                                                        float *__restrict__ lse) {
  grid_dependency_wait();  // the partials come from the previous kernel
  grid_launch_dependents();
  const int h = blockIdx.x, t = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long base = (long long)t * n_splits;
  const int d = 64 * warp + 2 * lane;
  const __half *src = ws_o + (base * 64 + h) * 512 + d;
  const long long step = 64LL * 512;
  const float2 ml = lane < n_splits ? ws_ml[(base + lane) * 64 + h] : make_float2(-INFINITY, 0.f);
  float2 x[kSmallMaxSplits];
#pragma unroll
  for (int i = 0; i < kSmallMaxSplits; ++i)
    x[i] = i < n_splits ? __half22float2(__ldg(reinterpret_cast<const __half2 *>(src + (long long)i * step)))
                        : make_float2(0.f, 0.f);
  float M = ml.x;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float w = (ml.x == -INFINITY || M == -INFINITY) ? 0.f : exp2f(ml.x - M) * ml.y;
  float L = w;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  // A split without visible rows left its o_part slot unwritten (stale bytes,
  // possibly NaN): the value is loaded, but its weight is 0 and the select
  // (never a multiply, which would turn 0 * NaN into NaN) drops it.
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kSmallMaxSplits; ++i) {
    const float wi = __shfl_sync(0xffffffffu, w, i);
    if (i < n_splits) {
      acc.x += wi != 0.f ? wi * x[i].x : 0.f;
      acc.y += wi != 0.f ? wi * x[i].y : 0.f;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  *reinterpret_cast<__half2 *>(o + (long long)t * o_tok_stride + h * 512 + d) =
      __floats2half2_rn(acc.x * inv, acc.y * inv);
  if (lse != nullptr && threadIdx.x == 0)
    lse[(long long)t * 64 + h] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

cudaError_t launch_combine(const __half *ws_o, const float2 *ws_ml, int n_splits, int T, __half *o,
                           long long o_tok_stride, float *lse, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (n_splits > kCombineMaxSplits) return cudaErrorInvalidValue;
  // Programmatic dependent launch: the merge is scheduled while the partial
  // kernel runs and waits for it inside (griddepcontrol.wait).
  cudaLaunchConfig_t cfg = {};
  const bool wide = n_splits >= kWideMinSplits, small = n_splits <= kSmallMaxSplits;
  cfg.gridDim = small ? dim3(64, T, 1) : dim3(wide ? kWideChunks : 2, 64, T);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (small) return cudaLaunchKernelEx(&cfg, combine_small_kernel, ws_o, ws_ml, n_splits, o, o_tok_stride, lse);
  if (wide) return cudaLaunchKernelEx(&cfg, combine_wide_kernel, ws_o, ws_ml, n_splits, o, o_tok_stride, lse);
  return cudaLaunchKernelEx(&cfg, combine_kernel, ws_o, ws_ml, n_splits, o, o_tok_stride, lse);
}

// ------------------------------------------------------------------ self test
// One CTA waits on a barrier that nothing ever completes; the bounded wait runs
// out, records the timeout and the kernel returns.

__global__ void selftest_wait_kernel(unsigned long long timeout_ns, unsigned int *err) {
  __shared__ alignas(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, timeout_ns, err, SITE_SELFTEST);
  __syncthreads();
}

cudaError_t launch_selftest_wait(unsigned long long timeout_ns, unsigned int *err, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(timeout_ns, err);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ FP8 K/V rows

// Per-row E4M3 quantisation ("DwarfStar 4 (DS4) - DeepSeek V4 Flash Inference
// Engine", sections "GPU Backend Architecture" and "Whole-Model Graph
// Execution": K/V rows are quantised to FP8 before they are stored; the
// format is this library's reading): scale = absmax / 448 and
// code = E4M3(x * (448 / absmax)), quotients and product in fp32 with round to
// nearest even, the code rounded to nearest even and saturated; an all-zero
// row gets scale 0 and codes 0.  One warp per row, 16 values per lane.
__global__ void quantize_fp8_kernel(const uint8_t *__restrict__ src, long long src_stride, int n_rows,
                                    uint8_t *__restrict__ dst, long long dst_stride, float *__restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < n_rows; r += warps) {
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src + (long long)r * src_stride) + 2 * lane;
    const uint4 a = __ldg(s4), b = __ldg(s4 + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float x[16];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
    // non-negative floats order like their bit patterns
    const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
    uint32_t out[4] = {0u, 0u, 0u, 0u};
    if (amax > 0.f) {
      const float inv = __fdiv_rn(448.f, amax);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint16_t h;
        // upper byte <- second operand's element 2i+1, lower byte <- element 2i
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
            : "=h"(h)
            : "f"(__fmul_rn(x[2 * i + 1], inv)), "f"(__fmul_rn(x[2 * i], inv)));
        out[i >> 1] |= static_cast<uint32_t>(h) << (16 * (i & 1));
      }
    }
    reinterpret_cast<uint4 *>(dst + (long long)r * dst_stride)[lane] = make_uint4(out[0], out[1], out[2], out[3]);
    if (lane == 0) scales[r] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
  }
}

// ------------------------------------------------------------------ E4M3 rows -> fp16 row values
// Rows of K and V codes to their values decode(code) * scale rounded to fp16
// (decode(code) itself is exact in fp16; the product is rounded once, as an
// fp16 row of the same values would be), [n][512] each.  Thread i handles 16
// codes (one 16-byte load, two 16-byte stores), grid-stride over both arrays.
// The next kernel may start at once: it waits for this grid before its reads.

__global__ void widen_e4m3_rows_kernel(const uint8_t *__restrict__ kc, const uint8_t *__restrict__ vc,
                                       const float *__restrict__ ks, const float *__restrict__ vs, long long stride,
                                       int n_rows, __half *__restrict__ ko, __half *__restrict__ vo) {
  grid_launch_dependents();
  const long long per = (long long)n_rows * 32;  // 16-code chunks per array
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < 2 * per;
       i += (long long)gridDim.x * blockDim.x) {
    const bool is_v = i >= per;
    const long long j = is_v ? i - per : i;
    const int row = (int)(j >> 5), c = (int)(j & 31);
    const uint4 w = __ldg(reinterpret_cast<const uint4 *>((is_v ? vc : kc) + row * stride) + c);
    const float sc = __ldg((is_v ? vs : ks) + row);
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t d = e4m3x2_to_f16x2(static_cast<uint16_t>(k & 1 ? wd[k >> 1] >> 16 : wd[k >> 1] & 0xFFFFu));
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&d));
      const __half2 r = __floats2half2_rn(f.x * sc, f.y * sc);
      h[k] = *reinterpret_cast<const uint32_t *>(&r);
    }
    uint4 *dst = reinterpret_cast<uint4 *>((is_v ? vo : ko) + (long long)row * 512 + 16 * c);
    dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
    dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

cudaError_t launch_widen_e4m3_rows(const void *k_codes, const void *v_codes, const float *k_scale,
                                   const float *v_scale, long long stride, int n_rows, __half *k_out, __half *v_out,
                                   cudaStream_t s) {
  if (n_rows <= 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = ((long long)n_rows * 64 + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  widen_e4m3_rows_kernel<<<(unsigned)blocks, threads, 0, s>>>(static_cast<const uint8_t *>(k_codes),
                                                              static_cast<const uint8_t *>(v_codes), k_scale, v_scale,
                                                              stride, n_rows, k_out, v_out);
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(const void *src, long long src_stride, int n_rows, void *dst, long long dst_stride,
                                float *scales, cudaStream_t s) {
  const int threads = 256, rows_per_block = threads / 32;
  long long blocks = (n_rows + rows_per_block - 1) / rows_per_block;
  if (blocks > 65535) blocks = 65535;
  quantize_fp8_kernel<<<(unsigned)blocks, threads, 0, s>>>(static_cast<const uint8_t *>(src), src_stride, n_rows,
                                                          static_cast<uint8_t *>(dst), dst_stride, scales);
  return cudaGetLastError();
}

// Loads the code of every kernel listed (lazy module loading would otherwise
// do it at a kernel's first launch, which may fall inside a stream capture).
cudaError_t preload_aux_kernels() {
  const void *k[] = {(const void *)pad_kernel,          (const void *)block_mask_struct_kernel,
                     (const void *)block_mask_dense_kernel, (const void *)combine_kernel,
                     (const void *)combine_wide_kernel, (const void *)combine_small_kernel,
                     (const void *)selftest_wait_kernel, (const void *)quantize_fp8_kernel,
                     (const void *)widen_e4m3_rows_kernel};
  for (const void *f : k) {
    cudaFuncAttributes a;
    const cudaError_t e = cudaFuncGetAttributes(&a, f);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ds4a
