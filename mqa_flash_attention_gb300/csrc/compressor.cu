// Compressor: pooled K/V rows at ratio boundaries, with a rolling state.
//
// "DwarfStar 4 (DS4) - DeepSeek V4 Flash Inference Engine", sections "Layer
// Compression" (a rolling K/V and score state; a pooled row is appended each
// time a ratio span completes) and "KV Cache Design" (attn_state_kv and
// attn_state_score).  Every position brings a row kv[i] and a score row s[i] of
// the same width; a completed span of `ratio` positions becomes
//     row[d] = sum_i exp(s[i][d] - m[d]) kv[i][d] / sum_i exp(s[i][d] - m[d]),
// m[d] = the span's largest score of dimension d.  Positions of an incomplete
// span wait in the state (oldest first) for the next call.
//
// The work is HBM-bound (8 bytes read per element, 2 written per pooled
// element), so it runs on the CUDA cores.  A lane owns 4 dimensions (one
// float4) of a run of consecutive rows of one span, keeps a running (max,
// sum, weighted sum) per dimension, and loads up to eight rows before it folds
// them in.  The rows of a span are cut over up to 4 row slots of a warp (the
// slot's lanes read one contiguous 128..512-byte piece of a row) and up to 8
// warps of a block, so that a lane holds about four rows and all its loads are
// in flight at once; the parts merge through shuffles and shared memory.
#include <cuda_fp16.h>

#include "internal.h"

namespace ds4a {

constexpr int kCompWarps = 8;
constexpr int kCompBatch = 8;  // rows loaded before they are folded in

__device__ __forceinline__ float4 ldg4(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

struct RunSum {
  float m, l, a;  // largest score so far, sum of weights, weighted sum of rows
};

__device__ __forceinline__ void fold_batch(RunSum &r, const float *sc, const float *kv, int nb) {
  float bm = r.m;
  for (int j = 0; j < nb; ++j) bm = fmaxf(bm, sc[j]);
  const float f = expf(r.m - bm);  // 0 on the first batch (r.m = -inf)
  float l = r.l * f, a = r.a * f;
  for (int j = 0; j < nb; ++j) {
    const float e = expf(sc[j] - bm);
    l += e;
    a = fmaf(e, kv[j], a);
  }
  r = RunSum{bm, l, a};
}

// Combines two running sums of disjoint row sets (either may be empty).
__device__ __forceinline__ RunSum merge(RunSum x, RunSum y) {
  const float M = fmaxf(x.m, y.m);
  const float fx = x.m == -INFINITY ? 0.f : expf(x.m - M);
  const float fy = y.m == -INFINITY ? 0.f : expf(y.m - M);
  return RunSum{M, x.l * fx + y.l * fy, x.a * fx + y.a * fy};
}

// Work: (span c, chunk q of 128/R dimensions) pairs; each pair is cut into
// S*R parts of consecutive rows: S warps of the block, R row slots per warp
// (lane = slot * 32/R + g, g owning 4 dimensions).  A part keeps a running
// sum; parts merge through shuffles (slots) and shared memory (warps).
__global__ void __launch_bounds__(kCompWarps * 32) compress_pool_kernel(CompressParams p) {
  __shared__ float4 sh_m[kCompWarps][32], sh_l[kCompWarps][32], sh_a[kCompWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.splits, R = p.slots;
  const int G = 32 / R;  // lanes per row slot
  const int slot = lane / G, g = lane % G;
  const int s = warp & (S - 1);
  const long long pair = (long long)blockIdx.x * (kCompWarps / S) + warp / S;
  const bool active = pair < (long long)p.n_out * p.chunks;
  const int c = active ? (int)(pair / p.chunks) : 0;
  const int q = active ? (int)(pair % p.chunks) : 0;
  const int d = q * (128 / R) + g * 4;
  const bool on = active && d < p.width;

  RunSum r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) r[k] = RunSum{-INFINITY, 0.f, 0.f};
  const int parts = S * R, part = s * R + slot;
  const int rpp = (p.ratio + parts - 1) / parts;
  const int r0 = min(part * rpp, p.ratio), r1 = min(r0 + rpp, p.ratio);
  if (on) {
    for (int rb = r0; rb < r1; rb += kCompBatch) {
      const int nb = min(kCompBatch, r1 - rb);
      float4 kv4[kCompBatch], sc4[kCompBatch];
#pragma unroll
      for (int j = 0; j < kCompBatch; ++j) {
        if (j < nb) {
          const long long i = (long long)c * p.ratio + rb + j - p.n_state;  // row of the new input, < 0: state
          if (i < 0) {
            const long long o = (i + p.n_state) * p.state_stride + d;
            kv4[j] = ld4(p.state_kv + o);
            sc4[j] = ld4(p.state_score + o);
          } else {
            const long long o = i * p.new_stride + d;
            kv4[j] = ldg4(p.kv + o);
            sc4[j] = ldg4(p.score + o);
          }
        }
      }
      float kv[4][kCompBatch], sc[4][kCompBatch];
#pragma unroll
      for (int j = 0; j < kCompBatch; ++j) {
        kv[0][j] = kv4[j].x; kv[1][j] = kv4[j].y; kv[2][j] = kv4[j].z; kv[3][j] = kv4[j].w;
        sc[0][j] = sc4[j].x; sc[1][j] = sc4[j].y; sc[2][j] = sc4[j].z; sc[3][j] = sc4[j].w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) fold_batch(r[k], sc[k], kv[k], nb);
    }
  }
  // row slots of the warp -> slot 0 (every lane takes part: the shuffles are warp-wide)
  for (int off = G; off < 32; off <<= 1) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const RunSum o{__shfl_xor_sync(0xffffffffu, r[k].m, off), __shfl_xor_sync(0xffffffffu, r[k].l, off),
                     __shfl_xor_sync(0xffffffffu, r[k].a, off)};
      r[k] = merge(r[k], o);
    }
  }

  if (S > 1 && slot == 0) {
    sh_m[warp][g] = make_float4(r[0].m, r[1].m, r[2].m, r[3].m);
    sh_l[warp][g] = make_float4(r[0].l, r[1].l, r[2].l, r[3].l);
    sh_a[warp][g] = make_float4(r[0].a, r[1].a, r[2].a, r[3].a);
  }
  __syncthreads();  // every read of the state rows of this block is done
  const bool writer = s == 0 && slot == 0 && on;
  if (S > 1 && writer) {
    for (int t = 1; t < S; ++t) {
      const float4 mt = sh_m[warp + t][g], lt = sh_l[warp + t][g], at = sh_a[warp + t][g];
      r[0] = merge(r[0], RunSum{mt.x, lt.x, at.x});
      r[1] = merge(r[1], RunSum{mt.y, lt.y, at.y});
      r[2] = merge(r[2], RunSum{mt.z, lt.z, at.z});
      r[3] = merge(r[3], RunSum{mt.w, lt.w, at.w});
    }
  }
  if (writer) {
    const __half2 lo = __floats2half2_rn(r[0].a / r[0].l, r[1].a / r[1].l);
    const __half2 hi = __floats2half2_rn(r[2].a / r[2].l, r[3].a / r[3].l);
    uint2 v;
    v.x = *reinterpret_cast<const uint32_t *>(&lo);
    v.y = *reinterpret_cast<const uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p.out + (long long)c * p.out_stride + d) = v;
  }

  // The rows after the last complete span become the state.  They all come
  // from the new input (the first span used up the old state), and only the
  // block that read the old state's rows of these dimensions (span 0) writes
  // them, after the barrier above.
  if (c == 0 && on && p.tail > 0) {
    for (int t = part; t < p.tail; t += parts) {
      const long long src = (long long)(p.n_new - p.tail + t) * p.new_stride + d;
      const long long dst = (long long)t * p.state_stride + d;
      st4(p.state_kv + dst, ldg4(p.kv + src));
      st4(p.state_score + dst, ldg4(p.score + src));
    }
  }
}

// No span completes: the new rows join the state after its n_state rows.
__global__ void compress_append_kernel(CompressParams p) {
  const int per_row = p.width / 4;
  const long long total = (long long)p.n_new * per_row;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / per_row;
    const int d = (int)(i - row * per_row) * 4;
    const long long src = row * p.new_stride + d;
    const long long dst = (row + p.n_state) * p.state_stride + d;
    st4(p.state_kv + dst, ldg4(p.kv + src));
    st4(p.state_score + dst, ldg4(p.score + src));
  }
}

// About four rows per part (one round of loads), at most 32 parts: row
// slots first (narrower chunks, more blocks), then warps.
void compress_shape(int ratio, int *splits, int *slots) {
  int parts = 1;
  while (parts < 32 && parts * 4 < ratio) parts *= 2;
  *slots = parts < 4 ? parts : 4;
  *splits = parts / *slots;
}

cudaError_t launch_compress(const CompressParams &p, cudaStream_t st) {
  if (p.n_new == 0) return cudaSuccess;
  if (p.n_out == 0) {
    const long long total = (long long)p.n_new * (p.width / 4);
    long long blocks = (total + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    compress_append_kernel<<<(int)blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
  }
  const long long pairs = (long long)p.n_out * p.chunks;
  const int per_block = kCompWarps / p.splits;
  const long long blocks = (pairs + per_block - 1) / per_block;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  compress_pool_kernel<<<(int)blocks, kCompWarps * 32, 0, st>>>(p);
  return cudaGetLastError();
}

// Loads the code of every kernel listed (lazy module loading would otherwise
// do it at a kernel's first launch, which may fall inside a stream capture).
cudaError_t preload_compressor_kernels() {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, (const void *)compress_pool_kernel);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, (const void *)compress_append_kernel);
  return e;
}

}  // namespace ds4a
