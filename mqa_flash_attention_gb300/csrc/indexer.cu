// Indexer kernels: scores of compressed rows for each query token, and the
// top-k selection that produces the attention's index lists.
//
// Source: "DwarfStar 4 (DS4) - DeepSeek V4 Flash Inference Engine", section
// "Layer Compression" (ratio-4 layers: a learned indexer selects the top-512
// compressed rows per query) and section "GPU Backend Architecture" (indexer
// scoring and top-k among the GPU ops).  The pages give no score formula; the
// reading implemented is s[t,c] = sum_h w[t,h] * f(scale * q[t,h,:] . k[c,:]),
// f the identity or max(0, x), over the candidate rows (c+1)*ratio <= p_t+1.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "indexer_params.h"
#include "internal.h"
#include "ptx.cuh"

namespace ds4a {

__device__ __forceinline__ int n_candidates(const IndexerGeom &g, int t) {
  const long long c = ((long long)g.q_pos0 + t + 1) / g.ratio;
  return (int)(c < g.n_comp ? c : g.n_comp);
}

__device__ __forceinline__ void bar_sync_n(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------ top-k

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;

// Order-preserving key of a score: larger score -> larger key.  NaN counts
// as -inf and -0 as +0, so equal IEEE values have equal keys.
__device__ __forceinline__ uint32_t score_key(float x) {
  if (x != x) x = -INFINITY;
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One CTA per token.  Exact radix select (4 passes of 8 bits) finds the key K*
// of the top_k-th largest candidate and how many keys equal to K* are taken;
// a final pass in row order writes every row with key > K* and the first such
// rows with key == K* (lower index first), so the list comes out ascending.
__global__ void __launch_bounds__(kTopkThreads) indexer_topk_kernel(const TopkParams p) {
  extern __shared__ uint32_t keys_s[];
  __shared__ uint32_t hist[kTopkWarps][256];
  __shared__ uint32_t tot[256];
  __shared__ uint32_t sh_prefix, sh_need;
  __shared__ uint32_t cnt[2][kTopkWarps];
  const int t = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = n_candidates(p.g, t);
  const int K = p.top_k;
  int32_t *out = p.idx + (long long)t * p.idx_stride;
  const float *row = p.scores + (long long)t * p.score_stride;
  if (n <= K) {
    for (int i = tid; i < K; i += kTopkThreads) out[i] = i < n ? i : -1;
    return;
  }
  const bool cached = n <= p.cached_keys;
  if (cached) {
    for (int i = tid; i < n; i += kTopkThreads) keys_s[i] = score_key(__ldg(row + i));
  }
  uint32_t prefix = 0, need = (uint32_t)K;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const uint32_t hi_mask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int i = tid; i < kTopkWarps * 256; i += kTopkThreads) (&hist[0][0])[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kTopkThreads) {
      const uint32_t k = cached ? keys_s[i] : score_key(__ldg(row + i));
      if ((k & hi_mask) == prefix) atomicAdd(&hist[warp][(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t s = 0;
#pragma unroll
      for (int w = 0; w < kTopkWarps; ++w) s += hist[w][tid];
      tot[tid] = s;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255-8l .. 248-8l (descending); find the bin where
      // the count of larger keys reaches `need`.
      uint32_t s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) s += tot[255 - 8 * lane - j];
      uint32_t incl = s;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const uint32_t above = incl - s;
      if (above < need && need <= incl) {
        uint32_t acc = above;
        for (int j = 0; j < 8; ++j) {
          const int d = 255 - 8 * lane - j;
          const uint32_t c = tot[d];
          if (acc + c >= need) {
            sh_prefix = prefix | ((uint32_t)d << shift);
            sh_need = need - acc;
            break;
          }
          acc += c;
        }
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    need = sh_need;
  }
  // Selection in row order, 512 rows at a time, with ballot scans.
  const uint32_t kstar = prefix;
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t run_eq = 0, run_sel = 0;
  for (int base = 0; base < n && run_sel < (uint32_t)K; base += kTopkThreads) {
    const int i = base + tid;
    const uint32_t k = i < n ? (cached ? keys_s[i] : score_key(__ldg(row + i))) : 0u;
    const bool gt = i < n && k > kstar, eq = i < n && k == kstar;
    const uint32_t b_eq = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) cnt[0][warp] = __popc(b_eq);
    __syncthreads();
    uint32_t eq_before = run_eq + __popc(b_eq & lt_mask), eq_tile = 0;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) {
      const uint32_t c = cnt[0][w];
      eq_before += w < warp ? c : 0u;
      eq_tile += c;
    }
    const bool take = gt || (eq && eq_before < need);
    const uint32_t b_sel = __ballot_sync(0xffffffffu, take);
    if (lane == 0) cnt[1][warp] = __popc(b_sel);
    __syncthreads();
    uint32_t pos = run_sel + __popc(b_sel & lt_mask), sel_tile = 0;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) {
      const uint32_t c = cnt[1][w];
      pos += w < warp ? c : 0u;
      sel_tile += c;
    }
    if (take && pos < (uint32_t)K) out[pos] = i;
    run_eq += eq_tile;
    run_sel += sel_tile;
    __syncthreads();  // cnt is rewritten by the next tile
  }
}

cudaError_t launch_indexer_topk(const TopkParams &p, int dyn_smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(indexer_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem);
  if (e != cudaSuccess) return e;
  indexer_topk_kernel<<<p.g.T, kTopkThreads, dyn_smem, s>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ scores

// Tile: M = 128 compressed rows (A = k rows, K-major), N = 256 = tokens x
// heads of one token group (B = q, K-major), K = head_dim in 64-dim boxes.
// The group's q stays in shared memory for the item; k boxes stream through a
// 4-stage ring; the fp32 accumulator is double-buffered in TMEM (2 x 256
// columns) so the epilogue of one tile overlaps the MMAs of the next.
constexpr int kScoreEpiWarps = 8;
constexpr int kScoreEpiThreads = 32 * kScoreEpiWarps;
constexpr int kScoreLoaderWarp = kScoreEpiWarps;
constexpr int kScoreMmaWarp = kScoreEpiWarps + 1;
constexpr int kScoreThreads = 32 * (kScoreMmaWarp + 1);
constexpr int kScoreStages = 4;
constexpr uint32_t kScoreQBox = 32768;   // [256 (token, head) rows][64 dims] fp16
constexpr uint32_t kScoreKBox = 16384;   // [128 rows][64 dims] fp16
constexpr uint32_t kScoreOffQ = 0;       // up to 4 boxes (head_dim 256)
constexpr uint32_t kScoreOffK = 4 * kScoreQBox;
constexpr uint32_t kScoreOffMisc = kScoreOffK + kScoreStages * kScoreKBox;

struct ScoreMisc {
  alignas(16) float w_s[256];
  alignas(8) uint64_t q_full, q_empty;
  uint64_t k_full[kScoreStages], k_empty[kScoreStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr uint32_t kScoreSmemBytes = kScoreOffMisc + ((sizeof(ScoreMisc) + 127) / 128) * 128 + 1024;

enum : unsigned int {
  SITE_IX_Q_EMPTY = 0x40, SITE_IX_K_EMPTY, SITE_IX_Q_FULL, SITE_IX_ACC_EMPTY, SITE_IX_K_FULL, SITE_IX_ACC_FULL,
  SITE_IX_DRAIN
};

// Work item -> token group, row tiles [r0, r1) and the tiles [r0, r_mma) that
// hold at least one candidate of the group's last token.
struct ScoreItem {
  int g, t0, nt, r0, r1, r_mma;
};

__device__ __forceinline__ ScoreItem score_item(const ScoreParams &p, int item, int G) {
  ScoreItem it;
  it.g = item / p.items_per_group;
  const int part = item - it.g * p.items_per_group;
  it.t0 = it.g * G;
  it.nt = min(G, p.g.T - it.t0);
  it.r0 = part * p.tiles_per_item;
  it.r1 = min(it.r0 + p.tiles_per_item, p.n_row_tiles);
  const int last = n_candidates(p.g, it.t0 + it.nt - 1);
  it.r_mma = min(it.r1, (last + 127) / 128);
  if (it.r_mma < it.r0) it.r_mma = it.r0;
  return it;
}

template <int NH>
__global__ void __launch_bounds__(kScoreThreads, 1) indexer_scores_kernel(const __grid_constant__ ScoreParams p) {
  constexpr int G = 256 / NH;  // tokens per group
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  ScoreMisc &ms = *reinterpret_cast<ScoreMisc *>(smem + kScoreOffMisc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_kc = p.head_dim / 64;
  const int n_items = p.n_groups * p.items_per_group;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ms.q_full), 1);
    mbar_init(smem_u32(&ms.q_empty), 1);
    for (int s = 0; s < kScoreStages; ++s) {
      mbar_init(smem_u32(&ms.k_full[s]), 1);
      mbar_init(smem_u32(&ms.k_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ms.acc_full[b]), 1);
      mbar_init(smem_u32(&ms.acc_empty[b]), kScoreEpiThreads);
    }
    mbar_init(smem_u32(&ms.mma_done), 1);
    ms.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kScoreMmaWarp) {
    tmem_alloc(smem_u32(&ms.tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == kScoreLoaderWarp && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  grid_launch_dependents();
  grid_dependency_wait();
  volatile int *abrt = &ms.abort_flag;

  if (warp == kScoreLoaderWarp) {
    if (lane == 0) {
      bool ok = true;
      uint32_t nq = 0, st = 0, ph = 0, filled = 0, last_par = 0;
      bool q_issued = false;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const ScoreItem it = score_item(p, item, G);
        if (it.r_mma == it.r0) continue;
        ok = mbar_wait(smem_u32(&ms.q_empty), (nq & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_IX_Q_EMPTY);
        if (!ok) break;
        mbar_arrive_expect_tx(smem_u32(&ms.q_full), kScoreQBox * n_kc);
        for (int kc = 0; kc < n_kc; ++kc)
          tma_load_3d(sbase + kScoreOffQ + kc * kScoreQBox, &p.tm_q, smem_u32(&ms.q_full), 64 * kc, 0, it.t0);
        q_issued = true;
        ++nq;
        for (int r = it.r0; r < it.r_mma && ok; ++r) {
          for (int kc = 0; kc < n_kc; ++kc) {
            ok = mbar_wait(smem_u32(&ms.k_empty[st]), ph ^ 1, abrt, p.timeout_ns, p.err, SITE_IX_K_EMPTY);
            if (!ok) break;
            mbar_arrive_expect_tx(smem_u32(&ms.k_full[st]), kScoreKBox);
            tma_load_2d(sbase + kScoreOffK + st * kScoreKBox, &p.tm_k, smem_u32(&ms.k_full[st]), 64 * kc, 128 * r);
            filled |= 1u << st;
            last_par = (last_par & ~(1u << st)) | (ph << st);
            if (++st == kScoreStages) {
              st = 0;
              ph ^= 1;
            }
          }
        }
      }
      if (!ok) {
        // Let every copy already issued land before the shared memory goes away.
        volatile int never = 0;
        for (int s = 0; s < kScoreStages; ++s)
          if (filled & (1u << s))
            mbar_wait(smem_u32(&ms.k_full[s]), (last_par >> s) & 1, &never, 100000000ull, p.err, SITE_IX_DRAIN);
        if (q_issued) mbar_wait(smem_u32(&ms.q_full), (nq - 1) & 1, &never, 100000000ull, p.err, SITE_IX_DRAIN);
      }
    }
    __syncwarp();
  } else if (warp == kScoreMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_f16_f32(128, 256, false, false);
      const uint64_t k_desc = sdesc_sw128(sbase + kScoreOffK, 16, 1024);
      const uint64_t q_desc = sdesc_sw128(sbase + kScoreOffQ, 16, 1024);
      bool ok = true;
      uint32_t nq = 0, st = 0, ph = 0, tc = 0;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const ScoreItem it = score_item(p, item, G);
        if (it.r_mma == it.r0) continue;
        ok = mbar_wait(smem_u32(&ms.q_full), nq & 1, abrt, p.timeout_ns, p.err, SITE_IX_Q_FULL);
        if (!ok) break;
        for (int r = it.r0; r < it.r_mma && ok; ++r) {
          const uint32_t buf = tc & 1;
          ok = mbar_wait(smem_u32(&ms.acc_empty[buf]), ((tc >> 1) & 1) ^ 1, abrt, p.timeout_ns, p.err,
                         SITE_IX_ACC_EMPTY);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + 256 * buf;
          for (int kc = 0; kc < n_kc && ok; ++kc) {
            ok = mbar_wait(smem_u32(&ms.k_full[st]), ph, abrt, p.timeout_ns, p.err, SITE_IX_K_FULL);
            if (!ok) break;
            tc_fence_after();
            const uint64_t a0 = sdesc_add(k_desc, st * kScoreKBox);
            const uint64_t b0 = sdesc_add(q_desc, kc * kScoreQBox);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t a = sdesc_add(a0, ks * 32), b = sdesc_add(b0, ks * 32);
              if (ks == 0)
                umma_f16(d, a, b, kIdesc, kc != 0 ? 1u : 0u);
              else
                umma_f16_acc(d, a, b, kIdesc);
            }
            umma_commit(smem_u32(&ms.k_empty[st]));
            if (++st == kScoreStages) {
              st = 0;
              ph ^= 1;
            }
          }
          if (!ok) break;
          umma_commit(smem_u32(&ms.acc_full[buf]));
          ++tc;
        }
        if (!ok) break;
        umma_commit(smem_u32(&ms.q_empty));
        ++nq;
      }
      // Every MMA issued so far must finish before TMEM is released.
      umma_commit(smem_u32(&ms.mma_done));
      volatile int never = 0;
      mbar_wait(smem_u32(&ms.mma_done), 0, &never, 100000000ull, p.err, SITE_IX_DRAIN);
    }
    __syncwarp();
  } else {
    // Epilogue: thread (q, l) of warp w reads TMEM lane 32q + l (row c of the
    // tile) and the 128 columns of half hf = w / 4 (tokens G/2 * hf ..).
    const int tid = threadIdx.x;
    const int q = warp & 3, hf = warp >> 2;
    const int lrow = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    constexpr int HW = NH < 32 ? NH : 32;       // heads of one token inside a 32-column chunk
    constexpr int TPC = 32 / HW;                 // tokens per chunk
    constexpr int CPT = NH < 32 ? 1 : NH / 32;   // chunks per token
    const float scale = p.scale;
    const bool relu = p.relu != 0;
    uint32_t tc = 0;
    bool bad = false;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const ScoreItem it = score_item(p, item, G);
      bar_sync_n(1, kScoreEpiThreads);  // the previous item's epilogue is done with w_s
      {
        const int tl = tid / NH, h = tid % NH;
        ms.w_s[tid] = tl < it.nt ? __ldg(p.w + (long long)(it.t0 + tl) * NH + h) : 0.f;
      }
      bar_sync_n(1, kScoreEpiThreads);
      // Row c is a candidate of token t iff (c+1)*ratio <= q_pos0 + t + 1.
      const long long pos1 = (long long)p.g.q_pos0 + it.t0 + 1;
      for (int r = it.r0; r < it.r_mma; ++r) {
        const uint32_t buf = tc & 1;
        bad = bad || !mbar_wait(smem_u32(&ms.acc_full[buf]), (tc >> 1) & 1, abrt, p.timeout_ns, p.err,
                                SITE_IX_ACC_FULL);
        tc_fence_after();
        const int c = 128 * r + lrow;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float v[32];
          tmem_ld32(tmem + 256 * buf + 128 * hf + 32 * j + lane_base, v);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < TPC; ++u) {
            float s = 0.f;
#pragma unroll
            for (int h = 0; h < HW; ++h) {
              const float x = scale * v[u * HW + h];
              s += ms.w_s[128 * hf + 32 * j + u * HW + h] * (relu ? fmaxf(x, 0.f) : x);
            }
            if (NH >= 32) {
              acc += s;
              if ((j + 1) % CPT == 0) {
                const int tl = (128 * hf + 32 * j) / NH;  // token of this chunk
                if (tl < it.nt && c < p.g.n_comp)
                  p.scores[(long long)(it.t0 + tl) * p.score_stride + c] =
                      (long long)(c + 1) * p.g.ratio <= pos1 + tl ? acc : -INFINITY;
                acc = 0.f;
              }
            } else {
              const int tl = (128 * hf + 32 * j) / NH + u;
              if (tl < it.nt && c < p.g.n_comp)
                p.scores[(long long)(it.t0 + tl) * p.score_stride + c] =
                    (long long)(c + 1) * p.g.ratio <= pos1 + tl ? s : -INFINITY;
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&ms.acc_empty[buf]));
        ++tc;
      }
      // Tiles past the group's last candidate: no MMA, every score is -inf.
      for (int r = it.r_mma; r < it.r1; ++r) {
        const int c = 128 * r + lrow;
        if (c >= p.g.n_comp) continue;
#pragma unroll
        for (int u = 0; u < G / 2; ++u) {
          const int tl = (G / 2) * hf + u;
          if (tl < it.nt) p.scores[(long long)(it.t0 + tl) * p.score_stride + c] = -INFINITY;
        }
      }
      if (bad) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kScoreMmaWarp) tmem_dealloc(tmem, 512);
}

template <int NH>
cudaError_t launch_scores_nh(const ScoreParams &p, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(indexer_scores_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kScoreSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kScoreThreads);
  cfg.dynamicSmemBytes = kScoreSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, indexer_scores_kernel<NH>, p);
}

cudaError_t launch_indexer_scores(const ScoreParams &p, int n_heads, int grid, cudaStream_t s) {
  switch (n_heads) {
    case 1: return launch_scores_nh<1>(p, grid, s);
    case 2: return launch_scores_nh<2>(p, grid, s);
    case 4: return launch_scores_nh<4>(p, grid, s);
    case 8: return launch_scores_nh<8>(p, grid, s);
    case 16: return launch_scores_nh<16>(p, grid, s);
    case 32: return launch_scores_nh<32>(p, grid, s);
    case 64: return launch_scores_nh<64>(p, grid, s);
    case 128: return launch_scores_nh<128>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ds4a
