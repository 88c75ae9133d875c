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

// One CTA per token.  Exact radix select on the score keys in three digits of
// 12, 10 and 10 bits (the first spans sign, exponent and 3 mantissa bits, so
// clustered scores spread over many bins and the shared atomics rarely
// collide).  The first pass histograms the first digit; it names the bin b0
// where the count of larger keys reaches top_k.  The second pass walks each
// warp's contiguous chunk of rows, counts the keys of larger bins (all of
// them are taken) and compacts bin b0's keys with their row numbers.  The
// other two digits run over those survivors alone and give K* (the top_k-th
// largest key) and how many keys equal to K* are taken; the survivors' own
// K* comparisons finish each chunk's counts.  A last pass in row order takes
// every row with key > K* and the first rows with key == K* (lower index
// first) up to top_k, from each chunk's offset and share of the ties.  When
// bin b0 is too large to compact, the last two digits and the counts run over
// all keys instead.
constexpr int kTopkCompact = 2048;  // (key, row) pairs of the crossing bin kept for the last two digits

// Block-wide: the bin (scanning from the top) where the count of keys in
// larger bins first reaches `need`; returns it and that count.
template <int NBINS>
__device__ __forceinline__ void find_bin(const uint32_t *hist, uint32_t need, uint32_t *sh_out, uint32_t *wsum,
                                         int tid) {
  constexpr int PER = NBINS / kTopkThreads;  // bins per thread, descending order
  const int lane = tid & 31, warp = tid >> 5;
  const int top = NBINS - 1 - PER * tid;
  uint32_t s = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) s += hist[top - j];
  uint32_t incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += x;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  uint32_t above = incl - s;
  for (int w = 0; w < warp; ++w) above += wsum[w];
  if (above < need && need <= above + s) {
    uint32_t acc = above;
    for (int j = 0; j < PER; ++j) {
      const uint32_t c = hist[top - j];
      if (acc + c >= need) {
        sh_out[0] = (uint32_t)(top - j);
        sh_out[1] = acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

template <bool CACHED>
__global__ void __launch_bounds__(kTopkThreads) indexer_topk_kernel(const TopkParams p) {
  extern __shared__ uint32_t keys_s[];
  // The first digit's histogram, then (once bin b0 is known) the compacted
  // (key, row) pairs of that bin: one array, so that four CTAs fit on an SM.
  __shared__ __align__(16) uint32_t hist[4096];
  __shared__ uint32_t hist2[1024];  // digits 2 and 3
  static_assert(2 * kTopkCompact <= 4096, "the survivors reuse the first histogram");
  uint2 *surv = reinterpret_cast<uint2 *>(hist);
  __shared__ uint32_t wsum[kTopkWarps];
  __shared__ uint32_t cnt[2][kTopkWarps];
  __shared__ uint32_t sh_bin[2];
  __shared__ uint32_t sh_count;
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
  auto key_at = [&](int i) -> uint32_t { return CACHED ? keys_s[i] : score_key(__ldg(row + i)); };
  for (int i = tid; i < 4096; i += kTopkThreads) hist[i] = 0u;
  if (tid < kTopkWarps) {
    cnt[0][tid] = 0u;
    cnt[1][tid] = 0u;
  }
  if (tid == 0) sh_count = 0;
  __syncthreads();
  // pass 1, digit 1: bits 31..20
  for (int i = tid; i < n; i += kTopkThreads) {
    const uint32_t k = score_key(__ldg(row + i));
    if (CACHED) keys_s[i] = k;
    atomicAdd(&hist[k >> 20], 1u);
  }
  __syncthreads();
  find_bin<4096>(hist, (uint32_t)K, sh_bin, wsum, tid);
  const uint32_t b0 = sh_bin[0];
  uint32_t need = (uint32_t)K - sh_bin[1];  // keys still to take from bin b0
  const uint32_t m = hist[b0];              // keys in bin b0
  const bool compact = m <= (uint32_t)kTopkCompact;
  __syncthreads();  // every thread has read hist[b0] before the survivors overwrite it
  const uint32_t lt_mask = (1u << lane) - 1u;
  // Each warp owns rows [r0, r1), a multiple of 32 long.
  const int chunk = ((n + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
  const int r0 = min(n, warp * chunk), r1 = min(n, r0 + chunk);
  // pass 2: keys of larger bins counted per chunk, bin b0 compacted with its rows
  if (compact) {
    uint32_t c_hi = 0;
    for (int base = r0; base < r1; base += 32) {
      const int i = base + lane;
      const uint32_t k = i < r1 ? key_at(i) : 0u;
      const uint32_t bin = k >> 20;
      c_hi += __popc(__ballot_sync(0xffffffffu, i < r1 && bin > b0));
      const bool hit = i < r1 && bin == b0;
      const uint32_t bal = __ballot_sync(0xffffffffu, hit);
      if (bal != 0u) {
        uint32_t off = 0;
        if (lane == 0) off = atomicAdd(&sh_count, (uint32_t)__popc(bal));
        off = __shfl_sync(0xffffffffu, off, 0);
        if (hit) surv[off + __popc(bal & lt_mask)] = make_uint2(k, (uint32_t)i);
      }
    }
    if (lane == 0) cnt[0][warp] = c_hi;
  }
  __syncthreads();  // surv and the larger-bin counts complete
  // digits 2 and 3: bits 19..10 and 9..0, over bin b0's keys
  uint32_t prefix = b0;
  for (int d = 0; d < 2; ++d) {
    const int shift = d == 0 ? 10 : 0;
    for (int i = tid; i < 1024; i += kTopkThreads) hist2[i] = 0u;
    __syncthreads();
    const int nsrc = compact ? (int)m : n;
    for (int i = tid; i < nsrc; i += kTopkThreads) {
      const uint32_t k = compact ? surv[i].x : key_at(i);
      if ((k >> (shift + 10)) == prefix) atomicAdd(&hist2[(k >> shift) & 1023u], 1u);
    }
    __syncthreads();
    find_bin<1024>(hist2, need, sh_bin, wsum, tid);
    prefix = (prefix << 10) | sh_bin[0];
    need -= sh_bin[1];
  }
  const uint32_t kstar = prefix;
  // Per chunk: keys > K* (cnt[0]) and keys == K* (cnt[1]).
  if (compact) {
    for (int i = tid; i < (int)m; i += kTopkThreads) {
      const uint2 e = surv[i];
      const int w = (int)e.y / chunk;
      if (e.x > kstar) atomicAdd(&cnt[0][w], 1u);
      else if (e.x == kstar) atomicAdd(&cnt[1][w], 1u);
    }
  } else {
    uint32_t c_gt = 0, c_eq = 0;
    for (int base = r0; base < r1; base += 32) {
      const int i = base + lane;
      const uint32_t k = i < r1 ? key_at(i) : 0u;
      c_gt += __popc(__ballot_sync(0xffffffffu, i < r1 && k > kstar));
      c_eq += __popc(__ballot_sync(0xffffffffu, i < r1 && k == kstar));
    }
    if (lane == 0) {
      cnt[0][warp] = c_gt;
      cnt[1][warp] = c_eq;
    }
  }
  __syncthreads();
  // pass 3: selection in row order
  uint32_t eq_run = 0, sel_run = 0;
  for (int w = 0; w < warp; ++w) {
    const uint32_t g = cnt[0][w], e = cnt[1][w];
    const uint32_t taken = eq_run >= need ? 0u : min(e, need - eq_run);
    sel_run += g + taken;
    eq_run += e;
  }
  for (int base = r0; base < r1; base += 32) {
    const int i = base + lane;
    const uint32_t k = i < r1 ? key_at(i) : 0u;
    const bool gt = i < r1 && k > kstar, eq = i < r1 && k == kstar;
    const uint32_t b_eq = __ballot_sync(0xffffffffu, eq);
    const bool take = gt || (eq && eq_run + __popc(b_eq & lt_mask) < need);
    const uint32_t b_sel = __ballot_sync(0xffffffffu, take);
    const uint32_t pos = sel_run + __popc(b_sel & lt_mask);
    if (take && pos < (uint32_t)K) out[pos] = i;
    eq_run += __popc(b_eq);
    sel_run += __popc(b_sel);
  }
}

cudaError_t launch_indexer_topk(const TopkParams &p, int dyn_smem, cudaStream_t s) {
  if (p.cached_keys > 0) {
    cudaError_t e =
        cudaFuncSetAttribute(indexer_topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem);
    if (e != cudaSuccess) return e;
    indexer_topk_kernel<true><<<p.g.T, kTopkThreads, dyn_smem, s>>>(p);
  } else {
    indexer_topk_kernel<false><<<p.g.T, kTopkThreads, 0, s>>>(p);
  }
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

// Scores of one tile for the thread's row c and half hf of the 256 columns
// (tokens G/2*hf ..): w_s holds w[t][h] * |scale| (or * scale without the
// max), so each TMEM value costs one max and one fma (one fma without max).
// Packed pair of fp32 lanes (fma.rn.f32x2: two fmas per instruction).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ float f2_sum(uint64_t r) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
  return a + b;
}

template <int NH, bool RELU, bool NEG>
__device__ __forceinline__ void score_tile(const ScoreParams &p, const ScoreItem &it, const float *w_s,
                                           uint32_t tcol, int hf, int c, long long pos1) {
  constexpr int HW = NH < 32 ? NH : 32;  // heads of one token inside a 32-column chunk
  constexpr int TPC = 32 / HW;            // tokens per chunk
  constexpr int CPT = NH < 32 ? 1 : NH / 32;  // chunks per token
  float acc = 0.f;
#pragma unroll
  for (int j2 = 0; j2 < 2; ++j2) {
    float v[64];
    tmem_ld64(tcol + 64 * j2, v);
    tmem_wait_ld();
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = 2 * j2 + jj;
      const float *ww = w_s + 128 * hf + 32 * j;
#pragma unroll
      for (int u = 0; u < TPC; ++u) {
        float sum = 0.f;
        if (HW == 1) {
          float x = v[32 * jj + u];
          if (RELU) x = fmaxf(NEG ? -x : x, 0.f);
          sum = ww[u] * x;
        } else {
          // two heads per packed fma: even and odd heads in separate partial sums
          uint64_t s2 = 0;
#pragma unroll
          for (int h = 0; h < HW; h += 2) {
            float x0 = v[32 * jj + u * HW + h], x1 = v[32 * jj + u * HW + h + 1];
            if (RELU) {
              x0 = fmaxf(NEG ? -x0 : x0, 0.f);
              x1 = fmaxf(NEG ? -x1 : x1, 0.f);
            }
            const float2 w2 = *reinterpret_cast<const float2 *>(ww + u * HW + h);
            s2 = f2_fma(f2_pack(w2.x, w2.y), f2_pack(x0, x1), s2);
          }
          sum = f2_sum(s2);
        }
        if (NH >= 32) {
          acc += sum;
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
                (long long)(c + 1) * p.g.ratio <= pos1 + tl ? sum : -INFINITY;
        }
      }
    }
  }
}

template <int NH, bool RELU>
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
    // relu(scale x) = |scale| relu(sign(scale) x): |scale| goes into the weights.
    const bool neg = RELU && p.scale < 0.f;
    const float wscale = RELU ? fabsf(p.scale) : p.scale;
    uint32_t tc = 0;
    bool bad = false;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const ScoreItem it = score_item(p, item, G);
      bar_sync_n(1, kScoreEpiThreads);  // the previous item's epilogue is done with w_s
      {
        const int tl = tid / NH, h = tid % NH;
        ms.w_s[tid] = tl < it.nt ? wscale * __ldg(p.w + (long long)(it.t0 + tl) * NH + h) : 0.f;
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
        const uint32_t tcol = tmem + 256 * buf + 128 * hf + lane_base;
        if (neg)
          score_tile<NH, RELU, true>(p, it, ms.w_s, tcol, hf, c, pos1);
        else
          score_tile<NH, RELU, false>(p, it, ms.w_s, tcol, hf, c, pos1);
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

template <int NH, bool RELU>
cudaError_t launch_scores_nh(const ScoreParams &p, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(indexer_scores_kernel<NH, RELU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  return cudaLaunchKernelEx(&cfg, indexer_scores_kernel<NH, RELU>, p);
}

template <bool RELU>
cudaError_t launch_scores_relu(const ScoreParams &p, int n_heads, int grid, cudaStream_t s) {
  switch (n_heads) {
    case 1: return launch_scores_nh<1, RELU>(p, grid, s);
    case 2: return launch_scores_nh<2, RELU>(p, grid, s);
    case 4: return launch_scores_nh<4, RELU>(p, grid, s);
    case 8: return launch_scores_nh<8, RELU>(p, grid, s);
    case 16: return launch_scores_nh<16, RELU>(p, grid, s);
    case 32: return launch_scores_nh<32, RELU>(p, grid, s);
    case 64: return launch_scores_nh<64, RELU>(p, grid, s);
    case 128: return launch_scores_nh<128, RELU>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_indexer_scores(const ScoreParams &p, int n_heads, int grid, cudaStream_t s) {
  return p.relu ? launch_scores_relu<true>(p, n_heads, grid, s) : launch_scores_relu<false>(p, n_heads, grid, s);
}

// Loads the code of every kernel listed (lazy module loading would otherwise
// do it at a kernel's first launch, which may fall inside a stream capture).
cudaError_t preload_indexer_kernels() {
  const void *k[] = {
      (const void *)indexer_topk_kernel<true>,          (const void *)indexer_topk_kernel<false>,
      (const void *)indexer_scores_kernel<1, false>,   (const void *)indexer_scores_kernel<1, true>,
      (const void *)indexer_scores_kernel<2, false>,   (const void *)indexer_scores_kernel<2, true>,
      (const void *)indexer_scores_kernel<4, false>,   (const void *)indexer_scores_kernel<4, true>,
      (const void *)indexer_scores_kernel<8, false>,   (const void *)indexer_scores_kernel<8, true>,
      (const void *)indexer_scores_kernel<16, false>,  (const void *)indexer_scores_kernel<16, true>,
      (const void *)indexer_scores_kernel<32, false>,  (const void *)indexer_scores_kernel<32, true>,
      (const void *)indexer_scores_kernel<64, false>,  (const void *)indexer_scores_kernel<64, true>,
      (const void *)indexer_scores_kernel<128, false>, (const void *)indexer_scores_kernel<128, true>};
  for (const void *f : k) {
    cudaFuncAttributes a;
    const cudaError_t e = cudaFuncGetAttributes(&a, f);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ds4a
