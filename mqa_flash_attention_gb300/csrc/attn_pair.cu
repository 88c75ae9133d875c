// Fused attention forward for pairs of consecutive query tokens over raw rows
// (structural rule, no compressed rows, window <= 128): the raw-only layers
// and the raw part of a prefill chunk ("DwarfStar 4 (DS4) - DeepSeek V4 Flash
// Inference Engine", sections "Layer Compression" and "Whole-Model Graph
// Execution"; fused as in "How DeepSeek V4 Flash Model Inference Works on
// Apple Silicon with Metal Backend", section "FlashAttention Kernel
// Architecture").  The result is the same attention as attn_fwd_kernel's.
//
// Why pairs.  Two consecutive tokens see windows that differ by one row, so
// one 128-row K/V tile serves both: the tile is the later token's window and
// the earlier token's one remaining row (below the tile) is folded in on the
// CUDA cores.  Every K/V row then enters the SM once per two tokens (Q 64 KB
// + K 64 KB + V 64 KB per token instead of 64 + 128 + 128), and both
// products run as N = 128 MMAs (two tokens x 64 heads), at the tensor core's
// full rate where a single token's N = 64 runs near half of it:
//   S^T[128 rows][128]      = K_tile[128][512] . Q_pair[128][512]^T   (K-major A, K-major B)
//   O^T_m[128 dims][128]    = V_tile^T[dims 128m..][128] . P^T          (MN-major A, MN-major B)
// TMEM: two S^T buffers (columns 0-127 and 128-255, by pair parity) and two
// 128-column O^T buffers (256-383 and 384-511) through which the four 128-dim
// blocks of a pair's O^T pass, drained by the epilogue as they complete; no
// block accumulates across tiles (the pair has one tile).  With two S^T
// buffers the QK^T of the next pair runs while the softmax reads this one.
//
// Shared memory: a ring of 10 slots of 16 KB through which every box streams
// in the order the MMAs take them: the Q and K boxes of pair 0, then for each
// pair n the Q and K boxes of pair n+1 (Q box b, K box b for b = 0..7) before
// the V boxes of pair n (0..7; a PV block takes two adjacent V slots), so the
// next pair's loads are not queued behind V boxes that wait for this pair's
// softmax.  Also P^T of a pair (32 KB), the extra row's K and V (two 2 KB
// buffers, by pair parity) and bookkeeping.
// Warp roles (352 threads):
//   warps 0-7  softmax + epilogue; thread (TMEM lane quarter w % 4, token w / 4)
//              handles one row (or dim) and that token's 64 heads in two halves
//   warp  8    loader (one thread issues every TMA copy)
//   warp  9    TMEM allocator and tcgen05.mma issuer
//   warp 10    extra row: reads its K and V rows (one pair ahead) and takes
//              token a's scores against it from the Q boxes as they pass
//              through the ring
// A Q slot is released by the MMA's commit and by the extra-row warp (it reads
// it), a K or V slot by the commit and a plain arrival of the MMA thread:
// every slot's "free" barrier counts two arrivals.  The extra-row warp learns
// that Q box b landed from the MMA thread (qx[b]), which waits on every slot
// in order: a parity wait must not fall more than one phase behind, and a
// ring position passes through K and V uses the extra-row warp never sees.
// For the same reason the MMA thread passes on Q box b of a pair only after
// the extra-row warp has finished box b of the previous pair (xdone[b]), and
// the extra-row scores are handed over through one barrier per pair parity.
// Every wait is bounded as in attn_fwd_kernel.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ds4a {
namespace {

constexpr int kPWarps = 8;
constexpr int kPThreadsC = 32 * kPWarps;
constexpr int kPLoaderWarp = 8;
constexpr int kPMmaWarp = 9;
constexpr int kPXWarp = 10;
constexpr int kPThreads = 32 * (kPXWarp + 1);
constexpr int kPSlots = 10;
constexpr uint32_t kPSlot = 16384;
constexpr int kPSlotsPerPair = 24;  // 8 Q + 8 K + 8 V boxes
constexpr uint32_t kPOffRing = 0;
constexpr uint32_t kPOffP = kPSlots * kPSlot;      // P^T: token a's box, then token b's
constexpr uint32_t kPOffX = kPOffP + 2 * kPSlot;   // extra rows by pair parity: K [512] fp16, then V [512]
constexpr uint32_t kPOffMisc = kPOffX + 2 * 2048;
static_assert(kPSlots % 2 == 0 && kPSlotsPerPair % 2 == 0, "V slot pairs must stay adjacent in the ring");

struct PairMisc {
  alignas(16) float red[4][128];  // per lane quarter: partial max, then partial sum, of each column
  alignas(16) float m_use[128];   // reference max of each column (log2 units), 0 when nothing is visible
  alignas(16) float m_true[128];  // the max itself (-inf when nothing is visible)
  alignas(16) float inv_l[128];
  alignas(16) float sx[2][64];    // extra row, by pair parity: scaled score of token a per head (log2 units)
  alignas(16) float px[64];       // extra row: its weight
  alignas(8) uint64_t full[kPSlots], empty[kPSlots];
  uint64_t s_full[2], s_empty[2], p_full, p_empty, o_full[2], o_empty[2], mma_done;
  uint64_t x_full[2], x_empty[2]; // by pair parity: extra-row scores ready; the row buffer free again
  uint64_t qx[8];                 // Q box b of the current pair has landed (passed on by the MMA thread)
  uint64_t xdone[8];              // the extra-row warp is done with Q box b of its current pair
  uint32_t tmem_base;
  int abort_flag;
};
constexpr uint32_t kPSmemBytes = kPOffMisc + ((sizeof(PairMisc) + 127) / 128) * 128 + 1024;
static_assert(kPSmemBytes <= 232448, "pair kernel shared memory");

enum : unsigned int {
  SITE_PR_EMPTY = 0x20, SITE_PR_FULL, SITE_PR_S_EMPTY, SITE_PR_S_FULL, SITE_PR_P_FULL, SITE_PR_P_EMPTY,
  SITE_PR_O_EMPTY, SITE_PR_O_FULL, SITE_PR_DRAIN, SITE_PR_X_FULL, SITE_PR_X_EMPTY
};

// The pair's tokens and rows.  Token a = 2 * pair, token b = a + 1 (absent for
// an odd last token).  Token t sees raw rows [lo, hi) (its window clipped to
// the rows given); the tile is the 128 rows ending at the later token's last
// row (it may start below row 0: the TMA fills those rows with zeros and the
// mask drops them); with a window of at most 128, token a reaches at most one
// row below the tile.
struct PairGeom {
  int ta;
  bool has_b;
  int lo[2], hi[2];
  int tile_lo;
  bool extra;
};

__device__ __forceinline__ PairGeom pair_geom(const PairParams &p, int pr) {
  PairGeom g;
  g.ta = 2 * pr;
  g.has_b = g.ta + 1 < p.T;
  int hi_max = 0;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    int lo = 0, hi = 0;
    if (u == 0 || g.has_b) {
      const long long pos = (long long)p.q_pos0 + g.ta + u;
      const long long a = pos - p.window + 1 - p.raw_pos0, b = pos + 1 - p.raw_pos0;
      lo = (int)(a < 0 ? 0 : a);
      hi = (int)(b > p.n_raw ? p.n_raw : b);
      if (hi < lo) hi = lo;
    }
    g.lo[u] = lo;
    g.hi[u] = hi;
    hi_max = max(hi_max, hi);
  }
  g.tile_lo = hi_max - 128;
  g.extra = g.lo[0] < g.hi[0] && g.lo[0] < g.tile_lo;
  return g;
}

__device__ __forceinline__ uint32_t slot_addr(uint32_t sbase, uint32_t sl) {
  return sbase + kPOffRing + (sl % kPSlots) * kPSlot;
}
__device__ __forceinline__ uint32_t slot_phase(uint32_t sl) { return (sl / kPSlots) & 1u; }
// TMEM columns: S^T of pair parity i at 128 i; O^T block m in buffer m & 1 at 256 + 128 (m & 1).
__device__ __forceinline__ uint32_t s_column(uint32_t n) { return 128u * (n & 1u); }
__device__ __forceinline__ uint32_t o_column(int m) { return 256u + 128u * (m & 1); }

// Ring slot of Q box 0 of the CTA's pair n: pair 0's Q and K boxes come
// first, then each pair step adds the next pair's 16 boxes and this pair's 8
// V boxes.
__device__ __forceinline__ uint32_t qk_base(uint32_t n) { return n == 0 ? 0u : 16u + 24u * (n - 1u); }

// ------------------------------------------------------------------ loader

__device__ __forceinline__ bool pair_fill(const PairParams &p, uint32_t sbase, PairMisc &ms, volatile int *abrt,
                                          const PairGeom &g, int i, uint32_t &sl, uint32_t &filled,
                                          uint32_t &last_par) {
  const uint32_t pos = sl % kPSlots, ph = slot_phase(sl);
  if (!mbar_wait(smem_u32(&ms.empty[pos]), ph ^ 1, abrt, p.timeout_ns, p.err, SITE_PR_EMPTY)) return false;
  const uint32_t dst = slot_addr(sbase, sl), bar = smem_u32(&ms.full[pos]);
  mbar_arrive_expect_tx(bar, kPSlot);
  if (i < 16) {
    const int b = i >> 1;
    if ((i & 1) == 0)
      tma_load_3d(dst, &p.tm_q2, bar, 64 * b, 0, g.ta);  // both tokens' heads, dims 64b ..
    else
      tma_load_2d(dst, &p.tm_k, bar, 64 * b, g.tile_lo);
  } else {
    tma_load_2d(dst, &p.tm_v, bar, 64 * (i - 16), g.tile_lo);
  }
  filled |= 1u << pos;
  last_par = (last_par & ~(1u << pos)) | (ph << pos);
  ++sl;
  return true;
}

__device__ __forceinline__ void pair_loader(const PairParams &p, uint32_t sbase, PairMisc &ms) {
  volatile int *abrt = &ms.abort_flag;
  const int n_pairs = (p.T + 1) / 2;
  uint32_t sl = 0, filled = 0, last_par = 0;
  bool ok = true;
  grid_dependency_wait();  // Q, K and V may come from the previous kernel
  if ((int)blockIdx.x < n_pairs) {
    const PairGeom g0 = pair_geom(p, blockIdx.x);
    for (int i = 0; i < 16 && ok; ++i) ok = pair_fill(p, sbase, ms, abrt, g0, i, sl, filled, last_par);
  }
  for (int pr = blockIdx.x; pr < n_pairs && ok; pr += gridDim.x) {
    if (pr + (int)gridDim.x < n_pairs) {  // the next pair's Q and K, then this pair's V
      const PairGeom gn = pair_geom(p, pr + gridDim.x);
#pragma unroll 1
      for (int i = 0; i < 16 && ok; ++i) ok = pair_fill(p, sbase, ms, abrt, gn, i, sl, filled, last_par);
    }
    const PairGeom g = pair_geom(p, pr);
#pragma unroll 1
    for (int i = 16; i < kPSlotsPerPair && ok; ++i) ok = pair_fill(p, sbase, ms, abrt, g, i, sl, filled, last_par);
  }
  if (!ok) {
    // Let every copy already issued land before the shared memory goes away.
    volatile int never = 0;
    for (int s = 0; s < kPSlots; ++s)
      if (filled & (1u << s))
        mbar_wait(smem_u32(&ms.full[s]), (last_par >> s) & 1, &never, 100000000ull, p.err, SITE_PR_DRAIN);
  }
}

// ------------------------------------------------------------------ MMA issuer

// QK^T of the CTA's pair j into S^T buffer j & 1, from the pair's 16 Q and K
// slots starting at `sl`.
__device__ __forceinline__ bool pair_qk(const PairParams &p, uint32_t sbase, uint32_t tmem, PairMisc &ms,
                                        volatile int *abrt, uint32_t j, uint32_t &sl) {
  constexpr uint32_t kIdescQK = idesc_f16_f32(128, 128, false, false);
  // K and Q boxes: K-major, SBO = one 8-row group.
  const uint64_t kq_desc = sdesc_sw128(sbase + kPOffRing, 16, 1024);
  if (!mbar_wait(smem_u32(&ms.s_empty[j & 1]), ((j >> 1) & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_PR_S_EMPTY))
    return false;
  tc_fence_after();
  const uint32_t d = tmem + s_column(j);
  for (int b = 0; b < 8; ++b, sl += 2) {
    const uint32_t pq = sl % kPSlots, pk = (sl + 1) % kPSlots;
    if (!mbar_wait(smem_u32(&ms.full[pq]), slot_phase(sl), abrt, p.timeout_ns, p.err, SITE_PR_FULL) ||
        !mbar_wait(smem_u32(&ms.full[pk]), slot_phase(sl + 1), abrt, p.timeout_ns, p.err, SITE_PR_FULL))
      return false;
    tc_fence_after();
    const uint64_t a0 = sdesc_add(kq_desc, pk * kPSlot), b0 = sdesc_add(kq_desc, pq * kPSlot);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      if (b == 0 && ks == 0)
        umma_f16(d, sdesc_add(a0, ks * 32), sdesc_add(b0, ks * 32), kIdescQK, 0u);
      else
        umma_f16_acc(d, sdesc_add(a0, ks * 32), sdesc_add(b0, ks * 32), kIdescQK);
    }
    // The extra-row warp may read Q box b once it is done with box b of the
    // previous pair (so qx[b] never runs two phases ahead of it).
    if (j > 0 && !mbar_wait(smem_u32(&ms.xdone[b]), (j - 1) & 1, abrt, p.timeout_ns, p.err, SITE_PR_X_EMPTY))
      return false;
    mbar_arrive(smem_u32(&ms.qx[b]));
    umma_commit(smem_u32(&ms.empty[pq]));  // the extra-row warp gives the Q slot's second arrival
    umma_commit(smem_u32(&ms.empty[pk]));
    mbar_arrive(smem_u32(&ms.empty[pk]));
  }
  umma_commit(smem_u32(&ms.s_full[j & 1]));
  return true;
}

// PV of the CTA's pair n once P^T is written: O^T block m into buffer m & 1
// (after the epilogue drained block m - 2), from the V slots starting at `sl`.
__device__ __forceinline__ bool pair_pv(const PairParams &p, uint32_t sbase, uint32_t tmem, PairMisc &ms,
                                        volatile int *abrt, uint32_t n, uint32_t &sl) {
  constexpr uint32_t kIdescPV = idesc_f16_f32(128, 128, true, true);
  // V^T: MN-major, its two 64-dim atoms in adjacent slots (LBO = one slot).
  // P^T: MN-major, token a's heads then token b's (LBO = one box).
  const uint64_t v_desc = sdesc_sw128(sbase + kPOffRing, kPSlot, 1024);
  const uint64_t p_desc = sdesc_sw128(sbase + kPOffP, kPSlot, 1024);
  if (!mbar_wait(smem_u32(&ms.p_full), n & 1, abrt, p.timeout_ns, p.err, SITE_PR_P_FULL)) return false;
  tc_fence_after();
  for (int m = 0; m < 4; ++m, sl += 2) {
    const uint32_t gb = 4 * n + m, buf = gb & 1;
    const uint32_t pa = sl % kPSlots, pb = (sl + 1) % kPSlots;  // pa even: pb = pa + 1
    if (!mbar_wait(smem_u32(&ms.o_empty[buf]), ((gb >> 1) & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_PR_O_EMPTY) ||
        !mbar_wait(smem_u32(&ms.full[pa]), slot_phase(sl), abrt, p.timeout_ns, p.err, SITE_PR_FULL) ||
        !mbar_wait(smem_u32(&ms.full[pb]), slot_phase(sl + 1), abrt, p.timeout_ns, p.err, SITE_PR_FULL))
      return false;
    tc_fence_after();
    const uint64_t a0 = sdesc_add(v_desc, pa * kPSlot);
    const uint32_t d = tmem + o_column(m);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      if (ks == 0)
        umma_f16(d, a0, p_desc, kIdescPV, 0u);
      else
        umma_f16_acc(d, sdesc_add(a0, ks * 2048), sdesc_add(p_desc, ks * 2048), kIdescPV);
    }
    umma_commit(smem_u32(&ms.empty[pa]));
    umma_commit(smem_u32(&ms.empty[pb]));
    mbar_arrive(smem_u32(&ms.empty[pa]));
    mbar_arrive(smem_u32(&ms.empty[pb]));
    umma_commit(smem_u32(&ms.o_full[buf]));
  }
  umma_commit(smem_u32(&ms.p_empty));
  return true;
}

// The MMA thread takes the slots in the loader's order: QK^T of pair 0, then
// for each pair n the QK^T of pair n+1 (while the softmax works on pair n)
// and the PV of pair n.
__device__ __forceinline__ void pair_mma(const PairParams &p, uint32_t sbase, uint32_t tmem, PairMisc &ms) {
  volatile int *abrt = &ms.abort_flag;
  const int n_pairs = (p.T + 1) / 2;
  uint32_t sl = 0, n = 0;
  bool ok = true;
  if ((int)blockIdx.x < n_pairs) ok = pair_qk(p, sbase, tmem, ms, abrt, 0, sl);
  for (int pr = blockIdx.x; pr < n_pairs && ok; pr += gridDim.x, ++n) {
    if (pr + (int)gridDim.x < n_pairs) ok = pair_qk(p, sbase, tmem, ms, abrt, n + 1, sl);
    ok = ok && pair_pv(p, sbase, tmem, ms, abrt, n, sl);
  }
  // Every MMA issued so far must finish before TMEM is released.
  umma_commit(smem_u32(&ms.mma_done));
  volatile int never = 0;
  mbar_wait(smem_u32(&ms.mma_done), 0, &never, 100000000ull, p.err, SITE_PR_DRAIN);
}

// ------------------------------------------------------------------ softmax and epilogue

// Lane l ends with the max (or sum) over the warp's 32 rows of column l of the
// 32 columns held in s[0..31].
template <bool kMax>
__device__ __forceinline__ float reduce_scatter32(const float (&s)[32], int lane) {
  float a[16];
  {
    const bool up = lane & 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float send = up ? s[i] : s[i + 16];
      const float keep = up ? s[i + 16] : s[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, 16);
      a[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int c = 16; c >= 2; c >>= 1) {
    const int half = c / 2;
    const bool up = lane & half;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? a[i] : a[i + half];
      const float keep = up ? a[i + half] : a[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, half);
      a[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return a[0];
}

__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kPThreadsC) : "memory"); }

__device__ __forceinline__ void pair_compute(const PairParams &p, uint8_t *smem, uint32_t tmem, PairMisc &ms,
                                             int tid) {
  volatile int *abrt = &ms.abort_flag;
  const int w = tid >> 5, l = tid & 31;
  const int q = w & 3;       // TMEM lane quarter: rows (or dims) 32q .. 32q+31
  const int tau = w >> 2;    // token of the pair whose columns this thread takes
  const int r = 32 * q + l;  // this thread's TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
  const int n_pairs = (p.T + 1) / 2;
  uint32_t n = 0;
  bool bad = false;
  grid_dependency_wait();  // the outputs may still be read by the previous kernel
  for (int pr = blockIdx.x; pr < n_pairs; pr += gridDim.x, ++n) {
    const PairGeom g = pair_geom(p, pr);
    const bool has_tok = tau == 0 || g.has_b;
    const float *sx = ms.sx[n & 1];
    const __half *vx = reinterpret_cast<const __half *>(smem + kPOffX + 2048 * (n & 1)) + 512;
    // The extra-row warp's scores of this pair (every pair, so the phases
    // stay in step).
    bad = bad || !mbar_wait(smem_u32(&ms.x_full[n & 1]), (n >> 1) & 1, abrt, p.timeout_ns, p.err, SITE_PR_X_FULL);

    // Softmax of the pair's tile.  Pass 1: column maxima.
    bad = bad || !mbar_wait(smem_u32(&ms.s_full[n & 1]), (n >> 1) & 1, abrt, p.timeout_ns, p.err, SITE_PR_S_FULL);
    tc_fence_after();
    const int row = g.tile_lo + r;
    const bool vis = has_tok && row >= g.lo[tau] && row < g.hi[tau];
#pragma unroll 1
    for (int u = 0; u < 2; ++u) {
      float s[32];
      tmem_ld32(tmem + s_column(n) + 64 * tau + 32 * u + lane_base, s);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < 32; ++h) s[h] = vis ? s[h] * p.scale_log2 : -INFINITY;
      ms.red[q][64 * tau + 32 * u + l] = reduce_scatter32<true>(s, l);
    }
    if (bar_red_or(1, kPThreadsC, bad)) break;
    if (tid < 128) {
      const int tt = tid >> 6, h = tid & 63;
      float mx = fmaxf(fmaxf(ms.red[0][tid], ms.red[1][tid]), fmaxf(ms.red[2][tid], ms.red[3][tid]));
      if (tt == 0 && g.extra) mx = fmaxf(mx, sx[h]);
      ms.m_true[tid] = mx;
      ms.m_use[tid] = mx == -INFINITY ? 0.f : mx;
    }
    csync();
    // Pass 2: P = 2^(s - m) in fp16 (P^T row r of token tau's box, 16-byte
    // chunk c at c ^ (r & 7): the 128-byte swizzle) and the row sums of the
    // same fp16 values.  P may be rewritten once the previous pair's PV is done.
    bad = bad || !mbar_wait(smem_u32(&ms.p_empty), (n & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_PR_P_EMPTY);
    uint8_t *prow = smem + kPOffP + tau * kPSlot + r * 128;
#pragma unroll 1
    for (int u = 0; u < 2; ++u) {
      float s[32];
      tmem_ld32(tmem + s_column(n) + 64 * tau + 32 * u + lane_base, s);
      tmem_wait_ld();
      const float *mu = ms.m_use + 64 * tau + 32 * u;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = 8 * c + 2 * i;
          const float e0 = vis ? exp2f(s[h] * p.scale_log2 - mu[h]) : 0.f;
          const float e1 = vis ? exp2f(s[h + 1] * p.scale_log2 - mu[h + 1]) : 0.f;
          const __half2 hp = __floats2half2_rn(e0, e1);
          const float2 f = __half22float2(hp);
          s[h] = f.x;
          s[h + 1] = f.y;
          w4[i] = *reinterpret_cast<const uint32_t *>(&hp);
        }
        const int chunk = 4 * u + c;
        *reinterpret_cast<uint4 *>(prow + ((chunk ^ (r & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      ms.red[q][64 * tau + 32 * u + l] = reduce_scatter32<false>(s, l);
    }
    tc_fence_before();
    mbar_arrive(smem_u32(&ms.s_empty[n & 1]));  // S^T read for the last time
    fence_proxy_async_smem();
    mbar_arrive(smem_u32(&ms.p_full));
    if (bar_red_or(1, kPThreadsC, bad)) break;
    if (tid < 128) {
      const int tt = tid >> 6, h = tid & 63;
      float lsum = ms.red[0][tid] + ms.red[1][tid] + ms.red[2][tid] + ms.red[3][tid];
      if (tt == 0 && g.extra) {
        const float px = exp2f(sx[h] - ms.m_use[tid]);
        ms.px[h] = px;
        lsum += px;
      }
      ms.inv_l[tid] = lsum > 0.f ? 1.f / lsum : 0.f;
      if (p.lse != nullptr && (tt == 0 || g.has_b))
        p.lse[(long long)(g.ta + tt) * kH + h] = lsum > 0.f ? (ms.m_true[tid] + log2f(lsum)) * kLn2 : -INFINITY;
    }
    csync();

    // Epilogue: O^T block m [128 dims][128] -> o of both tokens, as each
    // block completes.  Lanes 2k and 2k+1 hold adjacent dims: for each pair
    // of heads they swap one value, so the even lane writes both dims of the
    // first head and the odd lane both dims of the second (32-bit stores).
    const bool odd = l & 1;
    const bool with_x = tau == 0 && g.extra;  // token a folds in its extra row
    __half *obase = p.o + (long long)(g.ta + tau) * p.o_tok_stride + (r & ~1);
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
      const uint32_t gb = 4 * n + m;
      bad = bad || !mbar_wait(smem_u32(&ms.o_full[m & 1]), (gb >> 1) & 1, abrt, p.timeout_ns, p.err, SITE_PR_O_FULL);
      tc_fence_after();
      const float xv = with_x ? __half2float(vx[128 * m + r]) : 0.f;
      // Both halves of the block leave TMEM before the buffer is handed back,
      // so the next PV into it need not wait for the stores.
      float o[2][32];
      tmem_ld32(tmem + o_column(m) + 64 * tau + lane_base, o[0]);
      tmem_ld32(tmem + o_column(m) + 64 * tau + 32 + lane_base, o[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(smem_u32(&ms.o_empty[m & 1]));  // the buffer may take block m + 2
      if (has_tok) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float4 *iv4 = reinterpret_cast<const float4 *>(ms.inv_l + 64 * tau + 32 * u);
          if (with_x) {
            const float4 *px4 = reinterpret_cast<const float4 *>(ms.px + 32 * u);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 iv = iv4[j], px = px4[j];
              o[u][4 * j] = fmaf(px.x, xv, o[u][4 * j]) * iv.x;
              o[u][4 * j + 1] = fmaf(px.y, xv, o[u][4 * j + 1]) * iv.y;
              o[u][4 * j + 2] = fmaf(px.z, xv, o[u][4 * j + 2]) * iv.z;
              o[u][4 * j + 3] = fmaf(px.w, xv, o[u][4 * j + 3]) * iv.w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 iv = iv4[j];
              o[u][4 * j] *= iv.x;
              o[u][4 * j + 1] *= iv.y;
              o[u][4 * j + 2] *= iv.z;
              o[u][4 * j + 3] *= iv.w;
            }
          }
#pragma unroll
          for (int h = 0; h < 32; h += 2) {
            const float got = __shfl_xor_sync(0xffffffffu, odd ? o[u][h] : o[u][h + 1], 1);
            const __half2 v = odd ? __floats2half2_rn(got, o[u][h + 1]) : __floats2half2_rn(o[u][h], got);
            *reinterpret_cast<__half2 *>(obase + (32 * u + h + (odd ? 1 : 0)) * kD + 128 * m) = v;
          }
        }
      }
    }
    if (bar_red_or(1, kPThreadsC, bad)) break;
    if (tid == 0) mbar_arrive(smem_u32(&ms.x_empty[n & 1]));  // every thread is done with this parity's rows
  }
}

// Warp 10: for each pair, token a's row below the tile (when there is one):
// its K and V rows, read from global memory one pair ahead into registers;
// token a's scores against the K row, taken from the Q boxes as they pass
// through the ring (lane l: heads l and l + 32), with the second release of
// every Q slot; then the V row into this parity's buffer once the softmax
// warps are done with the pair two back.  Only the V row waits for them, so
// the Q slots go back to the ring as soon as the MMA has read them.  Lane l
// takes heads l and l + 32: the eight lanes of a group then read eight
// different 16-byte columns of the swizzled box, all 32 banks.
__device__ __forceinline__ void load_extra_row(const PairParams &p, const PairGeom &g, int lane, uint4 (&kr)[2],
                                               uint4 (&vr)[2]) {
  if (!g.extra) return;
  const long long off = (long long)(g.tile_lo - 1) * p.raw_row_stride;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = lane + 32 * i;  // 16-byte chunk of the 1024-byte row
    kr[i] = *reinterpret_cast<const uint4 *>(p.k_raw + off + 16 * c);
    vr[i] = *reinterpret_cast<const uint4 *>(p.v_raw + off + 16 * c);
  }
}

__device__ __forceinline__ void pair_extra_row(const PairParams &p, uint8_t *smem, PairMisc &ms, int lane) {
  volatile int *abrt = &ms.abort_flag;
  const int n_pairs = (p.T + 1) / 2;
  uint32_t n = 0;
  bool ok = true;
  grid_dependency_wait();  // the extra rows are read from global memory
  uint4 kr[2], vr[2];
  if ((int)blockIdx.x < n_pairs) load_extra_row(p, pair_geom(p, blockIdx.x), lane, kr, vr);
  for (int pr = blockIdx.x; pr < n_pairs && ok; pr += gridDim.x, ++n) {
    const PairGeom g = pair_geom(p, pr);
    uint8_t *xb = smem + kPOffX + 2048 * (n & 1);
    if (g.extra) {
      // The K half of this parity's buffer is read only by this warp.
#pragma unroll
      for (int i = 0; i < 2; ++i) *reinterpret_cast<uint4 *>(xb + 16 * (lane + 32 * i)) = kr[i];
      __syncwarp();
    }
    const __half *kx = reinterpret_cast<const __half *>(xb);
    float acc0 = 0.f, acc1 = 0.f;
    uint32_t sl = qk_base(n);
    for (int b = 0; b < 8; ++b, sl += 2) {
      const uint32_t pq = sl % kPSlots;
      ok = mbar_wait(smem_u32(&ms.qx[b]), n & 1, abrt, p.timeout_ns, p.err, SITE_PR_FULL);
      if (!ok) break;
      if (g.extra) {
        // Q box b: row (token a, head h) at h * 128, 16-byte chunk c (dims
        // 64b + 8c ..) at column c ^ (h & 7).
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 kv = *reinterpret_cast<const uint4 *>(kx + 64 * b + 8 * c);
          const __half2 *k2 = reinterpret_cast<const __half2 *>(&kv);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int h = lane + 32 * j;
            const uint4 qv = *reinterpret_cast<const uint4 *>(smem + kPOffRing + pq * kPSlot + h * 128 +
                                                              ((c ^ (h & 7)) << 4));
            const __half2 *q2 = reinterpret_cast<const __half2 *>(&qv);
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 x = __half22float2(q2[e]), y = __half22float2(k2[e]);
              a = fmaf(x.x, y.x, fmaf(x.y, y.y, a));
            }
            if (j == 0) acc0 += a; else acc1 += a;
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&ms.empty[pq]));
        mbar_arrive(smem_u32(&ms.xdone[b]));
      }
    }
    if (!ok) break;
    if (g.extra) {
      ok = mbar_wait(smem_u32(&ms.x_empty[n & 1]), ((n >> 1) & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_PR_X_EMPTY);
      if (!ok) break;
#pragma unroll
      for (int i = 0; i < 2; ++i) *reinterpret_cast<uint4 *>(xb + 1024 + 16 * (lane + 32 * i)) = vr[i];
    }
    // The next pair's rows travel while this pair finishes.
    if (pr + (int)gridDim.x < n_pairs) load_extra_row(p, pair_geom(p, pr + gridDim.x), lane, kr, vr);
    ms.sx[n & 1][lane] = acc0 * p.scale_log2;
    ms.sx[n & 1][lane + 32] = acc1 * p.scale_log2;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ms.x_full[n & 1]));
  }
}

__global__ void __launch_bounds__(kPThreads, 1) attn_pair_kernel(const __grid_constant__ PairParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  PairMisc &ms = *reinterpret_cast<PairMisc *>(smem + kPOffMisc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPSlots; ++s) {
      mbar_init(smem_u32(&ms.full[s]), 1);
      mbar_init(smem_u32(&ms.empty[s]), 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ms.s_full[b]), 1);
      mbar_init(smem_u32(&ms.s_empty[b]), kPThreadsC);
      mbar_init(smem_u32(&ms.o_full[b]), 1);
      mbar_init(smem_u32(&ms.o_empty[b]), kPThreadsC);
      mbar_init(smem_u32(&ms.x_full[b]), 1);
      mbar_init(smem_u32(&ms.x_empty[b]), 1);
    }
    mbar_init(smem_u32(&ms.p_full), kPThreadsC);
    mbar_init(smem_u32(&ms.p_empty), 1);
    mbar_init(smem_u32(&ms.mma_done), 1);
    for (int b = 0; b < 8; ++b) {
      mbar_init(smem_u32(&ms.qx[b]), 1);
      mbar_init(smem_u32(&ms.xdone[b]), 1);
    }
    ms.abort_flag = 0;
    for (int i = 0; i < 64; ++i) ms.px[i] = 0.f;
    fence_barrier_init();
  }
  if (warp == kPMmaWarp) {
    tmem_alloc(smem_u32(&ms.tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == kPLoaderWarp && lane == 0) {
    tma_prefetch_desc(&p.tm_q2);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  grid_launch_dependents();
  if (warp < kPWarps) {
    pair_compute(p, smem, tmem, ms, threadIdx.x);
  } else if (warp == kPLoaderWarp) {
    if (lane == 0) pair_loader(p, sbase, ms);
    __syncwarp();
  } else if (warp == kPMmaWarp) {
    if (lane == 0) pair_mma(p, sbase, tmem, ms);
    __syncwarp();
  } else {
    pair_extra_row(p, smem, ms, lane);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kPMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t prepare_pair_kernel() {
  return cudaFuncSetAttribute(attn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmemBytes);
}

cudaError_t launch_pair(const PairParams &p, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_pair_kernel, p);
}

}  // namespace ds4a
