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
// products run as N = 128 MMAs at the tensor core's full rate, with the
// pair's 128 query rows (two tokens x 64 heads) on the M side:
//   S[128 q][128 rows]      = Q_pair[128][512] . K_tile[128][512]^T        (K-major A and B, shared memory)
//   O_m[128 q][128 dims]    = P[128 q][128 rows] . V_tile[rows][dims 128m..] (A = P in tensor memory, MN-major B)
// A query row lives in one TMEM lane, so its softmax needs no exchange
// between threads: the thread that owns the lane reads the row's 128 scores,
// writes the row of P (fp16, two per 32-bit column) over the first 64
// columns of the same S buffer, and PV takes P from there as its A operand.
// TMEM: two S buffers (columns 0-127 and 128-255, by pair parity; a buffer is
// free again once the pair's PV has read its P) and two 128-column O buffers
// (256-383 and 384-511) through which the four 128-dim blocks of a pair's O
// pass, drained by the epilogue as they complete; no block accumulates across
// tiles (the pair has one tile).  With two S buffers the QK^T of the next
// pair runs while the softmax reads this one.
//
// Shared memory: a ring of 10 slots of 16 KB through which every box streams
// in the order the MMAs take them: the Q and K boxes of pair 0, then for each
// pair n the Q and K boxes of pair n+1 (Q box b, K box b for b = 0..7) before
// the V boxes of pair n (0..7; a PV block takes two adjacent V slots), so the
// next pair's loads are not queued behind V boxes that wait for this pair's
// softmax.  Also the extra row's K and V (two 2 KB buffers, by pair parity)
// and bookkeeping; P needs no shared memory.  (12 slots ran no faster.)
//
// Measured against the earlier form of this kernel (S^T with the rows on the
// lanes, the softmax reducing over lanes and warps, P^T in shared memory, the
// eight compute warps doing softmax and epilogue in turn): 66.7 -> 64.0 us for
// the 2048-token chunk.  The output stores are what remains: without them
// the same kernel takes 57.5 us.  Each epilogue thread owns a (token, head)
// row of o, so a warp's store touches 32 rows; 32-byte stores
// (st.global.v8) halve the transactions of 16-byte ones (72.0 us), and
// staging the rows in shared memory for TMA stores cost more than it saved
// (66.9-69.3 us: the staging writes, proxy fences and barriers).
// Warp roles (352 threads):
//   warps 0-3  softmax: thread 32w + l owns query row r = 32w + l (token r / 64,
//              head r % 64) in TMEM lane r
//   warps 4-7  epilogue: thread 32(w-4) + l drains row r of each O block
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

constexpr int kPSoftWarps = 4;    // warps 0-3
constexpr int kPEpiWarp0 = 4;     // warps 4-7
constexpr int kPRowThreads = 128;  // one thread per query row in each of the two roles
constexpr int kPLoaderWarp = 8;
constexpr int kPMmaWarp = 9;
constexpr int kPXWarp = 10;
constexpr int kPThreads = 32 * (kPXWarp + 1);
constexpr int kPSlots = 10;
constexpr uint32_t kPSlot = 16384;
constexpr int kPSlotsPerPair = 24;  // 8 Q + 8 K + 8 V boxes
constexpr uint32_t kPOffRing = 0;
constexpr uint32_t kPOffX = kPSlots * kPSlot;  // extra rows by pair parity: K [512] fp16, then V [512]
constexpr uint32_t kPOffMisc = kPOffX + 2 * 2048;
static_assert(kPSlots % 2 == 0 && kPSlotsPerPair % 2 == 0, "V slot pairs must stay adjacent in the ring");

struct PairMisc {
  alignas(16) float inv_l[2][128];  // by pair parity: 1 / row sum of each query row (0 when nothing is visible)
  alignas(16) float px[2][64];      // by pair parity: token a's extra-row weight per head
  alignas(16) float sx[2][64];      // extra row, by pair parity: scaled score of token a per head (log2 units)
  alignas(8) uint64_t full[kPSlots], empty[kPSlots];
  uint64_t s_full[2], s_empty[2], p_full[2], o_full[2], o_empty[2], mma_done;  // p_full by pair parity
  uint64_t x_full[2], x_empty[2];  // by pair parity: extra-row scores ready; the row buffer free again
  uint64_t st_full[2], st_empty[2];  // by pair parity: inv_l / px written; read by the epilogue
  uint64_t qx[8];                 // Q box b of the current pair has landed (passed on by the MMA thread)
  uint64_t xdone[8];              // the extra-row warp is done with Q box b of its current pair
  uint32_t tmem_base;
  int abort_flag;
};
constexpr uint32_t kPSmemBytes = kPOffMisc + ((sizeof(PairMisc) + 127) / 128) * 128 + 1024;
static_assert(kPSmemBytes <= 232448, "pair kernel shared memory");

enum : unsigned int {
  SITE_PR_EMPTY = 0x20, SITE_PR_FULL, SITE_PR_S_EMPTY, SITE_PR_S_FULL, SITE_PR_P_FULL,
  SITE_PR_P_EMPTY,  // (no longer waited on: P lives in its S buffer)
  SITE_PR_O_EMPTY, SITE_PR_O_FULL, SITE_PR_DRAIN, SITE_PR_X_FULL, SITE_PR_X_EMPTY, SITE_PR_ST_FULL,
  SITE_PR_ST_EMPTY
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
// TMEM columns: S (then P) of pair parity i at 128 i; O block m in buffer m & 1 at 256 + 128 (m & 1).
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

// D(tmem) (+)= A(tmem) * B(smem desc)^T: A in tensor memory, row i of A in
// lane i of the 128 lanes, K packed along the 32-bit columns (two fp16 values
// per column, the lower K index in the low half).
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// QK^T of the CTA's pair j into S buffer j & 1 (query rows on the lanes), from
// the pair's 16 Q and K slots starting at `sl`.  The buffer is free once the
// PV of pair j - 2 has read the P written over it.
__device__ __forceinline__ bool pair_qk(const PairParams &p, uint32_t sbase, uint32_t tmem, PairMisc &ms,
                                        volatile int *abrt, uint32_t j, uint32_t &sl) {
  constexpr uint32_t kIdescQK = idesc_f16_f32(128, 128, false, false);
  // Q and K boxes: K-major, SBO = one 8-row group.
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
    const uint64_t a0 = sdesc_add(kq_desc, pq * kPSlot), b0 = sdesc_add(kq_desc, pk * kPSlot);
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

// PV of the CTA's pair n once P is written over its S buffer: O block m into
// buffer m & 1 (after the epilogue drained block m - 2), from the V slots
// starting at `sl`; then the S buffer is free for pair n + 2.
__device__ __forceinline__ bool pair_pv(const PairParams &p, uint32_t sbase, uint32_t tmem, PairMisc &ms,
                                        volatile int *abrt, uint32_t n, uint32_t &sl) {
  constexpr uint32_t kIdescPV = idesc_f16_f32(128, 128, false, true);
  // V: MN-major B (dims contiguous), its two 64-dim atoms in adjacent slots
  // (LBO = one slot), 16 rows of K per MMA = two 8-row groups of 1024 bytes.
  const uint64_t v_desc = sdesc_sw128(sbase + kPOffRing, kPSlot, 1024);
  const uint32_t p_tmem = tmem + s_column(n);  // P: 64 columns, 8 per 16 rows of K
  // By pair parity: the softmax of pair n + 1 may finish before this wait.
  if (!mbar_wait(smem_u32(&ms.p_full[n & 1]), (n >> 1) & 1, abrt, p.timeout_ns, p.err, SITE_PR_P_FULL)) return false;
  tc_fence_after();
  for (int m = 0; m < 4; ++m, sl += 2) {
    const uint32_t gb = 4 * n + m, buf = gb & 1;
    const uint32_t pa = sl % kPSlots, pb = (sl + 1) % kPSlots;  // pa even: pb = pa + 1
    if (!mbar_wait(smem_u32(&ms.o_empty[buf]), ((gb >> 1) & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_PR_O_EMPTY) ||
        !mbar_wait(smem_u32(&ms.full[pa]), slot_phase(sl), abrt, p.timeout_ns, p.err, SITE_PR_FULL) ||
        !mbar_wait(smem_u32(&ms.full[pb]), slot_phase(sl + 1), abrt, p.timeout_ns, p.err, SITE_PR_FULL))
      return false;
    tc_fence_after();
    const uint64_t b0 = sdesc_add(v_desc, pa * kPSlot);
    const uint32_t d = tmem + o_column(m);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) umma_f16_ts(d, p_tmem + 8 * ks, sdesc_add(b0, ks * 2048), kIdescPV, ks > 0);
    umma_commit(smem_u32(&ms.empty[pa]));
    umma_commit(smem_u32(&ms.empty[pb]));
    mbar_arrive(smem_u32(&ms.empty[pa]));
    mbar_arrive(smem_u32(&ms.empty[pb]));
    umma_commit(smem_u32(&ms.o_full[buf]));
  }
  umma_commit(smem_u32(&ms.s_empty[n & 1]));
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

// The visible columns [c0, c1) of a query row of token tau in the pair's tile.
__device__ __forceinline__ void visible_columns(const PairGeom &g, int tau, int &c0, int &c1) {
  if (tau == 1 && !g.has_b) {
    c0 = c1 = 0;
    return;
  }
  c0 = max(g.lo[tau] - g.tile_lo, 0);
  c1 = min(g.hi[tau] - g.tile_lo, 128);
  if (c1 < c0) c1 = c0;
}

// Warps 0-3: thread r owns query row r (token tau = r / 64, head h = r % 64)
// in TMEM lane r.  Pass 1 takes the row's maximum over its visible scores
// (and token a's extra-row score), pass 2 writes P = 2^(s - m) in fp16 over
// the first 64 columns of the S buffer (columns 32u .. 32u+31 hold rows
// 64u .. 64u+63 of the tile, two per column) and sums the same fp16 values.
// A thread rewrites only its own lane, and only columns it has already read.
__device__ __forceinline__ void pair_softmax(const PairParams &p, uint32_t tmem, PairMisc &ms, int r) {
  volatile int *abrt = &ms.abort_flag;
  const int tau = r >> 6, h = r & 63;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
  const int n_pairs = (p.T + 1) / 2;
  uint32_t n = 0;
  grid_dependency_wait();  // lse may still be read by the previous kernel
  for (int pr = blockIdx.x; pr < n_pairs; pr += gridDim.x, ++n) {
    const PairGeom g = pair_geom(p, pr);
    int c0, c1;
    visible_columns(g, tau, c0, c1);
    const bool with_x = tau == 0 && g.extra;
    // The extra-row warp's scores of this pair (every pair, so the phases
    // stay in step), then the pair's S.
    // (Decisions to leave are made per warp: the TMEM accesses below are
    // warp-collective.)
    const bool ready =
        mbar_wait(smem_u32(&ms.x_full[n & 1]), (n >> 1) & 1, abrt, p.timeout_ns, p.err, SITE_PR_X_FULL) &&
        mbar_wait(smem_u32(&ms.s_full[n & 1]), (n >> 1) & 1, abrt, p.timeout_ns, p.err, SITE_PR_S_FULL);
    if (!__all_sync(0xffffffffu, ready)) break;
    tc_fence_after();
    const uint32_t sb = tmem + s_column(n) + lane_base;
    const float sxv = with_x ? ms.sx[n & 1][h] : -INFINITY;
    float mx = sxv;
#pragma unroll 1
    for (int u = 0; u < 2; ++u) {
      float s[64];
      tmem_ld64(sb + 64 * u, s);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const int col = 64 * u + c;
        if (col >= c0 && col < c1) mx = fmaxf(mx, s[c] * p.scale_log2);
      }
    }
    const float mu = mx == -INFINITY ? 0.f : mx;
    float lsum = 0.f;
#pragma unroll 1
    for (int u = 0; u < 2; ++u) {
      float s[64];
      tmem_ld64(sb + 64 * u, s);
      tmem_wait_ld();
      float pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int col = 64 * u + 2 * i;
        const float e0 = (col >= c0 && col < c1) ? exp2f(s[2 * i] * p.scale_log2 - mu) : 0.f;
        const float e1 = (col + 1 >= c0 && col + 1 < c1) ? exp2f(s[2 * i + 1] * p.scale_log2 - mu) : 0.f;
        const __half2 hp = __floats2half2_rn(e0, e1);
        const float2 f = __half22float2(hp);
        lsum += f.x + f.y;
        pk[i] = __uint_as_float(*reinterpret_cast<const uint32_t *>(&hp));
      }
      tmem_st32(sb + 32 * u, pk);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(smem_u32(&ms.p_full[n & 1]));
    float px = 0.f;
    if (with_x) {
      px = exp2f(sxv - mu);
      lsum += px;
    }
    // Row statistics for the epilogue, once it is done with this parity's
    // previous pair.
    const bool free_st =
        mbar_wait(smem_u32(&ms.st_empty[n & 1]), ((n >> 1) & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_PR_ST_EMPTY);
    if (!__all_sync(0xffffffffu, free_st)) break;
    ms.inv_l[n & 1][r] = lsum > 0.f ? 1.f / lsum : 0.f;
    if (tau == 0) ms.px[n & 1][h] = px;
    mbar_arrive(smem_u32(&ms.st_full[n & 1]));
    if (p.lse != nullptr && (tau == 0 || g.has_b))
      p.lse[(long long)(g.ta + tau) * kH + h] = lsum > 0.f ? (mx + log2f(lsum)) * kLn2 : -INFINITY;
  }
}

// 32 bytes to global memory (the address 32-byte aligned).
__device__ __forceinline__ void stg_v8(void *p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Warps 4-7: thread r drains query row r of each O block [128 q][128 dims]
// as the PV completes it, scales it by 1 / l (adding token a's extra row,
// weight px times the V row) and writes the block's 128 dims (256 bytes) of
// its (token, head) row of o, 32 bytes per store when o allows it.
__device__ __forceinline__ void pair_epilogue(const PairParams &p, uint8_t *smem, uint32_t tmem, PairMisc &ms,
                                              int r) {
  volatile int *abrt = &ms.abort_flag;
  const int tau = r >> 6, h = r & 63;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
  const int n_pairs = (p.T + 1) / 2;
  uint32_t n = 0;
  grid_dependency_wait();  // the outputs may still be read by the previous kernel
  for (int pr = blockIdx.x; pr < n_pairs; pr += gridDim.x, ++n) {
    const PairGeom g = pair_geom(p, pr);
    const bool has_tok = tau == 0 || g.has_b;
    const bool with_x = tau == 0 && g.extra;
    const __half *vx = reinterpret_cast<const __half *>(smem + kPOffX + 2048 * (n & 1)) + 512;
    const bool ready =
        mbar_wait(smem_u32(&ms.st_full[n & 1]), (n >> 1) & 1, abrt, p.timeout_ns, p.err, SITE_PR_ST_FULL);
    if (!__all_sync(0xffffffffu, ready)) break;  // per warp: the TMEM loads are warp-collective
    const float il = ms.inv_l[n & 1][r];
    const float px = with_x ? ms.px[n & 1][h] : 0.f;
    __half *orow = p.o + (long long)(g.ta + tau) * p.o_tok_stride + (long long)h * kD;
    bool bad = false;
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
      const uint32_t gb = 4 * n + m;
      const bool done =
          mbar_wait(smem_u32(&ms.o_full[m & 1]), (gb >> 1) & 1, abrt, p.timeout_ns, p.err, SITE_PR_O_FULL);
      if (!__all_sync(0xffffffffu, done)) {
        bad = true;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int u = 0; u < 2; ++u) {
        float o[64];
        tmem_ld64(tmem + o_column(m) + 64 * u + lane_base, o);
        tmem_wait_ld();
        if (u == 1) {
          tc_fence_before();
          mbar_arrive(smem_u32(&ms.o_empty[m & 1]));  // the buffer may take block m + 2
        }
        if (!has_tok) continue;
        const int d0 = 128 * m + 64 * u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int e = 16 * c + 2 * i;
            float a = o[e], b = o[e + 1];
            if (with_x) {
              const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(vx + d0 + e));
              a = fmaf(px, v.x, a);
              b = fmaf(px, v.y, b);
            }
            const __half2 hv = __floats2half2_rn(a * il, b * il);
            w8[i] = *reinterpret_cast<const uint32_t *>(&hv);
          }
          __half *dst = orow + d0 + 16 * c;
          if (p.o_v8) {
            stg_v8(dst, w8);
          } else {
            reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
            reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
          }
        }
      }
    }
    if (bad) break;
    mbar_arrive(smem_u32(&ms.st_empty[n & 1]));
    mbar_arrive(smem_u32(&ms.x_empty[n & 1]));  // done with this parity's extra V row
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
      mbar_init(smem_u32(&ms.s_empty[b]), 1);
      mbar_init(smem_u32(&ms.o_full[b]), 1);
      mbar_init(smem_u32(&ms.o_empty[b]), kPRowThreads);
      mbar_init(smem_u32(&ms.x_full[b]), 1);
      mbar_init(smem_u32(&ms.x_empty[b]), kPRowThreads);
      mbar_init(smem_u32(&ms.st_full[b]), kPRowThreads);
      mbar_init(smem_u32(&ms.st_empty[b]), kPRowThreads);
    }
    for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&ms.p_full[b]), kPRowThreads);
    mbar_init(smem_u32(&ms.mma_done), 1);
    for (int b = 0; b < 8; ++b) {
      mbar_init(smem_u32(&ms.qx[b]), 1);
      mbar_init(smem_u32(&ms.xdone[b]), 1);
    }
    ms.abort_flag = 0;
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
  if (warp < kPSoftWarps) {
    pair_softmax(p, tmem, ms, threadIdx.x);
  } else if (warp < kPEpiWarp0 + 4) {
    pair_epilogue(p, smem, tmem, ms, threadIdx.x - 32 * kPEpiWarp0);
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
