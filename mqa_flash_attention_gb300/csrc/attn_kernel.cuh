// Fused multi-query attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes: for every query token t and head h,
//   o[t][h] = sum_j softmax_j(scale * q[t][h].k_j + bias_j) v_j
// over the rows the token may see (ds4 page "DwarfStar 4 (DS4) - DeepSeek V4
// Flash Inference Engine", sections "Fixed Model Shape" and "Layer
// Compression"; fused as in "How DeepSeek V4 Flash Model Inference Works on
// Apple Silicon with Metal Backend", section "FlashAttention Kernel
// Architecture").
//
// Orientation.  The 64 heads share one K/V row, so a token's scores against a
// 128-row K tile form a 128 x 64 product.  The kernel keeps the KV rows on the
// M side of every MMA, so each instruction is a full M = 128 tcgen05 tile:
//   S^T[128 rows][64 heads]  = K_tile[128][512] . Q_t[64][512]^T   (K-major A, K-major B)
//   O^T[512 dims][64 heads] += V_tile^T[512][128] . P^T[64][128]^T (MN-major A, MN-major B)
// TMEM holds O^T (4 x 64 columns, fp32) and two S^T buffers (64 columns each):
// 384 of the 512 columns.  Lane r of TMEM is KV row r (for S) or dim r of a
// 128-dim slice (for O).  The softmax is over TMEM lanes, i.e. across threads:
// a warp reduce-scatter gives each lane two heads, a 4-warp exchange in shared
// memory finishes the per-head max.
//
// Rows are loaded by TMA at the exact row where a token's window starts (a
// tile need not be 32-row aligned), so a raw-only token issues exactly its 128
// window rows.  The pages' 32-row block skip is kept for dense masks, where the
// caller's status bytes decide which 128-row tiles are loaded at all.
//
// Online softmax with a lazy reference: the running reference max of a head
// moves only when a tile's max exceeds it by more than 2^8 (kTau in log2
// units); then O^T and the partial sums are rescaled.  Values of P stay below
// 2^8 and are stored as fp16, and the row sums add the same fp16 values, so
// o = sum(p v) / sum(p) is an exact convex combination up to fp32 rounding.
//
// Warp roles (512 threads, one CTA per SM, persistent over work items):
//   warps 0-7   softmax + epilogue: warp w owns TMEM lane quarter w % 4 (32
//               KV rows or dims) and heads 32*(w/4) .. +31
//   warps 8-14  loaders: Q once per item, every K/V stage in ring order (TMA
//               tiles, or 16-byte cp.async gathers of index-listed rows by
//               all seven warps: a TMA gather moves only 512 bytes per
//               instruction); in a CTA with a single item warps 9-14 copy its
//               Q.  With E4M3 rows (the FP8 instantiation) the codes of each
//               part land in the upper half of its stage and warps 9-12
//               convert them in place, one row per thread
//   epilogue    a whole token: o (fp16) and its log-sum-exp; a split of a
//               token: the split's own normalised o (fp16) and (m, l)
//   warp  15    TMEM allocator and tcgen05.mma issuer
// Each mbarrier is waited on only by a role that cannot fall more than one
// phase behind it, which a parity wait needs.
#pragma once

#include "attn_params.h"
#include "ptx.cuh"

namespace ds4a {

// ------------------------------------------------------------------ tile plan

struct Tile {
  int seg;    // 0 raw rows, 1 compressed rows, 2 compressed rows named by the index list
  int start;  // first row (seg 0/1) or first list slot (seg 2)
  int count;  // rows (or slots) of the tile that exist, <= 128
  int open;   // dense mask: every covered block has status 2 (visible, zero bias)
};

struct TokenTiles {
  int t, pos;
  int raw_lo, raw_hi;  // raw rows [raw_lo, raw_hi)
  int comp_rows;       // compressed rows (seg 1) or list slots (seg 2)
  int n_rt, n_ct;      // raw / compressed tile candidates
};

__device__ __forceinline__ TokenTiles token_tiles(const AttnParams &p, int t) {
  TokenTiles z;
  z.t = t;
  int pos = p.q_pos0 + t, n_raw = p.n_raw, raw_pos0 = p.raw_pos0, n_comp = p.n_comp;
  if (p.batch_geom != nullptr) {
    // Batched decode: token t is sequence t, with its own position and row
    // counts (clamped to the rows its K/V tensors hold).
    const int4 g = __ldg(p.batch_geom + t);
    pos = max(g.x, 0);
    n_raw = min(max(g.y, 0), p.n_raw);
    raw_pos0 = max(g.z, 0);
    n_comp = min(max(g.w, 0), p.n_comp);
  }
  z.pos = pos;
  if (p.mode == MODE_MASK) {
    z.raw_lo = 0;
    z.raw_hi = n_raw;
    z.comp_rows = n_comp;
  } else {
    // Raw row i sits at raw_pos0 + i; the window is pos - window + 1 .. pos.
    const long long a = (long long)pos - p.window + 1 - raw_pos0;
    const long long b = (long long)pos + 1 - raw_pos0;
    long long lo = a < 0 ? 0 : a;
    long long hi = b > n_raw ? n_raw : b;
    if (hi < lo) hi = lo;
    z.raw_lo = (int)lo;
    z.raw_hi = (int)hi;
    if (p.mode == MODE_INDEXED) {
      z.comp_rows = n_comp > 0 ? p.top_k : 0;
    } else {
      // Compressed row c is pooled from positions c*ratio .. (c+1)*ratio-1.
      const long long c = n_comp > 0 ? ((long long)pos + 1) / p.ratio : 0;
      z.comp_rows = (int)(c < n_comp ? c : n_comp);
    }
  }
  z.n_rt = (z.raw_hi - z.raw_lo + p.tile_rows - 1) / p.tile_rows;
  z.n_ct = (z.comp_rows + p.tile_rows - 1) / p.tile_rows;
  return z;
}

__device__ __forceinline__ Tile tile_candidate(const AttnParams &p, const TokenTiles &z, int i, bool &skip) {
  Tile tl;
  skip = false;
  tl.open = 0;
  if (i < z.n_rt) {
    tl.seg = 0;
    tl.start = z.raw_lo + i * p.tile_rows;
    tl.count = min(p.tile_rows, z.raw_hi - tl.start);
  } else {
    tl.seg = p.mode == MODE_INDEXED ? 2 : 1;
    tl.start = (i - z.n_rt) * p.tile_rows;
    tl.count = min(p.tile_rows, z.comp_rows - tl.start);
  }
  if (p.mode == MODE_MASK && p.status != nullptr) {
    const int base = tl.seg == 0 ? 0 : p.nbr;
    const int b0 = base + tl.start / 32;
    const int b1 = base + (tl.start + tl.count - 1) / 32;
    const uint8_t *srow = p.status + (long long)(z.t / p.q_tile) * p.n_blocks;
    bool all0 = true, all2 = true;
    for (int b = b0; b <= b1; ++b) {
      const uint8_t s = srow[b];
      all0 = all0 && s == 0;
      all2 = all2 && s == 2;
    }
    skip = all0;
    tl.open = all2 ? 1 : 0;
  }
  return tl;
}

__device__ __forceinline__ int count_tiles(const AttnParams &p, const TokenTiles &z) {
  const int n = z.n_rt + z.n_ct;
  if (p.mode != MODE_MASK || p.status == nullptr) return n;
  int c = 0;
  for (int i = 0; i < n; ++i) {
    bool skip;
    tile_candidate(p, z, i, skip);
    c += skip ? 0 : 1;
  }
  return c;
}


// A tile's parts arrive as E4M3 codes (compressed rows; raw rows too when
// they are E4M3) or as fp16 boxes.  Used by the FP8 instantiation only.
__device__ __forceinline__ bool tile_codes(const AttnParams &p, const Tile &tl) {
  return tl.seg == 0 ? p.raw_fp8 != 0 : true;
}

struct TileCursor {
  TokenTiles z;
  int cand;
  __device__ __forceinline__ Tile next(const AttnParams &p) {
    const int n = z.n_rt + z.n_ct;
    while (cand < n) {
      bool skip;
      Tile tl = tile_candidate(p, z, cand++, skip);
      if (!skip) return tl;
    }
    Tile none{0, 0, 0, 0};
    return none;
  }
};

// The plan of an item reads memory the caller (or the previous kernel in the
// stream) wrote: status bytes in dense-mask mode, the per-sequence geometry in
// batched decode.  Roles then wait for the previous grid before planning.
__device__ __forceinline__ bool plan_reads_inputs(const AttnParams &p) {
  return (p.mode == MODE_MASK && p.status != nullptr) || p.batch_geom != nullptr;
}

// Work item -> token, tile range [j0, j1) and a cursor positioned at j0.
struct ItemPlan {
  int t, j0, j1;
  TileCursor cur;
};

__device__ __forceinline__ ItemPlan plan_item(const AttnParams &p, int item) {
  ItemPlan ip;
  ip.t = item / p.n_splits;
  const int sp = item - ip.t * p.n_splits;
  ip.cur.z = token_tiles(p, ip.t);
  ip.cur.cand = 0;
  const int n = count_tiles(p, ip.cur.z);
  ip.j0 = (int)(((long long)sp * n) / p.n_splits);
  ip.j1 = (int)(((long long)(sp + 1) * n) / p.n_splits);
  if (p.mode == MODE_MASK && p.status != nullptr) {
    for (int j = 0; j < ip.j0; ++j) ip.cur.next(p);  // skipped blocks: walk the candidates
  } else {
    ip.cur.cand = ip.j0;  // every candidate is a tile: jump straight to the split's first
  }
  return ip;
}

// ------------------------------------------------------------------ warp reductions

// Lane l ends with the max (or sum) over the warp's 32 rows of head l of the
// 32 heads held in s[0..31].
template <bool kMax>
__device__ __forceinline__ float warp_reduce_scatter32(const float (&s)[32], int lane) {
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
  for (int c = 16; c >= 2; c >>= 1) {  // 16 -> 8 -> 4 -> 2 -> 1 values, xor 8, 4, 2, 1
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

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Ring position bookkeeping shared by every role.
struct Ring {
  uint32_t st = 0, ph = 0;
  __device__ __forceinline__ void advance() {
    if (++st == kStages) {
      st = 0;
      ph ^= 1;
    }
  }
};

// ------------------------------------------------------------------ loaders

// Ring order of an item's parts (the kernel's LA parameter).  With look-ahead
// the K parts of the next tile come before the V parts of this one, so the
// next QK^T runs while the softmax works on this tile and the ring keeps
// loading meanwhile: K(0), then K(j+1) and V(j) for each tile j.  Without it
// each tile's parts come together (always when parts are held from QK^T until
// PV: K = V rows, paired stages).  Measured (one GB300): look-ahead takes the
// indexed r4 prefill chunk from 366 to 332 us, the E4M3 256K decode from 102
// to 98 us and, with the sixteen-warp layout, the fp16 split-KV decodes too
// (65,536 rows 33.8 -> 32.2 us, 64 batched sequences 22.9 -> 21.8 us), but
// slows the E4M3 prefill (106 -> 117 us), so it is a separate instantiation
// chosen per call (launch_attn), which leaves the code of the others as it
// was: split-KV decode and indexed calls.
__host__ __device__ __forceinline__ bool look_ahead_suits(const AttnParams &p) {
  return !p.alias_kv && !p.kv_pair && (p.mode == MODE_INDEXED || p.partial);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Arrive on `bar` when every cp.async this thread issued so far has completed;
// the arrival counts toward the barrier's expected count (.noinc).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Q through the load/store path, for a CTA with a single work item (a short
// decode: Q's latency is then paid once, at the head of the chain).  Loader
// warps 9-14 copy the item's Q while thread 0 issues the K/V tiles, so Q does
// not queue in front of them on the SM's TMA engine: 8.8 -> 8.5 us for a
// 384-row decode split over 3 CTAs.  (In a long prefill, where each CTA runs
// many items, it made no difference: there every TMA load takes ~2.7 us under
// load whatever is queued with it.)  4096 chunks of 16 bytes: chunk (head h,
// 16-byte column c of the 1024-byte head row) lands in box c/8 at row h,
// column (c%8) ^ (h%8) (the 128-byte swizzle TMA applies).  Each thread's
// copies arrive on q_full by themselves when they land.
constexpr int kQCopyThreads = kLoaderThreads - 32;
constexpr int kConvThreads = kTile;  // E4M3 converters: one row of a part per thread (warps 9-12)

// Loader threads that gather index-listed rows: all of them, or with E4M3
// rows (where warps 9-12 convert) warps 8, 13 and 14.  The barrier the
// gathered copies complete (kv_full in the fp16 kernel, code_full in the
// E4M3 one) then counts one arrival per gathering thread.
template <bool FP8>
__host__ __device__ constexpr int gather_threads() { return FP8 ? kLoaderThreads - kConvThreads : kLoaderThreads; }
template <bool FP8>
__device__ __forceinline__ uint32_t stage_fill_count(const AttnParams &p) {
  return (p.mode == MODE_INDEXED && p.n_comp > 0) ? (uint32_t)gather_threads<FP8>() : 1u;
}

__device__ __forceinline__ bool q_by_lsu(const AttnParams &p, bool fp8) {
  return !fp8 && !(p.mode == MODE_INDEXED && p.n_comp > 0) && p.q_ptr != nullptr &&
         (long long)p.T * p.n_splits <= (long long)gridDim.x;
}

__device__ __noinline__ void q_copy_role(const AttnParams &p, uint32_t sbase, Misc &ms, int qtid) {
  volatile int *abrt = &ms.abort_flag;
  const uint32_t b_q_full = smem_u32(&ms.q_full), b_q_empty = smem_u32(&ms.q_empty);
  const int n_items = p.T * p.n_splits;
  const bool plan_reads_status = plan_reads_inputs(p);
  if (plan_reads_status) grid_dependency_wait();
  uint32_t n_item = 0;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const ItemPlan ip = plan_item(p, item);
    if (ip.j1 == ip.j0) continue;
    if (n_item == 0 && !plan_reads_status) grid_dependency_wait();
    if (!mbar_wait(b_q_empty, (n_item & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_Q_EMPTY)) break;
    const uint8_t *q = p.q_ptr + (long long)ip.t * p.q_tok_bytes;
#pragma unroll 4
    for (int i = qtid; i < 4096; i += kQCopyThreads) {
      const int h = i >> 6, c = i & 63;
      cp_async16(sbase + kOffQ + (c >> 3) * kQBoxBytes + h * 128 + (((c & 7) ^ (h & 7)) << 4), q + 16 * i);
    }
    cp_async_arrive_noinc(b_q_full);
    ++n_item;
  }
  cp_async_wait<0>();  // no copy may still be landing at exit
}

// The loader warps fill Q (once per work item) and every K/V ring stage, in
// ring order.  Only fillers wait on a "stage free" barrier: a parity wait is
// unambiguous only for a waiter at most one phase behind, and a filler cannot
// fall behind a barrier that only advances after its own fills.
//
// TMA tiles: thread 0 issues one copy per 32 KB stage (the row maps' boxes
// span two 64-dim blocks), Q in one 64 KB copy.
// Gathered tiles (index-listed compressed rows): per stage (128 rows x 128
// dims) the loader threads copy 2048 chunks of 16 bytes: thread (row group
// rsub, column c8) copies column c8 of both 64-dim boxes of rows rsub,
// rsub + 28, rsub + 56, ... (224 threads: four or five rows each), so a
// warp instruction covers four rows x 128 contiguous bytes and each listed
// row's address is formed once per stage for two copies (forming it for
// every copy held the gather rate near 43 GB/s per SM: indexed attention
// 452 -> 366 us).  Chunk (row r, 16-byte column c of a
// 64-dim box) lands at column c ^ (r & 7): the 128-byte swizzle TMA applies, so
// the MMA reads gathered and TMA-loaded stages alike.  Each thread's copies
// arrive on the stage's barrier by themselves when they complete
// (cp.async.mbarrier.arrive.noinc), so no loader thread waits for its own
// copies and stages stay in flight up to the ring depth.  In this mode a
// stage barrier expects one arrival per loader thread (TMA stages: thread 0's
// arrive.expect_tx plus a plain arrival from every other thread).
template <bool FP8, bool LA>
__device__ __forceinline__ void loader_role(const AttnParams &p, uint32_t sbase, Misc &ms, int ltid) {
  volatile int *abrt = &ms.abort_flag;
  const bool group = p.mode == MODE_INDEXED && p.n_comp > 0;  // all loader threads needed
  const bool q_lsu = q_by_lsu(p, FP8);
  if (!group && ltid != 0) {
    if (q_lsu && ltid >= 32) q_copy_role(p, sbase, ms, ltid - 32);
    return;
  }
  const uint32_t b_q_full = smem_u32(&ms.q_full), b_q_empty = smem_u32(&ms.q_empty);
  Ring ring;
  uint32_t n_item = 0;
  uint32_t filled = 0, last_par = 0;  // TMA stages issued (thread 0), for draining on abort
  uint32_t code_ph = 0, cfilled = 0, clast_par = 0;  // E4M3 code copies: per-stage phase bits
  bool q_issued = false;
  uint32_t q_par = 0;
  bool ok = true;
  constexpr int kGroup = gather_threads<FP8>();
  const int gtid = (FP8 && ltid >= 32) ? ltid - kConvThreads : ltid;  // 0 .. kGroup-1 (warps 8, 13, 14 with E4M3)
  constexpr int kRowStep = kGroup / 8;  // rows copied per pass of the group
  const int c8 = gtid & 7;     // 16-byte column c8 of both 128-byte boxes of a stage's 256-byte row slice
  const int rsub = gtid >> 3;  // row within each group of kRowStep
  const uint8_t *kbase = reinterpret_cast<const uint8_t *>(p.k_comp);
  const uint8_t *vbase = reinterpret_cast<const uint8_t *>(p.v_comp);

  const int n_items = p.T * p.n_splits;
  const bool plan_reads_status = plan_reads_inputs(p);
  if (plan_reads_status) grid_dependency_wait();  // the plan reads status bytes or sequence geometry
  for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
    ItemPlan ip = plan_item(p, item);
    if (ip.j1 == ip.j0) continue;
    if (n_item == 0 && !plan_reads_status) grid_dependency_wait();  // first global read follows
    bool bad = false;
    if (ltid == 0 && !q_lsu) bad = !mbar_wait(b_q_empty, (n_item & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_Q_EMPTY);
    if (group) bad = bar_red_or(2, kGroup, bad);
    if (bad) {
      ok = false;
      break;
    }
    if (ltid == 0 && !q_lsu) {
      mbar_arrive_expect_tx(b_q_full, kQBytes);
      tma_load_4d(sbase + kOffQ, &p.tm_q, b_q_full, 0, 0, ip.t, 0);  // the eight boxes in one copy
    }
    q_issued = !q_lsu;
    q_par = n_item & 1;
    // One K/V part of tile `tl` into the next ring stage (parts 0-3: K dims
    // 128*part, parts 4-7: V); gathered tiles read their rows from list `ib`.
    auto emit = [&](const Tile &tl, int part, int ib) -> bool {
      // Every thread waits for the slot itself (bounded); a thread that gives
      // up stops filling, and the group meets at the next tile's barrier.
      if (!mbar_wait(smem_u32(&ms.kv_empty[ring.st]), ring.ph ^ 1, abrt, p.timeout_ns, p.err, SITE_KV_EMPTY))
        return false;
      const uint32_t stage = sbase + kOffKV + ring.st * kStageBytes;
      const uint32_t b_full = smem_u32(&ms.kv_full[ring.st]);
      if (FP8 && tile_codes(p, tl)) {
        // E4M3 rows: the codes of this part (128 rows x 128 bytes) land in
        // the stage's upper half; the converter warps turn them into the
        // fp16 stage and arrive on kv_full.
        const uint32_t b_code = smem_u32(&ms.code_full[ring.st]);
        if (tl.seg == 2) {
          // Gathered E4M3 rows: thread (rsub, c8) copies codes 16 c8 .. +15 of
          // the part's 128 codes of its rows, into the dense [row][128 codes]
          // layout the TMA copy of a code box produces.
          const uint8_t *cbase = (part >= 4 ? vbase : kbase) + 128 * (part & 3) + 16 * c8;
#pragma unroll
          for (int it = 0; it < (kTile + kRowStep - 1) / kRowStep; ++it) {
            const int row = kRowStep * it + rsub;
            if (kTile % kRowStep != 0 && row >= kTile) break;
            cp_async16(stage + kBoxBytes + row * 128 + 16 * c8,
                       cbase + (long long)ms.idx_s[ib][row] * p.comp_row_stride);
          }
          cp_async_arrive_noinc(b_code);
        } else if (ltid == 0) {
          mbar_arrive_expect_tx(b_code, kBoxBytes);
          tma_load_2d(stage + kBoxBytes, part >= 4 ? &p.tm_v8[tl.seg] : &p.tm_k8[tl.seg], b_code, 128 * (part & 3),
                      tl.start);
          cfilled |= 1u << ring.st;
          clast_par = (clast_par & ~(1u << ring.st)) | (((code_ph >> ring.st) & 1u) << ring.st);
          code_ph ^= 1u << ring.st;
        } else {
          mbar_arrive(b_code);  // a gathering group: one arrival per thread
        }
      } else if (tl.seg != 2) {
        if (ltid == 0) {
          const int dim0 = 128 * (part & 3);
          const CUtensorMap *m = part >= 4 ? &p.tm_v[tl.seg] : &p.tm_k[tl.seg];
          mbar_arrive_expect_tx(b_full, kStageBytes);
          if (FP8) mbar_arrive_cnt(b_full, kConvThreads - 1);  // the stage counts the converter threads
          if (p.kv_pair) {
            // 64-row tile: the K and the V slice of dims dim0 .. dim0+127 in
            // one stage, four [64 rows][64 dims] boxes of 8 KB (two copies:
            // the maps' boxes span two 64-dim blocks).
            tma_load_3d(stage, &p.tm_k[tl.seg], b_full, 0, tl.start, dim0 / 64);
            tma_load_3d(stage + kBoxBytes, &p.tm_v[tl.seg], b_full, 0, tl.start, dim0 / 64);
          } else if (p.batch_geom != nullptr) {  // [sequences][rows][512]: the sequence is the third coordinate
            tma_load_3d(stage, m, b_full, dim0, tl.start, ip.t);
            tma_load_3d(stage + kBoxBytes, m, b_full, dim0 + 64, tl.start, ip.t);
          } else {
            tma_load_3d(stage, m, b_full, 0, tl.start, dim0 / 64);  // both 64-dim boxes of the part
          }
          filled |= 1u << ring.st;
          last_par = (last_par & ~(1u << ring.st)) | (ring.ph << ring.st);
        } else if (!FP8) {
          mbar_arrive(b_full);
        }
      } else {
        const uint8_t *base = (part >= 4 ? vbase : kbase) + 256 * (part & 3) + 16 * c8;
#pragma unroll
        for (int it = 0; it < (kTile + kRowStep - 1) / kRowStep; ++it) {
          const int row = kRowStep * it + rsub;
          if (kTile % kRowStep != 0 && row >= kTile) break;  // the last pass covers part of the rows
          const uint8_t *src = base + (long long)ms.idx_s[ib][row] * p.comp_row_stride;
          const uint32_t dst = stage + row * 128 + ((c8 ^ (row & 7)) << 4);
          cp_async16(dst, src);                    // dims 0-63 of the part: the first box
          cp_async16(dst + kBoxBytes, src + 128);  // dims 64-127: the second box
        }
        cp_async_arrive_noinc(b_full);
      }
      ring.advance();
      return true;
    };
    // The compressed rows a gathered tile lists, into list `ib`.  A list may
    // be rewritten once every thread has issued the copies of the tile that
    // used it last (a copy takes its address when it is issued).
    auto load_list = [&](const Tile &tl, int ib) {
      named_bar_sync(2, kGroup);
      const int32_t *lst = p.idx + (long long)ip.t * p.idx_stride;
      for (int k = gtid; k < 128; k += kGroup) {
        const int slot = tl.start + k;
        const int c = slot < p.top_k ? __ldg(lst + slot) : -1;
        ms.idx_s[ib][k] = (c >= 0 && c < p.n_comp) ? c : 0;  // empty slots load row 0, masked later
      }
      named_bar_sync(2, kGroup);
    };
    // With E4M3 rows the group is 96 threads and each reads two slots of a
    // list: there the slots are read into registers one tile ahead of their
    // use (fetch_list), so the reads' latency passes while the group copies
    // the tile before, and store_list writes them into the list (indexed
    // E4M3 chunk 457 -> 423 us).  The fp16 kernel keeps load_list: the same
    // read-ahead left its indexed time unchanged and, by its mere presence,
    // slowed its long decodes by 1-2%.
    auto fetch_list = [&](const Tile &tl, int (&v)[2]) {
      const int32_t *lst = p.idx + (long long)ip.t * p.idx_stride;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int k = gtid + u * kGroup, slot = tl.start + k;
        v[u] = (k < 128 && slot < p.top_k) ? __ldg(lst + slot) : -1;
      }
    };
    auto store_list = [&](const int (&v)[2], int ib) {
      named_bar_sync(2, kGroup);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int k = gtid + u * kGroup;
        if (k < 128) ms.idx_s[ib][k] = (v[u] >= 0 && v[u] < p.n_comp) ? v[u] : 0;  // empty slots: row 0, masked
      }
      named_bar_sync(2, kGroup);
    };
    static_assert(!FP8 || 2 * kGroup >= 128, "two list slots per thread cover a tile");
    // The tile after the cursor's position, without moving the cursor.
    auto peek = [&]() -> Tile {
      TileCursor c = ip.cur;
      return c.next(p);
    };
    const int nt = ip.j1 - ip.j0;
    int lv[2] = {-1, -1};  // (E4M3) list slots of the next gathered tile, read ahead
    Tile cur = ip.cur.next(p);
    if (cur.seg == 2) {
      if (FP8) {
        fetch_list(cur, lv);
        store_list(lv, 0);
      } else {
        load_list(cur, 0);
      }
    }
    if (FP8 && group && nt > 1) {
      const Tile t1 = peek();
      if (t1.seg == 2) fetch_list(t1, lv);
    }
    if (LA) {
      // Ring order: the K parts of tile 0, then for each tile the K parts of
      // the next tile before its own V parts (see mma_role).
      for (int part = 0; part < 4; ++part) ok = ok && emit(cur, part, 0);
      for (int jj = 0; jj < nt; ++jj) {
        if (group) ok = !bar_red_or(2, kGroup, !ok);  // uniform decision before the next list
        if (!ok) break;
        Tile nxt = cur;
        if (jj + 1 < nt) {
          nxt = ip.cur.next(p);
          if (nxt.seg == 2) {
            if (FP8)
              store_list(lv, (jj + 1) & 1);
            else
              load_list(nxt, (jj + 1) & 1);
          }
          if (FP8 && group && jj + 2 < nt) {
            const Tile t2 = peek();
            if (t2.seg == 2) fetch_list(t2, lv);
          }
          for (int part = 0; part < 4; ++part) ok = ok && emit(nxt, part, (jj + 1) & 1);
        }
        for (int part = 4; part < 8; ++part) ok = ok && emit(cur, part, jj & 1);
        cur = nxt;
      }
    } else {
      // K/V parts of a tile in ring order: 4 K parts then 4 V parts, or only
      // the 4 K parts when K and V are the same rows (see mma_role).
      const int n_parts = (p.alias_kv | p.kv_pair) ? 4 : 8;
      for (int jj = 0; jj < nt; ++jj) {
        if (jj > 0) {
          cur = ip.cur.next(p);
          if (cur.seg == 2) {
            if (FP8)
              store_list(lv, 0);
            else
              load_list(cur, 0);
          }
          if (FP8 && group && jj + 1 < nt) {
            const Tile t1 = peek();
            if (t1.seg == 2) fetch_list(t1, lv);
          }
        }
#pragma unroll 1
        for (int part = 0; part < n_parts; ++part) ok = ok && emit(cur, part, 0);
        if (group) ok = !bar_red_or(2, kGroup, !ok);  // uniform decision before the next list
        if (!ok) break;
      }
    }
    // Every group thread reaches this point (the loops above leave together),
    // so the last step's outcome is made uniform here too.
    if (group) ok = !bar_red_or(2, kGroup, !ok);
    ++n_item;
  }
  if (group) cp_async_wait<0>();  // no gathered copy may still be landing at exit
  if (!ok && ltid == 0) {
    // Let every TMA copy already issued land before the CTA's shared memory goes away.
    volatile int never = 0;
    for (int s = 0; s < kStages; ++s)
      if (filled & (1u << s))
        mbar_wait(smem_u32(&ms.kv_full[s]), (last_par >> s) & 1, &never, 100000000ull, p.err, SITE_DRAIN);
    if (q_issued) mbar_wait(b_q_full, q_par, &never, 100000000ull, p.err, SITE_DRAIN);
    for (int st = 0; st < kStages; ++st)
      if (cfilled & (1u << st))
        mbar_wait(smem_u32(&ms.code_full[st]), (clast_par >> st) & 1, &never, 100000000ull, p.err, SITE_DRAIN);
  }
}

// ------------------------------------------------------------------ E4M3 converters


// Warps 9..12 when K/V rows are E4M3 (one row of a part per thread): for each such K/V part,
// wait for its codes (upper half of the stage), then convert them (exactly)
// into the fp16 stage in the swizzled layout the TMA would have produced, and
// arrive on kv_full.  A thread converts whole rows: row r's fp16 values in the
// upper box overwrite only row r's own codes, which the thread has read
// first; chunks are visited in a per-thread rotated order (no bank
// conflicts).  The threads never wait for one another: each arrives on
// kv_full after its own row (a stage of the E4M3 kernel counts 128
// arrivals; an fp16 stage gets them from the loader thread at once), which
// made the 262,144-row E4M3 decode 78.8 -> 75.1 us against a barrier among the
// converters per part.  The same walk of items, tiles and parts as the
// loader, so both agree on stage and phase.
template <bool LA>
__device__ __forceinline__ void converter_role(const AttnParams &p, uint32_t sbase, Misc &ms, int ctid) {
  volatile int *abrt = &ms.abort_flag;
  Ring ring;
  uint32_t code_ph = 0;
  bool ok = true;
  const int n_items = p.T * p.n_splits;
  if (plan_reads_inputs(p)) grid_dependency_wait();
  for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
    ItemPlan ip = plan_item(p, item);
    if (ip.j1 == ip.j0) continue;
    // One part of tile `tl` in ring order: convert its codes if it has any.
    auto convert = [&](const Tile &tl, int part) -> bool {
      (void)part;
      if (tile_codes(p, tl)) {
        const uint32_t st = ring.st;
        bool w = mbar_wait(smem_u32(&ms.code_full[st]), (code_ph >> st) & 1u, abrt, p.timeout_ns, p.err,
                           SITE_KV_FULL);
        code_ph ^= 1u << st;
        if (!w) return false;
        const uint32_t stage = sbase + kOffKV + st * kStageBytes;
#pragma unroll 1
        for (int row = ctid; row < kTile; row += kConvThreads) {
          uint4 raw[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int c = (k + row) & 7;
            const uint32_t a = stage + kBoxBytes + row * 128 + 16 * c;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(raw[k].x), "=r"(raw[k].y), "=r"(raw[k].z), "=r"(raw[k].w)
                         : "r"(a));
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int c = (k + row) & 7;
            const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              h[2 * i] = e4m3x2_to_f16x2(static_cast<uint16_t>(w4[i] & 0xFFFFu));
              h[2 * i + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w4[i] >> 16));
            }
            // dims 16c .. 16c+15 of the part: box c/4, 16-byte chunks 2(c%4), 2(c%4)+1
            const uint32_t drow = stage + (c >> 2) * kBoxBytes + row * 128;
            const int col = 2 * (c & 3);
            sts_v4(drow + ((col ^ (row & 7)) << 4), h[0], h[1], h[2], h[3]);
            sts_v4(drow + (((col + 1) ^ (row & 7)) << 4), h[4], h[5], h[6], h[7]);
          }
        }
        fence_proxy_async_smem();  // generic stores -> visible to the tensor core
        mbar_arrive(smem_u32(&ms.kv_full[st]));
      }
      ring.advance();
      return true;
    };
    const int nt = ip.j1 - ip.j0;
    Tile cur = ip.cur.next(p);
    if (LA) {  // the loader's order: K(0), then K(j+1) and V(j) for each tile j
      for (int part = 0; part < 4 && ok; ++part) ok = convert(cur, part);
      for (int jj = 0; jj < nt && ok; ++jj) {
        Tile nxt = cur;
        if (jj + 1 < nt) {
          nxt = ip.cur.next(p);
          for (int part = 0; part < 4 && ok; ++part) ok = convert(nxt, part);
        }
        for (int part = 4; part < 8 && ok; ++part) ok = convert(cur, part);
        cur = nxt;
      }
    } else {
      const int n_parts = p.alias_kv ? 4 : 8;  // the E4M3 path never aliases
      for (int jj = 0; jj < nt && ok; ++jj) {
        if (jj > 0) cur = ip.cur.next(p);
        for (int part = 0; part < n_parts && ok; ++part) ok = convert(cur, part);
      }
    }
  }
}

// ------------------------------------------------------------------ MMA issuer

template <bool LA>
__device__ __forceinline__ void mma_role(const AttnParams &p, uint32_t sbase, uint32_t tmem, Misc &ms, int lane) {
  if (lane == 0) {
    volatile int *abrt = &ms.abort_flag;
    constexpr uint32_t kIdescQK = idesc_f16_f32(128, 64, false, false);
    constexpr uint32_t kIdescPV = idesc_f16_f32(128, 64, true, true);
    // Base descriptors, built once; the issue loops only add byte offsets.
    // K tiles and Q: K-major.  V tiles: MN-major, LBO = one 64-dim box.
    // P^T: one 64-head MN atom, LBO unused.
    const uint64_t k_desc = sdesc_sw128(sbase + kOffKV, 16, 1024);
    const uint64_t v_desc = sdesc_sw128(sbase + kOffKV, kBoxBytes, 1024);
    static_assert(kBoxBytes == (1u << 14), "K box distances are taken as shifts");
    // Paired stages (64-row tiles): K boxes at +0 and +8 KB, V boxes at +16 KB
    // and +24 KB of the stage, so V^T's two 64-dim atoms are 8 KB apart.
    const uint64_t pv_desc = p.kv_pair ? sdesc_sw128(sbase + kOffKV + kBoxBytes, kBoxBytes / 2, 1024) : v_desc;
    const uint32_t kbox_shift = p.kv_pair ? 13 : 14;  // log2 of the distance of a part's two K boxes
    const uint64_t q_desc = sdesc_sw128(sbase + kOffQ, 16, 1024);
    const uint64_t p_desc = sdesc_sw128(sbase + kOffP, 16, 1024);
    Ring ring;
    uint32_t g = 0, n_item = 0;
    bool ok = true;
    const int n_items = p.T * p.n_splits;
    if (plan_reads_inputs(p)) grid_dependency_wait();  // the plan reads status bytes or sequence geometry
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      ItemPlan ip = plan_item(p, item);
      if (ip.j1 == ip.j0) continue;
      ok = mbar_wait(smem_u32(&ms.q_full), n_item & 1, abrt, p.timeout_ns, p.err, SITE_Q_FULL);
      if (!ok) break;
      const int nt = ip.j1 - ip.j0;
      // K and V the same rows: each K part stays in the ring after QK^T and
      // serves PV as V^T.  A part holds 128 dims of every row of the tile,
      // the K-major A operand of QK^T and the MN-major A operand of PV alike,
      // so each row crosses into the SM once.  Paired stages hold the K and
      // the V slice of a 64-row tile: they too stay from QK^T until PV.  With
      // 64 rows the M = 128 QK^T reads 64 more rows (the next boxes of the
      // stage): their scores are dropped by the mask, and PV only takes the
      // tile's own rows.
      const bool hold = p.alias_kv != 0 || p.kv_pair != 0;
      uint32_t k0 = 0;  // held: part m sits in stage (k0 + m) % kStages until PV m
      // S^T of tile jj (global tile gj) = K_tile . Q^T over the 512 dims, 128 dims per stage.
      auto qk = [&](uint32_t gj, int jj) -> bool {
        k0 = ring.st;
        const uint32_t sb = gj & 1;
        if (!mbar_wait(smem_u32(&ms.s_empty[sb]), ((gj >> 1) & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_S_EMPTY))
          return false;
        tc_fence_after();
        const uint32_t d_s = tmem + kTmemS + 64 * sb;
        for (int c = 0; c < 4; ++c) {
          if (!mbar_wait(smem_u32(&ms.kv_full[ring.st]), ring.ph, abrt, p.timeout_ns, p.err, SITE_KV_FULL)) return false;
          tc_fence_after();
          const uint64_t a0 = sdesc_add(k_desc, ring.st * kStageBytes);
          const uint64_t b0 = sdesc_add(q_desc, 2 * c * kQBoxBytes);
#pragma unroll
          for (int b2 = 0; b2 < 2; ++b2) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t a = sdesc_add(a0, (b2 << kbox_shift) + ks * 32);
              const uint64_t b = sdesc_add(b0, b2 * kQBoxBytes + ks * 32);
              if (b2 == 0 && ks == 0)
                umma_f16(d_s, a, b, kIdescQK, c != 0 ? 1u : 0u);
              else
                umma_f16_acc(d_s, a, b, kIdescQK);
            }
          }
          if (!hold) umma_commit(smem_u32(&ms.kv_empty[ring.st]));  // held for PV otherwise
          ring.advance();
        }
        umma_commit(smem_u32(&ms.s_full[sb]));
        if (jj == nt - 1) umma_commit(smem_u32(&ms.q_empty));
        return true;
      };
      // O^T[m] += V_tile^T[dims 128m..] . P^T of tile jj (global tile gj), 16 rows per instruction.
      auto pv = [&](uint32_t gj, int jj) -> bool {
        if (!mbar_wait(smem_u32(&ms.p_full), gj & 1, abrt, p.timeout_ns, p.err, SITE_P_FULL)) return false;
        if (jj == 0 &&
            !mbar_wait(smem_u32(&ms.o_empty), (n_item & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_O_EMPTY))
          return false;
        tc_fence_after();
        for (int m = 0; m < 4; ++m) {
          uint32_t vst = (k0 + m) % kStages;  // held: the part of the same dims, already landed
          if (!hold) {
            if (!mbar_wait(smem_u32(&ms.kv_full[ring.st]), ring.ph, abrt, p.timeout_ns, p.err, SITE_KV_FULL))
              return false;
            tc_fence_after();
            vst = ring.st;
          }
          const uint64_t a0 = sdesc_add(pv_desc, vst * kStageBytes);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            if (ks == 4 && p.kv_pair) break;  // a 64-row tile: its rows only
            const uint64_t a = sdesc_add(a0, ks * 2048);
            const uint64_t b = sdesc_add(p_desc, ks * 2048);
            if (ks == 0)
              umma_f16(tmem + 64 * m, a, b, kIdescPV, jj > 0 ? 1u : 0u);
            else
              umma_f16_acc(tmem + 64 * m, a, b, kIdescPV);
          }
          umma_commit(smem_u32(&ms.kv_empty[vst]));
          // After the item's last tile, block m of O^T is final: the epilogue
          // drains it while the remaining blocks are still being computed.
          if (jj == nt - 1) umma_commit(smem_u32(&ms.o_full[m]));
          if (!hold) ring.advance();
        }
        umma_commit(smem_u32(&ms.p_empty));
        return true;
      };
      if (LA) {
        // The loader's order: QK^T of tile 0, then per tile the QK^T of the
        // next tile (into the other S^T buffer, while the softmax works on
        // this one) and the PV of this one.
        ok = qk(g, 0);
        for (int jj = 0; jj < nt && ok; ++jj, ++g) {
          if (jj + 1 < nt) ok = qk(g + 1, jj + 1);
          ok = ok && pv(g, jj);
        }
      } else {
        for (int jj = 0; jj < nt && ok; ++jj, ++g) ok = qk(g, jj) && pv(g, jj);
      }
      if (!ok) break;
      ++n_item;
    }
    // Every MMA issued so far must finish before TMEM is released.
    umma_commit(smem_u32(&ms.mma_done));
    volatile int never = 0;
    mbar_wait(smem_u32(&ms.mma_done), 0, &never, 100000000ull, p.err, SITE_DRAIN);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ softmax / epilogue

__device__ __forceinline__ void row_visibility(const AttnParams &p, int t, const Tile &tl, int r, bool &vis,
                                               float &bias_l2) {
  bias_l2 = 0.f;
  vis = r < tl.count;
  if (!vis) return;
  if (p.mode == MODE_MASK) {
    if (tl.open) return;
    const int col = (tl.seg == 0 ? 0 : p.nbr * 32) + tl.start + r;
    const float m = __half2float(p.mask[(long long)t * p.mask_stride + col]);
    vis = m != -INFINITY;
    bias_l2 = vis ? m * kLog2e : 0.f;
  } else if (tl.seg == 2) {
    const int c = __ldg(p.idx + (long long)t * p.idx_stride + tl.start + r);
    vis = c >= 0 && c < p.n_comp;
  }
}

__device__ __forceinline__ void write_empty_item(const AttnParams &p, int item, int t, int tid) {
  if (p.partial) {
    if (tid < kH) p.ws_ml[(long long)item * kH + tid] = make_float2(-INFINITY, 0.f);
    return;
  }
  __half *orow = p.o + (long long)t * p.o_tok_stride;
  for (int i = tid; i < kH * kD; i += kComputeThreads) orow[(i >> 9) * kD + (i & 511)] = __float2half_rn(0.f);
  if (p.lse != nullptr && tid < kH) p.lse[(long long)t * kH + tid] = -INFINITY;
}

__device__ __forceinline__ void load32(const float *src, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 x = reinterpret_cast<const float4 *>(src)[i];
    v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
  }
}

template <bool FP8>
__device__ __forceinline__ void compute_role(const AttnParams &p, uint8_t *smem, uint32_t tmem, Misc &ms, int tid) {
  volatile int *abrt = &ms.abort_flag;
  const int w = tid >> 5, l = tid & 31;
  const int q = w & 3;            // TMEM lane quarter: rows (or dims) 32q .. 32q+31
  const int hh = w >> 2;          // head half: heads 32hh .. 32hh+31
  const int r = 32 * q + l;       // this thread's TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
  const uint32_t col0 = 32 * hh;
  uint32_t g = 0, n_item = 0;
  bool bad = false, aborted = false;
  const int n_items = p.T * p.n_splits;
  grid_dependency_wait();  // outputs and index lists may be shared with the previous kernel
  for (int item = blockIdx.x; item < n_items && !aborted; item += gridDim.x) {
    ItemPlan ip = plan_item(p, item);
    const int t = ip.t;
    if (ip.j1 == ip.j0) {
      write_empty_item(p, item, t, tid);
      continue;
    }
    float m_ref = -INFINITY;  // reference max of head `tid` (threads < 64), log2 units
    float lpart[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) lpart[h] = 0.f;
    const int nt = ip.j1 - ip.j0;
    for (int jj = 0; jj < nt; ++jj) {
      const Tile tl = ip.cur.next(p);
      const uint32_t sb = g & 1;
      bad = bad || !mbar_wait(smem_u32(&ms.s_full[sb]), (g >> 1) & 1, abrt, p.timeout_ns, p.err, SITE_S_FULL);
      tc_fence_after();
      float s[32];
      tmem_ld32(tmem + kTmemS + 64 * sb + col0 + lane_base, s);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(smem_u32(&ms.s_empty[sb]));

      bool vis;
      float bias;
      row_visibility(p, t, tl, r, vis, bias);
      // E4M3 rows: the MMA saw the unscaled codes; the row scales come in here
      // (K's on the scores, V's on P below).
      const bool f8 = FP8 && tile_codes(p, tl);
      const float *ksc = tl.seg == 0 ? p.k_scale[0] : p.k_scale[1];
      const float *vsp = tl.seg == 0 ? p.v_scale[0] : p.v_scale[1];
      // (a gathered row's scale is that of the compressed row it lists)
      const int srow = (f8 && vis && tl.seg == 2) ? __ldg(p.idx + (long long)t * p.idx_stride + tl.start + r)
                                                  : tl.start + r;
      const float sl2 = f8 && vis ? p.scale_log2 * __ldg(ksc + srow) : p.scale_log2;
      const float vsc = f8 && vis ? __ldg(vsp + srow) : 1.f;
#pragma unroll
      for (int h = 0; h < 32; ++h) s[h] = vis ? fmaf(s[h], sl2, bias) : -INFINITY;

      ms.red[q][col0 + l] = warp_reduce_scatter32<true>(s, l);
      if (bar_red_or(1, kComputeThreads, bad)) {
        aborted = true;
        break;
      }
      if (tid < kH) {
        const float tmax = fmaxf(fmaxf(ms.red[0][tid], ms.red[1][tid]), fmaxf(ms.red[2][tid], ms.red[3][tid]));
        float alpha = 1.f;
        if (m_ref == -INFINITY) {
          m_ref = tmax;
        } else if (tmax > m_ref + kTau) {
          alpha = exp2f(m_ref - tmax);
          m_ref = tmax;
        }
        ms.m_use[tid] = m_ref == -INFINITY ? 0.f : m_ref;
        ms.alpha[tid] = alpha;
        if (alpha != 1.f) ms.resc_flag[g & 1] = 1;
      }
      named_bar_sync(1, kComputeThreads);
      const int resc = ms.resc_flag[g & 1];
      if (tid == 0) ms.resc_flag[(g + 1) & 1] = 0;

      // P (fp16) may only be rewritten once the previous PV has consumed it.
      bad = bad || !mbar_wait(smem_u32(&ms.p_empty), (g & 1) ^ 1, abrt, p.timeout_ns, p.err, SITE_P_EMPTY);
      if (resc) {
        float al[32];
        load32(ms.alpha + col0, al);
#pragma unroll
        for (int h = 0; h < 32; ++h) lpart[h] *= al[h];
      }
      // P^T row r, heads 32hh .. +31 = 16-byte chunks 4hh .. 4hh+3 of the
      // 128-byte row, stored at chunk c ^ (r & 7) (128-byte swizzle).
      {
        uint8_t *prow = smem + kOffP + r * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 m0 = reinterpret_cast<const float4 *>(ms.m_use + col0)[2 * c];
          const float4 m1 = reinterpret_cast<const float4 *>(ms.m_use + col0)[2 * c + 1];
          const float mu[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
          uint32_t w4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int h = 8 * c + 2 * i;
            const float e0 = exp2f(s[h] - mu[2 * i]), e1 = exp2f(s[h + 1] - mu[2 * i + 1]);
            const __half2 hp = __floats2half2_rn(e0, e1);
            const float2 f = __half22float2(hp);
            lpart[h] += f.x;
            lpart[h + 1] += f.y;
            if (f8) {  // P times the row's V scale feeds the MMA; the sums keep P
              const __half2 hv = __floats2half2_rn(e0 * vsc, e1 * vsc);
              w4[i] = *reinterpret_cast<const uint32_t *>(&hv);
            } else {
              w4[i] = *reinterpret_cast<const uint32_t *>(&hp);
            }
          }
          const int chunk = 4 * hh + c;
          *reinterpret_cast<uint4 *>(prow + ((chunk ^ (r & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      if (resc && jj > 0) {
        // O^T holds the previous tiles against the old reference: scale column h by alpha[h].
        float al[32];
        load32(ms.alpha + col0, al);
        tc_fence_after();
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
          float o[32];
          tmem_ld32(tmem + 64 * m + col0 + lane_base, o);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) o[h] *= al[h];
          tmem_st32(tmem + 64 * m + col0 + lane_base, o);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&ms.p_full));
      ++g;
    }
    if (aborted) break;

    // Epilogue: sum the row partials per head (they do not depend on O), then
    // normalise one O^T block at a time as each block of the last PV
    // completes.  A split-KV item hands out its own normalised o (fp16) and
    // (m, l); a whole token writes o and the log-sum-exp.
    ms.red[q][col0 + l] = warp_reduce_scatter32<false>(lpart, l);
    if (bar_red_or(1, kComputeThreads, bad)) {
      aborted = true;
      break;
    }
    if (tid < kH) {
      const float lsum = ms.red[0][tid] + ms.red[1][tid] + ms.red[2][tid] + ms.red[3][tid];
      ms.inv_l[tid] = lsum > 0.f ? 1.f / lsum : 0.f;
      if (p.partial) {
        p.ws_ml[(long long)item * kH + tid] = make_float2(lsum > 0.f ? m_ref : -INFINITY, lsum);
      } else if (p.lse != nullptr) {
        p.lse[(long long)t * kH + tid] = lsum > 0.f ? (m_ref + log2f(lsum)) * kLn2 : -INFINITY;
      }
    }
    named_bar_sync(1, kComputeThreads);
    {
      // O^T[128 dims][64 heads] -> fp16 o.  Lanes 2k and 2k+1 hold adjacent
      // dims: for each pair of heads they swap one value, so the even lane
      // writes both dims of the first head and the odd lane both dims of the
      // second (32-bit stores, 64 contiguous bytes per head per warp).
      float inv[32];
      load32(ms.inv_l + col0, inv);
      const bool odd = l & 1;
      __half *obase = p.partial ? p.ws_o + ((long long)item * kH + col0) * kD + (r & ~1)
                                : p.o + (long long)t * p.o_tok_stride + (long long)col0 * kD + (r & ~1);
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        bad = bad || !mbar_wait(smem_u32(&ms.o_full[m]), n_item & 1, abrt, p.timeout_ns, p.err, SITE_O_FULL);
        tc_fence_after();
        float o[32];
        tmem_ld32(tmem + 64 * m + col0 + lane_base, o);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 32; h += 2) {
          const float a = o[h] * inv[h], b = o[h + 1] * inv[h + 1];
          const float got = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
          const __half2 v = odd ? __floats2half2_rn(got, b) : __floats2half2_rn(a, got);
          *reinterpret_cast<__half2 *>(obase + (h + (odd ? 1 : 0)) * kD + 128 * m) = v;
        }
      }
    }
    tc_fence_before();
    mbar_arrive(smem_u32(&ms.o_empty));
    ++n_item;
    if (bar_red_or(1, kComputeThreads, bad)) {  // a block wait ran out: leave together
      aborted = true;
      break;
    }
  }
  if (tid == 0) bulk_wait_all();
}

// ------------------------------------------------------------------ kernel

template <bool FP8, bool LA>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Align by pointer arithmetic on the __shared__ array (not through an
  // integer cast) so every access below stays a shared-memory access.
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  Misc &ms = *reinterpret_cast<Misc *>(smem + kOffMisc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ms.q_full), q_by_lsu(p, FP8) ? kQCopyThreads : 1);
    mbar_init(smem_u32(&ms.q_empty), 1);
    const uint32_t fill_count = stage_fill_count<FP8>(p);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ms.kv_full[s]), FP8 ? (uint32_t)kConvThreads : fill_count);
      mbar_init(smem_u32(&ms.kv_empty[s]), 1);
      mbar_init(smem_u32(&ms.code_full[s]), fill_count);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ms.s_full[s]), 1);
      mbar_init(smem_u32(&ms.s_empty[s]), kComputeThreads);
    }
    mbar_init(smem_u32(&ms.p_full), kComputeThreads);
    mbar_init(smem_u32(&ms.p_empty), 1);
    for (int m = 0; m < 4; ++m) mbar_init(smem_u32(&ms.o_full[m]), 1);
    mbar_init(smem_u32(&ms.o_empty), kComputeThreads);
    mbar_init(smem_u32(&ms.mma_done), 1);
    ms.abort_flag = 0;
    ms.resc_flag[0] = 0;
    ms.resc_flag[1] = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&ms.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kLoaderWarp0 && lane == 0) {
    // Fetch the tensor maps this call uses while the prologue runs.
    tma_prefetch_desc(&p.tm_q);
    if (p.n_raw > 0) {
      tma_prefetch_desc(&p.tm_k[0]);
      tma_prefetch_desc(&p.tm_v[0]);
    }
    if (p.n_comp > 0 && p.mode != MODE_INDEXED) {
      tma_prefetch_desc(FP8 ? &p.tm_k8[1] : &p.tm_k[1]);
      tma_prefetch_desc(FP8 ? &p.tm_v8[1] : &p.tm_v[1]);
    }
    if (FP8 && p.raw_fp8) {
      tma_prefetch_desc(&p.tm_k8[0]);
      tma_prefetch_desc(&p.tm_v8[0]);
    }
    if (!p.partial) tma_prefetch_desc(&p.tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  // Let the next kernel in the stream start its own prologue.  Inputs may come
  // from the previous kernel: each role waits for it just before its first
  // global access (the loader after planning its first item, so that work
  // overlaps the previous kernel's tail, unless the plan itself reads inputs:
  // status bytes in dense-mask mode, the sequences' geometry in batched
  // decode).
  grid_launch_dependents();

  if (warp < kComputeWarps) {
    compute_role<FP8>(p, smem, tmem, ms, threadIdx.x);
  } else if (warp == kMmaWarp) {
    mma_role<LA>(p, sbase, tmem, ms, lane);
  } else {
    const int ltid = threadIdx.x - 32 * kLoaderWarp0;
    if (FP8 && ltid >= 32 && ltid < 32 + kConvThreads)
      converter_role<LA>(p, sbase, ms, ltid - 32);
    else
      loader_role<FP8, LA>(p, sbase, ms, ltid);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace ds4a
