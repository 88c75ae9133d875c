// C ABI of the library (declared in include/ds4a.h): argument checks, TMA
// tensor maps, work splitting and kernel launches.  No device memory is
// allocated here; every buffer belongs to the caller.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "ds4a.h"
#include "internal.h"

// Device error word: set by a kernel whose bounded wait ran out.  Its address
// is looked up once per device and handed to the kernels as a parameter.
__device__ unsigned int g_ds4a_device_error;

// Split-KV scratch of ds4a_attn_decode_noalloc, for callers that cannot
// allocate device memory.  Every device that loads the library holds these
// 8 MiB until the process exits.  In host code the name is only a stand-in:
// the device address comes from cudaGetSymbolAddress (see current_device).
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

namespace {

using ds4a::AttnParams;

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  unsigned int *err = nullptr;
  void *scratch = nullptr;  // device address of g_decode_scratch
  bool loaded = false;      // every kernel's code loaded (before a recording)
};

std::mutex g_mu;

// What the latest DS4A_ERR_CUDA of this thread came from (empty when none).
thread_local char g_cuda_detail[192] = "";

ds4a_status cuda_failed(const char *call, int code, const char *text) {
  std::snprintf(g_cuda_detail, sizeof(g_cuda_detail), "%s: error %d%s%s", call, code, text ? " " : "",
                text ? text : "");
  return DS4A_ERR_CUDA;
}
ds4a_status cuda_failed(const char *call, cudaError_t e) { return cuda_failed(call, (int)e, cudaGetErrorString(e)); }
#define DS4A_CUDA_TRY(call)                              \
  do {                                                   \
    const cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_failed(#call, e_); \
  } while (0)

DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Looks up the current device once: compute capability, SM count, the error
// word's address, the kernel's shared-memory opt-in and the tensor-map encoder.
ds4a_status current_device(DeviceState **out) {
  int dev = -1;
  DS4A_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return DS4A_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState &d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    DS4A_CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    DS4A_CUDA_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    DS4A_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    d.sm_count = sms;
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
      DS4A_CUDA_TRY(ds4a::prepare_attn_kernel());
      DS4A_CUDA_TRY(ds4a::prepare_pair_kernel());
      DS4A_CUDA_TRY(cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err), g_ds4a_device_error));
      DS4A_CUDA_TRY(cudaGetSymbolAddress(&d.scratch, g_decode_scratch));
      if (g_encode == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        DS4A_CUDA_TRY(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
        if (q != cudaDriverEntryPointSuccess || fn == nullptr)
          return cuda_failed("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", (int)q, nullptr);
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
    }
    d.ready = true;
  }
  if (!d.supported) return DS4A_ERR_UNSUPPORTED;
  *out = &d;
  return DS4A_OK;
}

cudaStream_t as_cuda(ds4a_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool row_stride_ok(int64_t s) { return s >= DS4A_ROW_BYTES && s % 16 == 0 && s < (1LL << 39); }
bool tok_stride_ok(int64_t s) { return s >= 64LL * DS4A_ROW_BYTES && s % 16 == 0 && s < (1LL << 39); }
int32_t ceil_div(int64_t a, int64_t b) { return (int32_t)((a + b - 1) / b); }

ds4a_status check_layout(const ds4a_layout *L) {
  if (L == nullptr) return DS4A_ERR_INVALID_ARG;
  if (L->T < 0 || L->q_pos0 < 0 || L->n_raw < 0 || L->raw_pos0 < 0 || L->n_comp < 0) return DS4A_ERR_INVALID_ARG;
  if (L->window < 1) return DS4A_ERR_INVALID_ARG;
  if (L->n_comp > 0 && L->ratio < 1) return DS4A_ERR_INVALID_ARG;
  if (!std::isfinite(L->scale)) return DS4A_ERR_INVALID_ARG;
  // Positions and row counts must stay inside int32 arithmetic.
  if ((int64_t)L->q_pos0 + L->T > INT32_MAX - 1 || (int64_t)L->raw_pos0 + L->n_raw > INT32_MAX - 1)
    return DS4A_ERR_INVALID_ARG;
  if (L->n_raw > (1 << 30) || L->n_comp > (1 << 30)) return DS4A_ERR_INVALID_ARG;
  return DS4A_OK;
}

ds4a_status check_tensors(const ds4a_layout *L, const ds4a_tensors *X) {
  if (X == nullptr) return DS4A_ERR_INVALID_ARG;
  if (X->q == nullptr || !aligned(X->q, 16) || !tok_stride_ok(X->q_tok_stride)) return DS4A_ERR_INVALID_ARG;
  if (X->o == nullptr || !aligned(X->o, 16) || !tok_stride_ok(X->o_tok_stride)) return DS4A_ERR_INVALID_ARG;
  if (X->lse != nullptr && !aligned(X->lse, 4)) return DS4A_ERR_INVALID_ARG;
  if (L->n_raw > 0) {
    if (X->k_raw == nullptr || X->v_raw == nullptr || !aligned(X->k_raw, 16) || !aligned(X->v_raw, 16) ||
        !row_stride_ok(X->raw_row_stride))
      return DS4A_ERR_INVALID_ARG;
  }
  if (L->n_comp > 0) {
    if (X->k_comp == nullptr || X->v_comp == nullptr || !aligned(X->k_comp, 16) || !aligned(X->v_comp, 16) ||
        !row_stride_ok(X->comp_row_stride))
      return DS4A_ERR_INVALID_ARG;
  }
  return DS4A_OK;
}

ds4a_status encode(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                   const cuuint32_t *box, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
                   CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_FLOAT16) {
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};  // element strides, up to rank 5
  const CUresult r = g_encode(m, dtype, (cuuint32_t)rank, const_cast<void *>(base), dims,
                              strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) return DS4A_OK;
  char what[160];
  int n = std::snprintf(what, sizeof(what), "cuTensorMapEncodeTiled(rank %d, dims", rank);
  for (int i = 0; i < rank && n < (int)sizeof(what); ++i)
    n += std::snprintf(what + n, sizeof(what) - n, " %llu", (unsigned long long)dims[i]);
  for (int i = 0; i + 1 < rank && n < (int)sizeof(what); ++i)
    n += std::snprintf(what + n, sizeof(what) - n, "%s%llu", i == 0 ? ", strides " : " ", (unsigned long long)strides[i]);
  for (int i = 0; i < rank && n < (int)sizeof(what); ++i)
    n += std::snprintf(what + n, sizeof(what) - n, "%s%u", i == 0 ? ", box " : " ", box[i]);
  if (n < (int)sizeof(what)) std::snprintf(what + n, sizeof(what) - n, ")");
  return cuda_failed(what, (int)r, nullptr);
}

// K/V rows: {512 dims, rows}, box {64 dims, box_rows rows}, 128-byte swizzle.
ds4a_status encode_rows(CUtensorMap *m, const void *base, int rows, int64_t stride, unsigned box_rows) {
  const cuuint64_t dims[2] = {DS4A_HEAD_DIM, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)stride};
  const cuuint32_t box[2] = {64, box_rows};
  return encode(m, base, 2, dims, strides, box);
}

// K/V rows as 64-dim column blocks: {64 dims, rows, 8 blocks} (block stride
// 128 bytes), box {64, box_rows, 2}: one copy brings a 128-dim part of a tile
// as two [box_rows][64] swizzled boxes, one after the other.  A thread's bulk
// copies start one after another, some 650 cycles apart whatever their size,
// so fewer, larger copies load a tile sooner.
ds4a_status encode_row_parts(CUtensorMap *m, const void *base, int rows, int64_t stride, unsigned box_rows) {
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, DS4A_HEAD_DIM / 64};
  const cuuint64_t strides[2] = {(cuuint64_t)stride, 128};
  const cuuint32_t box[3] = {64, box_rows, 2};
  return encode(m, base, 3, dims, strides, box);
}

// Q of every token (or sequence) at once per copy: {64 dims, 64 heads, n,
// 8 blocks}, box {64, 64, 1, 8}: the eight [64 heads][64 dims] boxes of a token.
ds4a_status encode_q_blocks(CUtensorMap *m, const void *base, int n, int64_t stride) {
  const cuuint64_t dims[4] = {64, DS4A_HEADS, (cuuint64_t)n, DS4A_HEAD_DIM / 64};
  const cuuint64_t strides[3] = {DS4A_ROW_BYTES, (cuuint64_t)stride, 128};
  const cuuint32_t box[4] = {64, 64, 1, DS4A_HEAD_DIM / 64};
  return encode(m, base, 4, dims, strides, box);
}

// Fills the parts of the kernel parameters every attention mode shares.
ds4a_status fill_params(AttnParams &p, const ds4a_layout *L, const ds4a_tensors *X, int mode, DeviceState *d) {
  std::memset(&p, 0, sizeof(p));
  {
    ds4a_status st = encode_q_blocks(&p.tm_q, X->q, L->T, X->q_tok_stride);
    if (st != DS4A_OK) return st;
  }
  if (X->o != nullptr) {
    // Output: fp16 [T][64][512]; the epilogue stores [64 heads][128 dims] boxes.
    const cuuint64_t dims[3] = {DS4A_HEAD_DIM, DS4A_HEADS, (cuuint64_t)L->T};
    const cuuint64_t strides[2] = {DS4A_ROW_BYTES, (cuuint64_t)X->o_tok_stride};
    const cuuint32_t box[3] = {128, 64, 1};
    ds4a_status st = encode(&p.tm_o, X->o, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != DS4A_OK) return st;
  }
  if (L->n_raw > 0) {
    ds4a_status st = encode_row_parts(&p.tm_k[0], X->k_raw, L->n_raw, X->raw_row_stride, 128);
    if (st == DS4A_OK) st = encode_row_parts(&p.tm_v[0], X->v_raw, L->n_raw, X->raw_row_stride, 128);
    if (st != DS4A_OK) return st;
  }
  if (L->n_comp > 0) {
    ds4a_status st = encode_row_parts(&p.tm_k[1], X->k_comp, L->n_comp, X->comp_row_stride, 128);
    if (st == DS4A_OK) st = encode_row_parts(&p.tm_v[1], X->v_comp, L->n_comp, X->comp_row_stride, 128);
    if (st != DS4A_OK) return st;
  }
  p.k_comp = X->k_comp;
  p.v_comp = X->v_comp;
  p.comp_row_stride = X->comp_row_stride;
  // One row serving as K and V in every segment that has rows (the pointers
  // are equal; a segment has one row stride): each tile part is loaded once
  // for both products.  A call whose segments differ reads K and V apart.
  p.alias_kv = ((L->n_raw == 0 || X->k_raw == X->v_raw) && (L->n_comp == 0 || X->k_comp == X->v_comp) &&
                L->n_raw + L->n_comp > 0) ? 1 : 0;
  p.q_ptr = static_cast<const uint8_t *>(X->q);
  p.q_tok_bytes = X->q_tok_stride;
  p.tile_rows = 128;
  p.T = L->T;
  p.q_pos0 = L->q_pos0;
  p.n_raw = L->n_raw;
  p.raw_pos0 = L->raw_pos0;
  p.n_comp = L->n_comp;
  p.ratio = L->n_comp > 0 ? L->ratio : 1;
  p.window = L->window;
  p.scale_log2 = L->scale * 1.4426950408889634f;
  p.mode = mode;
  p.n_splits = 1;
  p.q_tile = 1;
  p.nbr = ceil_div(L->n_raw, DS4A_BLOCK_ROWS);
  p.n_blocks = p.nbr + ceil_div(L->n_comp, DS4A_BLOCK_ROWS);
  p.o = static_cast<__half *>(X->o);
  p.o_tok_stride = X->o_tok_stride / 2;
  p.lse = X->lse;
  p.timeout_ns = kDefaultTimeoutNs;
  p.err = d->err;
  return DS4A_OK;
}

ds4a_status launched(cudaError_t e) { return e == cudaSuccess ? DS4A_OK : cuda_failed("kernel launch", e); }

int32_t max_tiles_per_token(const ds4a_layout *L, int rows = 128) {
  const int64_t raw = L->window < L->n_raw ? L->window : L->n_raw;
  return ceil_div(raw, rows) + ceil_div(L->n_comp, rows);
}

// A short decode: every (token, split) item fits on its own SM even with
// 64-row tiles, and a token has at most 32 of them.  Then each CTA runs one
// item, and tiles of 64 rows whose K and V share a ring stage let a CTA issue
// all its loads at once (its Q, K and V fit in shared memory together),
// instead of loading V only as the K parts are consumed.  Longer rows gain
// less than the wider merge of twice the splits costs (8192 compressed rows:
// 13.8 us with 65 splits of 128-row tiles, 16.8 us with 130 of 64 rows).  The
// default split count and the kernel use the same rule.
bool short_decode(const ds4a_layout *L, int sm_count) {
  const int64_t half_tiles = (int64_t)2 * max_tiles_per_token(L);
  return half_tiles <= 32 && half_tiles * L->T <= sm_count;
}

// Raw rows only, window <= 128, T >= 2: pairs of consecutive tokens share one
// 128-row tile (attn_pair.cu); the result is the structural attention.
ds4a_status prefill_pairs(const ds4a_layout *L, const ds4a_tensors *X, DeviceState *d, ds4a_stream_t stream) {
  ds4a::PairParams p;
  std::memset(&p, 0, sizeof(p));
  {
    const cuuint64_t dims[3] = {DS4A_HEAD_DIM, DS4A_HEADS, (cuuint64_t)L->T};
    const cuuint64_t strides[2] = {DS4A_ROW_BYTES, (cuuint64_t)X->q_tok_stride};
    const cuuint32_t box[3] = {64, 64, 2};
    ds4a_status st = encode(&p.tm_q2, X->q, 3, dims, strides, box);
    if (st != DS4A_OK) return st;
  }

  ds4a_status st = encode_rows(&p.tm_k, X->k_raw, L->n_raw, X->raw_row_stride, 128);
  if (st == DS4A_OK) st = encode_rows(&p.tm_v, X->v_raw, L->n_raw, X->raw_row_stride, 128);
  if (st != DS4A_OK) return st;
  p.T = L->T;
  p.q_pos0 = L->q_pos0;
  p.n_raw = L->n_raw;
  p.raw_pos0 = L->raw_pos0;
  p.window = L->window;
  p.scale_log2 = L->scale * 1.4426950408889634f;
  p.k_raw = static_cast<const uint8_t *>(X->k_raw);
  p.v_raw = static_cast<const uint8_t *>(X->v_raw);
  p.raw_row_stride = X->raw_row_stride;
  p.o = static_cast<__half *>(X->o);
  p.o_tok_stride = X->o_tok_stride / 2;
  p.o_v8 = (aligned(X->o, 32) && X->o_tok_stride % 32 == 0) ? 1 : 0;
  p.lse = X->lse;
  p.timeout_ns = kDefaultTimeoutNs;
  p.err = d->err;
  const int pairs = (L->T + 1) / 2;
  const int grid = pairs < d->sm_count ? pairs : d->sm_count;
  return launched(ds4a::launch_pair(p, grid, as_cuda(stream)));
}

}  // namespace

extern "C" {

const char *ds4a_status_string(int status) {
  switch (status) {
    case DS4A_OK: return "ok";
    case DS4A_ERR_INVALID_ARG: return "invalid argument";
    case DS4A_ERR_UNSUPPORTED: return "unsupported (needs an sm_103a device)";
    case DS4A_ERR_WORKSPACE: return "workspace missing or too small";
    case DS4A_ERR_CUDA: return "CUDA error";
    case DS4A_ERR_TIMEOUT: return "a bounded device wait ran out";
    default: return "unknown status";
  }
}

const char *ds4a_version(void) { return "ds4a 0.2 sm_103a"; }

const char *ds4a_last_cuda_error(void) { return g_cuda_detail; }

ds4a_status ds4a_pad_kv(const void *src, int64_t src_row_stride, int32_t n_rows, void *dst, int64_t dst_row_stride,
                        ds4a_stream_t stream) {
  if (n_rows < 0) return DS4A_ERR_INVALID_ARG;
  if (n_rows == 0) return DS4A_OK;
  if (src == nullptr || dst == nullptr || !aligned(src, 16) || !aligned(dst, 16) || !row_stride_ok(src_row_stride) ||
      !row_stride_ok(dst_row_stride))
    return DS4A_ERR_INVALID_ARG;
  const bool in_place = src == dst;
  if (in_place && src_row_stride != dst_row_stride) return DS4A_ERR_INVALID_ARG;
  if (!in_place) {
    // Other overlaps are not allowed.
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
    const uintptr_t s1 = s0 + (uintptr_t)(n_rows - 1) * src_row_stride + DS4A_ROW_BYTES;
    const uintptr_t d1 = d0 + (uintptr_t)(ceil_div(n_rows, 32) * 32 - 1) * dst_row_stride + DS4A_ROW_BYTES;
    if (s0 < d1 && d0 < s1) return DS4A_ERR_INVALID_ARG;
  }
  DeviceState *d = nullptr;
  ds4a_status st = current_device(&d);
  if (st != DS4A_OK) return st;
  return launched(ds4a::launch_pad(src, src_row_stride, n_rows, dst, dst_row_stride, in_place ? n_rows : 0,
                                   as_cuda(stream)));
}

ds4a_status ds4a_quantize_kv_fp8(const void *src, int64_t src_row_stride, int32_t n_rows, void *dst_codes,
                                 int64_t dst_row_stride, float *scales, ds4a_stream_t stream) {
  if (n_rows < 0) return DS4A_ERR_INVALID_ARG;
  if (n_rows == 0) return DS4A_OK;
  if (src == nullptr || !aligned(src, 16) || !row_stride_ok(src_row_stride)) return DS4A_ERR_INVALID_ARG;
  if (dst_codes == nullptr || !aligned(dst_codes, 16) || dst_row_stride < DS4A_HEAD_DIM || dst_row_stride % 16 != 0 ||
      dst_row_stride >= (1LL << 39))
    return DS4A_ERR_INVALID_ARG;
  if (scales == nullptr || !aligned(scales, 4)) return DS4A_ERR_INVALID_ARG;
  DeviceState *d = nullptr;
  ds4a_status st = current_device(&d);
  if (st != DS4A_OK) return st;
  return launched(ds4a::launch_quantize_fp8(src, src_row_stride, n_rows, dst_codes, dst_row_stride, scales,
                                            as_cuda(stream)));
}

int32_t ds4a_compress_rows(int32_t n_state, int32_t n_new, int32_t ratio) {
  if (ratio < 1 || ratio > 65536 || n_state < 0 || n_state >= ratio || n_new < 0) return -1;
  return (int32_t)(((int64_t)n_state + n_new) / ratio);
}

ds4a_status ds4a_compress_append(int32_t width, int32_t ratio, int32_t n_state, const float *kv, const float *score,
                                 int64_t new_row_stride, int32_t n_new, float *state_kv, float *state_score,
                                 int64_t state_row_stride, void *out, int64_t out_row_stride, ds4a_stream_t stream) {
  const int32_t n_out = ds4a_compress_rows(n_state, n_new, ratio);
  if (n_out < 0 || width < 4 || width > 65536 || width % 4 != 0) return DS4A_ERR_INVALID_ARG;
  if (n_new == 0) return DS4A_OK;
  auto stride_ok = [](int64_t s, int64_t row) { return s >= row && s % 16 == 0 && s < (1LL << 39); };
  if (kv == nullptr || score == nullptr || !aligned(kv, 16) || !aligned(score, 16) ||
      !stride_ok(new_row_stride, 4LL * width))
    return DS4A_ERR_INVALID_ARG;
  if (ratio > 1 && (state_kv == nullptr || state_score == nullptr || !aligned(state_kv, 16) ||
                    !aligned(state_score, 16) || !stride_ok(state_row_stride, 4LL * width)))
    return DS4A_ERR_INVALID_ARG;
  if (n_out > 0 && (out == nullptr || !aligned(out, 16) || out_row_stride < 2LL * width || out_row_stride % 8 != 0 ||
                    out_row_stride >= (1LL << 39)))
    return DS4A_ERR_INVALID_ARG;
  // Byte ranges: the new rows are read while the state and the output are
  // written, so none of the written ranges may meet a read one or each other.
  struct Span {
    uintptr_t lo, hi;
  };
  auto span = [](const void *ptr, int64_t rows, int64_t stride, int64_t row_bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr);
    return Span{lo, rows > 0 ? lo + (uintptr_t)((rows - 1) * stride + row_bytes) : lo};
  };
  auto meet = [](Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; };
  const Span rd[2] = {span(kv, n_new, new_row_stride, 4LL * width), span(score, n_new, new_row_stride, 4LL * width)};
  const Span wr[3] = {span(state_kv, ratio > 1 ? ratio - 1 : 0, state_row_stride, 4LL * width),
                      span(state_score, ratio > 1 ? ratio - 1 : 0, state_row_stride, 4LL * width),
                      span(out, n_out, out_row_stride, 2LL * width)};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 2; ++j)
      if (meet(wr[i], rd[j])) return DS4A_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (meet(wr[i], wr[j])) return DS4A_ERR_INVALID_ARG;
  }
  DeviceState *d = nullptr;
  ds4a_status st = current_device(&d);
  if (st != DS4A_OK) return st;
  ds4a::CompressParams p;
  p.kv = kv;
  p.score = score;
  p.new_stride = new_row_stride / 4;
  p.state_kv = state_kv;
  p.state_score = state_score;
  p.state_stride = ratio > 1 ? state_row_stride / 4 : 0;
  p.out = static_cast<__half *>(out);
  p.out_stride = n_out > 0 ? out_row_stride / 2 : 0;
  p.width = width;
  p.ratio = ratio;
  p.n_state = n_state;
  p.n_new = n_new;
  p.n_out = n_out;
  p.tail = (int32_t)(((int64_t)n_state + n_new) % ratio);
  ds4a::compress_shape(ratio, &p.splits, &p.slots);
  const int chunk = 128 / p.slots;
  p.chunks = (width + chunk - 1) / chunk;
  return launched(ds4a::launch_compress(p, as_cuda(stream)));
}

int32_t ds4a_block_count(const ds4a_layout *L) {
  if (L == nullptr || L->n_raw < 0 || L->n_comp < 0) return -1;
  return ceil_div(L->n_raw, DS4A_BLOCK_ROWS) + ceil_div(L->n_comp, DS4A_BLOCK_ROWS);
}

ds4a_status ds4a_block_mask(const ds4a_layout *L, const void *dense_mask, int64_t mask_row_stride, int32_t q_tile,
                            uint8_t *status, ds4a_stream_t stream) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (q_tile < 1) return DS4A_ERR_INVALID_ARG;
  const int32_t n_blocks = ds4a_block_count(L);
  if (L->T == 0 || n_blocks == 0) return DS4A_OK;
  if (status == nullptr) return DS4A_ERR_INVALID_ARG;
  if (dense_mask != nullptr &&
      (!aligned(dense_mask, 16) || mask_row_stride < (int64_t)n_blocks * 64 || mask_row_stride % 16 != 0))
    return DS4A_ERR_INVALID_ARG;
  DeviceState *d = nullptr;
  st = current_device(&d);
  if (st != DS4A_OK) return st;
  const ds4a::GeomScalars g{L->T, L->q_pos0, L->n_raw, L->raw_pos0, L->n_comp, L->n_comp > 0 ? L->ratio : 1,
                            L->window};
  if (dense_mask == nullptr) return launched(ds4a::launch_block_mask_struct(g, q_tile, status, as_cuda(stream)));
  return launched(ds4a::launch_block_mask_dense(g, static_cast<const __half *>(dense_mask), mask_row_stride / 2,
                                                q_tile, status, as_cuda(stream)));
}

ds4a_status ds4a_attn_prefill(const ds4a_layout *L, const ds4a_tensors *X, const void *dense_mask,
                              int64_t mask_row_stride, const uint8_t *status, int32_t q_tile, ds4a_stream_t stream) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (L->T == 0) return DS4A_OK;
  st = check_tensors(L, X);
  if (st != DS4A_OK) return st;
  const int32_t n_blocks = ds4a_block_count(L);
  if (dense_mask != nullptr &&
      (!aligned(dense_mask, 16) || mask_row_stride < (int64_t)n_blocks * 64 || mask_row_stride % 16 != 0))
    return DS4A_ERR_INVALID_ARG;
  if (status != nullptr && q_tile < 1) return DS4A_ERR_INVALID_ARG;
  DeviceState *d = nullptr;
  st = current_device(&d);
  if (st != DS4A_OK) return st;
  if (dense_mask == nullptr && L->n_comp == 0 && L->n_raw > 0 && L->window <= 128 && L->T >= 2)
    return prefill_pairs(L, X, d, stream);
  AttnParams p;
  st = fill_params(p, L, X, dense_mask != nullptr ? ds4a::MODE_MASK : ds4a::MODE_STRUCT, d);
  if (st != DS4A_OK) return st;
  if (dense_mask != nullptr) {
    p.mask = static_cast<const __half *>(dense_mask);
    p.mask_stride = mask_row_stride / 2;
    p.status = status;
    p.q_tile = status != nullptr ? q_tile : 1;
  }
  const int grid = L->T < d->sm_count ? L->T : d->sm_count;
  return launched(ds4a::launch_attn(p, grid, as_cuda(stream)));
}

int32_t ds4a_attn_decode_default_splits(const ds4a_layout *L) {
  if (check_layout(L) != DS4A_OK || L->T == 0) return 1;
  int sms = 148;
  int dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  }
  int32_t s = ceil_div(sms, L->T);
  const int32_t mt = max_tiles_per_token(L, short_decode(L, sms) ? 64 : 128);
  if (s > mt) s = mt;
  if (s < 1) return 1;
  // The fewest splits whose longest range has as many tiles as with s splits:
  // the same longest chain, fewer partials to write and merge (65,536
  // compressed rows, 513 tiles: 129 splits of at most 4 tiles 37.1 us per
  // call, 152 splits 39.6 us; 262,144 rows: 147 splits 97.8 us, 152 98.9 us).
  return ceil_div(mt, ceil_div(mt, s));
}

size_t ds4a_attn_decode_workspace_size(const ds4a_layout *L, int32_t n_splits) {
  if (check_layout(L) != DS4A_OK) return 0;
  if (n_splits <= 0) n_splits = ds4a_attn_decode_default_splits(L);
  return (size_t)L->T * (size_t)n_splits * DS4A_HEADS * (DS4A_HEAD_DIM * sizeof(__half) + 2 * sizeof(float));
}

namespace {

// Shared checks of the decode calls; fills the partial-output pointers.
ds4a_status decode_setup(const ds4a_layout *L, const ds4a_tensors *X, int32_t &n_splits, const void *workspace,
                         size_t workspace_bytes, bool need_inputs, bool need_outputs, __half **ws_o,
                         float2 **ws_ml) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (L->T == 0) return DS4A_OK;
  if (X == nullptr) return DS4A_ERR_INVALID_ARG;
  if (need_inputs) {
    ds4a_tensors probe = *X;
    if (!need_outputs) {  // the outputs are not touched: check the inputs only
      probe.o = const_cast<void *>(X->q);
      probe.o_tok_stride = X->q_tok_stride;
      probe.lse = nullptr;
    }
    st = check_tensors(L, &probe);
    if (st != DS4A_OK) return st;
  } else {
    if (X->o == nullptr || !aligned(X->o, 16) || !tok_stride_ok(X->o_tok_stride)) return DS4A_ERR_INVALID_ARG;
    if (X->lse != nullptr && !aligned(X->lse, 4)) return DS4A_ERR_INVALID_ARG;
  }
  if (n_splits <= 0) n_splits = ds4a_attn_decode_default_splits(L);
  if (n_splits > 4096) return DS4A_ERR_INVALID_ARG;
  const size_t need = ds4a_attn_decode_workspace_size(L, n_splits);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)) return DS4A_ERR_WORKSPACE;
  const size_t n_items = (size_t)L->T * n_splits;
  if (n_items > (size_t)INT32_MAX) return DS4A_ERR_INVALID_ARG;
  *ws_o = static_cast<__half *>(const_cast<void *>(workspace));
  *ws_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(const_cast<void *>(workspace)) +
                                      n_items * DS4A_HEADS * DS4A_HEAD_DIM * sizeof(__half));
  return DS4A_OK;
}

ds4a_status decode_partials(const ds4a_layout *L, const ds4a_tensors *X, int32_t n_splits, __half *ws_o,
                            float2 *ws_ml, ds4a_stream_t stream) {
  DeviceState *d = nullptr;
  ds4a_status st = current_device(&d);
  if (st != DS4A_OK) return st;
  ds4a_tensors Xi = *X;
  if (Xi.o == nullptr) {  // the partial kernel never writes o; the tensor map needs none either
    Xi.o = const_cast<void *>(X->q);
    Xi.o_tok_stride = X->q_tok_stride;
  }
  AttnParams p;
  st = fill_params(p, L, &Xi, ds4a::MODE_STRUCT, d);
  if (st != DS4A_OK) return st;
  const size_t n_items = (size_t)L->T * n_splits;
  if (!p.alias_kv && short_decode(L, d->sm_count) && n_items <= (size_t)d->sm_count) {
    p.kv_pair = 1;
    p.tile_rows = 64;
    // K/V rows in 64-row boxes for the paired stages.
    if (L->n_raw > 0) {
      if ((st = encode_row_parts(&p.tm_k[0], X->k_raw, L->n_raw, X->raw_row_stride, 64)) != DS4A_OK) return st;
      if ((st = encode_row_parts(&p.tm_v[0], X->v_raw, L->n_raw, X->raw_row_stride, 64)) != DS4A_OK) return st;
    }
    if (L->n_comp > 0) {
      if ((st = encode_row_parts(&p.tm_k[1], X->k_comp, L->n_comp, X->comp_row_stride, 64)) != DS4A_OK) return st;
      if ((st = encode_row_parts(&p.tm_v[1], X->v_comp, L->n_comp, X->comp_row_stride, 64)) != DS4A_OK) return st;
    }
  }
  p.n_splits = n_splits;
  p.partial = 1;
  p.o = nullptr;
  p.lse = nullptr;
  p.ws_o = ws_o;
  p.ws_ml = ws_ml;
  const int grid = (int)(n_items < (size_t)d->sm_count ? n_items : (size_t)d->sm_count);
  return launched(ds4a::launch_attn(p, grid, as_cuda(stream)));
}

}  // namespace

ds4a_status ds4a_attn_decode_partials(const ds4a_layout *L, const ds4a_tensors *X, int32_t n_splits,
                                      void *workspace, size_t workspace_bytes, ds4a_stream_t stream) {
  __half *ws_o = nullptr;
  float2 *ws_ml = nullptr;
  ds4a_status st = decode_setup(L, X, n_splits, workspace, workspace_bytes, true, false, &ws_o, &ws_ml);
  if (st != DS4A_OK || L->T == 0) return st;
  return decode_partials(L, X, n_splits, ws_o, ws_ml, stream);
}

ds4a_status ds4a_attn_decode_merge(const ds4a_layout *L, const ds4a_tensors *X, int32_t n_splits,
                                   const void *workspace, size_t workspace_bytes, ds4a_stream_t stream) {
  __half *ws_o = nullptr;
  float2 *ws_ml = nullptr;
  ds4a_status st = decode_setup(L, X, n_splits, workspace, workspace_bytes, false, true, &ws_o, &ws_ml);
  if (st != DS4A_OK || L->T == 0) return st;
  DeviceState *d = nullptr;
  st = current_device(&d);
  if (st != DS4A_OK) return st;
  return launched(ds4a::launch_combine(ws_o, ws_ml, n_splits, L->T, static_cast<__half *>(X->o),
                                       X->o_tok_stride / 2, X->lse, as_cuda(stream)));
}

ds4a_status ds4a_attn_decode(const ds4a_layout *L, const ds4a_tensors *X, int32_t n_splits, void *workspace,
                             size_t workspace_bytes, ds4a_stream_t stream) {
  __half *ws_o = nullptr;
  float2 *ws_ml = nullptr;
  ds4a_status st = decode_setup(L, X, n_splits, workspace, workspace_bytes, true, true, &ws_o, &ws_ml);
  if (st != DS4A_OK || L->T == 0) return st;
  st = decode_partials(L, X, n_splits, ws_o, ws_ml, stream);
  if (st != DS4A_OK) return st;
  return launched(ds4a::launch_combine(ws_o, ws_ml, n_splits, L->T, static_cast<__half *>(X->o),
                                       X->o_tok_stride / 2, X->lse, as_cuda(stream)));
}

}  // extern "C"

namespace {

bool e4m3_rows_ok(const void *k, const void *v, int64_t stride) {
  return k != nullptr && v != nullptr && aligned(k, 16) && aligned(v, 16) && stride >= DS4A_HEAD_DIM &&
         stride % 16 == 0 && stride < (1LL << 39);
}

bool scales_ok(const float *k, const float *v) { return k != nullptr && v != nullptr && aligned(k, 4) && aligned(v, 4); }

// E4M3 rows as bytes: {512, rows}, box {128 codes, 128 rows}, no swizzle.
ds4a_status encode_codes(CUtensorMap *m, const void *codes, int rows, int64_t stride) {
  const cuuint64_t dims[2] = {DS4A_HEAD_DIM, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)stride};
  const cuuint32_t box[2] = {128, 128};
  return encode(m, codes, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

// Checks and kernel parameters of an attention call whose compressed rows (and
// raw rows, when S->k_raw is given) are E4M3 codes with per-row scales.
ds4a_status e4m3_params(AttnParams &p, const ds4a_layout *L, const ds4a_tensors *X, const ds4a_fp8_scales *S,
                        DeviceState **dev, int mode = ds4a::MODE_STRUCT) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (X == nullptr || S == nullptr) return DS4A_ERR_INVALID_ARG;
  const bool raw_fp8 = S->k_raw != nullptr || S->v_raw != nullptr;
  // Q, O and the fp16 rows as usual (checked with the E4M3 segments left out).
  ds4a_layout L0 = *L;
  L0.n_comp = 0;
  if (raw_fp8) L0.n_raw = 0;
  st = check_tensors(&L0, X);
  if (st != DS4A_OK) return st;
  if (L->n_comp > 0 && (!e4m3_rows_ok(X->k_comp, X->v_comp, X->comp_row_stride) || !scales_ok(S->k_comp, S->v_comp)))
    return DS4A_ERR_INVALID_ARG;
  if (raw_fp8 && L->n_raw > 0 && (!e4m3_rows_ok(X->k_raw, X->v_raw, X->raw_row_stride) || !scales_ok(S->k_raw, S->v_raw)))
    return DS4A_ERR_INVALID_ARG;
  st = current_device(dev);
  if (st != DS4A_OK) return st;
  st = fill_params(p, &L0, X, mode, *dev);  // fp16 tensor maps only for fp16 segments
  if (st != DS4A_OK) return st;
  p.n_raw = L->n_raw;
  p.n_comp = L->n_comp;
  p.ratio = L->n_comp > 0 ? L->ratio : 1;
  p.nbr = ceil_div(L->n_raw, DS4A_BLOCK_ROWS);
  p.n_blocks = p.nbr + ceil_div(L->n_comp, DS4A_BLOCK_ROWS);
  p.comp_fp8 = 1;  // selects the E4M3 instantiation of the kernel
  p.raw_fp8 = raw_fp8 ? 1 : 0;
  p.alias_kv = 0;  // the E4M3 path reads K and V as two arrays
  if (L->n_comp > 0) {
    if ((st = encode_codes(&p.tm_k8[1], X->k_comp, L->n_comp, X->comp_row_stride)) != DS4A_OK) return st;
    if ((st = encode_codes(&p.tm_v8[1], X->v_comp, L->n_comp, X->comp_row_stride)) != DS4A_OK) return st;
  }
  if (raw_fp8 && L->n_raw > 0) {
    if ((st = encode_codes(&p.tm_k8[0], X->k_raw, L->n_raw, X->raw_row_stride)) != DS4A_OK) return st;
    if ((st = encode_codes(&p.tm_v8[0], X->v_raw, L->n_raw, X->raw_row_stride)) != DS4A_OK) return st;
  }
  p.k_scale[0] = S->k_raw;
  p.v_scale[0] = S->v_raw;
  p.k_scale[1] = S->k_comp;
  p.v_scale[1] = S->v_comp;
  return DS4A_OK;
}

}  // namespace

extern "C" {

ds4a_status ds4a_attn_decode_fp8kv(const ds4a_layout *L, const ds4a_tensors *X, const ds4a_fp8_scales *S,
                                   int32_t n_splits, void *workspace, size_t workspace_bytes, ds4a_stream_t stream) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (L->T == 0) return DS4A_OK;
  AttnParams p;
  DeviceState *d = nullptr;
  st = e4m3_params(p, L, X, S, &d);
  if (st != DS4A_OK) return st;
  if (n_splits <= 0) n_splits = ds4a_attn_decode_default_splits(L);
  if (n_splits > 4096) return DS4A_ERR_INVALID_ARG;
  const size_t need = ds4a_attn_decode_workspace_size(L, n_splits);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)) return DS4A_ERR_WORKSPACE;
  const size_t n_items = (size_t)L->T * n_splits;
  if (n_items > (size_t)INT32_MAX) return DS4A_ERR_INVALID_ARG;
  __half *ws_o = static_cast<__half *>(workspace);
  float2 *ws_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(workspace) +
                                             n_items * DS4A_HEADS * DS4A_HEAD_DIM * sizeof(__half));
  p.n_splits = n_splits;
  p.partial = 1;
  p.o = nullptr;
  p.lse = nullptr;
  p.ws_o = ws_o;
  p.ws_ml = ws_ml;
  const int grid = (int)(n_items < (size_t)d->sm_count ? n_items : (size_t)d->sm_count);
  st = launched(ds4a::launch_attn(p, grid, as_cuda(stream)));
  if (st != DS4A_OK) return st;
  return launched(ds4a::launch_combine(ws_o, ws_ml, n_splits, L->T, static_cast<__half *>(X->o),
                                       X->o_tok_stride / 2, X->lse, as_cuda(stream)));
}

ds4a_status ds4a_attn_decode_fp8(const ds4a_layout *L, const ds4a_tensors *X, const float *k_comp_scale,
                                 const float *v_comp_scale, int32_t n_splits, void *workspace,
                                 size_t workspace_bytes, ds4a_stream_t stream) {
  const ds4a_fp8_scales S = {nullptr, nullptr, k_comp_scale, v_comp_scale};
  return ds4a_attn_decode_fp8kv(L, X, &S, n_splits, workspace, workspace_bytes, stream);
}

ds4a_status ds4a_attn_prefill_fp8kv(const ds4a_layout *L, const ds4a_tensors *X, const ds4a_fp8_scales *S,
                                    ds4a_stream_t stream) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (L->T == 0) return DS4A_OK;
  AttnParams p;
  DeviceState *d = nullptr;
  st = e4m3_params(p, L, X, S, &d);
  if (st != DS4A_OK) return st;
  const int grid = L->T < d->sm_count ? L->T : d->sm_count;
  return launched(ds4a::launch_attn(p, grid, as_cuda(stream)));
}

}  // extern "C"

namespace {

// The raw rows [lo, hi) that some query of a raw-only E4M3 prefill sees, when
// the call takes the pair kernel (window <= 128, T >= 2; the window rule
// t - window < position <= t); false otherwise.
bool fp8_pair_rows(const ds4a_layout *L, int64_t *lo, int64_t *hi) {
  if (L->n_comp != 0 || L->n_raw <= 0 || L->window > 128 || L->T < 2) return false;
  const int64_t a = (int64_t)L->q_pos0 - L->window + 1 - L->raw_pos0;
  const int64_t b = (int64_t)L->q_pos0 + L->T - L->raw_pos0;
  *lo = a < 0 ? 0 : a;
  *hi = b > L->n_raw ? L->n_raw : b;
  return *hi > *lo;
}

}  // namespace

extern "C" {

size_t ds4a_attn_prefill_fp8kv_workspace_size(const ds4a_layout *L) {
  int64_t lo = 0, hi = 0;
  if (check_layout(L) != DS4A_OK || !fp8_pair_rows(L, &lo, &hi)) return 0;
  return (size_t)(hi - lo) * 2 * DS4A_ROW_BYTES;
}

ds4a_status ds4a_attn_prefill_fp8kv_ws(const ds4a_layout *L, const ds4a_tensors *X, const ds4a_fp8_scales *S,
                                       void *workspace, size_t workspace_bytes, ds4a_stream_t stream) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (L->T == 0) return DS4A_OK;
  int64_t lo = 0, hi = 0;
  if (X == nullptr || S == nullptr || S->k_raw == nullptr || !fp8_pair_rows(L, &lo, &hi))
    return ds4a_attn_prefill_fp8kv(L, X, S, stream);
  // Q and O as usual (checked with the E4M3 rows left out), then the codes.
  ds4a_layout L0 = *L;
  L0.n_raw = 0;
  st = check_tensors(&L0, X);
  if (st != DS4A_OK) return st;
  if (!e4m3_rows_ok(X->k_raw, X->v_raw, X->raw_row_stride) || !scales_ok(S->k_raw, S->v_raw))
    return DS4A_ERR_INVALID_ARG;
  const int32_t rows = (int32_t)(hi - lo);
  const size_t need = (size_t)rows * 2 * DS4A_ROW_BYTES;
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)) return DS4A_ERR_WORKSPACE;
  DeviceState *d = nullptr;
  st = current_device(&d);
  if (st != DS4A_OK) return st;
  // Each visible row's values decoded once, into fp16 rows of the workspace (K then V).
  __half *kw = static_cast<__half *>(workspace);
  __half *vw = kw + (size_t)rows * DS4A_HEAD_DIM;
  const uint8_t *kc = static_cast<const uint8_t *>(X->k_raw) + lo * X->raw_row_stride;
  const uint8_t *vc = static_cast<const uint8_t *>(X->v_raw) + lo * X->raw_row_stride;
  st = launched(ds4a::launch_widen_e4m3_rows(kc, vc, S->k_raw + lo, S->v_raw + lo, X->raw_row_stride, rows, kw, vw,
                                             as_cuda(stream)));
  if (st != DS4A_OK) return st;
  ds4a_layout L1 = *L;
  L1.raw_pos0 = (int32_t)(L->raw_pos0 + lo);
  L1.n_raw = rows;
  ds4a_tensors X1 = *X;
  X1.k_raw = kw;
  X1.v_raw = vw;
  X1.raw_row_stride = DS4A_ROW_BYTES;
  return prefill_pairs(&L1, &X1, d, stream);
}

// ------------------------------------------------------------------ batched decode

namespace {

// K/V rows of a batch: {512 dims, rows, sequences}, box {64, 128, 1}, 128-byte swizzle.
ds4a_status encode_batch_rows(CUtensorMap *m, const void *base, int rows, int64_t row_stride, int n_seq,
                              int64_t seq_stride) {
  const cuuint64_t dims[3] = {DS4A_HEAD_DIM, (cuuint64_t)rows, (cuuint64_t)n_seq};
  const cuuint64_t strides[2] = {(cuuint64_t)row_stride, (cuuint64_t)seq_stride};
  const cuuint32_t box[3] = {64, 128, 1};
  return encode(m, base, 3, dims, strides, box);
}

bool batch_rows_ok(const void *k, const void *v, int32_t rows, int64_t row_stride, int64_t seq_stride) {
  if (rows == 0) return true;
  return k != nullptr && v != nullptr && aligned(k, 16) && aligned(v, 16) && row_stride_ok(row_stride) &&
         seq_stride % 16 == 0 && seq_stride >= (int64_t)rows * row_stride && seq_stride < (1LL << 39);
}

}  // namespace

int32_t ds4a_attn_decode_batch_default_splits(int32_t n_seq, const ds4a_layout *shape, int32_t raw_rows,
                                              int32_t comp_rows) {
  if (n_seq <= 0 || shape == nullptr || raw_rows < 0 || comp_rows < 0 || shape->window < 1) return 1;
  int sms = 148, dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  }
  const int64_t raw = raw_rows < shape->window ? raw_rows : shape->window;
  const int32_t mt = ceil_div(raw, 128) + (raw > 0 ? 1 : 0) + ceil_div(comp_rows, 128);
  // Whole SMs per sequence (rounded down): with many sequences, extra splits
  // cost more (another wave of short items, a wider merge) than they gain.
  int32_t s = sms / n_seq;
  if (s > mt) s = mt;
  return s < 1 ? 1 : s;
}

size_t ds4a_attn_decode_batch_workspace_size(int32_t n_seq, int32_t n_splits) {
  if (n_seq <= 0 || n_splits <= 0) return 0;
  return (size_t)n_seq * (size_t)n_splits * DS4A_HEADS * (DS4A_HEAD_DIM * sizeof(__half) + 2 * sizeof(float));
}

ds4a_status ds4a_attn_decode_batch(int32_t n_seq, const ds4a_layout *shape, const int32_t *seq_geom,
                                   const ds4a_batch_tensors *X, int32_t n_splits, void *workspace,
                                   size_t workspace_bytes, ds4a_stream_t stream) {
  if (n_seq < 0 || shape == nullptr || X == nullptr) return DS4A_ERR_INVALID_ARG;
  if (n_seq == 0) return DS4A_OK;
  if (shape->window < 1 || !std::isfinite(shape->scale) || X->raw_rows < 0 || X->comp_rows < 0 ||
      X->raw_rows > (1 << 30) || X->comp_rows > (1 << 30) || (X->comp_rows > 0 && shape->ratio < 1))
    return DS4A_ERR_INVALID_ARG;
  if (seq_geom == nullptr || !aligned(seq_geom, 16)) return DS4A_ERR_INVALID_ARG;
  if (X->q == nullptr || !aligned(X->q, 16) || !tok_stride_ok(X->q_seq_stride)) return DS4A_ERR_INVALID_ARG;
  if (X->o == nullptr || !aligned(X->o, 16) || !tok_stride_ok(X->o_seq_stride)) return DS4A_ERR_INVALID_ARG;
  if (X->lse != nullptr && !aligned(X->lse, 4)) return DS4A_ERR_INVALID_ARG;
  if (!batch_rows_ok(X->k_raw, X->v_raw, X->raw_rows, X->raw_row_stride, X->raw_seq_stride) ||
      !batch_rows_ok(X->k_comp, X->v_comp, X->comp_rows, X->comp_row_stride, X->comp_seq_stride))
    return DS4A_ERR_INVALID_ARG;
  if (n_splits <= 0) n_splits = ds4a_attn_decode_batch_default_splits(n_seq, shape, X->raw_rows, X->comp_rows);
  if (n_splits > 4096) return DS4A_ERR_INVALID_ARG;
  const size_t n_items = (size_t)n_seq * n_splits;
  if (n_items > (size_t)INT32_MAX) return DS4A_ERR_INVALID_ARG;
  const size_t need = ds4a_attn_decode_batch_workspace_size(n_seq, n_splits);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)) return DS4A_ERR_WORKSPACE;
  DeviceState *d = nullptr;
  ds4a_status st = current_device(&d);
  if (st != DS4A_OK) return st;
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  if ((st = encode_q_blocks(&p.tm_q, X->q, n_seq, X->q_seq_stride)) != DS4A_OK) return st;
  if (X->raw_rows > 0) {
    st = encode_batch_rows(&p.tm_k[0], X->k_raw, X->raw_rows, X->raw_row_stride, n_seq, X->raw_seq_stride);
    if (st == DS4A_OK)
      st = encode_batch_rows(&p.tm_v[0], X->v_raw, X->raw_rows, X->raw_row_stride, n_seq, X->raw_seq_stride);
    if (st != DS4A_OK) return st;
  }
  if (X->comp_rows > 0) {
    st = encode_batch_rows(&p.tm_k[1], X->k_comp, X->comp_rows, X->comp_row_stride, n_seq, X->comp_seq_stride);
    if (st == DS4A_OK)
      st = encode_batch_rows(&p.tm_v[1], X->v_comp, X->comp_rows, X->comp_row_stride, n_seq, X->comp_seq_stride);
    if (st != DS4A_OK) return st;
  }
  p.q_ptr = static_cast<const uint8_t *>(X->q);
  p.q_tok_bytes = X->q_seq_stride;
  p.tile_rows = 128;
  p.T = n_seq;
  p.n_raw = X->raw_rows;
  p.n_comp = X->comp_rows;
  p.ratio = X->comp_rows > 0 ? shape->ratio : 1;
  p.window = shape->window;
  p.scale_log2 = shape->scale * 1.4426950408889634f;
  p.mode = ds4a::MODE_STRUCT;
  p.n_splits = n_splits;
  p.q_tile = 1;
  p.batch_geom = reinterpret_cast<const int4 *>(seq_geom);
  p.alias_kv = ((X->raw_rows == 0 || X->k_raw == X->v_raw) && (X->comp_rows == 0 || X->k_comp == X->v_comp) &&
                X->raw_rows + X->comp_rows > 0) ? 1 : 0;
  p.partial = 1;
  __half *ws_o = static_cast<__half *>(workspace);
  float2 *ws_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(workspace) +
                                             n_items * DS4A_HEADS * DS4A_HEAD_DIM * sizeof(__half));
  p.ws_o = ws_o;
  p.ws_ml = ws_ml;
  p.timeout_ns = kDefaultTimeoutNs;
  p.err = d->err;
  const int grid = (int)(n_items < (size_t)d->sm_count ? n_items : (size_t)d->sm_count);
  st = launched(ds4a::launch_attn(p, grid, as_cuda(stream)));
  if (st != DS4A_OK) return st;
  return launched(ds4a::launch_combine(ws_o, ws_ml, n_splits, n_seq, static_cast<__half *>(X->o),
                                       X->o_seq_stride / 2, X->lse, as_cuda(stream)));
}

ds4a_status ds4a_attn_decode_noalloc(const ds4a_layout *L, const ds4a_tensors *X, int32_t n_splits,
                                     ds4a_stream_t stream) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (L->T == 0) return DS4A_OK;
  // Items (token, split) that fit in the scratch array.
  const size_t per_item = ds4a_attn_decode_workspace_size(L, 1) / (size_t)L->T;
  const size_t max_items = kNoAllocScratchBytes / per_item;
  if ((size_t)L->T > max_items) return DS4A_ERR_WORKSPACE;
  if (n_splits <= 0) {
    n_splits = ds4a_attn_decode_default_splits(L);
    const int32_t cap = (int32_t)(max_items / (size_t)L->T);
    if (n_splits > cap) n_splits = cap;
  } else if ((size_t)L->T * (size_t)n_splits > max_items) {
    return DS4A_ERR_WORKSPACE;
  }
  DeviceState *d = nullptr;
  st = current_device(&d);  // the first call on a device looks up the scratch address
  if (st != DS4A_OK) return st;
  __half *ws_o = nullptr;
  float2 *ws_ml = nullptr;
  st = decode_setup(L, X, n_splits, d->scratch, kNoAllocScratchBytes, true, true, &ws_o, &ws_ml);
  if (st != DS4A_OK) return st;
  st = decode_partials(L, X, n_splits, ws_o, ws_ml, stream);
  if (st != DS4A_OK) return st;
  return launched(ds4a::launch_combine(ws_o, ws_ml, n_splits, L->T, static_cast<__half *>(X->o),
                                       X->o_tok_stride / 2, X->lse, as_cuda(stream)));
}

ds4a_status ds4a_attn_indexed(const ds4a_layout *L, const ds4a_tensors *X, const int32_t *idx,
                              int64_t idx_row_stride, int32_t top_k, ds4a_stream_t stream) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (top_k < 1 || top_k > 4096) return DS4A_ERR_INVALID_ARG;
  if (L->T == 0) return DS4A_OK;
  st = check_tensors(L, X);
  if (st != DS4A_OK) return st;
  if (idx == nullptr || !aligned(idx, 16) || idx_row_stride < 4LL * top_k || idx_row_stride % 16 != 0)
    return DS4A_ERR_INVALID_ARG;
  DeviceState *d = nullptr;
  st = current_device(&d);
  if (st != DS4A_OK) return st;
  AttnParams p;
  st = fill_params(p, L, X, ds4a::MODE_INDEXED, d);
  if (st != DS4A_OK) return st;
  // Gathered rows come from L2, where the look-ahead ring order (the K parts
  // of the next tile before the V parts of this one) gains more than loading
  // each row once for both products, which holds a tile's parts in the ring
  // from QK^T to PV (2048 tokens, top-512 of 8192 rows, K = V rows: 343 us
  // loaded once, 313 us read apart): K and V are read apart even when they
  // are the same rows.
  p.alias_kv = 0;
  p.idx = idx;
  p.idx_stride = idx_row_stride / 4;
  p.top_k = top_k;
  const int grid = L->T < d->sm_count ? L->T : d->sm_count;
  return launched(ds4a::launch_attn(p, grid, as_cuda(stream)));
}

ds4a_status ds4a_attn_indexed_fp8kv(const ds4a_layout *L, const ds4a_tensors *X, const ds4a_fp8_scales *S,
                                   const int32_t *idx, int64_t idx_row_stride, int32_t top_k, ds4a_stream_t stream) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (top_k < 1 || top_k > 4096) return DS4A_ERR_INVALID_ARG;
  if (L->T == 0) return DS4A_OK;
  if (S == nullptr || (L->n_comp > 0 && (S->k_comp == nullptr || S->v_comp == nullptr)))
    return DS4A_ERR_INVALID_ARG;  // the listed rows are E4M3
  if (idx == nullptr || !aligned(idx, 16) || idx_row_stride < 4LL * top_k || idx_row_stride % 16 != 0)
    return DS4A_ERR_INVALID_ARG;
  AttnParams p;
  DeviceState *d = nullptr;
  st = e4m3_params(p, L, X, S, &d, ds4a::MODE_INDEXED);
  if (st != DS4A_OK) return st;
  p.idx = idx;
  p.idx_stride = idx_row_stride / 4;
  p.top_k = top_k;
  const int grid = L->T < d->sm_count ? L->T : d->sm_count;
  return launched(ds4a::launch_attn(p, grid, as_cuda(stream)));
}

ds4a_status ds4a_device_error_word(ds4a_stream_t stream, uint32_t *word, int clear) {
  if (word == nullptr) return DS4A_ERR_INVALID_ARG;
  *word = 0;
  DeviceState *d = nullptr;
  ds4a_status st = current_device(&d);
  if (st != DS4A_OK) return st;
  DS4A_CUDA_TRY(cudaStreamSynchronize(as_cuda(stream)));
  unsigned int v = 0;
  DS4A_CUDA_TRY(cudaMemcpy(&v, d->err, sizeof(v), cudaMemcpyDeviceToHost));
  if (clear && v != 0) {
    const unsigned int zero = 0;
    DS4A_CUDA_TRY(cudaMemcpy(d->err, &zero, sizeof(zero), cudaMemcpyHostToDevice));
  }
  *word = v;
  return DS4A_OK;
}

ds4a_status ds4a_device_status(ds4a_stream_t stream, int clear) {
  uint32_t v = 0;
  const ds4a_status st = ds4a_device_error_word(stream, &v, clear);
  if (st != DS4A_OK) return st;
  return v != 0 ? DS4A_ERR_TIMEOUT : DS4A_OK;
}

ds4a_status ds4a_selftest_wait_timeout(uint64_t timeout_ns, ds4a_stream_t stream) {
  if (timeout_ns < 1000ull || timeout_ns > 10000000000ull) return DS4A_ERR_INVALID_ARG;
  DeviceState *d = nullptr;
  ds4a_status st = current_device(&d);
  if (st != DS4A_OK) return st;
  return launched(ds4a::launch_selftest_wait(timeout_ns, d->err, as_cuda(stream)));
}

}  // extern "C"

// ------------------------------------------------------------------ indexer

namespace {

bool indexer_heads_ok(int32_t n) { return n >= 1 && n <= 128 && (n & (n - 1)) == 0; }

}  // namespace

ds4a_status ds4a_indexer_scores(const ds4a_layout *L, const void *q_idx, int64_t q_tok_stride, int32_t n_heads,
                                int32_t head_dim, const void *k_idx, int64_t k_row_stride,
                                const float *head_weights, float scale, int32_t relu, float *scores,
                                int64_t score_row_stride, ds4a_stream_t stream) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (!indexer_heads_ok(n_heads) || (head_dim != 64 && head_dim != 128 && head_dim != 256)) return DS4A_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return DS4A_ERR_INVALID_ARG;
  if (L->T == 0 || L->n_comp == 0) return DS4A_OK;
  const int64_t q_row = 2LL * n_heads * head_dim;
  if (q_idx == nullptr || !aligned(q_idx, 16) || q_tok_stride % 16 != 0 || q_tok_stride < q_row ||
      q_tok_stride >= (1LL << 39))
    return DS4A_ERR_INVALID_ARG;
  if (k_idx == nullptr || !aligned(k_idx, 16) || k_row_stride % 16 != 0 || k_row_stride < 2LL * head_dim ||
      k_row_stride >= (1LL << 39))
    return DS4A_ERR_INVALID_ARG;
  if (head_weights == nullptr || !aligned(head_weights, 4)) return DS4A_ERR_INVALID_ARG;
  if (scores == nullptr || !aligned(scores, 16) || score_row_stride % 16 != 0 ||
      score_row_stride < 4LL * L->n_comp || score_row_stride >= (1LL << 39))
    return DS4A_ERR_INVALID_ARG;
  DeviceState *d = nullptr;
  st = current_device(&d);
  if (st != DS4A_OK) return st;
  ds4a::ScoreParams p;
  std::memset(&p, 0, sizeof(p));
  p.g = ds4a::IndexerGeom{L->T, L->q_pos0, L->n_comp, L->ratio};
  const int G = 256 / n_heads;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_heads, (cuuint64_t)L->T};
    const cuuint64_t strides[2] = {(cuuint64_t)(2 * head_dim), (cuuint64_t)q_tok_stride};
    const cuuint32_t box[3] = {64, (cuuint32_t)n_heads, (cuuint32_t)G};
    if ((st = encode(&p.tm_q, q_idx, 3, dims, strides, box)) != DS4A_OK) return st;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)L->n_comp};
    const cuuint64_t strides[1] = {(cuuint64_t)k_row_stride};
    const cuuint32_t box[2] = {64, 128};
    if ((st = encode(&p.tm_k, k_idx, 2, dims, strides, box)) != DS4A_OK) return st;
  }
  p.w = head_weights;
  p.scores = scores;
  p.score_stride = score_row_stride / 4;
  p.scale = scale;
  p.relu = relu != 0;
  p.head_dim = head_dim;
  p.n_groups = ceil_div(L->T, G);
  p.n_row_tiles = ceil_div(L->n_comp, 128);
  // Cut each group's row tiles into items so that there are a few per SM.
  int ipg = ceil_div(4LL * d->sm_count, p.n_groups);
  if (ipg < 1) ipg = 1;
  if (ipg > p.n_row_tiles) ipg = p.n_row_tiles;
  p.tiles_per_item = ceil_div(p.n_row_tiles, ipg);
  p.items_per_group = ceil_div(p.n_row_tiles, p.tiles_per_item);
  p.timeout_ns = kDefaultTimeoutNs;
  p.err = d->err;
  const long long items = (long long)p.n_groups * p.items_per_group;
  if (items > INT32_MAX) return DS4A_ERR_INVALID_ARG;
  const int grid = (int)(items < d->sm_count ? items : d->sm_count);
  return launched(ds4a::launch_indexer_scores(p, n_heads, grid, as_cuda(stream)));
}

ds4a_status ds4a_indexer_topk(const ds4a_layout *L, const float *scores, int64_t score_row_stride, int32_t top_k,
                              int32_t *idx, int64_t idx_row_stride, ds4a_stream_t stream) {
  ds4a_status st = check_layout(L);
  if (st != DS4A_OK) return st;
  if (top_k < 1 || top_k > 4096) return DS4A_ERR_INVALID_ARG;
  if (L->T == 0) return DS4A_OK;
  if (idx == nullptr || !aligned(idx, 16) || idx_row_stride % 16 != 0 || idx_row_stride < 4LL * top_k ||
      idx_row_stride >= (1LL << 39))
    return DS4A_ERR_INVALID_ARG;
  if (L->n_comp > 0 && (scores == nullptr || !aligned(scores, 4) || score_row_stride % 4 != 0 ||
                        score_row_stride < 4LL * L->n_comp || score_row_stride >= (1LL << 39)))
    return DS4A_ERR_INVALID_ARG;
  DeviceState *d = nullptr;
  st = current_device(&d);
  if (st != DS4A_OK) return st;
  ds4a::TopkParams p;
  std::memset(&p, 0, sizeof(p));
  const int ratio = L->n_comp > 0 ? L->ratio : 1;
  p.g = ds4a::IndexerGeom{L->T, L->q_pos0, L->n_comp, ratio};
  p.scores = scores;
  p.score_stride = score_row_stride / 4;
  p.idx = idx;
  p.idx_stride = idx_row_stride / 4;
  p.top_k = top_k;
  // The last token has the most candidates.
  int64_t max_n = ((int64_t)L->q_pos0 + L->T) / ratio;
  if (max_n > L->n_comp) max_n = L->n_comp;
  // Keys in shared memory when every token's candidates fit; otherwise every
  // pass rereads the scores (the kernel variant without the cache).
  p.cached_keys = (max_n <= top_k || max_n > ds4a::kTopkMaxCachedKeys) ? 0 : (int)max_n;
  return launched(ds4a::launch_indexer_topk(p, p.cached_keys * 4, as_cuda(stream)));
}

// ------------------------------------------------------------------ recorded call sequences

struct ds4a_graph_s {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

extern "C" {

ds4a_status ds4a_graph_begin(ds4a_stream_t stream) {
  if (stream == nullptr) return DS4A_ERR_INVALID_ARG;  // the legacy default stream cannot be recorded
  DeviceState *d = nullptr;
  ds4a_status st = current_device(&d);
  if (st != DS4A_OK) return st;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!d->loaded) {
      // A kernel's first launch loads its code, which a recording does not allow.
      DS4A_CUDA_TRY(ds4a::preload_aux_kernels());
      DS4A_CUDA_TRY(ds4a::preload_indexer_kernels());
      DS4A_CUDA_TRY(ds4a::preload_compressor_kernels());
      d->loaded = true;
    }
  }
  DS4A_CUDA_TRY(cudaStreamBeginCapture(as_cuda(stream), cudaStreamCaptureModeThreadLocal));
  return DS4A_OK;
}

ds4a_status ds4a_graph_end(ds4a_stream_t stream, ds4a_graph *graph) {
  if (graph != nullptr) *graph = nullptr;
  if (stream == nullptr) return DS4A_ERR_INVALID_ARG;
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(as_cuda(stream), &g);  // ends the recording in every case
  if (e != cudaSuccess) {
    if (g != nullptr) cudaGraphDestroy(g);
    return cuda_failed("cudaStreamEndCapture", e);
  }
  if (graph == nullptr) {
    cudaGraphDestroy(g);
    return DS4A_ERR_INVALID_ARG;
  }
  cudaGraphExec_t x = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&x, g, 0);
  if (ei != cudaSuccess) {
    cudaGraphDestroy(g);
    return cuda_failed("cudaGraphInstantiate", ei);
  }
  ds4a_graph h = new (std::nothrow) ds4a_graph_s{g, x};
  if (h == nullptr) {
    cudaGraphExecDestroy(x);
    cudaGraphDestroy(g);
    return cuda_failed("allocation of the graph handle", (int)cudaErrorMemoryAllocation, nullptr);
  }
  *graph = h;
  return DS4A_OK;
}

ds4a_status ds4a_graph_launch(ds4a_graph graph, ds4a_stream_t stream) {
  if (graph == nullptr) return DS4A_ERR_INVALID_ARG;
  const cudaError_t e = cudaGraphLaunch(graph->exec, as_cuda(stream));
  return e == cudaSuccess ? DS4A_OK : cuda_failed("cudaGraphLaunch", e);
}

void ds4a_graph_destroy(ds4a_graph graph) {
  if (graph == nullptr) return;
  cudaGraphExecDestroy(graph->exec);
  cudaGraphDestroy(graph->graph);
  delete graph;
}

}  // extern "C"
