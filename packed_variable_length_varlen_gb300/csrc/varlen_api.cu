// varlen_api.cu -- the C ABI of libvarlen_attn (declared in varlen_attn.h):
// argument validation, 64-bit TMA descriptor encoding, grid sizing, launch,
// and the device status word.
//
// Lessons from the pages built in here:
//   * Every stride and extent handed to a TMA descriptor is computed in
//     64-bit (the "NVFP4 sm_120 persist-D path" pull request on ffpa-attn,
//     sections "Error" and "Root cause": int32 layout extents wrapped and the
//     descriptor's stride assertion aborted).  Strides are checked against
//     the real hardware limit (2^40 bytes) instead.
//   * Every operand, dout included, keeps its own row / head strides; nothing
//     is made contiguous ("[FA4] cute varlen backward: int32 overflow in
//     _bwd_preprocess", sections "Root cause" and "User-side workaround").
#include <cmath>
#include <cstring>
#include <climits>
#include <cstdint>
#include <algorithm>
#include <atomic>
#include <mutex>

#include "varlen_attn.h"
#include "varlen_internal.h"

namespace varlen {

__device__ unsigned int g_device_error = 0;

// Last CUDA error an entry point saw on this host thread (for diagnostics).
thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return VARLEN_ERR_CUDA;
}

namespace {
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
}  // namespace

int current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  *id = 0;
  if (get_current == nullptr || get_id == nullptr) return cuda_fail(cudaErrorNotSupported);
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cuda_fail(cudaErrorUnknown);
  if (ctx == nullptr) return VARLEN_OK;
  if (get_id(ctx, id) != CUDA_SUCCESS) return cuda_fail(cudaErrorUnknown);
  return VARLEN_OK;
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct DeviceInfo {
  int sms = 0;
  int major = 0, minor = 0;
  unsigned int* err = nullptr;      // device address of g_device_error in the context below
  unsigned long long ctx_id = 0;    // the context err was looked up in (0: none yet)
};

constexpr int kMaxDevices = 64;

// Per-device attribute cache (the only host state of the library besides
// the optional profiling events).  The device address of g_device_error
// belongs to a CUDA context, not to the device: it is looked up again
// whenever the context current on the calling thread differs from the one
// it was looked up in (after cudaDeviceReset, or under a caller's own
// driver-API context on the same device).
int device_info(DeviceInfo* out) {
  static DeviceInfo cache[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = cache[dev];
  if (d.sms == 0) {
    int sms = 0, major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    d.major = major;
    d.minor = minor;
    d.sms = sms;
  }
  if (d.major != 10 || d.minor != 3) {
    *out = d;
    return VARLEN_ERR_ARCH;
  }
  unsigned long long ctx = 0;
  int st = current_context_id(&ctx);
  if (st != VARLEN_OK) return st;
  if (ctx == 0 || ctx != d.ctx_id || d.err == nullptr) {
    // (the lookup makes the device's primary context current when no
    // context was, so the identity is read again afterwards)
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_device_error)) != cudaSuccess) return cuda_fail(e);
    if ((st = current_context_id(&ctx)) != VARLEN_OK) return st;
    d.err = static_cast<unsigned int*>(p);
    d.ctx_id = ctx;
  }
  *out = d;
  return VARLEN_OK;
}

}  // namespace

int device_ready() {
  DeviceInfo d;
  return device_info(&d);
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates one NHD operand (pointer, strides) of `rows` rows.
int check_operand(const void* ptr, varlen_stride s, int64_t rows, int32_t H, int32_t D) {
  if (rows > 0 && ptr == nullptr) return VARLEN_ERR_NULL;
  if (ptr != nullptr && !aligned16(ptr)) return VARLEN_ERR_ALIGN;
  if (s.row < 0 || s.head < 0 || (s.row & 7) != 0 || (s.head & 7) != 0) return VARLEN_ERR_STRIDE;
  // Highest element touched must be addressable with a 64-bit offset, and
  // each byte stride must fit the TMA descriptor's 40-bit field.
  if (s.row >= (int64_t(1) << 39) || s.head >= (int64_t(1) << 39)) return VARLEN_ERR_STRIDE;
  (void)H;
  (void)D;
  return VARLEN_OK;
}

// An output operand must also not overlap itself: its rows * H vectors of
// D elements go to distinct addresses (else two CTAs would race on one
// element).  Sufficient condition, over the dimensions of extent > 1
// ordered by stride: the smaller stride is at least D and the larger at
// least the smaller's extent times the smaller stride.  (Inputs may
// overlap: they are only read.)
int check_output(const void* ptr, varlen_stride s, int64_t rows, int32_t H, int32_t D) {
  int st = check_operand(ptr, s, rows, H, D);
  if (st != VARLEN_OK) return st;
  const bool many_rows = rows > 1, many_heads = H > 1;
  if (many_rows && many_heads) {
    const bool heads_inner = s.head <= s.row;
    const int64_t small = heads_inner ? s.head : s.row, big = heads_inner ? s.row : s.head;
    const int64_t n_small = heads_inner ? (int64_t)H : rows;
    if (small < D || big / n_small < small) return VARLEN_ERR_STRIDE;
  } else if (many_rows) {
    if (s.row < D) return VARLEN_ERR_STRIDE;
  } else if (many_heads) {
    if (s.head < D) return VARLEN_ERR_STRIDE;
  }
  return VARLEN_OK;
}

// A 3-D bf16 tensor map {D, H, rows} with byte strides {2*head, 2*row} and a
// {64, 1, box_rows} box in the 128-byte swizzle.  All arithmetic is 64-bit.
int encode_nhd(CUtensorMap* map, const void* base, varlen_stride s, int64_t rows, int32_t H, int32_t D,
               int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return VARLEN_ERR_CUDA;
  // A stride over a dimension of extent 1 is never used; give it a legal value.
  int64_t hs = (H > 1) ? s.head : (int64_t)D;
  int64_t rs = (rows > 1) ? s.row : (int64_t)H * hs;
  if (hs == 0 || rs == 0) return VARLEN_ERR_STRIDE;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)hs * 2u, (cuuint64_t)rs * 2u};
  cuuint32_t box[3] = {64u, 1u, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  // A zero-row operand is never loaded, but the descriptor needs an address.
  static const uint4 dummy_host = {0, 0, 0, 0};
  void* addr = const_cast<void*>(base != nullptr ? base : static_cast<const void*>(&dummy_host));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, addr, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VARLEN_OK : VARLEN_ERR_STRIDE;
}

// The fp32 dQ accumulator [total_q, H, D] as a 3-D tensor map for bulk
// reduce-add of 32 (d) x 1 (head) x 64 (rows) boxes.
int encode_dq_acc(CUtensorMap* map, float* base, int64_t rows, int32_t H, int32_t D) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return VARLEN_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4u, (cuuint64_t)H * (cuuint64_t)D * 4u};
  cuuint32_t box[3] = {32u, 1u, 64u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VARLEN_OK : VARLEN_ERR_STRIDE;
}

int check_common(int32_t batch, int32_t total_q, int32_t total_k, int32_t H, int32_t D, float scale) {
  if (batch < 1 || total_q < 0 || total_k < 0 || H < 1) return VARLEN_ERR_SHAPE;
  if (D != 64 && D != 96 && D != 128) return VARLEN_ERR_HEAD_DIM;
  if (!(scale > 0.f) || !std::isfinite(scale)) return VARLEN_ERR_SHAPE;
  // H*total fits comfortably in int64; H itself bounded for TMA (<= 2^32).
  return VARLEN_OK;
}

constexpr float kLog2e = 1.4426950408889634f;

// Optional profiling events for the three backward kernels (process-wide).
cudaEvent_t g_phase_events[4] = {nullptr, nullptr, nullptr, nullptr};
std::mutex g_phase_mu;

// Debug knobs (process-wide): bytes taken off every operand span (the
// bounds checker's self test) and the load the forward / backward producer
// of CTA 0 leaves out (the failure test).
std::atomic<int64_t> g_span_slack{0};
std::atomic<int64_t> g_skip_fwd_load{-1}, g_skip_bwd_step{-1};

// Bytes an NHD operand of `rows` rows occupies from its base: up to the end
// of its last (row, head) vector.
Span nhd_span(const void* base, varlen_stride s, int64_t rows, int32_t H, int32_t D) {
  if (base == nullptr || rows <= 0 || H <= 0) return Span{base, 0};
  const int64_t last = (rows - 1) * s.row + (int64_t)(H - 1) * s.head + D;
  return Span{base, std::max<int64_t>(0, 2 * last - g_span_slack.load())};
}
Span flat_span(const void* base, int64_t bytes) {
  return Span{base, std::max<int64_t>(0, bytes - g_span_slack.load())};
}
int32_t skip_knob(const std::atomic<int64_t>& k) {
  const int64_t v = k.load();
  return v < 0 || v > INT32_MAX ? -1 : (int32_t)v;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// E4M3 codes [rows][H][128] as a 3-D uint8 tensor map {128, H, rows} with
// {128, 1, 128} boxes in the 128-byte swizzle.
int encode_codes_nhd(CUtensorMap* map, void* base, int64_t rows, int32_t H) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return VARLEN_ERR_CUDA;
  cuuint64_t dims[3] = {128u, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {128u, (cuuint64_t)H * 128u};
  cuuint32_t box[3] = {128u, 1u, 128u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VARLEN_OK : VARLEN_ERR_STRIDE;
}

// V^T codes [H][128][kp] as {kp, 128, H} with {128, 128, 1} boxes.
int encode_codes_vt(CUtensorMap* map, void* base, int64_t kp, int32_t H) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return VARLEN_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)kp, 128u, (cuuint64_t)H};
  cuuint64_t strides[2] = {(cuuint64_t)kp, (cuuint64_t)kp * 128u};
  cuuint32_t box[3] = {128u, 128u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VARLEN_OK : VARLEN_ERR_STRIDE;
}

// Workspace sections of the E4M3 forward: amax [3][batch * H] fp32, then
// the Q and K codes, then V^T; each section 256-byte aligned.
void fp8_sections(int32_t batch, int32_t total_q, int32_t total_k, int32_t H, size_t off[5]) {
  const size_t kp = (size_t)fp8_vt_cols(batch, total_k);
  off[0] = 0;
  off[1] = off[0] + round256((size_t)3 * batch * H * sizeof(float));
  off[2] = off[1] + round256((size_t)total_q * H * 128);
  off[3] = off[2] + round256((size_t)total_k * H * 128);
  off[4] = off[3] + round256((size_t)H * 128 * kp);
}

}  // namespace
}  // namespace varlen

using namespace varlen;

namespace {

// The visibility band of a launch from the public window sides (negative:
// unbounded).  No bounded side means no mask: the unmasked kernels run.
struct Band {
  int32_t masked;
  int64_t left, right;
};

Band band_of(int32_t window_left, int32_t window_right) {
  return Band{(window_left >= 0 || window_right >= 0) ? 1 : 0, window_left < 0 ? kWinUnbounded : window_left,
              window_right < 0 ? kWinUnbounded : window_right};
}

constexpr Band kNoMask{0, kWinUnbounded, kWinUnbounded};
constexpr Band kCausal{1, kWinUnbounded, 0};

int fwd_impl(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v, varlen_stride sv,
             CuView cu_q, CuView cu_k, int32_t batch, int32_t total_q, int32_t total_k, int32_t num_heads,
             int32_t head_dim, int32_t max_seqlen_q, int32_t max_seqlen_k, float scale, void* out,
             varlen_stride so, float* lse, void* stream, Band band) {
  (void)max_seqlen_q;  // advisory only: the kernels derive lengths from cu_seqlens
  (void)max_seqlen_k;
  int st = check_common(batch, total_q, total_k, num_heads, head_dim, scale);
  if (st != VARLEN_OK) return st;
  if ((st = check_operand(q, sq, total_q, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_operand(k, sk, total_k, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_operand(v, sv, total_k, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_output(out, so, total_q, num_heads, head_dim)) != VARLEN_OK) return st;
  if (total_q > 0 && lse == nullptr) return VARLEN_ERR_NULL;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != VARLEN_OK) return st;
  if (total_q == 0) return VARLEN_OK;
  FwdLaunch L;
  std::memset(&L, 0, sizeof(L));
  if ((st = encode_nhd(&L.tm_q, q, sq, total_q, num_heads, head_dim, kTileM)) != VARLEN_OK) return st;
  if ((st = encode_nhd(&L.tm_k, k, sk, total_k, num_heads, head_dim, kTileN)) != VARLEN_OK) return st;
  if ((st = encode_nhd(&L.tm_v, v, sv, total_k, num_heads, head_dim, kTileN)) != VARLEN_OK) return st;
  L.p.out = static_cast<__nv_bfloat16*>(out);
  L.p.o_rs = so.row;
  L.p.o_hs = so.head;
  L.p.lse = lse;
  L.p.cu_q = cu_q;
  L.p.cu_k = cu_k;
  L.p.batch = batch;
  L.p.total_q = total_q;
  L.p.total_k = total_k;
  L.p.num_heads = num_heads;
  L.p.masked = band.masked;
  L.p.win_left = band.left;
  L.p.win_right = band.right;
  L.p.scale_log2 = scale * kLog2e;
  L.p.err = dev.err;
  L.p.out_span = nhd_span(out, so, total_q, num_heads, head_dim);
  L.p.lse_span = flat_span(lse, (int64_t)num_heads * total_q * 4);
  L.p.debug_skip_load = skip_knob(g_skip_fwd_load);
  L.head_dim = head_dim;
  L.grid = dev.sms;
  cudaError_t e = launch_fwd(L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VARLEN_OK : cuda_fail(e);
}

}  // namespace

extern "C" int varlen_attn_fwd(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                               varlen_stride sv, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                               int32_t batch, int32_t total_q, int32_t total_k, int32_t num_heads, int32_t head_dim,
                               int32_t max_seqlen_q, int32_t max_seqlen_k, float scale, void* out,
                               varlen_stride so, float* lse, void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return VARLEN_ERR_NULL;
  return fwd_impl(q, sq, k, sk, v, sv, CuView{cu_seqlens_q, 0}, CuView{cu_seqlens_k, 0}, batch, total_q, total_k,
                  num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, out, so, lse, stream, kNoMask);
}

extern "C" int varlen_attn_fwd_causal(const void* q, varlen_stride sq, const void* k, varlen_stride sk,
                                      const void* v, varlen_stride sv, const int32_t* cu_seqlens_q,
                                      const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q, int32_t total_k,
                                      int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q,
                                      int32_t max_seqlen_k, float scale, void* out, varlen_stride so, float* lse,
                                      void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return VARLEN_ERR_NULL;
  return fwd_impl(q, sq, k, sk, v, sv, CuView{cu_seqlens_q, 0}, CuView{cu_seqlens_k, 0}, batch, total_q, total_k,
                  num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, out, so, lse, stream, kCausal);
}

extern "C" int varlen_attn_fwd_window(const void* q, varlen_stride sq, const void* k, varlen_stride sk,
                                      const void* v, varlen_stride sv, const int32_t* cu_seqlens_q,
                                      const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q, int32_t total_k,
                                      int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q,
                                      int32_t max_seqlen_k, float scale, int32_t window_left, int32_t window_right,
                                      void* out, varlen_stride so, float* lse, void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return VARLEN_ERR_NULL;
  return fwd_impl(q, sq, k, sk, v, sv, CuView{cu_seqlens_q, 0}, CuView{cu_seqlens_k, 0}, batch, total_q, total_k,
                  num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, out, so, lse, stream,
                  band_of(window_left, window_right));
}

extern "C" size_t varlen_attn_bwd_workspace_size(int32_t batch, int32_t total_q, int32_t num_heads,
                                                 int32_t head_dim) {
  if (batch < 0 || total_q < 0 || num_heads < 0 || head_dim < 0) return 0;
  const size_t rows = (size_t)total_q;
  const size_t prow = (size_t)varlen::bwd_pad_rows(batch, total_q);
  return round256(rows * num_heads * head_dim * sizeof(float)) + 2 * round256(prow * num_heads * sizeof(float));
}

namespace {

int bwd_impl(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v, varlen_stride sv,
             const void* out, varlen_stride so, const void* dout, varlen_stride sdo, const float* lse,
             CuView cu_q, CuView cu_k, int32_t batch, int32_t total_q, int32_t total_k, int32_t num_heads,
             int32_t head_dim, int32_t max_seqlen_q, int32_t max_seqlen_k, float scale, void* dq, varlen_stride sdq,
             void* dk, varlen_stride sdk, void* dv, varlen_stride sdv, void* workspace, size_t workspace_bytes,
             void* stream, Band band, int deterministic = 0) {
  (void)max_seqlen_q;
  (void)max_seqlen_k;
  int st = check_common(batch, total_q, total_k, num_heads, head_dim, scale);
  if (st != VARLEN_OK) return st;
  if ((st = check_operand(q, sq, total_q, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_operand(k, sk, total_k, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_operand(v, sv, total_k, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_operand(out, so, total_q, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_operand(dout, sdo, total_q, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_output(dq, sdq, total_q, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_output(dk, sdk, total_k, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_output(dv, sdv, total_k, num_heads, head_dim)) != VARLEN_OK) return st;
  if (total_q > 0 && lse == nullptr) return VARLEN_ERR_NULL;
  const size_t need = varlen_attn_bwd_workspace_size(batch, total_q, num_heads, head_dim);
  if (need > 0 && (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                   workspace_bytes < need))
    return VARLEN_ERR_WORKSPACE;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != VARLEN_OK) return st;
  if (total_q == 0 && total_k == 0) return VARLEN_OK;
  BwdLaunch L;
  std::memset(&L, 0, sizeof(L));
  if ((st = encode_nhd(&L.tm_q, q, sq, total_q, num_heads, head_dim, kBwdTileQ)) != VARLEN_OK) return st;
  if ((st = encode_nhd(&L.tm_do, dout, sdo, total_q, num_heads, head_dim, kBwdTileQ)) != VARLEN_OK) return st;
  if ((st = encode_nhd(&L.tm_k, k, sk, total_k, num_heads, head_dim, kTileM)) != VARLEN_OK) return st;
  if ((st = encode_nhd(&L.tm_v, v, sv, total_k, num_heads, head_dim, kTileM)) != VARLEN_OK) return st;
  char* ws = static_cast<char*>(workspace);
  float* dq_acc = reinterpret_cast<float*>(ws);
  const int64_t pad_rows = bwd_pad_rows(batch, total_q);
  float* delta = reinterpret_cast<float*>(ws + round256((size_t)total_q * num_heads * head_dim * sizeof(float)));
  float* lse2 = reinterpret_cast<float*>(reinterpret_cast<char*>(delta) +
                                         round256((size_t)pad_rows * num_heads * sizeof(float)));
  if ((st = encode_dq_acc(&L.tm_dq, dq_acc, total_q, num_heads, head_dim)) != VARLEN_OK) return st;
  L.prep = PrepParams{static_cast<const __nv_bfloat16*>(out), so.row, so.head,
                      static_cast<const __nv_bfloat16*>(dout), sdo.row, sdo.head,
                      lse, delta, lse2, deterministic ? nullptr : dq_acc, cu_q, batch, total_q, num_heads,
                      head_dim, pad_rows};
  L.p.dk = static_cast<__nv_bfloat16*>(dk);
  L.p.dk_rs = sdk.row;
  L.p.dk_hs = sdk.head;
  L.p.dv = static_cast<__nv_bfloat16*>(dv);
  L.p.dv_rs = sdv.row;
  L.p.dv_hs = sdv.head;
  L.p.delta = delta;
  L.p.lse2 = lse2;
  L.p.dq_acc = dq_acc;
  L.p.dq = static_cast<__nv_bfloat16*>(dq);
  L.p.dq_rs = sdq.row;
  L.p.dq_hs = sdq.head;
  L.p.cu_q = cu_q;
  L.p.cu_k = cu_k;
  L.p.batch = batch;
  L.p.total_q = total_q;
  L.p.total_k = total_k;
  L.p.num_heads = num_heads;
  L.p.pad_rows = pad_rows;
  L.p.masked = band.masked;
  L.p.win_left = band.left;
  L.p.win_right = band.right;
  L.p.scale_log2 = scale * kLog2e;
  L.p.scale = scale;
  L.p.err = dev.err;
  L.post = PostParams{dq_acc, static_cast<__nv_bfloat16*>(dq), sdq.row, sdq.head, cu_q, batch,
                      total_q, num_heads, head_dim, scale};
  const int64_t acc_bytes = (int64_t)total_q * num_heads * head_dim * 4;
  const int64_t row_bytes = pad_rows * num_heads * 4;
  L.prep.out_span = nhd_span(out, so, total_q, num_heads, head_dim);
  L.prep.dout_span = nhd_span(dout, sdo, total_q, num_heads, head_dim);
  L.prep.lse_span = flat_span(lse, (int64_t)num_heads * total_q * 4);
  L.prep.delta_span = flat_span(delta, row_bytes);
  L.prep.lse2_span = flat_span(lse2, row_bytes);
  L.prep.acc_span = flat_span(dq_acc, acc_bytes);
  L.prep.err = dev.err;
  L.p.dk_span = nhd_span(dk, sdk, total_k, num_heads, head_dim);
  L.p.dv_span = nhd_span(dv, sdv, total_k, num_heads, head_dim);
  L.p.dq_span = nhd_span(dq, sdq, total_q, num_heads, head_dim);
  L.p.debug_skip_step = skip_knob(g_skip_bwd_step);
  L.post.acc_span = flat_span(dq_acc, acc_bytes);
  L.post.dq_span = nhd_span(dq, sdq, total_q, num_heads, head_dim);
  L.post.err = dev.err;
  L.head_dim = head_dim;
  L.grid = dev.sms;
  L.deterministic = deterministic;
  {
    std::lock_guard<std::mutex> lock(g_phase_mu);
    for (int i = 0; i < 4; ++i) L.phase_events[i] = g_phase_events[i];
  }
  cudaError_t e = launch_bwd(L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VARLEN_OK : cuda_fail(e);
}

}  // namespace

extern "C" int varlen_attn_bwd(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                               varlen_stride sv, const void* out, varlen_stride so, const void* dout,
                               varlen_stride sdo, const float* lse, const int32_t* cu_seqlens_q,
                               const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q, int32_t total_k,
                               int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q, int32_t max_seqlen_k,
                               float scale, void* dq, varlen_stride sdq, void* dk, varlen_stride sdk, void* dv,
                               varlen_stride sdv, void* workspace, size_t workspace_bytes, void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return VARLEN_ERR_NULL;
  return bwd_impl(q, sq, k, sk, v, sv, out, so, dout, sdo, lse, CuView{cu_seqlens_q, 0}, CuView{cu_seqlens_k, 0},
                  batch, total_q, total_k, num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, dq, sdq, dk, sdk,
                  dv, sdv, workspace, workspace_bytes, stream, kNoMask);
}

extern "C" int varlen_attn_bwd_causal(const void* q, varlen_stride sq, const void* k, varlen_stride sk,
                                      const void* v, varlen_stride sv, const void* out, varlen_stride so,
                                      const void* dout, varlen_stride sdo, const float* lse,
                                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                                      int32_t total_q, int32_t total_k, int32_t num_heads, int32_t head_dim,
                                      int32_t max_seqlen_q, int32_t max_seqlen_k, float scale, void* dq,
                                      varlen_stride sdq, void* dk, varlen_stride sdk, void* dv, varlen_stride sdv,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return VARLEN_ERR_NULL;
  return bwd_impl(q, sq, k, sk, v, sv, out, so, dout, sdo, lse, CuView{cu_seqlens_q, 0}, CuView{cu_seqlens_k, 0},
                  batch, total_q, total_k, num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, dq, sdq, dk, sdk,
                  dv, sdv, workspace, workspace_bytes, stream, kCausal);
}

extern "C" int varlen_attn_bwd_window(const void* q, varlen_stride sq, const void* k, varlen_stride sk,
                                      const void* v, varlen_stride sv, const void* out, varlen_stride so,
                                      const void* dout, varlen_stride sdo, const float* lse,
                                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                                      int32_t total_q, int32_t total_k, int32_t num_heads, int32_t head_dim,
                                      int32_t max_seqlen_q, int32_t max_seqlen_k, float scale, int32_t window_left,
                                      int32_t window_right, void* dq, varlen_stride sdq, void* dk, varlen_stride sdk,
                                      void* dv, varlen_stride sdv, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return VARLEN_ERR_NULL;
  return bwd_impl(q, sq, k, sk, v, sv, out, so, dout, sdo, lse, CuView{cu_seqlens_q, 0}, CuView{cu_seqlens_k, 0},
                  batch, total_q, total_k, num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, dq, sdq, dk, sdk,
                  dv, sdv, workspace, workspace_bytes, stream, band_of(window_left, window_right));
}

extern "C" int varlen_attn_bwd_deterministic(
    const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v, varlen_stride sv,
    const void* out, varlen_stride so, const void* dout, varlen_stride sdo, const float* lse,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q, int32_t total_k,
    int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q, int32_t max_seqlen_k, float scale,
    int32_t window_left, int32_t window_right, void* dq, varlen_stride sdq, void* dk, varlen_stride sdk, void* dv,
    varlen_stride sdv, void* workspace, size_t workspace_bytes, void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return VARLEN_ERR_NULL;
  return bwd_impl(q, sq, k, sk, v, sv, out, so, dout, sdo, lse, CuView{cu_seqlens_q, 0}, CuView{cu_seqlens_k, 0},
                  batch, total_q, total_k, num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, dq, sdq, dk, sdk,
                  dv, sdv, workspace, workspace_bytes, stream, band_of(window_left, window_right), 1);
}

// ------------------------------------------------------------ dense batched

namespace {

// The dense layout [batch, seqlen, H, D] is the packed [batch * seqlen, H, D]
// layout when the batch stride is seqlen row strides (checked here), so the
// varlen kernels run it unchanged with uniform segments b * seqlen.
int dense_view(varlen_dense_stride s, int32_t seqlen, int32_t batch, varlen_stride* out) {
  if (batch > 1 && s.batch != (int64_t)seqlen * s.row) return VARLEN_ERR_STRIDE;
  *out = varlen_stride{s.row, s.head};
  return VARLEN_OK;
}

int dense_shape(int32_t batch, int32_t seqlen_q, int32_t seqlen_k, int32_t causal, int32_t* total_q,
                int32_t* total_k) {
  if (batch < 1 || seqlen_q < 0 || seqlen_k < 0 || (causal != 0 && causal != 1)) return VARLEN_ERR_SHAPE;
  const int64_t tq = (int64_t)batch * seqlen_q, tk = (int64_t)batch * seqlen_k;
  if (tq > INT32_MAX || tk > INT32_MAX) return VARLEN_ERR_SHAPE;
  *total_q = (int32_t)tq;
  *total_k = (int32_t)tk;
  return VARLEN_OK;
}

}  // namespace

extern "C" int varlen_attn_fwd_dense(const void* q, varlen_dense_stride sq, const void* k, varlen_dense_stride sk,
                                     const void* v, varlen_dense_stride sv, int32_t batch, int32_t seqlen_q,
                                     int32_t seqlen_k, int32_t num_heads, int32_t head_dim, float scale,
                                     int32_t causal, void* out, varlen_dense_stride so, float* lse, void* stream) {
  int32_t total_q = 0, total_k = 0;
  int st = dense_shape(batch, seqlen_q, seqlen_k, causal, &total_q, &total_k);
  if (st != VARLEN_OK) return st;
  varlen_stride vq, vk, vv, vo;
  if ((st = dense_view(sq, seqlen_q, batch, &vq)) != VARLEN_OK) return st;
  if ((st = dense_view(sk, seqlen_k, batch, &vk)) != VARLEN_OK) return st;
  if ((st = dense_view(sv, seqlen_k, batch, &vv)) != VARLEN_OK) return st;
  if ((st = dense_view(so, seqlen_q, batch, &vo)) != VARLEN_OK) return st;
  return fwd_impl(q, vq, k, vk, v, vv, CuView{nullptr, seqlen_q}, CuView{nullptr, seqlen_k}, batch, total_q, total_k,
                  num_heads, head_dim, seqlen_q, seqlen_k, scale, out, vo, lse, stream, causal ? kCausal : kNoMask);
}

extern "C" size_t varlen_attn_bwd_dense_workspace_size(int32_t batch, int32_t seqlen_q, int32_t num_heads,
                                                      int32_t head_dim) {
  if (batch < 0 || seqlen_q < 0) return 0;
  const int64_t tq = (int64_t)batch * seqlen_q;
  if (tq > INT32_MAX) return 0;
  return varlen_attn_bwd_workspace_size(batch, (int32_t)tq, num_heads, head_dim);
}

extern "C" int varlen_attn_bwd_dense(const void* q, varlen_dense_stride sq, const void* k, varlen_dense_stride sk,
                                     const void* v, varlen_dense_stride sv, const void* out, varlen_dense_stride so,
                                     const void* dout, varlen_dense_stride sdo, const float* lse, int32_t batch,
                                     int32_t seqlen_q, int32_t seqlen_k, int32_t num_heads, int32_t head_dim,
                                     float scale, int32_t causal, void* dq, varlen_dense_stride sdq, void* dk,
                                     varlen_dense_stride sdk, void* dv, varlen_dense_stride sdv, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  int32_t total_q = 0, total_k = 0;
  int st = dense_shape(batch, seqlen_q, seqlen_k, causal, &total_q, &total_k);
  if (st != VARLEN_OK) return st;
  varlen_stride vq, vk, vv, vo, vdo, vdq, vdk, vdv;
  if ((st = dense_view(sq, seqlen_q, batch, &vq)) != VARLEN_OK) return st;
  if ((st = dense_view(sk, seqlen_k, batch, &vk)) != VARLEN_OK) return st;
  if ((st = dense_view(sv, seqlen_k, batch, &vv)) != VARLEN_OK) return st;
  if ((st = dense_view(so, seqlen_q, batch, &vo)) != VARLEN_OK) return st;
  if ((st = dense_view(sdo, seqlen_q, batch, &vdo)) != VARLEN_OK) return st;
  if ((st = dense_view(sdq, seqlen_q, batch, &vdq)) != VARLEN_OK) return st;
  if ((st = dense_view(sdk, seqlen_k, batch, &vdk)) != VARLEN_OK) return st;
  if ((st = dense_view(sdv, seqlen_k, batch, &vdv)) != VARLEN_OK) return st;
  return bwd_impl(q, vq, k, vk, v, vv, out, vo, dout, vdo, lse, CuView{nullptr, seqlen_q}, CuView{nullptr, seqlen_k},
                  batch, total_q, total_k, num_heads, head_dim, seqlen_q, seqlen_k, scale, dq, vdq, dk, vdk, dv, vdv,
                  workspace, workspace_bytes, stream, causal ? kCausal : kNoMask);
}

// ------------------------------------------------------------ FP8 (E4M3)

extern "C" size_t varlen_attn_fwd_fp8_workspace_size(int32_t batch, int32_t total_q, int32_t total_k,
                                                     int32_t num_heads, int32_t head_dim) {
  if (batch < 0 || total_q < 0 || total_k < 0 || num_heads < 0 || head_dim != 128) return 0;
  size_t off[5];
  fp8_sections(batch, total_q, total_k, num_heads, off);
  return off[4];
}

extern "C" int varlen_attn_fwd_fp8_workspace_layout(int32_t batch, int32_t total_q, int32_t total_k,
                                                    int32_t num_heads, int32_t head_dim, size_t* offsets,
                                                    int64_t* vt_cols) {
  if (offsets == nullptr || vt_cols == nullptr) return VARLEN_ERR_NULL;
  if (batch < 1 || total_q < 0 || total_k < 0 || num_heads < 1) return VARLEN_ERR_SHAPE;
  if (head_dim != 128) return VARLEN_ERR_HEAD_DIM;
  size_t off[5];
  fp8_sections(batch, total_q, total_k, num_heads, off);
  for (int i = 0; i < 4; ++i) offsets[i] = off[i];
  *vt_cols = fp8_vt_cols(batch, total_k);
  return VARLEN_OK;
}

namespace {

// The E4M3 forward on segments given by cu_seqlens arrays, or (dense) by
// uniform lengths (CuView with a null pointer).
int fwd_fp8_impl(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v, varlen_stride sv,
                 CuView cu_q, CuView cu_k, int32_t batch, int32_t total_q, int32_t total_k, int32_t num_heads,
                 int32_t head_dim, float scale, void* out, varlen_stride so, float* lse, void* workspace,
                 size_t workspace_bytes, void* stream, Band band) {
  int st = check_common(batch, total_q, total_k, num_heads, head_dim, scale);
  if (st != VARLEN_OK) return st;
  if (head_dim != 128) return VARLEN_ERR_HEAD_DIM;
  if (fp8_vt_cols(batch, total_k) > INT32_MAX) return VARLEN_ERR_SHAPE;  // V^T columns are TMA coordinates
  if ((st = check_operand(q, sq, total_q, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_operand(k, sk, total_k, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_operand(v, sv, total_k, num_heads, head_dim)) != VARLEN_OK) return st;
  if ((st = check_output(out, so, total_q, num_heads, head_dim)) != VARLEN_OK) return st;
  if (total_q > 0 && lse == nullptr) return VARLEN_ERR_NULL;
  size_t off[5];
  fp8_sections(batch, total_q, total_k, num_heads, off);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < off[4])
    return VARLEN_ERR_WORKSPACE;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != VARLEN_OK) return st;
  if (total_q == 0 && total_k == 0) return VARLEN_OK;
  char* ws = static_cast<char*>(workspace);
  Fp8Launch L;
  std::memset(&L, 0, sizeof(L));
  L.p.q = static_cast<const __nv_bfloat16*>(q);
  L.p.k = static_cast<const __nv_bfloat16*>(k);
  L.p.v = static_cast<const __nv_bfloat16*>(v);
  L.p.q_rs = sq.row;
  L.p.q_hs = sq.head;
  L.p.k_rs = sk.row;
  L.p.k_hs = sk.head;
  L.p.v_rs = sv.row;
  L.p.v_hs = sv.head;
  L.p.out = static_cast<__nv_bfloat16*>(out);
  L.p.o_rs = so.row;
  L.p.o_hs = so.head;
  L.p.lse = lse;
  L.p.amax = reinterpret_cast<float*>(ws + off[0]);
  L.p.q8 = reinterpret_cast<uint8_t*>(ws + off[1]);
  L.p.k8 = reinterpret_cast<uint8_t*>(ws + off[2]);
  L.p.vt = reinterpret_cast<uint8_t*>(ws + off[3]);
  L.p.kp = fp8_vt_cols(batch, total_k);
  L.p.cu_q = cu_q;
  L.p.cu_k = cu_k;
  L.p.batch = batch;
  L.p.total_q = total_q;
  L.p.total_k = total_k;
  L.p.num_heads = num_heads;
  L.p.scale = scale;
  L.p.masked = band.masked;
  L.p.win_left = band.left;
  L.p.win_right = band.right;
  L.p.err = dev.err;
  L.p.q_span = nhd_span(q, sq, total_q, num_heads, head_dim);
  L.p.k_span = nhd_span(k, sk, total_k, num_heads, head_dim);
  L.p.v_span = nhd_span(v, sv, total_k, num_heads, head_dim);
  L.p.out_span = nhd_span(out, so, total_q, num_heads, head_dim);
  L.p.lse_span = flat_span(lse, (int64_t)num_heads * total_q * 4);
  L.p.amax_span = flat_span(L.p.amax, (int64_t)3 * batch * num_heads * 4);
  L.p.q8_span = flat_span(L.p.q8, (int64_t)total_q * num_heads * 128);
  L.p.k8_span = flat_span(L.p.k8, (int64_t)total_k * num_heads * 128);
  L.p.vt_span = flat_span(L.p.vt, (int64_t)num_heads * 128 * L.p.kp);
  L.grid = dev.sms;
  if ((st = encode_codes_nhd(&L.tm_q8, L.p.q8, total_q, num_heads)) != VARLEN_OK) return st;
  if ((st = encode_codes_nhd(&L.tm_k8, L.p.k8, total_k, num_heads)) != VARLEN_OK) return st;
  if ((st = encode_codes_vt(&L.tm_vt, L.p.vt, L.p.kp, num_heads)) != VARLEN_OK) return st;
  cudaError_t e = launch_fwd_fp8(L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VARLEN_OK : cuda_fail(e);
}

}  // namespace

extern "C" int varlen_attn_fwd_fp8(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                                   varlen_stride sv, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                   int32_t batch, int32_t total_q, int32_t total_k, int32_t num_heads,
                                   int32_t head_dim, int32_t max_seqlen_q, int32_t max_seqlen_k, float scale,
                                   void* out, varlen_stride so, float* lse, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  (void)max_seqlen_q;
  (void)max_seqlen_k;
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return VARLEN_ERR_NULL;
  return fwd_fp8_impl(q, sq, k, sk, v, sv, CuView{cu_seqlens_q, 0}, CuView{cu_seqlens_k, 0}, batch, total_q, total_k,
                      num_heads, head_dim, scale, out, so, lse, workspace, workspace_bytes, stream, kNoMask);
}

extern "C" int varlen_attn_fwd_fp8_window(const void* q, varlen_stride sq, const void* k, varlen_stride sk,
                                          const void* v, varlen_stride sv, const int32_t* cu_seqlens_q,
                                          const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q,
                                          int32_t total_k, int32_t num_heads, int32_t head_dim,
                                          int32_t max_seqlen_q, int32_t max_seqlen_k, float scale,
                                          int32_t window_left, int32_t window_right, void* out, varlen_stride so,
                                          float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  (void)max_seqlen_q;
  (void)max_seqlen_k;
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return VARLEN_ERR_NULL;
  return fwd_fp8_impl(q, sq, k, sk, v, sv, CuView{cu_seqlens_q, 0}, CuView{cu_seqlens_k, 0}, batch, total_q, total_k,
                      num_heads, head_dim, scale, out, so, lse, workspace, workspace_bytes, stream,
                      band_of(window_left, window_right));
}

extern "C" size_t varlen_attn_fwd_fp8_dense_workspace_size(int32_t batch, int32_t seqlen_q, int32_t seqlen_k,
                                                           int32_t num_heads, int32_t head_dim) {
  if (batch < 0 || seqlen_q < 0 || seqlen_k < 0) return 0;
  const int64_t tq = (int64_t)batch * seqlen_q, tk = (int64_t)batch * seqlen_k;
  if (tq > INT32_MAX || tk > INT32_MAX) return 0;
  return varlen_attn_fwd_fp8_workspace_size(batch, (int32_t)tq, (int32_t)tk, num_heads, head_dim);
}

extern "C" int varlen_attn_fwd_fp8_dense(const void* q, varlen_dense_stride sq, const void* k, varlen_dense_stride sk,
                                         const void* v, varlen_dense_stride sv, int32_t batch, int32_t seqlen_q,
                                         int32_t seqlen_k, int32_t num_heads, int32_t head_dim, float scale,
                                         int32_t causal, void* out, varlen_dense_stride so, float* lse,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  int32_t total_q = 0, total_k = 0;
  int st = dense_shape(batch, seqlen_q, seqlen_k, causal, &total_q, &total_k);
  if (st != VARLEN_OK) return st;
  varlen_stride vq, vk, vv, vo;
  if ((st = dense_view(sq, seqlen_q, batch, &vq)) != VARLEN_OK) return st;
  if ((st = dense_view(sk, seqlen_k, batch, &vk)) != VARLEN_OK) return st;
  if ((st = dense_view(sv, seqlen_k, batch, &vv)) != VARLEN_OK) return st;
  if ((st = dense_view(so, seqlen_q, batch, &vo)) != VARLEN_OK) return st;
  return fwd_fp8_impl(q, vq, k, vk, v, vv, CuView{nullptr, seqlen_q}, CuView{nullptr, seqlen_k}, batch, total_q,
                      total_k, num_heads, head_dim, scale, out, vo, lse, workspace, workspace_bytes, stream,
                      causal ? kCausal : kNoMask);
}

extern "C" int varlen_attn_get_device_status(void* stream) {
  const cudaError_t se = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (se != cudaSuccess) return cuda_fail(se);
  unsigned int word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_device_error, sizeof(word)) != cudaSuccess) return VARLEN_ERR_CUDA;
  if (word != 0 && cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return VARLEN_ERR_CUDA;
  if (word & kErrTimeout) return VARLEN_ERR_TIMEOUT;
  if (word & kErrBounds) return VARLEN_ERR_DEVICE_BOUNDS;
  return VARLEN_OK;
}

extern "C" const char* varlen_attn_status_string(int status) {
  switch (status) {
    case VARLEN_OK: return "ok";
    case VARLEN_ERR_NULL: return "required pointer is NULL";
    case VARLEN_ERR_SHAPE: return "batch, totals, heads or scale out of range";
    case VARLEN_ERR_HEAD_DIM: return "head_dim must be 64, 96 or 128";
    case VARLEN_ERR_ALIGN: return "base pointer not 16-byte aligned";
    case VARLEN_ERR_STRIDE: return "stride negative, not a multiple of 8 elements, or too large for TMA";
    case VARLEN_ERR_WORKSPACE: return "workspace NULL, not 256-byte aligned, or too small";
    case VARLEN_ERR_CUDA: return "CUDA runtime or driver call failed";
    case VARLEN_ERR_TIMEOUT: return "device-side bounded wait timed out";
    case VARLEN_ERR_DEVICE_BOUNDS: return "device-side bounds check failed";
    case VARLEN_ERR_ARCH: return "current device is not sm_103";
    default: return "unknown status";
  }
}

extern "C" int64_t varlen_attn_tile_count(const int32_t* cu, int32_t batch, int32_t total, int32_t num_heads,
                                          int32_t tile) {
  if (cu == nullptr || batch < 0 || total < 0 || num_heads < 0 || tile <= 0) return -1;
  int64_t n = 0;
  for (int32_t b = 0; b < batch; ++b) {
    int64_t a = std::min<int64_t>(std::max<int64_t>(cu[b], 0), total);
    int64_t e = std::min<int64_t>(std::max<int64_t>(cu[b + 1], 0), total);
    int64_t len = std::max<int64_t>(e - a, 0);
    n += (len + tile - 1) / tile;
  }
  return n * num_heads;
}

extern "C" int varlen_attn_debug_schedule(const int32_t* cu, int32_t batch, int32_t total, int32_t num_heads,
                                          int32_t tile, int32_t grid, int32_t* out, int64_t max_records,
                                          void* stream) {
  if (cu == nullptr || out == nullptr) return VARLEN_ERR_NULL;
  if (batch < 1 || total < 0 || num_heads < 1 || grid < 1 || max_records < 0) return VARLEN_ERR_SHAPE;
  if (tile != 64 && tile != 128 && tile != 256) return VARLEN_ERR_SHAPE;
  DeviceInfo dev;
  int st = device_info(&dev);
  if (st != VARLEN_OK) return st;
  cudaError_t e = launch_debug_schedule(cu, batch, total, num_heads, tile, grid, out, max_records,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VARLEN_OK : VARLEN_ERR_CUDA;
}

extern "C" int varlen_attn_selftest_wait_timeout(uint64_t budget_ns, void* stream) {
  DeviceInfo dev;
  int st = device_info(&dev);
  if (st != VARLEN_OK) return st;
  cudaError_t e = launch_selftest_timeout(budget_ns, dev.err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VARLEN_OK : VARLEN_ERR_CUDA;
}

extern "C" int varlen_attn_debug_mma_cycles(int32_t n_mma, int32_t n_cols, int32_t mode,
                                            unsigned long long* cycles, void* stream) {
  if (cycles == nullptr) return VARLEN_ERR_NULL;
  if (n_mma < 4 || n_mma > (1 << 20) || n_mma % 4 != 0) return VARLEN_ERR_SHAPE;
  if (n_cols != 64 && n_cols != 128 && n_cols != 256) return VARLEN_ERR_SHAPE;
  if (mode < 0 || mode > 7 || (mode == 5 && n_cols > 128)) return VARLEN_ERR_SHAPE;
  DeviceInfo dev;
  int st = device_info(&dev);
  if (st != VARLEN_OK) return st;
  cudaError_t e = launch_debug_mma_rate(n_mma, n_cols, mode, cycles, dev.err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VARLEN_OK : cuda_fail(e);
}

extern "C" int varlen_attn_debug_set_phase_events(void* const* events, int count) {
  if (count != 0 && count != 4) return VARLEN_ERR_SHAPE;
  if (count == 4 && events == nullptr) return VARLEN_ERR_NULL;
  std::lock_guard<std::mutex> lock(g_phase_mu);
  for (int i = 0; i < 4; ++i) g_phase_events[i] = count ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  return VARLEN_OK;
}

extern "C" const char* varlen_attn_last_cuda_error(void) {
  return g_last_cuda_error == 0 ? "no error" : cudaGetErrorString(static_cast<cudaError_t>(g_last_cuda_error));
}

extern "C" int varlen_attn_num_sms(void) {
  DeviceInfo dev;
  int st = device_info(&dev);
  if (st != VARLEN_OK && st != VARLEN_ERR_ARCH) return st;
  return dev.sms;
}

extern "C" int varlen_attn_bounds_checked(void) {
#ifdef VARLEN_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

extern "C" int varlen_attn_debug_set_span_slack(int64_t bytes) {
  if (bytes < 0) return VARLEN_ERR_SHAPE;
  g_span_slack.store(bytes);
  return VARLEN_OK;
}

extern "C" int varlen_attn_debug_skip_load(int which, int64_t n) {
  if (which == 0) g_skip_fwd_load.store(n < 0 ? -1 : n);
  else if (which == 1) g_skip_bwd_step.store(n < 0 ? -1 : n);
  else return VARLEN_ERR_SHAPE;
  return VARLEN_OK;
}
