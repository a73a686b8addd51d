// varlen_internal.h -- declarations shared by the C-ABI layer and the
// kernel translation units (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace varlen {

// Bits of the device error word (read and cleared by
// varlen_attn_get_device_status).
enum : unsigned int {
  kErrTimeout = 1u,  // a bounded mbarrier wait gave up
  kErrBounds = 2u,   // a debug bounds check failed
};

// The bytes [base, base + bytes) one operand of a launch occupies.  In a
// build with -DVARLEN_DEBUG_BOUNDS every plain (non-TMA) global load and
// store of the kernels checks the bytes it touches against its operand's
// span (in_span); an access outside is skipped (a load reads 0) and
// kErrBounds is recorded in the device error word.  In the normal build the
// check compiles away.
struct Span {
  const void* base;
  int64_t bytes;
};

__device__ __forceinline__ bool in_span(const Span& s, const void* p, int n, unsigned int* err) {
#ifdef VARLEN_DEBUG_BOUNDS
  const int64_t off = static_cast<const char*>(p) - static_cast<const char*>(s.base);
  if (off < 0 || off + n > s.bytes) {
    if (err != nullptr) atomicOr(err, (unsigned int)kErrBounds);
    return false;
  }
#else
  (void)s;
  (void)p;
  (void)n;
  (void)err;
#endif
  return true;
}

// Where a launch finds its segment bounds: cu_seqlens in device memory
// (`ptr`), or, when ptr is null, uniform segments of `uni` rows each (the
// bounds b * uni of the dense batched entry points, never stored).
struct CuView {
  const int32_t* ptr;
  int32_t uni;
};

// Visibility band of a masked launch.  With d = Sk - Sq of a segment, its q
// row i (0-based) sees the keys j (0-based) with
//     i + d - win_left  <=  j  <=  i + d + win_right;
// an unbounded side holds kWinUnbounded, so one formula serves every mask
// (causal: win_left unbounded, win_right 0).
constexpr int64_t kWinUnbounded = int64_t(1) << 40;

// Keys [*lo, *hi) of a segment (Sq q rows, Sk keys) seen by at least one of
// its q rows i0..i1; *lo == *hi when none.
__host__ __device__ __forceinline__ void band_keys(int64_t i0, int64_t i1, int32_t Sq, int32_t Sk, int64_t win_left,
                                                   int64_t win_right, int32_t* lo, int32_t* hi) {
  const int64_t d = (int64_t)Sk - Sq;
  int64_t a = i0 + d - win_left, e = i1 + d + win_right + 1;
  a = a < 0 ? 0 : (a > Sk ? Sk : a);
  e = e < a ? a : (e > Sk ? Sk : e);
  *lo = (int32_t)a;
  *hi = (int32_t)e;
}

// q rows [*lo, *hi) of a segment that see at least one of its keys j0..j1.
__host__ __device__ __forceinline__ void band_rows(int64_t j0, int64_t j1, int32_t Sq, int32_t Sk, int64_t win_left,
                                                   int64_t win_right, int32_t* lo, int32_t* hi) {
  const int64_t d = (int64_t)Sk - Sq;
  int64_t a = j0 - d - win_right, e = j1 - d + win_left + 1;
  a = a < 0 ? 0 : (a > Sq ? Sq : a);
  e = e < a ? a : (e > Sq ? Sq : e);
  *lo = (int32_t)a;
  *hi = (int32_t)e;
}

// Records `e` as the calling thread's last CUDA error (reported by
// varlen_attn_last_cuda_error) and returns VARLEN_ERR_CUDA.
int cuda_fail(cudaError_t e);

// Identity (cuCtxGetId) of the CUDA context current on the calling thread,
// 0 when none is.  Device addresses of __device__ symbols belong to a
// context; caches of them are keyed by this identity, which, unlike the
// CUcontext handle, is never reused by a later context.
int current_context_id(unsigned long long* id);

// VARLEN_OK when the current device is an sm_103 GPU whose library state
// (attributes, device error word) is set up for the current context;
// VARLEN_ERR_ARCH on another device; VARLEN_ERR_CUDA when a call failed.
int device_ready();

constexpr int kTileM = 128;  // q rows per forward tile / kv rows per backward tile
constexpr int kTileN = 128;  // kv rows per forward inner step
constexpr int kBwdTileQ = 128; // q rows per backward inner step

struct FwdParams {
  __nv_bfloat16* out;
  int64_t o_rs, o_hs;
  float* lse;
  Span out_span, lse_span;     // checked in a bounds-checking build
  CuView cu_q;
  CuView cu_k;
  int32_t batch, total_q, total_k, num_heads;
  int32_t masked;              // 0: every key of the segment is visible
  int64_t win_left, win_right; // the band when masked (kWinUnbounded: that side open)
  float scale_log2;  // softmax scale * log2(e)
  unsigned int* err; // device error word
  int32_t debug_skip_load;  // < 0: off; else CTA 0's producer skips its K/V load number n (failure test)
};

struct FwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v;
  FwdParams p;
  int head_dim;
  int grid;
};

cudaError_t launch_fwd(const FwdLaunch& L, cudaStream_t stream);

struct PrepParams {
  const __nv_bfloat16* out;
  int64_t o_rs, o_hs;
  const __nv_bfloat16* dout;
  int64_t do_rs, do_hs;
  const float* lse;
  float* delta;     // [H, pad_rows], segment-padded (see bwd_pad_rows)
  float* lse2;      // [H, pad_rows], segment-padded
  float* dq_acc;    // [total_q, H, D], zeroed here; null: no accumulator (deterministic dQ)
  CuView cu_q;
  int32_t batch, total_q, num_heads, head_dim;
  int64_t pad_rows;
  int32_t rows_per_tile;  // q rows per CTA (set at launch)
  Span out_span, dout_span, lse_span, delta_span, lse2_span, acc_span;  // checked in a bounds-checking build
  unsigned int* err;      // device error word
};

struct BwdParams {
  __nv_bfloat16* dk;
  int64_t dk_rs, dk_hs;
  __nv_bfloat16* dv;
  int64_t dv_rs, dv_hs;
  const float* delta;  // [H, pad_rows]
  const float* lse2;   // [H, pad_rows]
  float* dq_acc;
  __nv_bfloat16* dq;   // written directly by the deterministic dQ kernel
  int64_t dq_rs, dq_hs;
  CuView cu_q;
  CuView cu_k;
  int32_t batch, total_q, total_k, num_heads;
  int32_t masked;              // 0: every key of the segment is visible
  int64_t win_left, win_right; // the band when masked (kWinUnbounded: that side open)
  int64_t pad_rows;
  float scale_log2;  // softmax scale * log2(e)
  float scale;       // softmax scale (applied to dK)
  unsigned int* err; // device error word
  Span dk_span, dv_span, dq_span;  // checked in a bounds-checking build
  int32_t debug_skip_step;  // < 0: off; else CTA 0's Q producer skips the load of this step (failure test)
};

struct PostParams {
  const float* dq_acc;
  __nv_bfloat16* dq;
  int64_t dq_rs, dq_hs;
  CuView cu_q;
  int32_t batch, total_q, num_heads, head_dim;
  float scale;
  Span acc_span, dq_span;  // checked in a bounds-checking build
  unsigned int* err;       // device error word
};

struct BwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  CUtensorMap tm_dq;  // fp32 dQ accumulator {D, H, total_q}, 32 x 1 x 64 boxes, for bulk reduce-add
  PrepParams prep;
  BwdParams p;
  PostParams post;
  int head_dim;
  int grid;
  int deterministic;  // 1: dK/dV main kernel + the q-major dQ kernel (no atomics), no post kernel
  cudaEvent_t phase_events[4];  // optional: recorded before prep / after prep / after main / after post (or dQ)
};

cudaError_t launch_bwd(const BwdLaunch& L, cudaStream_t stream);

// The deterministic dQ kernel (varlen_bwd_dq.cu) for head size D, masked or not.
cudaError_t launch_bwd_dq(const BwdLaunch& L, cudaStream_t stream);

// Length of one head's row of the segment-padded delta / lse2 arrays.
// Segment b's entries start at 4 * ceil(o0_b / 4) + 4 b (o0_b its first q
// row), 16-byte aligned; a backward step reads whole 128-row blocks of a
// segment, so up to 127 entries past its end, which this length covers for
// any cu_seqlens.
inline int64_t bwd_pad_rows(int32_t batch, int32_t total_q) {
  return 4 * (((int64_t)total_q + 3) / 4) + 4 * (int64_t)batch + 128;
}

// First index of segment b's entries in the padded per-row arrays (delta,
// lse2), o0 its first q row: a multiple of 4 (16 bytes), at least the
// previous segment's end for non-decreasing cu_seqlens, and below
// bwd_pad_rows() - 127 - len_b for any cu_seqlens (len_b + o0 <= total_q).
__host__ __device__ __forceinline__ int64_t pad_base(int32_t o0, int32_t b) {
  return 4 * (((int64_t)o0 + 3) / 4) + 4 * (int64_t)b;
}

// ------------------------------------------------------------------ FP8

// The E4M3 forward: bf16 operands quantised per (segment, head) into a
// workspace, then attention on the codes.  Head size 128, unmasked or under
// a band (masked, win_left, win_right as in FwdParams).
struct Fp8Params {
  const __nv_bfloat16 *q, *k, *v;
  int64_t q_rs, q_hs, k_rs, k_hs, v_rs, v_hs;
  __nv_bfloat16* out;
  int64_t o_rs, o_hs;
  float* lse;
  float* amax;     // [3][batch * H]: max |x| of q, k, v per (segment, head)
  uint8_t* q8;     // [total_q][H][128] codes
  uint8_t* k8;     // [total_k][H][128] codes
  uint8_t* vt;     // [H][128][kp] codes, V transposed (see fp8_vt_base)
  int64_t kp;      // row length of vt
  CuView cu_q, cu_k;
  int32_t batch, total_q, total_k, num_heads;
  float scale;     // softmax scale
  int32_t masked;              // 0: every key of the segment is visible
  int64_t win_left, win_right; // the band when masked (kWinUnbounded: that side open)
  unsigned int* err;
  Span q_span, k_span, v_span, out_span, lse_span, amax_span, q8_span, k8_span, vt_span;  // bounds-checking build
};

struct Fp8Launch {
  CUtensorMap tm_q8, tm_k8, tm_vt;
  Fp8Params p;
  int grid;
};

cudaError_t launch_fwd_fp8(const Fp8Launch& L, cudaStream_t stream);

// V^T layout of the E4M3 forward: segment b's key j (0-based) sits at column
// fp8_vt_base(k0_b, b) + j of every (head, d) row, k0_b its first key row.
// Each segment starts on a multiple of 128 columns and owns
// 128 * ceil(len_b / 128) of them (zero past its end): the start is at
// least the previous segment's end for non-decreasing cu_seqlens, and below
// fp8_vt_cols() - 128 * ceil(len_b / 128) for any.
__host__ __device__ __forceinline__ int64_t fp8_vt_base(int32_t k0, int32_t b) {
  return 128 * ((int64_t)b + ((int64_t)k0 + 127) / 128);
}
inline int64_t fp8_vt_cols(int32_t batch, int32_t total_k) {
  return 128 * ((int64_t)batch + ((int64_t)total_k + 127) / 128 + 1);
}

cudaError_t launch_debug_schedule(const int32_t* cu, int32_t batch, int32_t total, int32_t num_heads, int32_t tile,
                                  int32_t grid, int32_t* out, int64_t max_records, cudaStream_t stream);

cudaError_t launch_selftest_timeout(uint64_t budget_ns, unsigned int* err, cudaStream_t stream);

cudaError_t launch_debug_mma_rate(int32_t n_mma, int32_t n_cols, int32_t mode, unsigned long long* cycles,
                                  unsigned int* err, cudaStream_t stream);

}  // namespace varlen
