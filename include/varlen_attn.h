/*
 * varlen_attn.h -- C ABI of libvarlen_attn: packed variable-length
 * (cu_seqlens) multi-head scaled-dot-product attention, forward and backward,
 * in bf16 with fp32 accumulation, for one NVIDIA GB300 (sm_103a).
 *
 * The operation is the packed "varlen" attention of flash_attn_varlen_func
 * as called on the flash-attention issue pages:
 *   - "[FA4][SM120] flash_attn_varlen_func / flash_attn_func illegal memory
 *     access at >=4 varlen segments", section "Bug 2 details" (packed q with
 *     cu_seqlens_q = [0, 4032, ..., 35280], 17580 kv rows per window, H=56,
 *     D=128, max_seqlen_q / max_seqlen_k, non-causal), and
 *   - "[FA4] cute varlen backward: int32 overflow in _bwd_preprocess corrupts
 *     dQ/dK/dV when dout has a large outer stride", sections "Summary" and
 *     "Minimal repro" (cu_seqlens_q = cu_seqlens_k, causal=False, gradients
 *     dQ/dK/dV for an upstream dout whose row stride exceeds H*D).
 *
 * For every segment b (q rows [cu_q[b], cu_q[b+1]), kv rows [cu_k[b],
 * cu_k[b+1])) and head h:
 *     O_b  = softmax(scale * Q_b K_b^T) V_b,
 *     LSE  = natural-log log-sum-exp of each score row (-inf for a segment
 *            with no keys, whose O rows are 0),
 * and the backward returns dQ, dK, dV of sum(O * dO).
 *
 * Entry points, by family (each declared below with its own contract):
 *   packed bf16        varlen_attn_fwd / _bwd (+ _bwd_workspace_size), their
 *                      causal and sliding-window forms (_causal, _window), the
 *                      deterministic backward, and a backward without a
 *                      workspace argument (_bwd_noalloc);
 *   dense batched bf16 varlen_attn_fwd_dense / _bwd_dense ([B, S, H, D]);
 *   E4M3 (FP8) forward varlen_attn_fwd_fp8, _fp8_window, _fp8_dense (D = 128,
 *                      quantised from bf16 into a caller workspace);
 *   status             varlen_attn_get_device_status, _status_string,
 *                      _last_cuda_error;
 *   diagnostics        tile counts and schedules, the bounded-wait self test,
 *                      phase events, the tensor-core issue-rate probe, and the
 *                      knobs of the bounds-checking build and failure tests.
 *
 * Conventions shared by every entry point
 *   Layout.  Every q/k/v/out/dout/dq/dk/dv tensor is "NHD": element (row r,
 *     head h, dim d) lives at  base + r*stride.row + h*stride.head + d
 *     (bf16 elements, int64 strides, innermost stride 1).  Row and head
 *     strides are arbitrary non-negative multiples of 8 elements (16 bytes)
 *     and base pointers are 16-byte aligned; no tensor is ever copied to make
 *     it contiguous.  All offset arithmetic is 64-bit, so strides times rows
 *     may exceed 2^31 elements.  Inputs may alias themselves (a zero head
 *     stride broadcasts one head); an output (out, dq, dk, dv) must not:
 *     ordering its dimensions of extent > 1 by stride, the smaller stride
 *     must be at least head_dim and the larger at least the smaller's extent
 *     times the smaller stride, else VARLEN_ERR_STRIDE.
 *   cu_seqlens_q / cu_seqlens_k: device int32 arrays of batch+1 entries.  The
 *     host never reads them (no synchronisation); device code clamps every
 *     entry into [0, total] and never reads index > batch.  Empty segments
 *     (length 0) are allowed anywhere.
 *   max_seqlen_q / max_seqlen_k: advisory only, never trusted for
 *     correctness (a caller that passes a too-small value gets the same
 *     result).
 *   lse: fp32, [num_heads, total_q] contiguous (lse[h*total_q + row]).
 *   head_dim: 64, 96 or 128.  scale: finite and > 0.
 *   Ownership: every buffer belongs to the caller; the library allocates no
 *     device memory and keeps only a per-device attribute cache and one
 *     device error word.
 *   Streams: `stream` is a cudaStream_t (NULL = legacy default stream).
 *     Work is enqueued asynchronously; argument errors are returned
 *     synchronously before anything is enqueued.
 *   Device-side failures (a bounded wait that timed out) are recorded in a
 *     device error word; varlen_attn_get_device_status reads it.
 */
#ifndef VARLEN_ATTN_H_
#define VARLEN_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VARLEN_OK = 0,
  VARLEN_ERR_NULL = -1,          /* a required pointer is NULL                  */
  VARLEN_ERR_SHAPE = -2,         /* batch / totals / heads / scale out of range */
  VARLEN_ERR_HEAD_DIM = -3,      /* head_dim not in {64, 96, 128}               */
  VARLEN_ERR_ALIGN = -4,         /* base pointer not 16-byte aligned            */
  VARLEN_ERR_STRIDE = -5,        /* stride negative, not a multiple of 8, too
                                    large for a TMA descriptor (>= 2^40 bytes),
                                    or an output layout that overlaps itself  */
  VARLEN_ERR_WORKSPACE = -6,     /* workspace NULL, misaligned or too small     */
  VARLEN_ERR_CUDA = -7,          /* a CUDA runtime/driver call failed           */
  VARLEN_ERR_TIMEOUT = -8,       /* a device-side bounded wait gave up          */
  VARLEN_ERR_DEVICE_BOUNDS = -9, /* a device-side bounds check failed           */
  VARLEN_ERR_ARCH = -10          /* current device is not sm_103                 */
} varlen_status;

/* Row and head strides of one NHD tensor, in elements. */
typedef struct {
  int64_t row;
  int64_t head;
} varlen_stride;

/*
 * Forward.  Writes out[total_q, H, D] (bf16, its own strides) and
 * lse[H, total_q] (fp32).  Rows of a segment with no keys get O = 0 and
 * LSE = -inf.  Rows of out outside every segment, and padding between rows,
 * are not written.
 */
int varlen_attn_fwd(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                    varlen_stride sv, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                    int32_t total_q, int32_t total_k, int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q,
                    int32_t max_seqlen_k, float scale, void* out, varlen_stride so, float* lse, void* stream);

/*
 * Bytes of device workspace varlen_attn_bwd needs (256-byte aligned base).
 * It holds the fp32 dQ accumulator ([total_q, H, D] floats) and the per-row
 * delta and log2-domain LSE ([H, P] floats each, P = 4 * ceil(total_q / 4)
 * + 4 * batch + 128: each segment's rows start at a 16-byte aligned index,
 * with room for whole 128-row blocks past its end), each region rounded up
 * to 256 bytes.  Returns 0 for negative arguments.
 */
size_t varlen_attn_bwd_workspace_size(int32_t batch, int32_t total_q, int32_t num_heads, int32_t head_dim);

/*
 * Backward.  Given q, k, v, the forward's out and lse, and the upstream
 * gradient dout (each with its own strides), writes dq[total_q,H,D],
 * dk[total_k,H,D], dv[total_k,H,D] (bf16, their own strides).  Segments with
 * no queries get dK = dV = 0; segments with no keys get dQ = 0.
 * Three kernels on `stream`: delta preprocess (delta = rowsum(dO * O)),
 * the main dQ/dK/dV kernel, and the dQ conversion.  `workspace` is
 * caller-owned scratch of at least varlen_attn_bwd_workspace_size() bytes;
 * its contents on entry do not matter.
 */
int varlen_attn_bwd(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                    varlen_stride sv, const void* out, varlen_stride so, const void* dout, varlen_stride sdo,
                    const float* lse, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                    int32_t total_q, int32_t total_k, int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q,
                    int32_t max_seqlen_k, float scale, void* dq, varlen_stride sdq, void* dk, varlen_stride sdk,
                    void* dv, varlen_stride sdv, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Causal forward and backward.  Arguments, layouts, ownership and errors are
 * those of varlen_attn_fwd / varlen_attn_bwd.  The pages call the varlen
 * function with causal=False only ("[FA4] cute varlen backward: int32
 * overflow in _bwd_preprocess", "Minimal repro"); for causal=True these take
 * the alignment of that API, the diagonal meeting the last key at the last
 * query: q row i of a segment (0-based within it) attends to kv rows
 * j <= i + Sk - Sq of the same segment.  A row that sees no key (possible
 * when Sq > Sk) gets O = 0, LSE = -inf and dQ = 0, and adds nothing to dK /
 * dV.  Work past the diagonal is skipped, not masked.
 */
int varlen_attn_fwd_causal(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                           varlen_stride sv, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                           int32_t batch, int32_t total_q, int32_t total_k, int32_t num_heads, int32_t head_dim,
                           int32_t max_seqlen_q, int32_t max_seqlen_k, float scale, void* out, varlen_stride so,
                           float* lse, void* stream);
int varlen_attn_bwd_causal(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                           varlen_stride sv, const void* out, varlen_stride so, const void* dout,
                           varlen_stride sdo, const float* lse, const int32_t* cu_seqlens_q,
                           const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q, int32_t total_k,
                           int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q, int32_t max_seqlen_k,
                           float scale, void* dq, varlen_stride sdq, void* dk, varlen_stride sdk, void* dv,
                           varlen_stride sdv, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Sliding-window forward and backward (not on the pages; the window_size
 * convention of the API they call).  Arguments, layouts, ownership and
 * errors are those of varlen_attn_fwd / varlen_attn_bwd plus the two sides
 * of the band: with d = Sk - Sq of a segment, its q row i (0-based) attends
 * to the kv rows j (0-based) with
 *     i + d - window_left  <=  j  <=  i + d + window_right,
 * a negative side being unbounded.  (-1, -1) is no mask (the unmasked
 * kernels run), (-1, 0) is the causal mask of varlen_attn_fwd_causal.  A row
 * whose band holds no key gets O = 0, LSE = -inf and dQ = 0, and adds
 * nothing to dK / dV.  Key tiles outside a q tile's band (and q steps
 * outside a kv tile's) are skipped, not masked.
 */
int varlen_attn_fwd_window(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                           varlen_stride sv, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                           int32_t batch, int32_t total_q, int32_t total_k, int32_t num_heads, int32_t head_dim,
                           int32_t max_seqlen_q, int32_t max_seqlen_k, float scale, int32_t window_left,
                           int32_t window_right, void* out, varlen_stride so, float* lse, void* stream);
int varlen_attn_bwd_window(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                           varlen_stride sv, const void* out, varlen_stride so, const void* dout,
                           varlen_stride sdo, const float* lse, const int32_t* cu_seqlens_q,
                           const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q, int32_t total_k,
                           int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q, int32_t max_seqlen_k,
                           float scale, int32_t window_left, int32_t window_right, void* dq, varlen_stride sdq,
                           void* dk, varlen_stride sdk, void* dv, varlen_stride sdv, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * Deterministic backward (not on the pages; a plain extension): the same
 * arguments, layouts, ownership, errors and band as varlen_attn_bwd_window
 * (window_left = window_right = -1 for no mask, (-1, 0) for causal), and the
 * same workspace (varlen_attn_bwd_workspace_size bytes).  dK and dV come from
 * the main backward kernel without its dQ products; dQ comes from a second,
 * q-major kernel that recomputes S and dP per kv tile and accumulates dQ in
 * on-chip memory in a fixed kv order, with no atomics.  Repeated calls on the
 * same inputs return the same bits for dQ, dK and dV (varlen_attn_bwd's dQ
 * may differ in its last bits from run to run).  Costs two extra matrix
 * products per (q tile, kv tile) pair.
 */
int varlen_attn_bwd_deterministic(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                                  varlen_stride sv, const void* out, varlen_stride so, const void* dout,
                                  varlen_stride sdo, const float* lse, const int32_t* cu_seqlens_q,
                                  const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q, int32_t total_k,
                                  int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q, int32_t max_seqlen_k,
                                  float scale, int32_t window_left, int32_t window_right, void* dq,
                                  varlen_stride sdq, void* dk, varlen_stride sdk, void* dv, varlen_stride sdv,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * E4M3 (FP8) forward (not on the pages, which quote quantised attention
 * only by its accuracy: the ffpa-attn NVFP4 pull request, "Summary", cos
 * ~0.982 against SDPA).  Arguments, layouts and errors as varlen_attn_fwd;
 * head_dim must be 128 (else VARLEN_ERR_HEAD_DIM); no mask (the window form
 * below takes one).  q, k, v (bf16)
 * are quantised per (segment, head) and tensor into the caller's workspace
 * (varlen_attn_fwd_fp8_workspace_size bytes, 256-byte aligned, contents on
 * entry irrelevant): descale = amax / 448 (1 for an all-zero block), code =
 * E4M3(x / descale), round to nearest even, saturating, in fp32.  Then, per
 * q row, s = scale * qd * kd * (q8 . k8), P = exp(s - max) (fp32),
 * O = vd * sum_j E4M3(P_j) v8_j / sum_j P_j (bf16 out), LSE = max + ln sum P.
 * P is rounded from a running row maximum, so results match that definition
 * up to the rounding of P (a relative 2^-4 per weight).
 *
 * varlen_attn_fwd_fp8_window is the same call under the band of
 * varlen_attn_fwd_window (window_left, window_right after scale; a negative
 * side unbounded, (-1, 0) causal, (-1, -1) no mask): the max, the sums and
 * O run over each row's visible keys only, and a row that sees none gets
 * O = 0 and LSE = -inf.  The quantisation is that of the unmasked call (amax
 * over every row of the segment).
 *
 * varlen_attn_fwd_fp8_workspace_layout returns the byte offsets of the
 * workspace sections after a call: offsets[0] amax fp32 [3][batch * H] (q,
 * k, v; entry b * H + h), offsets[1] q codes [total_q][H][128], offsets[2] k
 * codes [total_k][H][128], offsets[3] V^T codes [H][128][*vt_cols], where
 * segment b's key j sits at column 128 * (b + ceil(cu_seqlens_k[b] / 128)) + j
 * (code 0 past the segment's end up to the next multiple of 128).
 */
size_t varlen_attn_fwd_fp8_workspace_size(int32_t batch, int32_t total_q, int32_t total_k, int32_t num_heads,
                                          int32_t head_dim);
int varlen_attn_fwd_fp8_workspace_layout(int32_t batch, int32_t total_q, int32_t total_k, int32_t num_heads,
                                         int32_t head_dim, size_t* offsets, int64_t* vt_cols);
int varlen_attn_fwd_fp8(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                        varlen_stride sv, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                        int32_t total_q, int32_t total_k, int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q,
                        int32_t max_seqlen_k, float scale, void* out, varlen_stride so, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream);
int varlen_attn_fwd_fp8_window(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                               varlen_stride sv, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                               int32_t batch, int32_t total_q, int32_t total_k, int32_t num_heads, int32_t head_dim,
                               int32_t max_seqlen_q, int32_t max_seqlen_k, float scale, int32_t window_left,
                               int32_t window_right, void* out, varlen_stride so, float* lse, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * Dense batched attention: q, out, dout, dq are [batch, seqlen_q, H, D] and
 * k, v, dk, dv are [batch, seqlen_k, H, D] (bf16), each with its own strides
 * in elements and a unit innermost stride; lse is [H, batch * seqlen_q]
 * fp32.  The pages' caller uses both this form and the packed one ("[FA4]
 * [SM120] flash_attn_varlen_func ... illegal memory access at >=4 varlen
 * segments", "Bug 2 details").  The result is that of the varlen call with
 * cu_seqlens = {0, S, 2S, ...}; the segment bounds are computed on the
 * device, never stored, so nothing is allocated.  Requires the batch stride
 * to be seqlen row strides (the tensor is then the packed
 * [batch * seqlen, H, D] layout; VARLEN_ERR_STRIDE otherwise) and
 * batch * seqlen < 2^31 (VARLEN_ERR_SHAPE).  `causal` is 0 or 1, with the
 * mask of varlen_attn_fwd_causal.
 */
typedef struct {
  int64_t batch;
  int64_t row;
  int64_t head;
} varlen_dense_stride;

int varlen_attn_fwd_dense(const void* q, varlen_dense_stride sq, const void* k, varlen_dense_stride sk,
                          const void* v, varlen_dense_stride sv, int32_t batch, int32_t seqlen_q, int32_t seqlen_k,
                          int32_t num_heads, int32_t head_dim, float scale, int32_t causal, void* out,
                          varlen_dense_stride so, float* lse, void* stream);
/* Workspace of varlen_attn_bwd_dense: that of the packed call (0 if
 * batch * seqlen_q overflows int32 or an argument is negative). */
size_t varlen_attn_bwd_dense_workspace_size(int32_t batch, int32_t seqlen_q, int32_t num_heads, int32_t head_dim);
int varlen_attn_bwd_dense(const void* q, varlen_dense_stride sq, const void* k, varlen_dense_stride sk,
                          const void* v, varlen_dense_stride sv, const void* out, varlen_dense_stride so,
                          const void* dout, varlen_dense_stride sdo, const float* lse, int32_t batch,
                          int32_t seqlen_q, int32_t seqlen_k, int32_t num_heads, int32_t head_dim, float scale,
                          int32_t causal, void* dq, varlen_dense_stride sdq, void* dk, varlen_dense_stride sdk,
                          void* dv, varlen_dense_stride sdv, void* workspace, size_t workspace_bytes, void* stream);

/*
 * E4M3 forward in the dense batched layout of varlen_attn_fwd_dense
 * ([batch, seqlen, H, 128] tensors with {batch, row, head} strides, batch
 * stride = seqlen row strides, causal 0 or 1; the same checks and status
 * codes): the result of varlen_attn_fwd_fp8 (causal: varlen_attn_fwd_fp8_window
 * with (-1, 0)) on cu_seqlens = [0, S, 2S, ...] over the same rows, segment
 * bounds computed on the device.  The workspace holds
 * varlen_attn_fwd_fp8_dense_workspace_size(batch, seqlen_q, seqlen_k, H, 128)
 * bytes (0 for a size that does not fit) and has the layout
 * varlen_attn_fwd_fp8_workspace_layout gives for batch, batch * seqlen_q and
 * batch * seqlen_k.
 */
size_t varlen_attn_fwd_fp8_dense_workspace_size(int32_t batch, int32_t seqlen_q, int32_t seqlen_k, int32_t num_heads,
                                                int32_t head_dim);
int varlen_attn_fwd_fp8_dense(const void* q, varlen_dense_stride sq, const void* k, varlen_dense_stride sk,
                              const void* v, varlen_dense_stride sv, int32_t batch, int32_t seqlen_q,
                              int32_t seqlen_k, int32_t num_heads, int32_t head_dim, float scale, int32_t causal,
                              void* out, varlen_dense_stride so, float* lse, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Backward without a workspace argument, for callers that cannot allocate
 * device memory (code inside a host framework that owns every device
 * allocation, or on a path where cudaMalloc is not allowed).  The attention
 * pages describe no such call: this is a deployment variant of varlen_attn_bwd.
 * Arguments, layouts and results are those of varlen_attn_bwd; the scratch
 * (the fp32 dQ accumulator, delta and log2-domain LSE) lives in a fixed
 * file-scope device array of VARLEN_NOALLOC_SCRATCH_BYTES bytes that every
 * GPU loading the library keeps until exit.  The call allocates nothing.
 * Returns VARLEN_ERR_WORKSPACE, before anything is enqueued, when the
 * problem needs more than that (varlen_attn_bwd_workspace_size() >
 * VARLEN_NOALLOC_SCRATCH_BYTES; at H=16, D=96 that is about 10,700 q rows).
 * The array's device address belongs to a CUDA context: the first call in
 * each context (the first call on a device, and the first one after the
 * caller reset the device or made another context current on it) looks it
 * up with that device current, so that call should come before any stream
 * capture.  Every call shares the one array: every entry a result depends
 * on is rewritten by each call before it is read (entries between segments
 * are read but masked out), but calls that overlap on the GPU (unordered
 * streams) race on it.  On a device that is not sm_103 the call returns
 * VARLEN_ERR_ARCH, like varlen_attn_bwd.
 */
#define VARLEN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* VARLEN_NOALLOC_SCRATCH_BYTES as compiled into the library. */
size_t varlen_attn_bwd_noalloc_scratch_bytes(void);

int varlen_attn_bwd_noalloc(const void* q, varlen_stride sq, const void* k, varlen_stride sk, const void* v,
                            varlen_stride sv, const void* out, varlen_stride so, const void* dout,
                            varlen_stride sdo, const float* lse, const int32_t* cu_seqlens_q,
                            const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q, int32_t total_k,
                            int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q, int32_t max_seqlen_k,
                            float scale, void* dq, varlen_stride sdq, void* dk, varlen_stride sdk, void* dv,
                            varlen_stride sdv, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device error word:
 * VARLEN_OK, VARLEN_ERR_TIMEOUT, VARLEN_ERR_DEVICE_BOUNDS, or VARLEN_ERR_CUDA
 * if the stream itself reports an error.
 */
int varlen_attn_get_device_status(void* stream);

/* Static description of a status code. */
const char* varlen_attn_status_string(int status);

/* Description of the CUDA error behind the last VARLEN_ERR_CUDA returned on
 * the calling host thread ("no error" if none). */
const char* varlen_attn_last_cuda_error(void);

/* ---------------------------------------------------------------------------
 * Diagnostics (host logic and scheduler checks; not needed for normal use).
 */

/*
 * Exact tile count of the varlen grid: num_heads * sum_b ceil(len_b / tile)
 * for a HOST copy of cu_seqlens (batch+1 entries, clamped to [0, total] like
 * the device does).  This is the count the persistent kernels walk; the
 * "[FA4][SM120] ... >=4 varlen segments" issue (section "Interpretation")
 * shows the over-provisioned alternative.  Returns -1 on bad arguments.
 */
int64_t varlen_attn_tile_count(const int32_t* cu_seqlens_host, int32_t batch, int32_t total, int32_t num_heads,
                               int32_t tile);

/*
 * Runs the device tile scheduler alone with `grid` persistent CTAs and writes
 * one record per visited tile into out_records (device int32, 4 per tile:
 * segment, row-block, head, cta).  Records are written at their global tile
 * index; records at index >= max_records are dropped.  Callers compare the
 * records against varlen_attn_tile_count.  `tile` is the row-block height:
 * 256 (forward: two 128-row halves per unit), 128 (backward kv tiles) or 64.
 */
int varlen_attn_debug_schedule(const int32_t* cu_seqlens, int32_t batch, int32_t total, int32_t num_heads,
                               int32_t tile, int32_t grid, int32_t* out_records, int64_t max_records,
                               void* stream);

/*
 * Failure-detection self test: launches one CTA whose bounded mbarrier wait
 * is never satisfied, with a budget of budget_ns nanoseconds.  The kernel
 * records VARLEN_ERR_TIMEOUT and returns; read it with
 * varlen_attn_get_device_status.
 */
int varlen_attn_selftest_wait_timeout(uint64_t budget_ns, void* stream);

/*
 * tcgen05 issue-rate probe (the measurements behind the kernels' MMA shapes
 * and their single issuing thread): one CTA, one thread issues n_mma MMAs of
 * M = 128, N = n_cols, K = 16 (bf16 x bf16 -> fp32, zero operands) into one
 * TMEM accumulator and writes to *cycles (a device pointer, 8 bytes) the
 * clock64 cycles from the first issue to the completion of the last.
 * mode 0: both operands from shared memory, descriptors kept as 32-bit low
 * words advanced by an immediate; 1: A from TMEM; 2: as 0, with both 64-bit
 * descriptors rebuilt from the shared-memory address for every MMA.
 * Modes 3 and 4 time TMEM <-> register traffic instead: each of four warps
 * loads (3) or stores (4) its 32 lanes x 32 columns (4 KB) n_mma times,
 * waiting for each; *cycles spans all four warps' loops.  Mode 5: as 1 with
 * B MN-major (the V operand layout of O += P V), n_cols 64 or 128.  Mode
 * 6: as 1 while four more warps keep loading TMEM columns the MMAs do not
 * use (as a softmax does beside the tensor core); 7: as 1 while four more
 * warps keep storing into a separate 16 KB of shared memory.
 * n_mma a multiple of 4 in [4, 2^20], n_cols 64, 128 or 256, else
 * VARLEN_ERR_SHAPE; a completion wait that gives up records
 * VARLEN_ERR_TIMEOUT (varlen_attn_get_device_status).
 */
int varlen_attn_debug_mma_cycles(int32_t n_mma, int32_t n_cols, int32_t mode, unsigned long long* cycles,
                                 void* stream);

/*
 * Profiling hook: with count == 4, every later varlen_attn_bwd call records
 * events[0] before its preprocess kernel, events[1] after it, events[2] after
 * the main kernel and events[3] after the dQ conversion, on the call's
 * stream (cudaEvent_t handles owned by the caller; they must outlive their
 * use).  count == 0 turns it off.  Process-wide setting.
 */
int varlen_attn_debug_set_phase_events(void* const* events, int count);

/*
 * The device address of varlen_attn_bwd_noalloc's scratch array in the
 * context current on the calling thread (*addr), and that context's
 * identity (cuCtxGetId; *ctx_id).  The address is the one the next
 * varlen_attn_bwd_noalloc call on this thread would use: it is looked up
 * again whenever the current context differs from the one it was last
 * looked up in.  Nothing is launched.  Errors as varlen_attn_bwd_noalloc.
 */
int varlen_attn_debug_noalloc_scratch(void** addr, unsigned long long* ctx_id);

/*
 * 1 when this library was built with device-side bounds checks
 * (-DVARLEN_DEBUG_BOUNDS; python -m packed_variable_length_varlen_gb300.build
 * --bounds): every plain (non-TMA) global load and store of its kernels is
 * checked against the bytes its operand occupies, and an access outside is
 * skipped (a load reads 0) and reported as VARLEN_ERR_DEVICE_BOUNDS by
 * varlen_attn_get_device_status.  0 for the normal build, whose kernels
 * carry no checks.
 */
int varlen_attn_bounds_checked(void);

/*
 * Bounds checker self test: every operand extent handed to the kernels of
 * later calls is `bytes` shorter (0 restores; negative: VARLEN_ERR_SHAPE).
 * In a bounds-checking build the last accesses of each operand then fail
 * their check, are skipped, and the call reports VARLEN_ERR_DEVICE_BOUNDS;
 * in the normal build it has no effect.  Process-wide; for tests only.
 */
int varlen_attn_debug_set_span_slack(int64_t bytes);

/*
 * Failure test of the bounded waits: with which = 0 the K/V producer of the
 * forward's CTA 0 leaves out its load number n (0-based, K and V loads
 * counted alike); with which = 1 the Q producer of the backward's CTA 0
 * leaves out the Q load of its step n.  The waits for that load give up
 * after their budget (2 s), every role of the CTA unwinds (the producer
 * waits, bounded, for its copies in flight; the MMA issuer drains its
 * products; TMEM is freed) and varlen_attn_get_device_status returns
 * VARLEN_ERR_TIMEOUT; the context stays usable.  n < 0 turns it off; an
 * unknown `which` returns VARLEN_ERR_SHAPE.  Process-wide; for tests only.
 */
int varlen_attn_debug_skip_load(int which, int64_t n);

/* Number of streaming multiprocessors the persistent kernels size their grid
 * by on the current device (cached). Returns <= 0 on failure. */
int varlen_attn_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* VARLEN_ATTN_H_ */
