// varlen_fp8.cu -- E4M3 (FP8) forward of packed variable-length attention on
// sm_103a, head size 128, unmasked or under a causal / sliding-window band.
//
// Four launches on the caller's stream:
//  1. varlen_fp8_amax_kernel: max |x| of Q, K and V per (segment, head),
//     by atomic max on the fp32 bit patterns (non-negative floats order as
//     unsigned integers); a grid-wide sweep, as a copy kernel reads.
//  2. varlen_fp8_quant_kernel: Q and K to E4M3 codes in NHD layout, code of
//     x = e4m3(x / descale), descale = amax / 448 (1 for an all-zero block),
//     round to nearest even, saturating (fp32 division and conversion: the
//     precision that decides each code); the same sweep.
//  3. varlen_fp8_vt_kernel: V to E4M3 codes transposed to [H][128][kp], one
//     128-key block of one head per CTA visit through shared memory, so that
//     V is a K-major operand of the P V product; segment starts are
//     multiples of 128 columns and the columns past a segment's end hold
//     code 0.
//  The fp32 quotient x / descale is the IEEE one; it is formed from the
//  correctly rounded reciprocal of the descale and one fma remainder
//  correction (Markstein's division step: q0 = x * y, r = x - q0 * d exact,
//  q = q0 + r * y, given x's sign; two lanes at a time with packed f32x2
//  operations, each lane rounded as the scalar ones), which gives the correctly rounded
//  quotient while the remainder stays a normal number: for descales below
//  2^-100 the kernels divide.  Checked for every positive bf16 amax and every
//  bf16 x of magnitude at most amax: the two quotients have the same sign and
//  differ only below 2^-11 in magnitude, where both codes are a signed 0.
//  4. varlen_fp8_fwd_kernel: the forward of the bf16 kernel (two 128-row
//     halves per scheduled unit sharing each key tile, online softmax with
//     lazy rescaling) on the codes:
//         S = Q8 K8^T          (tcgen05 kind::f8f6f4, E4M3 x E4M3 -> fp32)
//         P = exp2(S * scale*log2e*qd*kd - m),  l += P   (fp32)
//         O += e4m3(P) V8      (P written into TMEM over S as E4M3 codes,
//                               read from there as the A operand)
//     and finally O * vd / l in bf16 and LSE = (m + log2 l) ln 2.  The row
//     sum l uses the unrounded P.  Under a band (the bf16 kernels' causal /
//     sliding-window reading) a unit walks only the key tiles some of its
//     rows see, and each row's keys outside its band are -inf by select.
//
// The quantised reading is that of the flash-attention family's FP8 forward
// (one descale per (segment, head) and tensor); the pages themselves quote
// quantised attention only by its accuracy (the ffpa-attn NVFP4 pull
// request, "Summary": cos ~0.982 against SDPA).
#include <cuda_fp8.h>

#include <algorithm>
#include <cfloat>

#include "sm103_ptx.cuh"
#include "varlen_internal.h"
#include "varlen_sched.cuh"

namespace varlen {

namespace {

constexpr float kE4m3Max = 448.0f;

__device__ __forceinline__ float descale_of(float amax) { return amax > 0.f ? amax / kE4m3Max : 1.f; }

// Segment holding `row` (the last b with clamp(cu[b]) <= row); false when the
// row lies in no segment.  Exact for non-decreasing cu_seqlens.
__device__ __forceinline__ bool segment_of_row(const CuView& cu, int32_t batch, int32_t total, int32_t row,
                                               int32_t& b) {
  int32_t b0 = 0, b1 = batch - 1;
  while (b0 < b1) {
    const int32_t mid = (b0 + b1 + 1) >> 1;
    if (clamp_row(cu_at(cu, mid), total) <= row) b0 = mid;
    else b1 = mid - 1;
  }
  b = b0;
  return row >= clamp_row(cu_at(cu, b0), total) && row < clamp_row(cu_at(cu, b0 + 1), total);
}

// x / d in fp32, correctly rounded, for one descale d and many x.
struct Divider {
  float d, y;  // descale and its correctly rounded reciprocal
  bool fast;   // d >= 2^-100: Markstein's step is exact
  // Two quotients at a time: q0 = x * y, r = x - q0 * d (exact), q = q0 + r * y,
  // by packed f32x2 multiply and fmas (each lane rounded as the scalar
  // operation rounds it); the quotient's sign, zeros included, is x's (d > 0).
  __device__ __forceinline__ float2 two(float2 x) const {
    if (!fast) return make_float2(x.x / d, x.y / d);
    const float2 q0 = fmul2_rn(x, make_float2(y, y));
    const float2 r = ffma2(q0, make_float2(-d, -d), x);
    const float2 q = ffma2(r, make_float2(y, y), q0);
    return make_float2(copysignf(q.x, x.x), copysignf(q.y, x.y));
  }
};

__device__ __forceinline__ Divider divider(float descale) {
  Divider v;
  v.d = descale;
  v.y = __frcp_rn(descale);
  v.fast = descale >= 0x1p-100f;
  return v;
}

// Four E4M3 codes of a / d, b / d, c / d, e / d packed low byte first.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float e, const Divider& d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(d.two(make_float2(a, b)), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(d.two(make_float2(c, e)), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// out[k] = byte k of in[0], in[1], in[2], in[3] (in[i] in byte i).
__device__ __forceinline__ void transpose4x4(const uint32_t (&in)[4], uint32_t* out) {
  const uint32_t t0 = __byte_perm(in[0], in[1], 0x5140), t1 = __byte_perm(in[2], in[3], 0x5140);
  const uint32_t t2 = __byte_perm(in[0], in[1], 0x7362), t3 = __byte_perm(in[2], in[3], 0x7362);
  out[0] = __byte_perm(t0, t1, 0x5410);
  out[1] = __byte_perm(t0, t1, 0x7632);
  out[2] = __byte_perm(t2, t3, 0x5410);
  out[3] = __byte_perm(t2, t3, 0x7632);
}

}  // namespace

// ------------------------------------------------------------------ amax, Q / K codes
//
// Both passes sweep q, k (and v) in turn with the whole grid, the way a copy
// kernel does: the threads are cut into slots of 16 lanes per (head, row),
// 16 bytes per lane, H * 16 slots per row and R = (threads / (H * 16)) rows
// per sweep step, so that each step reads R consecutive rows, all heads, and
// every lane keeps its head and 8-value slice for the whole sweep while its
// row advances by R.  A lane keeps the state of its current segment (the
// running max, or the descale) in registers and looks the segment up again
// only when its row leaves it.  Each lane issues kSweepUnroll rows' loads
// before it uses any.

constexpr int kSweepThreads = 256;
constexpr int kAmaxBlocksPerSm = 5;   // CTAs per SM (48 registers)
constexpr int kQuantBlocksPerSm = 4;  // CTAs per SM (64 registers)
constexpr int kSweepUnroll = 4;

struct Sweep {
  const __nv_bfloat16* x;
  int64_t rs, hs;
  CuView cu;
  int32_t total, lo, hi;
  Span span;
};

__device__ __forceinline__ Sweep sweep_of(const Fp8Params& p, int which) {
  Sweep t;
  t.x = which == 0 ? p.q : (which == 1 ? p.k : p.v);
  t.rs = which == 0 ? p.q_rs : (which == 1 ? p.k_rs : p.v_rs);
  t.hs = which == 0 ? p.q_hs : (which == 1 ? p.k_hs : p.v_hs);
  t.cu = which == 0 ? p.cu_q : p.cu_k;
  t.total = which == 0 ? p.total_q : p.total_k;
  t.span = which == 0 ? p.q_span : (which == 1 ? p.k_span : p.v_span);
  t.lo = clamp_row(cu_at(t.cu, 0), t.total);
  t.hi = clamp_row(cu_at(t.cu, p.batch), t.total);
  return t;
}

// Slot of this thread: head h, lane gl of the head's 16, first row offset
// row_off, rows per step R; false for the few threads past the last whole row
// of slots (they still take part in warp shuffles).
__device__ __forceinline__ bool sweep_slot(int32_t H, int& h, int& gl, int64_t& row_off, int64_t& R) {
  const int64_t S = (int64_t)H * 16;
  const int64_t T = (int64_t)gridDim.x * blockDim.x;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  R = T / S;
  const bool active = g < R * S;
  h = (int)((g % S) / 16);
  gl = (int)(g % 16);
  row_off = active ? g / S : INT64_MAX / 4;  // inactive: no row
  return active;
}

__device__ __forceinline__ float absmax8(const uint4& u) {
  const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(hv[i]);
    m = fmaxf(m, fmaxf(fabsf(t.x), fabsf(t.y)));
  }
  return m;
}

// amax: max |x| per (segment, head) of q, k and v, by an atomic max on the
// fp32 bit pattern (non-negative floats order as unsigned integers) into a
// zeroed [3][batch * H] array: a 16-lane slot group reduces its lanes' maxima
// by shuffles and adds one atomic each time its row leaves a segment, and
// once at the end.
__global__ void __launch_bounds__(kSweepThreads, kAmaxBlocksPerSm) varlen_fp8_amax_kernel(const Fp8Params p) {
  const int32_t B = p.batch, H = p.num_heads;
  int h, gl;
  int64_t row_off, R;
  sweep_slot(H, h, gl, row_off, R);
  for (int which = 0; which < 3; ++which) {
    const Sweep X = sweep_of(p, which);
    unsigned int* amax = reinterpret_cast<unsigned int*>(p.amax) + (int64_t)which * B * H;
    const __nv_bfloat16* base = X.x + (int64_t)h * X.hs + gl * 8;
    int32_t b = -1, seg_lo = 0, seg_hi = 0;  // current segment and its rows
    float m = 0.f;
    for (int64_t r = X.lo + row_off;; r += kSweepUnroll * R) {
      if (!__any_sync(0xffffffffu, r < X.hi)) break;
      uint4 u[kSweepUnroll];
#pragma unroll
      for (int k = 0; k < kSweepUnroll; ++k) {
        const int64_t rk = r + k * R;
        const __nv_bfloat16* a = base + rk * X.rs;
        u[k] = (rk < X.hi && in_span(X.span, a, 16, p.err)) ? __ldg(reinterpret_cast<const uint4*>(a))
                                                            : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < kSweepUnroll; ++k) {
        const int64_t rk = r + k * R;
        const bool valid = rk < X.hi;
        const bool leave = valid && (rk < seg_lo || rk >= seg_hi);  // same for the 16 lanes of a slot group
        if (__any_sync(0xffffffffu, leave)) {
          float mx = m;
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (leave) {
            if (gl == 0 && b >= 0) {
              unsigned int* slot = amax + (int64_t)b * H + h;
              if (in_span(p.amax_span, slot, 4, p.err)) atomicMax(slot, __float_as_uint(mx));
            }
            m = 0.f;
            if (segment_of_row(X.cu, B, X.total, (int32_t)rk, b)) {
              seg_lo = clamp_row(cu_at(X.cu, b), X.total);
              seg_hi = clamp_row(cu_at(X.cu, b + 1), X.total);
            } else {  // no segment holds the row: look again at the next one
              b = -1;
              seg_lo = (int32_t)rk;
              seg_hi = (int32_t)rk + 1;
            }
          }
        }
        if (valid && b >= 0) m = fmaxf(m, absmax8(u[k]));
      }
    }
    float mx = m;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (gl == 0 && b >= 0) {
      unsigned int* slot = amax + (int64_t)b * H + h;
      if (in_span(p.amax_span, slot, 4, p.err)) atomicMax(slot, __float_as_uint(mx));
    }
  }
}

// Q and K to E4M3 codes [rows][H][128]: code = e4m3(x / descale), an IEEE
// fp32 division, descale = amax / 448 of the row's (segment, head).  Each
// lane writes the 8 codes of its 8 values: a slot group writes the 128-byte
// code row of its (row, head).
__global__ void __launch_bounds__(kSweepThreads, kQuantBlocksPerSm) varlen_fp8_quant_kernel(const Fp8Params p) {
  const int32_t B = p.batch, H = p.num_heads;
  int h, gl;
  int64_t row_off, R;
  if (!sweep_slot(H, h, gl, row_off, R)) return;  // no warp collectives below
  for (int which = 0; which < 2; ++which) {
    const Sweep X = sweep_of(p, which);
    uint8_t* dst8 = (which == 0 ? p.q8 : p.k8) + (int64_t)h * 128 + gl * 8;
    const Span ds = which == 0 ? p.q8_span : p.k8_span;
    const float* amax = p.amax + (int64_t)which * B * H + h;
    const __nv_bfloat16* base = X.x + (int64_t)h * X.hs + gl * 8;
    int32_t b = -1, seg_lo = 0, seg_hi = 0;
    Divider dsc = divider(1.f);
    for (int64_t r = X.lo + row_off; r < X.hi; r += kSweepUnroll * R) {
      uint4 u[kSweepUnroll];
#pragma unroll
      for (int k = 0; k < kSweepUnroll; ++k) {
        const int64_t rk = r + k * R;
        const __nv_bfloat16* a = base + rk * X.rs;
        u[k] = (rk < X.hi && in_span(X.span, a, 16, p.err)) ? __ldg(reinterpret_cast<const uint4*>(a))
                                                            : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < kSweepUnroll; ++k) {
        const int64_t rk = r + k * R;
        if (rk >= X.hi) break;
        if (rk < seg_lo || rk >= seg_hi) {
          if (segment_of_row(X.cu, B, X.total, (int32_t)rk, b)) {
            seg_lo = clamp_row(cu_at(X.cu, b), X.total);
            seg_hi = clamp_row(cu_at(X.cu, b + 1), X.total);
            const float* am = amax + (int64_t)b * H;
            dsc = divider(descale_of(in_span(p.amax_span, am, 4, p.err) ? *am : 0.f));
          } else {
            b = -1;
            seg_lo = (int32_t)rk;
            seg_hi = (int32_t)rk + 1;
          }
        }
        if (b < 0) continue;  // no segment holds the row
        const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u[k]);
        float f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 t2 = __bfloat1622float2(hv[i]);
          f[2 * i] = t2.x;
          f[2 * i + 1] = t2.y;
        }
        uint2* out = reinterpret_cast<uint2*>(dst8 + rk * H * 128);
        if (in_span(ds, out, 8, p.err))
          *out = make_uint2(e4m3x4(f[0], f[1], f[2], f[3], dsc), e4m3x4(f[4], f[5], f[6], f[7], dsc));
      }
    }
  }
}

// ------------------------------------------------------------------ V^T codes

// One CTA visit = one 128-key block of one (segment, head).  Thread
// (row group g = lane, d slice s = warp) quantises keys 4g..4g+3 at
// d = 16s..16s+15 and packs, per d, the four keys' codes into one 32-bit
// word of the transposed tile (a warp's words fill a 128-byte tile row:
// conflict-free); the tile then leaves as 128-byte rows of vt.
__global__ void __launch_bounds__(256, 4) varlen_fp8_vt_kernel(const Fp8Params p) {
  __shared__ __align__(16) uint32_t tile[128 * 32];  // [d][128 keys] codes
  const int g = threadIdx.x & 31, s = threadIdx.x >> 5;
  const int32_t B = p.batch, H = p.num_heads;
  const float* amax = p.amax + 2 * (int64_t)B * H;
  SegCursor c;
  cursor_init<128>(c, p.cu_k, p.cu_q, B, p.total_k, p.total_q);
  for (int64_t t = blockIdx.x; cursor_seek<128>(c, t, H, p.cu_k, p.cu_q, B, p.total_k, p.total_q);
       t += gridDim.x) {
    // the segment's tiles in (key block, head) order, heads fastest: the
    // grid's concurrent visits read whole rows of adjacent key blocks
    Tile tl;
    tl.b = c.b;
    tl.m = (int32_t)((t - c.first) / H);
    tl.h = (int32_t)(t - c.first - (int64_t)tl.m * H);
    const int32_t valid = min(128, c.len - tl.m * 128);
    const float* am = amax + (int64_t)c.b * H + tl.h;
    const Divider dsc = divider(descale_of(in_span(p.amax_span, am, 4, p.err) ? *am : 0.f));
    const __nv_bfloat16* src =
        p.v + ((int64_t)c.r0 + tl.m * 128 + 4 * g) * p.v_rs + (int64_t)tl.h * p.v_hs + s * 16;
    uint4 u[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const __nv_bfloat16* a = src + i * p.v_rs + hf * 8;
        u[i][hf] = (4 * g + i < valid && in_span(p.v_span, a, 16, p.err)) ? __ldg(reinterpret_cast<const uint4*>(a))
                                                                          : make_uint4(0, 0, 0, 0);
      }
    uint32_t w[16];  // w[j]: codes of keys 4g..4g+3 at d = 16s + j (keys past the segment end: 0)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t a[4], e[4];  // key 4g+i: codes of d = 16s + 8hf + 0..3 (a) and + 4..7 (e), low byte first
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u[i][hf]);
        float f[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 t2 = __bfloat1622float2(hv[k]);
          f[2 * k] = t2.x;
          f[2 * k + 1] = t2.y;
        }
        const bool in = 4 * g + i < valid;
        a[i] = in ? e4m3x4(f[0], f[1], f[2], f[3], dsc) : 0u;
        e[i] = in ? e4m3x4(f[4], f[5], f[6], f[7], dsc) : 0u;
      }
      // 4 x 4 byte transposes: word k of the result holds byte k of the
      // four keys' words, key 4g+i in byte i
      transpose4x4(a, &w[hf * 8]);
      transpose4x4(e, &w[hf * 8 + 4]);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) tile[(s * 16 + j) * 32 + g] = w[j];
    __syncthreads();
    // tile row dd (128 codes) -> vt[h][dd][base + 128 m ...]: 8 lanes per row, 16 bytes each
    const int64_t col0 = fp8_vt_base(c.r0, c.b) + (int64_t)tl.m * 128;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int dd = s * 16 + k * 4 + (g >> 3), part = g & 7;
      uint4* dst = reinterpret_cast<uint4*>(p.vt + ((int64_t)tl.h * 128 + dd) * p.kp + col0) + part;
      if (in_span(p.vt_span, dst, 16, p.err)) *dst = reinterpret_cast<const uint4*>(tile + dd * 32)[part];
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ forward

namespace {

constexpr int kF8Unit = 2 * kTileM;           // q rows per scheduled unit (two halves)
constexpr int kF8Tile = 128 * 128;            // one tile: 128 rows of 128 codes
constexpr int kF8Slots = 8;                   // K / V^T ring slots
constexpr int kF8OrderOff = 1024 + kF8Tile * (2 + kF8Slots);  // LPT order table (from the aligned base)
constexpr int kF8SmemBytes = 1024 + kF8OrderOff + 2 * kLptCapWide;  // align, barriers, Q_A Q_B, ring, order
constexpr int kF8OCol = 256;                  // TMEM column of O_A (O_B at +128); S_A at 0, S_B at 128

struct F8Barriers {
  uint64_t q_full, q_empty;
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t mma_done;
  uint64_t kv_full[kF8Slots], kv_empty[kF8Slots];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(F8Barriers) <= 1024, "barrier block too large");

// Registers: 384 threads at 168; control warpgroup 112, softmax 192.
constexpr uint32_t kF8RegsLaunch = 168, kF8RegsCtl = 112, kF8RegsSoftmax = 192;
static_assert(kF8RegsCtl + 2 * kF8RegsSoftmax <= 3 * kF8RegsLaunch, "register split exceeds the launch allocation");

// kv tiles [j_lo, j_lo + n) a unit (kF8Unit q rows of one segment and
// head) works through, n returned.  With a mask (the band of Fp8Params) only
// the tiles holding keys that some row of the unit sees; 0 means no row of
// the unit sees a key (O = 0, LSE = -inf).
template <bool MASKED>
__device__ __forceinline__ int32_t fp8_kv_tiles(const SegCursor& c, int32_t unit, const Fp8Params& p,
                                                int32_t& j_lo) {
  j_lo = 0;
  int32_t nkv = (c.olen + kTileN - 1) / kTileN;
  if (MASKED) {
    const int64_t q0 = (int64_t)unit * kF8Unit;
    const int64_t q1 = min((int64_t)c.len, q0 + kF8Unit) - 1;
    int32_t lo, hi;
    band_keys(q0, q1, c.len, c.olen, p.win_left, p.win_right, &lo, &hi);
    if (hi <= lo) return 0;
    j_lo = lo / kTileN;
    nkv = (hi + kTileN - 1) / kTileN - j_lo;
  }
  return nkv;
}

}  // namespace

template <bool MASKED>
__global__ void __launch_bounds__(384, 1)
    varlen_fp8_fwd_kernel(const __grid_constant__ CUtensorMap tm_q8, const __grid_constant__ CUtensorMap tm_k8,
                          const __grid_constant__ CUtensorMap tm_vt, const Fp8Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  F8Barriers& bar = *reinterpret_cast<F8Barriers*>(smem);
  uint8_t* q_smem = smem + 1024;              // Q_A, Q_B
  uint8_t* ring = q_smem + 2 * kF8Tile;
  volatile int* abort = &bar.abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.p_full[i], 128);
      mbar_init(&bar.pv_done[i], 1);
    }
    mbar_init(&bar.mma_done, 1);
    for (int i = 0; i < kF8Slots; ++i) {
      mbar_init(&bar.kv_full[i], 1);
      mbar_init(&bar.kv_empty[i], 1);
    }
    bar.abort = 0;
    fence_barrier_init();
  }
  const WalkOrder order{reinterpret_cast<const uint16_t*>(smem + kF8OrderOff), kLptCapWide};
  build_lpt_order(order, p.cu_k, p.batch, p.total_k);
  if (warp == 1) tmem_alloc(&bar.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  const int64_t G = gridDim.x;
  const int32_t H = p.num_heads;

  if (warp < 4) {
    warpgroup_set_regs<kF8RegsCtl, kF8RegsLaunch>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tm_q8);
      tma_prefetch_desc(&tm_k8);
      tma_prefetch_desc(&tm_vt);
      SegCursor c;
      cursor_init<kF8Unit>(c, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order);
      uint32_t q_loads = 0, ring_pos = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x;
           ok && cursor_seek<kF8Unit>(c, t, H, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order); t += G) {
        const Tile tl = cursor_tile(c, t);
        int32_t j_lo;
        const int32_t nkv = fp8_kv_tiles<MASKED>(c, tl.m, p, j_lo);
        if (nkv == 0) continue;
        const int32_t qrow = c.r0 + tl.m * kF8Unit;
        if (q_loads > 0 && !mbar_wait(&bar.q_empty, (q_loads - 1) & 1, abort)) break;
        mbar_arrive_expect_tx(&bar.q_full, 2 * kF8Tile);
        tma_load_3d(q_smem, &tm_q8, &bar.q_full, 0, tl.h, qrow);
        tma_load_3d(q_smem + kF8Tile, &tm_q8, &bar.q_full, 0, tl.h, qrow + kTileM);
        ++q_loads;
        const int32_t vt0 = (int32_t)fp8_vt_base(c.o0, c.b);
        for (int32_t j = 0; ok && j < nkv; ++j) {
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            const uint32_t slot = ring_pos % kF8Slots;
            if (!mbar_wait(&bar.kv_empty[slot], ((ring_pos / kF8Slots) & 1) ^ 1, abort)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bar.kv_full[slot], kF8Tile);
            uint8_t* dst = ring + slot * kF8Tile;
            if (which == 0) tma_load_3d(dst, &tm_k8, &bar.kv_full[slot], 0, tl.h, c.o0 + (j_lo + j) * kTileN);
            else tma_load_3d(dst, &tm_vt, &bar.kv_full[slot], vt0 + (j_lo + j) * kTileN, 0, tl.h);
            ++ring_pos;
          }
        }
      }
      if (*abort) {
        for (uint32_t s = 0; s < (uint32_t)kF8Slots && s < ring_pos; ++s) {
          const uint32_t last = ring_pos - 1 - ((ring_pos - 1 - s) % kF8Slots);
          int dummy = 0;
          mbar_wait(&bar.kv_full[s], (last / kF8Slots) & 1, &dummy, 100000000ull);
        }
        if (q_loads > 0) {
          int dummy = 0;
          mbar_wait(&bar.q_full, (q_loads - 1) & 1, &dummy, 100000000ull);
        }
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      // Per kv step j and half: O += P V_j (P from TMEM, E4M3 codes written
      // over the first 32 of the half's S columns), then S = Q K_{j+1}^T,
      // which overwrites them only after the product has read them (the
      // MMAs of one thread execute in issue order); 4 k-steps of 32 codes
      // per product.
      constexpr uint32_t kIdesc = idesc_e4m3_f32(128, 128);
      SegCursor c;
      cursor_init<kF8Unit>(c, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order);
      uint32_t tiles = 0, g = 0, ring0 = 0;
      bool ok = true;
      const uint32_t qlo = sw128_desc_lo(smem_addr(q_smem), 16);
      const uint32_t rlo = sw128_desc_lo(smem_addr(ring), 16);
      auto issue_s = [&](int hf, uint32_t kslot) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f8_ss_lo(tmem + hf * 128, qlo + ((hf * kF8Tile + kk * 32) >> 4), rlo + ((kslot * kF8Tile + kk * 32) >> 4),
                       kIdesc, kk > 0 ? 1u : 0u);
        mma_commit(&bar.s_full[hf]);
      };
      auto issue_pv = [&](int hf, uint32_t vslot, bool first) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f8_ts_lo(tmem + kF8OCol + hf * 128, tmem + hf * 128 + kk * 8, rlo + ((vslot * kF8Tile + kk * 32) >> 4),
                       kIdesc, (!first || kk > 0) ? 1u : 0u);
        mma_commit(&bar.pv_done[hf]);
      };
      for (int64_t t = blockIdx.x;
           ok && cursor_seek<kF8Unit>(c, t, H, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order); t += G) {
        int32_t j_lo;
        const int32_t nkv = fp8_kv_tiles<MASKED>(c, cursor_tile(c, t).m, p, j_lo);
        if (nkv == 0) continue;
        if (!mbar_wait(&bar.q_full, tiles & 1, abort)) break;
        ++tiles;
        {
          const uint32_t kslot = ring0 % kF8Slots;
          if (!mbar_wait(&bar.kv_full[kslot], (ring0 / kF8Slots) & 1, abort)) break;
          tc_fence_after();
          issue_s(0, kslot);
          issue_s(1, kslot);
          mma_commit(&bar.kv_empty[kslot]);
          if (nkv == 1) mma_commit(&bar.q_empty);
        }
        for (int32_t j = 0; j < nkv; ++j) {
          const uint32_t gj = g + j;
          const uint32_t vpos = ring0 + 2 * j + 1;
          const uint32_t vslot = vpos % kF8Slots;
          const bool more = j + 1 < nkv;
          const uint32_t kpos = vpos + 1;
          const uint32_t kslot = kpos % kF8Slots;
          if (!mbar_wait(&bar.kv_full[vslot], (vpos / kF8Slots) & 1, abort)) { ok = false; break; }
          if (more && !mbar_wait(&bar.kv_full[kslot], (kpos / kF8Slots) & 1, abort)) { ok = false; break; }
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            if (!mbar_wait(&bar.p_full[hf], gj & 1, abort)) { ok = false; break; }
            tc_fence_after();
            issue_pv(hf, vslot, j == 0);
            if (more) issue_s(hf, kslot);
          }
          if (!ok) break;
          mma_commit(&bar.kv_empty[vslot]);
          if (more) {
            mma_commit(&bar.kv_empty[kslot]);
            if (j + 1 == nkv - 1) mma_commit(&bar.q_empty);
          }
        }
        g += nkv;
        ring0 += 2 * nkv;
      }
      mma_commit(&bar.mma_done);
      int dummy = 0;
      mbar_wait(&bar.mma_done, 0, &dummy);
    }
  } else {
    warpgroup_set_regs<kF8RegsSoftmax, kF8RegsLaunch>();
    // ------------------------------------------------------------ softmax
    const int hf = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_col = hf * 128, o_col = kF8OCol + hf * 128;
    SegCursor c;
    cursor_init<kF8Unit>(c, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order);
    uint32_t g = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x;
         ok && cursor_seek<kF8Unit>(c, t, H, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order); t += G) {
      const Tile tl = cursor_tile(c, t);
      int32_t j_lo;
      const int32_t nkv = fp8_kv_tiles<MASKED>(c, tl.m, p, j_lo);
      const int32_t r_seg = tl.m * kF8Unit + hf * kTileM + row;
      const bool row_valid = r_seg < c.len;
      const int64_t grow = (int64_t)c.r0 + r_seg;
      __nv_bfloat16* orow = p.out + grow * p.o_rs + (int64_t)tl.h * p.o_hs;
      float* lse_out = p.lse + (int64_t)tl.h * p.total_q + grow;
      if (nkv == 0) {
        if (row_valid) {
#pragma unroll
          for (int d = 0; d < 128; d += 8)
            if (in_span(p.out_span, orow + d, 16, p.err)) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0, 0, 0, 0);
          if (in_span(p.lse_span, lse_out, 4, p.err)) *lse_out = -INFINITY;
        }
        continue;
      }
      const int64_t bh = (int64_t)c.b * H + tl.h;
      const int64_t nbh = (int64_t)p.batch * H;
      const float* aq = p.amax + bh;
      const float* ak = p.amax + nbh + bh;
      const float* av = p.amax + 2 * nbh + bh;
      const float qd = descale_of(in_span(p.amax_span, aq, 4, p.err) ? __ldg(aq) : 0.f);
      const float kd = descale_of(in_span(p.amax_span, ak, 4, p.err) ? __ldg(ak) : 0.f);
      const float vd = descale_of(in_span(p.amax_span, av, 4, p.err) ? __ldg(av) : 0.f);
      // The score factor in the log2 domain, floored at the smallest normal
      // float: a masked score (-inf) times c2 must stay -inf when
      // scale * qd * kd underflows.  The scores are then below 3e-31 in
      // magnitude, so P is 1 either way.
      const float c2 = fmaxf(p.scale * 1.4426950408889634f * qd * kd, FLT_MIN);
      // keys [key_lo, key_hi) this row sees: all Sk, or with a mask its band
      int32_t key_lo = 0, key_hi = c.olen;
      if (MASKED) band_keys(r_seg, r_seg, c.len, c.olen, p.win_left, p.win_right, &key_lo, &key_hi);
      float m_use = -INFINITY, l = 0.f;
      for (int32_t j = 0; j < nkv; ++j) {
        const uint32_t gj = g + j;
        if (!mbar_wait(&bar.s_full[hf], gj & 1, abort)) { ok = false; break; }
        tc_fence_after();
        float x[128];
        {
          // the four 32-column loads in flight together, one wait
          uint32_t s[128];
          uint32_t(&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
          uint32_t(&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
          uint32_t(&s2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[64]);
          uint32_t(&s3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[96]);
          const uint32_t ta = tmem + lane_off + s_col;
          tmem_ld32(ta + 0, s0);
          tmem_ld32(ta + 32, s1);
          tmem_ld32(ta + 64, s2);
          tmem_ld32(ta + 96, s3);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 128; ++i) x[i] = __uint_as_float(s[i]);
        }
        // keys the row does not see (past the segment end, or outside the
        // mask's band) are -inf, by select
        const int32_t lim = key_hi - (j_lo + j) * kTileN;
        if constexpr (MASKED) {
          const int32_t lim_lo = key_lo - (j_lo + j) * kTileN;
          if (__any_sync(0xffffffffu, lim_lo > 0)) {  // the band's left edge crosses this tile
#pragma unroll
            for (int i = 0; i < 128; ++i) x[i] = (i < lim && i >= lim_lo) ? x[i] : -INFINITY;
          } else if (__any_sync(0xffffffffu, lim < kTileN)) {
#pragma unroll
            for (int i = 0; i < 128; ++i) x[i] = (i < lim) ? x[i] : -INFINITY;
          }
        } else if (lim < kTileN) {
#pragma unroll
          for (int i = 0; i < 128; ++i) x[i] = (i < lim) ? x[i] : -INFINITY;
        }
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int i = 0; i < 128; i += 8) {
          m0 = fmax3(m0, x[i], x[i + 1]);
          m1 = fmax3(m1, x[i + 2], x[i + 3]);
          m2 = fmax3(m2, x[i + 4], x[i + 5]);
          m3 = fmax3(m3, x[i + 6], x[i + 7]);
        }
        const float m_new = fmaxf(m_use, fmaxf(fmax3(m0, m1, m2), m3) * c2);
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_use = m_new;
        } else if (m_new > m_use + 8.0f) {
          alpha = ex2(m_use - m_new);
          m_use = m_new;
          rescale = true;
        }
        // P = exp2(S c - m) in fp32, row sum of the unrounded P; the codes of
        // P go into TMEM over the first 32 S columns (already read), four
        // consecutive keys per 32-bit column, the A operand of P V.
        // (two lanes at a time: packed fma / add, as in the bf16 kernel)
        // a row that has seen no key yet keeps m = -inf; subtracting 0 then
        // gives P = exp2(-inf) = 0 instead of NaN
        const float m_sub = (MASKED && m_use == -INFINITY) ? 0.f : m_use;
        const float2 cc2 = make_float2(c2, c2), negm = make_float2(-m_sub, -m_sub);
        float2 rs2a = make_float2(0.f, 0.f), rs2b = make_float2(0.f, 0.f);
        uint32_t pw[32];
        // each 16-word half goes to TMEM as soon as it is packed, so the
        // first store overlaps the second half's arithmetic
#pragma unroll
        for (int hk = 0; hk < 2; ++hk) {
#pragma unroll
          for (int k = hk * 16; k < hk * 16 + 16; ++k) {
            const int e = k * 4;
            float2 t0 = ffma2(make_float2(x[e], x[e + 1]), cc2, negm);
            float2 t1 = ffma2(make_float2(x[e + 2], x[e + 3]), cc2, negm);
            t0.x = ex2(t0.x);
            t0.y = ex2(t0.y);
            t1.x = ex2(t1.x);
            t1.y = ex2(t1.y);
            rs2a = fadd2(rs2a, t0);
            rs2b = fadd2(rs2b, t1);
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(t0, __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(t1, __NV_SATFINITE, __NV_E4M3);
            pw[k] = lo | (hi << 16);
          }
          tmem_st16(tmem + lane_off + s_col + hk * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pw[hk * 16]));
        }
        const float rs = (rs2a.x + rs2a.y) + (rs2b.x + rs2b.y);
        l = fmaf(l, alpha, rs);
        if (__any_sync(0xffffffffu, rescale)) {
          // S_j was issued after O += P_{j-1} V_{j-1} of this half (issue
          // order), so O is complete here
#pragma unroll
          for (int d0 = 0; d0 < 128; d0 += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + o_col + d0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tmem + lane_off + o_col + d0, o);
          }
        }
        tmem_wait_st();  // P (and a rescaled O) are in TMEM
        tc_fence_before();
        mbar_arrive(&bar.p_full[hf]);
      }
      if (!ok) break;
      // epilogue: the last P V of this half, then O * vd / l and LSE
      const uint32_t gl = g + nkv - 1;
      if (!mbar_wait(&bar.pv_done[hf], gl & 1, abort)) break;
      tc_fence_after();
      const float f = l > 0.f ? vd / l : 0.f;
#pragma unroll
      for (int d0 = 0; d0 < 128; d0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + o_col + d0, o);
        tmem_wait_ld();
        if (row_valid) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * f, __uint_as_float(o[2 * i + 1]) * f);
          uint4* dst = reinterpret_cast<uint4*>(orow + d0);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (in_span(p.out_span, dst + i, 16, p.err)) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (row_valid && in_span(p.lse_span, lse_out, 4, p.err))
        *lse_out = l > 0.f ? (m_use + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      tc_fence_before();
      g += nkv;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && bar.abort) record_error(p.err, kErrTimeout);
}

cudaError_t launch_fwd_fp8(const Fp8Launch& L, cudaStream_t stream) {
  const Fp8Params& p = L.p;
  const int64_t nbh = (int64_t)p.batch * p.num_heads;
  cudaError_t e = cudaMemsetAsync(p.amax, 0, 3 * nbh * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  // grid-wide sweeps: a few CTAs per SM, and at least one row of slots (H * 16 threads)
  const int64_t min_blocks = ((int64_t)p.num_heads * 16 + kSweepThreads - 1) / kSweepThreads;
  const int64_t amax_blocks = std::max<int64_t>((int64_t)L.grid * kAmaxBlocksPerSm, min_blocks);
  const int64_t quant_blocks = std::max<int64_t>((int64_t)L.grid * kQuantBlocksPerSm, min_blocks);
  varlen_fp8_amax_kernel<<<(unsigned)amax_blocks, kSweepThreads, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  varlen_fp8_quant_kernel<<<(unsigned)quant_blocks, kSweepThreads, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  varlen_fp8_vt_kernel<<<L.grid * 4, 256, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.total_q == 0) return cudaSuccess;
  auto kern = p.masked ? varlen_fp8_fwd_kernel<true> : varlen_fp8_fwd_kernel<false>;
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  if (fa.numRegs != (int)kF8RegsLaunch) return cudaErrorInvalidConfiguration;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8SmemBytes)) != cudaSuccess)
    return e;
  kern<<<L.grid, 384, kF8SmemBytes, stream>>>(L.tm_q8, L.tm_k8, L.tm_vt, p);
  return cudaGetLastError();
}

}  // namespace varlen
