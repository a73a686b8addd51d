// varlen_bwd.cu -- backward of packed variable-length attention on sm_103a.
//
// Three kernels on the caller's stream:
//
//  1. varlen_bwd_prep_kernel (HBM-bound): for every q row i and head h,
//       delta[h,i] = sum_d dO[i,h,d] * O[i,h,d]      (fp32, from bf16)
//       lse2[h,i]  = LSE[h,i] * log2(e)
//     stored at segment-padded positions (segment b's rows start at the
//     16-byte aligned index pad_base(b)), and zero the fp32 dQ accumulator.
//     dO and O are read through their own row / head strides with 64-bit
//     offsets: the preprocess is where the "[FA4] cute varlen backward: int32
//     overflow in _bwd_preprocess" issue (sections "Summary", "Root cause")
//     wrapped cu_seqlens[b]*stride past 2^31.
//
//  2. varlen_bwd_main_kernel (tensor-bound), persistent over kv tiles
//     (segment b, 128 kv rows, head h) of an exact varlen schedule.  K and V
//     stay in shared memory; for each 128-row q step of the segment it issues
//     five tcgen05 MMAs, every one 128 rows by 128 (or D) columns, with TMEM
//     accumulators:
//         S^T  = K Q^T          (K = D)
//         dP^T = V dO^T         (K = D)
//         dV  += P^T dO         (K = 128; P^T read from TMEM, where it replaced S^T)
//         dK  += dS^T Q         (K = 128)
//         dQ^T = K^T dS^T       (K = 128; into the dP^T columns once dP^T was read)
//     (the contractions over q or kv skip 16-row k-steps past the segment end).
//     P^T = exp2(S^T * scale*log2e - lse2) and dS^T = P^T (dP^T - delta) are
//     computed by eight compute warps (thread = kv row, 64 of the 128 q
//     columns); P^T goes back to TMEM as bf16, dS^T to shared memory.  A
//     drain warpgroup reads each dQ^T out of TMEM, stages it in the Q / dO
//     stages the step is done with, and adds it into the fp32 accumulator
//     with TMA bulk reduce-adds, off the compute warps' path.  At the end of a kv tile,
//     dK * scale and dV go to their strided outputs; a segment without
//     queries writes zeros.
//
//  3. varlen_bwd_post_kernel (HBM-bound): dq = bf16(scale * dq_acc), strided.
//
// The deterministic form runs the main kernel without dQ^T (template flag
// DQ = false): dS^T goes into TMEM over the dP^T columns and dK reads it
// from there, the drain warpgroup idles, and the shared-memory dS^T buffer
// becomes a third Q stage; dQ then comes from the q-major kernel of
// varlen_bwd_dq.cu, and neither the accumulator zeroing nor the post kernel
// runs.  Masks (causal, sliding windows) are the template flag MASKED with
// the band in BwdParams: kv tiles run only the q steps whose rows see them.
//
// The gradient formulas are the standard ones for O = softmax(scale QK^T) V:
// dP = dO V^T, dS = P (dP - rowsum(dO o O)), dQ = scale dS K,
// dK = scale dS^T Q, dV = P^T dO.
#include <algorithm>

#include "sm103_ptx.cuh"
#include "varlen_internal.h"
#include "varlen_sched.cuh"

namespace varlen {

// ------------------------------------------------------------------ prep

// Persistent CTAs walk tiles of R consecutive q rows (all heads), tile t, t +
// gridDim.x, ...; small tiles keep the CTAs' shares even.  Every global
// access is coalesced:
//   * the tile's slice of the fp32 dQ accumulator is one contiguous region
//     (rows x H x D floats), zeroed with 16-byte stores;
//   * each (row, head) pair's O and dO vectors are read by a group of G lanes
//     (16 bytes per lane, D / 8 lanes active), adjacent groups taking
//     adjacent heads of the same row, so a warp reads whole rows;
//   * delta is reduced within the group by shuffles, transposed through
//     shared memory, and written with LSE * log2(e) head by head, rows
//     fastest, at the segment-padded positions (a row's segment is found once
//     per row by a binary search over cu_seqlens_q).
// All offsets are 64-bit.
constexpr int kPrepThreads = 256;
constexpr int kPrepBlocksPerSm = 8;  // persistent CTAs per SM (32 registers per thread)

template <int D>
__global__ void __launch_bounds__(kPrepThreads, kPrepBlocksPerSm) varlen_bwd_prep_kernel(const PrepParams p) {
  constexpr int G = D == 64 ? 8 : 16;  // lanes per (row, head) pair
  constexpr int NCH = D / 8;           // 16-byte chunks per vector
  constexpr int PAIRS_PER_WARP = 32 / G;
  extern __shared__ __align__(16) uint8_t prep_smem[];
  const int H = p.num_heads, R = p.rows_per_tile;
  int64_t* s_pidx = reinterpret_cast<int64_t*>(prep_smem);           // [R] padded index, -1: no segment
  float* s_delta = reinterpret_cast<float*>(prep_smem + 8 * R);      // [H][R]
  const int32_t B = p.batch;
  const int32_t lo = clamp_row(cu_at(p.cu_q, 0), p.total_q);
  const int32_t hi = clamp_row(cu_at(p.cu_q, B), p.total_q);
  const int tid = threadIdx.x;
  for (int64_t row0 = (int64_t)lo + (int64_t)blockIdx.x * R; row0 < hi; row0 += (int64_t)gridDim.x * R) {
  const int nrows = (int)min((int64_t)R, (int64_t)hi - row0);

  // 1. the accumulator rows of the tile, one contiguous region
  if (p.dq_acc != nullptr) {
    float4* z = reinterpret_cast<float4*>(p.dq_acc + row0 * H * D);
    const int64_t n4 = (int64_t)nrows * H * (D / 4);
    for (int64_t i = tid; i < n4; i += kPrepThreads)
      if (in_span(p.acc_span, z + i, 16, p.err)) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // 2. padded index of each row: the last b with clamp(cu_q[b]) <= row
  //    (exact for non-decreasing cu_seqlens); -1 when no segment holds it
  for (int r = tid; r < nrows; r += kPrepThreads) {
    const int32_t row = (int32_t)(row0 + r);
    int32_t b0 = 0, b1 = B - 1;
    while (b0 < b1) {
      const int32_t mid = (b0 + b1 + 1) >> 1;
      if (clamp_row(cu_at(p.cu_q, mid), p.total_q) <= row) b0 = mid;
      else b1 = mid - 1;
    }
    const int32_t o0 = clamp_row(cu_at(p.cu_q, b0), p.total_q);
    const int32_t e = clamp_row(cu_at(p.cu_q, b0 + 1), p.total_q);
    s_pidx[r] = (row >= o0 && row < e) ? pad_base(o0, b0) + (row - o0) : -1;
  }
  // 3. delta of every (row, head) pair of the tile; all lanes of a warp run
  //    the same iterations (the shuffles need the whole warp)
  const int warp = tid >> 5, lane = tid & 31;
  const int sub = lane / G, gl = lane % G;
  const int npairs = nrows * H;
  constexpr int kWarps = kPrepThreads / 32;
  for (int base = warp * PAIRS_PER_WARP; base < npairs; base += 2 * kWarps * PAIRS_PER_WARP) {
    float acc[2] = {0.f, 0.f};
    uint4 a[2], c[2];
    int pr[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {  // both pairs' loads are issued before the arithmetic
      pr[u] = base + u * kWarps * PAIRS_PER_WARP + sub;
      a[u] = c[u] = make_uint4(0, 0, 0, 0);
      if (pr[u] < npairs && gl < NCH) {
        const int r = pr[u] / H, h = pr[u] - r * H;
        const int64_t row = row0 + r;
        const uint4* pa = reinterpret_cast<const uint4*>(p.out + row * p.o_rs + (int64_t)h * p.o_hs + gl * 8);
        const uint4* pc = reinterpret_cast<const uint4*>(p.dout + row * p.do_rs + (int64_t)h * p.do_hs + gl * 8);
        if (in_span(p.out_span, pa, 16, p.err)) a[u] = __ldg(pa);
        if (in_span(p.dout_span, pc, 16, p.err)) c[u] = __ldg(pc);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
      const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(&c[u]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(a2[i]);
        const float2 y = __bfloat1622float2(c2[i]);
        acc[u] = fmaf(x.x, y.x, acc[u]);
        acc[u] = fmaf(x.y, y.y, acc[u]);
      }
#pragma unroll
      for (int o = G / 2; o >= 1; o >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
      if (gl == 0 && pr[u] < npairs) {
        const int r = pr[u] / H, h = pr[u] - r * H;
        s_delta[h * R + r] = acc[u];
      }
    }
  }
  __syncthreads();
  // 4. delta and lse2 head by head, rows fastest
  const float kLog2e = 1.4426950408889634f;
  for (int i = tid; i < npairs; i += kPrepThreads) {
    const int h = i / nrows, r = i - h * nrows;
    const int64_t pi = s_pidx[r];
    if (pi >= 0) {
      const int64_t idx = (int64_t)h * p.pad_rows + pi;
      const float* pl = p.lse + (int64_t)h * p.total_q + row0 + r;
      const float lv = in_span(p.lse_span, pl, 4, p.err) ? __ldg(pl) : 0.f;
      if (in_span(p.delta_span, p.delta + idx, 4, p.err)) p.delta[idx] = s_delta[h * R + r];
      if (in_span(p.lse2_span, p.lse2 + idx, 4, p.err)) p.lse2[idx] = lv * kLog2e;
    }
  }
  __syncthreads();  // the next tile rewrites s_pidx and s_delta
  }
}

// Rows per preprocess tile: 8 (32-byte runs of delta per head), fewer for
// many heads so that the transposed delta tile stays within 16 KB of shared
// memory.
inline int prep_rows_per_tile(int H) { return H >= 4096 ? 1 : min(8, 4096 / H); }
inline size_t prep_smem_bytes(int H, int R) { return (size_t)8 * R + (size_t)4 * H * R; }

// ------------------------------------------------------------------ post

__global__ void __launch_bounds__(256) varlen_bwd_post_kernel(const PostParams p) {
  const int32_t B = p.batch;
  const int32_t lo = clamp_row(cu_at(p.cu_q, 0), p.total_q);
  const int32_t hi = clamp_row(cu_at(p.cu_q, B), p.total_q);
  if (hi <= lo) return;
  const int H = p.num_heads, D = p.head_dim, V = D / 8;
  const int64_t n = (int64_t)(hi - lo) * H * V;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t rh = t / V;
    const int v = (int)(t - rh * V);
    const int64_t row = lo + rh / H;
    const int h = (int)(rh % H);
    const float4* s = reinterpret_cast<const float4*>(p.dq_acc + (row * H + h) * D + v * 8);
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 a = in_span(p.acc_span, s, 16, p.err) ? s[0] : z4;
    const float4 b = in_span(p.acc_span, s + 1, 16, p.err) ? s[1] : z4;
    uint4 w;
    w.x = pack_bf16x2(a.x * p.scale, a.y * p.scale);
    w.y = pack_bf16x2(a.z * p.scale, a.w * p.scale);
    w.z = pack_bf16x2(b.x * p.scale, b.y * p.scale);
    w.w = pack_bf16x2(b.z * p.scale, b.w * p.scale);
    uint4* dst = reinterpret_cast<uint4*>(p.dq + row * p.dq_rs + (int64_t)h * p.dq_hs + v * 8);
    if (in_span(p.dq_span, dst, 16, p.err)) *dst = w;
  }
}

// ------------------------------------------------------------------ main

constexpr int QT_ROWS = 128;  // q rows per backward step (kBwdTileQ)

// DQ: the kernel computes dQ^T (the default form); without it (the
// deterministic form) dS^T lives in TMEM and its shared-memory buffer
// becomes a third Q stage.
template <int D, bool DQ>
struct BwdCfg {
  static constexpr int NC = (D + 63) / 64;       // 64-column chunks of Q / dO / V
  static constexpr int KCH = 2;                  // K tile always holds 128 columns (dQ^T uses M = 128)
  static constexpr int CHUNK = 128 * 128;        // 128 rows x 128 B
  static constexpr int K_BYTES = KCH * CHUNK;
  static constexpr int V_BYTES = NC * CHUNK;
  static constexpr int T_BYTES = NC * CHUNK;     // one Q or dO tile (128 rows)
  static constexpr int NQ = (NC == 1 || !DQ) ? 3 : 2;  // Q ring depth
  static constexpr int NDO = NC == 1 ? 3 : 2;    // dO ring depth
  static constexpr int DS_BYTES = DQ ? 2 * CHUNK : 0;  // dS^T: 128 kv rows x 128 q (bf16), two 64-q chunks
  static constexpr int ROWV_BYTES = QT_ROWS * 4; // one step's lse2 or delta (128 floats)
  // Tiles from the (1024-byte aligned) base, then the barriers and the
  // per-stage lse2 / delta rows.
  static constexpr int TILE_BYTES = K_BYTES + V_BYTES + (NQ + NDO) * T_BYTES + DS_BYTES;
  static constexpr int BAR_OFF = TILE_BYTES;
  static constexpr int LSE_OFF = BAR_OFF + 256;
  static constexpr int DELTA_OFF = LSE_OFF + NQ * ROWV_BYTES;
  static constexpr int ORDER_OFF = DELTA_OFF + NDO * ROWV_BYTES;  // LPT order table
  static constexpr int ORDER_ROOM = (227 * 1024 - ORDER_OFF) / 2;    // entries that still fit
  static constexpr int ORDER_CAP = ORDER_ROOM < kLptCapNarrow ? ORDER_ROOM / 8 * 8 : kLptCapNarrow;
  static constexpr int SMEM_BYTES = ORDER_OFF + 2 * ORDER_CAP;
  static_assert(SMEM_BYTES <= 227 * 1024, "backward tile does not fit one CTA's shared memory");
  // TMEM columns: S^T (later P^T, bf16), dP^T (later dQ^T), dV, dK
  static constexpr int S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 384;
  static constexpr int TMEM_COLS = 512;
};

// The q steps [j0, nq) a kv tile works through (128 q rows each).  With a
// mask (the band of BwdParams) only the steps holding q rows that see some
// key of the tile; j0 == nq means no query sees the tile (dK = dV = 0).
// The cursor's scheduled side is kv.
template <bool MASKED>
__device__ __forceinline__ void bwd_q_steps(const SegCursor& c, int32_t tile_m, const BwdParams& p, int32_t& j0,
                                            int32_t& nq) {
  nq = (c.olen + kBwdTileQ - 1) / kBwdTileQ;
  j0 = 0;
  if (MASKED) {
    const int64_t k0 = (int64_t)tile_m * kTileM;
    const int64_t k1 = min((int64_t)c.len, k0 + kTileM) - 1;
    int32_t lo, hi;
    band_rows(k0, k1, c.olen, c.len, p.win_left, p.win_right, &lo, &hi);
    if (hi <= lo) {
      j0 = nq = 0;
      return;
    }
    j0 = lo / kBwdTileQ;
    nq = (hi + kBwdTileQ - 1) / kBwdTileQ;
  }
}

// 512 threads: warpgroup 0 = Q/K/V producer (warp 0), MMA issuer (warp 1),
// dO producer (warp 2); warpgroups 1-2 = compute; warpgroup 3 = dQ drain.
constexpr int kBwdThreads = 512;
constexpr uint32_t kBwdRegsLaunch = 128;   // 65536 / 512, the launch allocation
constexpr uint32_t kBwdRegsCtl = 104;
constexpr uint32_t kBwdRegsCompute = 144;
constexpr uint32_t kBwdRegsDrain = 112;
static_assert(128 * kBwdRegsCtl + 256 * kBwdRegsCompute + 128 * kBwdRegsDrain <= 512 * kBwdRegsLaunch,
              "register split exceeds the launch allocation");

struct BwdBarriers {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[3], q_empty[3], do_full[3], do_empty[3];
  uint64_t s_full, p_ready, dp_full, ds_ready, ps_free, ds_free, dq_full, dq_free, acc_ready, acc_free, mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(BwdBarriers) <= 256, "barrier block overflows its slot");

// Clears rows [row_from, row_to) of a tile made of `chunks` chunks of
// 128-byte rows (one thread; at most 15 rows per call).
__device__ __forceinline__ void clear_rows(uint8_t* tile, int chunks, int chunk_bytes, int row_from, int row_to) {
  for (int cc = 0; cc < chunks; ++cc) {
    uint4* base = reinterpret_cast<uint4*>(tile + cc * chunk_bytes + row_from * 128);
    for (int u = 0; u < (row_to - row_from) * 8; ++u) base[u] = make_uint4(0, 0, 0, 0);
  }
}

template <int D, bool MASKED, bool DQ>
__global__ void __launch_bounds__(kBwdThreads, 1)
    varlen_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                           const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D, DQ>;
  constexpr int QT = kBwdTileQ;  // 128
  static_assert(QT == QT_ROWS, "step rows");
  // The 128-byte swizzled tiles need 1024-byte alignment; the declaration
  // asks for it and the kernel refuses to run without it (there is no
  // room to pad: the tiles and rows take the whole 227 KB).
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_addr(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(p.err, kErrBounds);
    return;
  }
  uint8_t* smem = smem_raw;
  BwdBarriers& bar = *reinterpret_cast<BwdBarriers*>(smem + C::BAR_OFF);
  float* lse_rows = reinterpret_cast<float*>(smem + C::LSE_OFF);      // [NQ][128] lse2 of the Q stage's step
  float* delta_rows = reinterpret_cast<float*>(smem + C::DELTA_OFF);  // [NDO][128] delta of the dO stage's step
  uint8_t* k_smem = smem;
  uint8_t* v_smem = k_smem + C::K_BYTES;
  uint8_t* q_smem = v_smem + C::V_BYTES;              // [NQ] Q tiles
  uint8_t* do_smem = q_smem + C::NQ * C::T_BYTES;     // [NDO] dO tiles
  uint8_t* ds_smem = do_smem + C::NDO * C::T_BYTES;   // dS^T
  volatile int* abort = &bar.abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = warp >> 2;

  if (threadIdx.x == 0) {
    mbar_init(&bar.kv_full, 1);
    mbar_init(&bar.kv_empty, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&bar.q_full[i], 1);
      mbar_init(&bar.q_empty[i], 1);
      mbar_init(&bar.do_full[i], 1);
      mbar_init(&bar.do_empty[i], DQ ? 4 : 1);  // the four drain warps, or the MMA commit after dV
    }
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.p_ready, 8);
    mbar_init(&bar.dp_full, 1);
    mbar_init(&bar.ds_ready, 8);
    mbar_init(&bar.ps_free, 1);
    mbar_init(&bar.ds_free, 4);  // the four drain warps (with dQ only)
    mbar_init(&bar.dq_full, 1);
    mbar_init(&bar.dq_free, 4);     // the four drain warps
    mbar_init(&bar.acc_ready, 1);
    mbar_init(&bar.acc_free, 8);
    mbar_init(&bar.mma_done, 1);
    bar.abort = 0;
    fence_barrier_init();
  }
  const WalkOrder order{reinterpret_cast<const uint16_t*>(smem_raw + C::ORDER_OFF), C::ORDER_CAP};
  build_lpt_order(order, p.cu_q, p.batch, p.total_q);
  if (warp == 1) tmem_alloc(&bar.tmem_base, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  const int64_t G = gridDim.x;

  if (wg == 0) {
    warpgroup_set_regs<kBwdRegsCtl, kBwdRegsLaunch>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------- Q / K / V producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      SegCursor c;
      cursor_init<kTileM>(c, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q, order);
      uint32_t tiles = 0, gs = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x;
           ok && cursor_seek<kTileM>(c, t, p.num_heads, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q, order); t += G) {
        const Tile tl = cursor_tile(c, t);
        int32_t j0, nq;
        bwd_q_steps<MASKED>(c, tl.m, p, j0, nq);
        if (j0 == nq) continue;  // no query sees the tile: dK = dV = 0, written by the compute warps
        const int32_t krow = c.r0 + tl.m * kTileM;
        if (tiles > 0 && !mbar_wait(&bar.kv_empty, (tiles - 1) & 1, abort)) break;
        mbar_arrive_expect_tx(&bar.kv_full, C::K_BYTES + C::V_BYTES);
#pragma unroll
        for (int cc = 0; cc < C::KCH; ++cc)
          tma_load_3d(k_smem + cc * C::CHUNK, &tm_k, &bar.kv_full, cc * 64, tl.h, krow);
#pragma unroll
        for (int cc = 0; cc < C::NC; ++cc)
          tma_load_3d(v_smem + cc * C::CHUNK, &tm_v, &bar.kv_full, cc * 64, tl.h, krow);
        ++tiles;
        for (int32_t j = j0; j < nq; ++j, ++gs) {
          const uint32_t st = gs % C::NQ;
          if (!mbar_wait(&bar.q_empty[st], ((gs / C::NQ) & 1) ^ 1, abort)) { ok = false; break; }
          // (failure test: CTA 0 leaves one step's Q load out; the waits for
          // it give up and the kernel unwinds, reporting a timeout)
          if (blockIdx.x == 0 && (int64_t)gs == (int64_t)p.debug_skip_step) continue;
          mbar_arrive_expect_tx(&bar.q_full[st], C::T_BYTES + C::ROWV_BYTES);
#pragma unroll
          for (int cc = 0; cc < C::NC; ++cc)
            tma_load_3d(q_smem + st * C::T_BYTES + cc * C::CHUNK, &tm_q, &bar.q_full[st], cc * 64, tl.h,
                        c.o0 + j * QT);
          bulk_load_1d(lse_rows + st * QT, p.lse2 + (int64_t)tl.h * p.pad_rows + pad_base(c.o0, c.b) + j * QT,
                       C::ROWV_BYTES, &bar.q_full[st]);
        }
      }
      if (*abort) {
        // let the loads in flight land before the CTA exits
        int dummy = 0;
        if (tiles > 0) mbar_wait(&bar.kv_full, (tiles - 1) & 1, &dummy, 100000000ull);
        for (uint32_t s = 0; s < (uint32_t)C::NQ && s < gs; ++s) {
          const uint32_t last = gs - 1 - ((gs - 1 - s) % C::NQ);
          mbar_wait(&bar.q_full[s], (last / C::NQ) & 1, &dummy, 100000000ull);
        }
      }
    } else if (warp == 2 && lane == 0) {
      // ---------------------------------------------------- dO producer
      tma_prefetch_desc(&tm_do);
      SegCursor c;
      cursor_init<kTileM>(c, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q, order);
      uint32_t gs = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x;
           ok && cursor_seek<kTileM>(c, t, p.num_heads, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q, order); t += G) {
        const Tile tl = cursor_tile(c, t);
        int32_t j0, nq;
        bwd_q_steps<MASKED>(c, tl.m, p, j0, nq);
        for (int32_t j = j0; j < nq; ++j, ++gs) {
          const uint32_t st = gs % C::NDO;
          if (!mbar_wait(&bar.do_empty[st], ((gs / C::NDO) & 1) ^ 1, abort)) { ok = false; break; }
          mbar_arrive_expect_tx(&bar.do_full[st], C::T_BYTES + C::ROWV_BYTES);
#pragma unroll
          for (int cc = 0; cc < C::NC; ++cc)
            tma_load_3d(do_smem + st * C::T_BYTES + cc * C::CHUNK, &tm_do, &bar.do_full[st], cc * 64, tl.h,
                        c.o0 + j * QT);
          bulk_load_1d(delta_rows + st * QT, p.delta + (int64_t)tl.h * p.pad_rows + pad_base(c.o0, c.b) + j * QT,
                       C::ROWV_BYTES, &bar.do_full[st]);
        }
      }
      if (*abort) {
        int dummy = 0;
        for (uint32_t s = 0; s < (uint32_t)C::NDO && s < gs; ++s) {
          const uint32_t last = gs - 1 - ((gs - 1 - s) % C::NDO);
          mbar_wait(&bar.do_full[s], (last / C::NDO) & 1, &dummy, 100000000ull);
        }
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------- MMA issuer
      // One thread issues every MMA of the CTA, straight through (the warp's
      // other lanes wait at the end): a warp that rejoins between MMA groups
      // or spends many integer instructions per MMA leaves the tensor pipe
      // idle.  Per q step g the pipe runs  dV_g, S^T_{g+1}, dQ^T_g, dK_g,
      // dP^T_{g+1}: S^T of the next step is computed while the compute warps
      // build dS_g, and dP^T of the next step goes in as soon as the drain
      // warps have read dQ^T_g out of the columns they share.
      constexpr uint32_t kIdS = idesc_bf16_f32(128, QT, false, false);  // S^T, dP^T
      constexpr uint32_t kIdG = idesc_bf16_f32(128, D, false, true);    // dV, dK
      constexpr uint32_t kIdQ = idesc_bf16_f32(128, QT, true, true);    // dQ^T
      SegCursor c;
      cursor_init<kTileM>(c, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q, order);
      uint32_t tiles = 0, gs = 0;
      // descriptor low words (the high word is the constant of the 128-byte swizzle)
      const uint32_t kK = sw128_desc_lo(smem_addr(k_smem), 16);        // K as K-major A
      const uint32_t vK = sw128_desc_lo(smem_addr(v_smem), 16);        // V as K-major A
      const uint32_t kM = sw128_desc_lo(smem_addr(k_smem), C::CHUNK);  // K^T as MN-major A
      const uint32_t sK = sw128_desc_lo(smem_addr(ds_smem), 16);       // dS^T as K-major A
      const uint32_t sM = sw128_desc_lo(smem_addr(ds_smem), C::CHUNK); // dS^T as MN-major B
      bool ok = true;

      // Waits for a Q or dO tile.  dK / dV contract over q in 16-row k-steps
      // and skip those wholly past the segment end; the rows of the last
      // partial k-step past the end meet dS^T = 0 (P^T = 0) and are cleared,
      // so that 0 * NaN cannot occur.
      auto ready = [&](uint64_t* full, uint32_t parity, uint8_t* tile, int32_t valid) -> bool {
        if (!mbar_wait(full, parity, abort)) return false;
        if (valid < QT) {
          clear_rows(tile, C::NC, C::CHUNK, valid, min(QT, (valid + 15) & ~15));
          fence_proxy_async_smem();
        }
        return true;
      };
      auto issue_s = [&](uint32_t g) {  // S^T_g = K Q_g^T, both K-major
        const uint32_t qK = sw128_desc_lo(smem_addr(q_smem + (g % C::NQ) * C::T_BYTES), 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          mma_ss_lo(tmem + C::S_COL, kK + o, qK + o, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar.s_full);
      };
      auto issue_dp = [&](uint32_t g) {  // dP^T_g = V dO_g^T, both K-major
        const uint32_t dK_ = sw128_desc_lo(smem_addr(do_smem + (g % C::NDO) * C::T_BYTES), 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          mma_ss_lo(tmem + C::DP_COL, vK + o, dK_ + o, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar.dp_full);
      };
      // dV += P^T_g (TMEM, bf16 where S^T was) dO_g (MN-major); nk q k-steps
      auto issue_dv = [&](uint32_t g, int nk, bool acc0) {
        const uint32_t dM = sw128_desc_lo(smem_addr(do_smem + (g % C::NDO) * C::T_BYTES), C::CHUNK);
#pragma unroll
        for (int kk = 0; kk < QT / 16; ++kk)
          if (kk < nk)
            mma_ts_lo(tmem + C::DV_COL, tmem + C::S_COL + (kk >> 2) * 64 + (kk & 3) * 8, dM + kk * 128, kIdG,
                      (acc0 || kk > 0) ? 1u : 0u);
      };
      // dQ^T = K^T (MN-major) dS^T (MN-major) into the dP^T columns; nk kv k-steps
      auto issue_dq = [&](int nk) {
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk)
          if (kk < nk) mma_ss_lo(tmem + C::DP_COL, kM + kk * 128, sM + kk * 128, kIdQ, kk > 0 ? 1u : 0u);
        mma_commit(&bar.dq_full);
      };
      // dK += dS^T_g Q_g (MN-major); nk q k-steps.  dS^T_g is the K-major
      // shared-memory buffer, or without dQ the bf16 copy the compute warps
      // wrote into the dP^T columns (q columns [0, 64) at [0, 32), [64, 128)
      // at [64, 96)); dP^T_{g+1} is issued after this product.
      auto issue_dk = [&](uint32_t g, int nk, bool acc0) {
        const uint32_t qM = sw128_desc_lo(smem_addr(q_smem + (g % C::NQ) * C::T_BYTES), C::CHUNK);
#pragma unroll
        for (int kk = 0; kk < QT / 16; ++kk) {
          const uint32_t ao = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          if (kk < nk) {
            if (DQ)
              mma_ss_lo(tmem + C::DK_COL, sK + ao, qM + kk * 128, kIdG, (acc0 || kk > 0) ? 1u : 0u);
            else
              mma_ts_lo(tmem + C::DK_COL, tmem + C::DP_COL + (kk >> 2) * 64 + (kk & 3) * 8, qM + kk * 128, kIdG,
                        (acc0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&bar.q_empty[g % C::NQ]);
      };

      for (int64_t t = blockIdx.x;
           ok && cursor_seek<kTileM>(c, t, p.num_heads, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q, order); t += G) {
        const Tile tl = cursor_tile(c, t);
        int32_t j0, nq;
        bwd_q_steps<MASKED>(c, tl.m, p, j0, nq);
        if (j0 == nq) continue;
        if (!mbar_wait(&bar.kv_full, tiles & 1, abort)) break;
        const int32_t kv_valid = min(kTileM, c.len - tl.m * kTileM);
        const int nk_kv = (kv_valid + 15) >> 4;  // kv k-steps of dQ^T
        if (kv_valid < kTileM) {
          // dQ^T = K^T dS^T contracts over kv: rows of the last partial
          // k-step past the segment end meet dS^T = 0; clear them.
          clear_rows(k_smem, C::KCH, C::CHUNK, kv_valid, min(kTileM, nk_kv * 16));
          fence_proxy_async_smem();
        }
        // prologue: S^T and dP^T of the tile's first step.  The S^T columns
        // were last read by dV of the previous step (earlier in this
        // thread's MMA order); the dP^T columns held the previous dQ^T.
        if (!ready(&bar.q_full[gs % C::NQ], (gs / C::NQ) & 1, q_smem + (gs % C::NQ) * C::T_BYTES,
                   c.olen - j0 * QT)) break;
        tc_fence_after();
        issue_s(gs);
        if (DQ && gs > 0 && !mbar_wait(&bar.dq_free, (gs - 1) & 1, abort)) break;
        if (!ready(&bar.do_full[gs % C::NDO], (gs / C::NDO) & 1, do_smem + (gs % C::NDO) * C::T_BYTES,
                   c.olen - j0 * QT)) break;
        tc_fence_after();
        issue_dp(gs);
        for (int32_t j = j0; j < nq; ++j, ++gs) {
          const bool more = j + 1 < nq;
          const int nk_q = (min(QT, c.olen - j * QT) + 15) >> 4;  // q k-steps of dV / dK
          // dV_g += P^T_g dO_g, P^T_g read from TMEM
          if (!mbar_wait(&bar.p_ready, gs & 1, abort)) { ok = false; break; }
          if (j == j0 && tiles > 0 && !mbar_wait(&bar.acc_free, (tiles - 1) & 1, abort)) { ok = false; break; }
          tc_fence_after();
          issue_dv(gs, nk_q, j > j0);  // the tile's first step starts the accumulation
          // S^T_{g+1}: overwrites P^T_g after dV_g has read it (same-thread MMA order)
          if (more) {
            const uint32_t g1 = gs + 1;
            if (!ready(&bar.q_full[g1 % C::NQ], (g1 / C::NQ) & 1, q_smem + (g1 % C::NQ) * C::T_BYTES,
                       c.olen - (j + 1) * QT)) { ok = false; break; }
            tc_fence_after();
            issue_s(g1);
          }
          // dQ^T_g = K^T dS^T_g into the dP^T columns; dK_g += dS^T_g Q_g
          if (!mbar_wait(&bar.ds_ready, gs & 1, abort)) { ok = false; break; }
          tc_fence_after();
          if (DQ) issue_dq(nk_kv);
          issue_dk(gs, nk_q, j > j0);
          if (DQ) mma_commit(&bar.ps_free);
          // Without dQ the dO stage (tile and delta row) is free once dK_g is
          // done: dK_g follows ds_ready_g, so the compute warps have read
          // this step's delta row, and dV_g, the tile's last reader, ran first.
          if (!DQ) mma_commit(&bar.do_empty[gs % C::NDO]);
          if (!more) {
            mma_commit(&bar.kv_empty);
            mma_commit(&bar.acc_ready);
          }
          // dP^T_{g+1} once the drain warps have read dQ^T_g
          if (more) {
            const uint32_t g1 = gs + 1;
            if (DQ && !mbar_wait(&bar.dq_free, gs & 1, abort)) { ok = false; break; }
            if (!ready(&bar.do_full[g1 % C::NDO], (g1 / C::NDO) & 1, do_smem + (g1 % C::NDO) * C::T_BYTES,
                       c.olen - (j + 1) * QT)) { ok = false; break; }
            tc_fence_after();
            issue_dp(g1);
          }
        }
        ++tiles;
      }
      mma_commit(&bar.mma_done);
      int dummy = 0;
      mbar_wait(&bar.mma_done, 0, &dummy);
    }
  } else if (wg <= 2) {
    warpgroup_set_regs<kBwdRegsCompute, kBwdRegsLaunch>();
    // ------------------------------------------------------------ compute
    const int quad = warp & 3;
    const int half = wg - 1;                       // which 64 q columns (and half of D in the epilogue)
    const int r = quad * 32 + lane;                // kv row in the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c2 = p.scale_log2;
    SegCursor c;
    cursor_init<kTileM>(c, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q, order);
    uint32_t gs = 0, tiles = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x;
         ok && cursor_seek<kTileM>(c, t, p.num_heads, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q, order); t += G) {
      const Tile tl = cursor_tile(c, t);
      const int32_t kv_valid = c.len - tl.m * kTileM;
      const bool row_valid = r < kv_valid;
      const int64_t krow = (int64_t)c.r0 + tl.m * kTileM + r;
      int32_t j0, nq;
      bwd_q_steps<MASKED>(c, tl.m, p, j0, nq);
      if (j0 == nq) {
        if (row_valid) {
          __nv_bfloat16* dvrow = p.dv + krow * p.dv_rs + (int64_t)tl.h * p.dv_hs;
          __nv_bfloat16* dkrow = p.dk + krow * p.dk_rs + (int64_t)tl.h * p.dk_hs;
          for (int d = half * (D / 2); d < (half + 1) * (D / 2); d += 8) {
            if (in_span(p.dv_span, dvrow + d, 16, p.err)) *reinterpret_cast<uint4*>(dvrow + d) = make_uint4(0, 0, 0, 0);
            if (in_span(p.dk_span, dkrow + d, 16, p.err)) *reinterpret_cast<uint4*>(dkrow + d) = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      // q rows [q_lo, q_hi) of the segment see this key: all of them, or
      // with a mask those whose band holds it
      int32_t q_lo = 0, q_hi = c.olen;
      if (MASKED) {
        const int64_t jr = (int64_t)tl.m * kTileM + r;
        band_rows(jr, jr, c.olen, c.len, p.win_left, p.win_right, &q_lo, &q_hi);
      }
      for (int32_t j = j0; j < nq; ++j, ++gs) {
        const int32_t qc0 = j * QT + half * 64;             // first q column of this thread (in the segment)
        const int32_t nvalid = row_valid ? max(0, min(64, q_hi - qc0)) : 0;
        const int32_t lo = MASKED ? min(64, max(0, q_lo - qc0)) : 0;  // columns [lo, nvalid) are visible
        // interior steps (every column of every lane visible) skip the per-element selects
        const bool all_vis = __all_sync(0xffffffffu, lo == 0 && nvalid == 64);
        // this step's lse2 / delta rows arrive with its Q / dO tiles
        const float4* l4 = reinterpret_cast<const float4*>(lse_rows + (gs % C::NQ) * QT + half * 64);
        const float4* d4 = reinterpret_cast<const float4*>(delta_rows + (gs % C::NDO) * QT + half * 64);
        // ---- P^T = exp2(S^T c - lse2), back into the S^T columns as bf16
        if (!mbar_wait(&bar.s_full, gs & 1, abort)) { ok = false; break; }
        if (!mbar_wait(&bar.q_full[gs % C::NQ], (gs / C::NQ) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        float pv[64];
        {
          uint32_t sv[64];
          tmem_ld32(tmem + lane_off + C::S_COL + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
          tmem_ld32(tmem + lane_off + C::S_COL + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 64; i += 4) {
            const float4 l = l4[i / 4];
            const float2 t0 = ffma2(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])),
                                    make_float2(c2, c2), make_float2(-l.x, -l.y));
            const float2 t1 = ffma2(make_float2(__uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3])),
                                    make_float2(c2, c2), make_float2(-l.z, -l.w));
            pv[i] = ex2(t0.x);
            pv[i + 1] = ex2(t0.y);
            pv[i + 2] = ex2(t1.x);
            pv[i + 3] = ex2(t1.y);
          }
          if (!all_vis) {
#pragma unroll
            for (int i = 0; i < 64; ++i) pv[i] = (i >= lo && i < nvalid) ? pv[i] : 0.f;
          }
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(pv[2 * i], pv[2 * i + 1]);
          tmem_st32(tmem + lane_off + C::S_COL + half * 64, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.p_ready);
        // ---- dS^T = P^T (dP^T - delta), into shared memory
        if (!mbar_wait(&bar.dp_full, gs & 1, abort)) { ok = false; break; }
        if (!mbar_wait(&bar.do_full[gs % C::NDO], (gs / C::NDO) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        uint32_t dk2[32];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t dpv[32];
          tmem_ld32(tmem + lane_off + C::DP_COL + half * 64 + h2 * 32, dpv);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 dl = d4[(h2 * 32 + i) / 4];
            const int ii = h2 * 32 + i;
            const float2 a = fmul2(make_float2(pv[ii], pv[ii + 1]),
                                   fadd2(make_float2(__uint_as_float(dpv[i]), __uint_as_float(dpv[i + 1])),
                                         make_float2(-dl.x, -dl.y)));
            const float2 b = fmul2(make_float2(pv[ii + 2], pv[ii + 3]),
                                   fadd2(make_float2(__uint_as_float(dpv[i + 2]), __uint_as_float(dpv[i + 3])),
                                         make_float2(-dl.z, -dl.w)));
            // select, not multiply: dP^T and delta past the segment end may hold NaN
            if (all_vis) {
              dk2[ii / 2] = pack_bf16x2(a.x, a.y);
              dk2[ii / 2 + 1] = pack_bf16x2(b.x, b.y);
            } else {
              dk2[ii / 2] = pack_bf16x2(ii >= lo && ii < nvalid ? a.x : 0.f, ii + 1 >= lo && ii + 1 < nvalid ? a.y : 0.f);
              dk2[ii / 2 + 1] = pack_bf16x2(ii + 2 >= lo && ii + 2 < nvalid ? b.x : 0.f,
                                            ii + 3 >= lo && ii + 3 < nvalid ? b.y : 0.f);
            }
          }
        }
        if (DQ) {
          // the dS^T buffer is free once dQ^T and dK of the previous step are
          // done and the drain has staged (and bulk-read) its dQ there
          if (gs > 0 && !mbar_wait(&bar.ds_free, (gs - 1) & 1, abort)) { ok = false; break; }
          // row r of chunk `half` (128-byte swizzle: 16-byte unit u of row r sits at u ^ (r % 8))
          uint8_t* dsrow = ds_smem + half * C::CHUNK + r * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(dsrow + ((u ^ (r & 7)) * 16)) =
                make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
          fence_proxy_async_smem();
        } else {
          // Without dQ, dS^T only feeds dK: it goes into TMEM over the first
          // 32 of the dP^T columns this thread read above.  dK_{g-1}, the
          // last reader of the previous copy, ran before dP^T_g.
          tmem_st32(tmem + lane_off + C::DP_COL + half * 64, dk2);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.ds_ready);
      }
      if (!ok) break;
      // ---- epilogue: dV and dK * scale of this kv tile
      if (!mbar_wait(&bar.acc_ready, tiles & 1, abort)) break;
      tc_fence_after();
#pragma unroll
      for (int d0 = half * (D / 2); d0 < (half + 1) * (D / 2); d0 += 16) {
        uint32_t a[16], b[16];
        tmem_ld16(tmem + lane_off + C::DV_COL + d0, a);
        tmem_ld16(tmem + lane_off + C::DK_COL + d0, b);
        tmem_wait_ld();
        if (row_valid) {
          uint32_t wa[8], wb[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            wa[i] = pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
            wb[i] = pack_bf16x2(__uint_as_float(b[2 * i]) * p.scale, __uint_as_float(b[2 * i + 1]) * p.scale);
          }
          uint4* dv4 = reinterpret_cast<uint4*>(p.dv + krow * p.dv_rs + (int64_t)tl.h * p.dv_hs + d0);
          uint4* dk4 = reinterpret_cast<uint4*>(p.dk + krow * p.dk_rs + (int64_t)tl.h * p.dk_hs + d0);
          if (in_span(p.dv_span, dv4, 16, p.err)) dv4[0] = make_uint4(wa[0], wa[1], wa[2], wa[3]);
          if (in_span(p.dv_span, dv4 + 1, 16, p.err)) dv4[1] = make_uint4(wa[4], wa[5], wa[6], wa[7]);
          if (in_span(p.dk_span, dk4, 16, p.err)) dk4[0] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
          if (in_span(p.dk_span, dk4 + 1, 16, p.err)) dk4[1] = make_uint4(wb[4], wb[5], wb[6], wb[7]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.acc_free);
      ++tiles;
    }
  } else {
    warpgroup_set_regs<kBwdRegsDrain, kBwdRegsLaunch>();
    // ------------------------------------------------------------ dQ drain
    // dQ^T_g (TMEM lane = d, column = q) is staged in shared memory the step
    // no longer needs -- q columns [0, 64) in the dO_g stage (free once dV_g
    // has run, which precedes dQ^T_g in MMA order), [64, 128) in the dS^T
    // buffer (free from the end of dQ^T_g and dK_g until the compute warps
    // write the next dS^T, which waits for ds_free) -- and added into
    // dq_acc by TMA bulk reduce-adds performed at L2.  Each warp owns 32
    // consecutive d: it stages a dense 64 (q) x 32 (d) fp32 block (8 KB) and
    // issues its own box, so the warps never wait for one another.  Rows of
    // q past the segment end are staged as exact zeros (dQ^T there is 0 * K,
    // NaN if K is), so whole boxes may be added: the next segment's rows are
    // unchanged.
    const int quad = warp & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const bool drains = quad * 32 < D;             // warp-uniform
    if (DQ) {  // (without dQ -- the deterministic form -- this warpgroup has no work)
      SegCursor c;
      cursor_init<kTileM>(c, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q, order);
      uint32_t gs = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x;
           ok && cursor_seek<kTileM>(c, t, p.num_heads, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q, order); t += G) {
        const Tile tl = cursor_tile(c, t);
        int32_t j0, nq;
        bwd_q_steps<MASKED>(c, tl.m, p, j0, nq);
        for (int32_t j = j0; j < nq; ++j, ++gs) {
          if (!mbar_wait(&bar.dq_full, gs & 1, abort)) { ok = false; break; }
          tc_fence_after();
          const int32_t n = min(QT, c.olen - j * QT);  // valid q columns of this step
          const int32_t row0 = c.o0 + j * QT;
          float* blk0 = reinterpret_cast<float*>(do_smem + (gs % C::NDO) * C::T_BYTES + quad * 8192);
          float* blk1 = reinterpret_cast<float*>(ds_smem + quad * 8192);
          uint32_t v[64];
          // q columns [0, 64) -> dO_g stage
          tmem_ld32(tmem + lane_off + C::DP_COL, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(tmem + lane_off + C::DP_COL + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_wait_ld();
          if (drains) {
  #pragma unroll
            for (int i = 0; i < 64; ++i) blk0[i * 32 + lane] = i < n ? __uint_as_float(v[i]) : 0.f;
            fence_proxy_async_smem();
          }
          // q columns [64, 128)
          tmem_ld32(tmem + lane_off + C::DP_COL + 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(tmem + lane_off + C::DP_COL + 96, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar.dq_free);  // every TMEM read done: the columns may take dP^T_{g+1}
          // ... into the dS^T buffer once dQ^T_g and dK_g are done with it
          if (!mbar_wait(&bar.ps_free, gs & 1, abort)) { ok = false; break; }
          if (drains && n > 64) {
  #pragma unroll
            for (int i = 0; i < 64; ++i) blk1[i * 32 + lane] = 64 + i < n ? __uint_as_float(v[i]) : 0.f;
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) {
            // The block in the dS^T buffer goes first, in a bulk group of its
            // own: the compute warps wait for that buffer (ds_free), while the
            // dO stage is not needed again until a later step.
            if (drains && n > 64) tma_reduce_add_3d(blk1, &tm_dq, quad * 32, tl.h, row0 + 64);
            bulk_commit();
            if (drains) tma_reduce_add_3d(blk0, &tm_dq, quad * 32, tl.h, row0);
            bulk_commit();
            bulk_wait_read_1();  // the dS^T-buffer block has been read
            mbar_arrive(&bar.ds_free);
            bulk_wait_read_all();  // the dO-stage block has been read
            mbar_arrive(&bar.do_empty[gs % C::NDO]);
          }
          __syncwarp();
        }
      }
      if (lane == 0) bulk_wait_all();  // this warp's reductions have completed
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && bar.abort) record_error(p.err, kErrTimeout);
}

template <int D, bool MASKED, bool DQ>
static cudaError_t launch_bwd_d(const BwdLaunch& L, cudaStream_t stream) {
  using C = BwdCfg<D, DQ>;
  const int elem_grid = L.grid * 8;
  PrepParams prep = L.prep;
  prep.rows_per_tile = prep_rows_per_tile(prep.num_heads);
  const size_t prep_smem = prep_smem_bytes(prep.num_heads, prep.rows_per_tile);
  const int32_t prep_rows = L.p.total_q;  // rows [cu[0], cu[B]) lie within [0, total_q)
  const unsigned prep_grid = (unsigned)std::max<int64_t>(
      1, std::min<int64_t>(((int64_t)prep_rows + prep.rows_per_tile - 1) / prep.rows_per_tile,
                           (int64_t)L.grid * kPrepBlocksPerSm));
  auto mark = [&](int i) {
    if (L.phase_events[i] != nullptr) cudaEventRecord(L.phase_events[i], stream);
  };
  auto kern = varlen_bwd_main_kernel<D, MASKED, DQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // The warpgroup register split assumes the kernel was compiled to exactly
  // the launch allocation; refuse to run it otherwise.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != (int)kBwdRegsLaunch) return cudaErrorInvalidConfiguration;
  mark(0);
  varlen_bwd_prep_kernel<D><<<prep_grid, kPrepThreads, prep_smem, stream>>>(prep);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mark(1);
  kern<<<L.grid, kBwdThreads, C::SMEM_BYTES, stream>>>(L.tm_q, L.tm_k, L.tm_v, L.tm_do, L.tm_dq, L.p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mark(2);
  if (DQ) {
    varlen_bwd_post_kernel<<<elem_grid, 256, 0, stream>>>(L.post);
    e = cudaGetLastError();
  } else {
    e = launch_bwd_dq(L, stream);
  }
  mark(3);
  return e;
}

template <int D>
static cudaError_t launch_bwd_dm(const BwdLaunch& L, cudaStream_t stream) {
  if (L.deterministic)
    return L.p.masked ? launch_bwd_d<D, true, false>(L, stream) : launch_bwd_d<D, false, false>(L, stream);
  return L.p.masked ? launch_bwd_d<D, true, true>(L, stream) : launch_bwd_d<D, false, true>(L, stream);
}

cudaError_t launch_bwd(const BwdLaunch& L, cudaStream_t stream) {
  switch (L.head_dim) {
    case 64: return launch_bwd_dm<64>(L, stream);
    case 96: return launch_bwd_dm<96>(L, stream);
    case 128: return launch_bwd_dm<128>(L, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace varlen
