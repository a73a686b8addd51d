// varlen_bwd_dq.cu -- deterministic dQ of packed variable-length attention
// on sm_103a.
//
// The main backward kernel adds each kv tile's dQ contribution into an fp32
// accumulator with reduce-adds performed at L2, so the order of the adds --
// and the low bits of dQ -- vary between runs.  The deterministic form runs
// that kernel without its dQ products and computes dQ here instead, q-major:
// persistent over q tiles (segment b, 128 q rows, head h) of an exact varlen
// schedule, each tile walks the kv tiles of its segment (under a mask only
// those inside its rows' bands) in increasing order and accumulates
//     S   = Q K_j^T             (K = D)
//     dP  = dO V_j^T            (K = D)
//     P   = exp2(S * scale*log2e - lse2),  dS = P (dP - delta)
//     dQ += dS K_j              (K = 128 kv rows, in TMEM)
// then writes bf16(scale * dQ) once.  Every dQ element is a sum in a fixed
// order: repeated runs give the same bits.  lse2 and delta come from the
// backward preprocess, in its segment-padded layout.
//
// Per CTA (384 threads, one CTA per SM):
//   warp 0       TMA producer: Q, dO and the tile's lse2 / delta rows, then
//                K_j and V_j into two rings of shared-memory slots (K is
//                read until dQ_j, V only by dP_j, so the K ring is deeper).
//   warp 1       MMA issuer (one lane); owns the TMEM allocation:
//                S_j (two 128-column buffers; dS_j is written over S_j as
//                bf16 and read by the dQ product from TMEM), dP_j, dQ.
//   warps 4..11  compute: warpgroup 1 takes kv columns [0, 64) of every step,
//                warpgroup 2 columns [64, 128); thread = one q row (its
//                TMEM lane).  P of a thread's 64 columns stays in registers;
//                its dS goes back into TMEM over the S columns it read.  At
//                the end of a tile each warpgroup writes half of dQ's
//                columns.
//   warps 2, 3   idle (they complete warpgroup 0 for the register split).
#include "sm103_ptx.cuh"
#include "varlen_internal.h"
#include "varlen_sched.cuh"

namespace varlen {

template <int D>
struct DqCfg {
  static constexpr int NC = (D + 63) / 64;        // 64-column chunks of Q, dO, K, V
  static constexpr int CHUNK = 128 * 128;         // 128 rows x 128 bytes
  static constexpr int TILE = NC * CHUNK;         // one 128-row Q / dO / K / V tile
  static constexpr int NK = NC == 1 ? 4 : 3;      // K ring slots
  static constexpr int NV = NC == 1 ? 4 : 2;      // V ring slots
  static constexpr int ROWV = 128 * 4;            // a tile's lse2 or delta (128 floats)
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = TILE;
  static constexpr int K_OFF = 2 * TILE;
  static constexpr int V_OFF = K_OFF + NK * TILE;
  static constexpr int BAR_OFF = V_OFF + NV * TILE;
  static constexpr int LSE_OFF = BAR_OFF + 256;
  static constexpr int DELTA_OFF = LSE_OFF + ROWV;
  static constexpr int ORDER_OFF = DELTA_OFF + ROWV;  // LPT order table
  static constexpr int SMEM_BYTES = ORDER_OFF + 2 * kLptCapNarrow;
  static_assert(SMEM_BYTES <= 227 * 1024, "dQ tiles do not fit one CTA's shared memory");
  // TMEM columns: S_0 / S_1 (double buffer, dS over S), dP, dQ (D columns)
  static constexpr int S_COL = 0, DP_COL = 256, DQ_COL = 384;
  static constexpr int TMEM_COLS = 512;
};

struct DqBarriers {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2];
  uint64_t dp_full, dp_free;
  uint64_t ds_ready;
  uint64_t dq_full, dq_free;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DqBarriers) <= 256, "barrier block overflows its slot");

// kv tiles [j_lo, j_lo + n) a q tile (128 rows of one segment and head)
// works through, n returned: all of the segment's, or under a mask those
// holding keys some row of the tile sees; 0 means no row sees a key
// (dQ = 0).  The cursor's scheduled side is q.
template <bool MASKED>
__device__ __forceinline__ int32_t dq_kv_tiles(const SegCursor& c, int32_t m, const BwdParams& p, int32_t& j_lo) {
  j_lo = 0;
  int32_t n = (c.olen + kTileN - 1) / kTileN;
  if (MASKED) {
    const int64_t q0 = (int64_t)m * kTileM;
    const int64_t q1 = min((int64_t)c.len, q0 + kTileM) - 1;
    int32_t lo, hi;
    band_keys(q0, q1, c.len, c.olen, p.win_left, p.win_right, &lo, &hi);
    if (hi <= lo) return 0;
    j_lo = lo / kTileN;
    n = (hi + kTileN - 1) / kTileN - j_lo;
  }
  return n;
}

// Registers: 384 threads launched at 168 (64,512); the control warpgroup
// drops to 112 and the two compute warpgroups rise to 192.
constexpr uint32_t kDqRegsLaunch = 168, kDqRegsCtl = 112, kDqRegsCompute = 192;
static_assert(kDqRegsCtl + 2 * kDqRegsCompute <= 3 * kDqRegsLaunch,
              "warpgroup register split exceeds the launch allocation");
static_assert(kDqRegsLaunch * 384 <= 65536, "launch register count too large for 384 threads");

template <int D, bool MASKED>
__global__ void __launch_bounds__(384, 1)
    varlen_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const BwdParams p) {
  using C = DqCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_addr(smem_raw) & 1023u) != 0) {  // the 128-byte swizzle needs 1024-byte aligned tiles
    if (threadIdx.x == 0) record_error(p.err, kErrBounds);
    return;
  }
  uint8_t* smem = smem_raw;
  DqBarriers& bar = *reinterpret_cast<DqBarriers*>(smem + C::BAR_OFF);
  uint8_t* q_smem = smem + C::Q_OFF;
  uint8_t* do_smem = smem + C::DO_OFF;
  uint8_t* k_ring = smem + C::K_OFF;
  uint8_t* v_ring = smem + C::V_OFF;
  float* lse_rows = reinterpret_cast<float*>(smem + C::LSE_OFF);
  float* delta_rows = reinterpret_cast<float*>(smem + C::DELTA_OFF);
  volatile int* abort = &bar.abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_empty, 1 + 8);  // the MMA commit after the tile's last S / dP, and the compute warps
    for (int i = 0; i < C::NK; ++i) {
      mbar_init(&bar.k_full[i], 1);
      mbar_init(&bar.k_empty[i], 1);
    }
    for (int i = 0; i < C::NV; ++i) {
      mbar_init(&bar.v_full[i], 1);
      mbar_init(&bar.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&bar.s_full[i], 1);
    mbar_init(&bar.dp_full, 1);
    mbar_init(&bar.dp_free, 8);
    mbar_init(&bar.ds_ready, 8);
    mbar_init(&bar.dq_full, 1);
    mbar_init(&bar.dq_free, 8);
    mbar_init(&bar.mma_done, 1);
    bar.abort = 0;
    fence_barrier_init();
  }
  const WalkOrder order{reinterpret_cast<const uint16_t*>(smem_raw + C::ORDER_OFF), kLptCapNarrow};
  build_lpt_order(order, p.cu_k, p.batch, p.total_k);
  if (warp == 1) tmem_alloc(&bar.tmem_base, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  const int64_t G = gridDim.x;

  if (warp < 4) {
    warpgroup_set_regs<kDqRegsCtl, kDqRegsLaunch>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      SegCursor c;
      cursor_init<kTileM>(c, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order);
      uint32_t tiles = 0, kn = 0, vn = 0;  // K and V loads issued (load n goes to slot n % NK / n % NV)
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && cursor_seek<kTileM>(c, t, p.num_heads, p.cu_q, p.cu_k, p.batch,
                                                                p.total_q, p.total_k, order);
           t += G) {
        const Tile tl = cursor_tile(c, t);
        int32_t j_lo;
        const int32_t nkv = dq_kv_tiles<MASKED>(c, tl.m, p, j_lo);
        if (nkv == 0) continue;  // no row sees a key: the compute warps write dQ = 0
        const int32_t qrow = c.r0 + tl.m * kTileM;
        if (tiles > 0 && !mbar_wait(&bar.q_empty, (tiles - 1) & 1, abort)) break;
        mbar_arrive_expect_tx(&bar.q_full, 2 * C::TILE + 2 * C::ROWV);
#pragma unroll
        for (int cc = 0; cc < C::NC; ++cc) {
          tma_load_3d(q_smem + cc * C::CHUNK, &tm_q, &bar.q_full, cc * 64, tl.h, qrow);
          tma_load_3d(do_smem + cc * C::CHUNK, &tm_do, &bar.q_full, cc * 64, tl.h, qrow);
        }
        const int64_t rows_at = (int64_t)tl.h * p.pad_rows + pad_base(c.r0, c.b) + (int64_t)tl.m * kTileM;
        bulk_load_1d(lse_rows, p.lse2 + rows_at, C::ROWV, &bar.q_full);
        bulk_load_1d(delta_rows, p.delta + rows_at, C::ROWV, &bar.q_full);
        ++tiles;
        for (int32_t j = 0; j < nkv; ++j) {
          const int32_t krow = c.o0 + (j_lo + j) * kTileN;
          const uint32_t ks = kn % C::NK, vs = vn % C::NV;
          if (!mbar_wait(&bar.k_empty[ks], ((kn / C::NK) & 1) ^ 1, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar.k_full[ks], C::TILE);
#pragma unroll
          for (int cc = 0; cc < C::NC; ++cc)
            tma_load_3d(k_ring + ks * C::TILE + cc * C::CHUNK, &tm_k, &bar.k_full[ks], cc * 64, tl.h, krow);
          ++kn;
          if (!mbar_wait(&bar.v_empty[vs], ((vn / C::NV) & 1) ^ 1, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar.v_full[vs], C::TILE);
#pragma unroll
          for (int cc = 0; cc < C::NC; ++cc)
            tma_load_3d(v_ring + vs * C::TILE + cc * C::CHUNK, &tm_v, &bar.v_full[vs], cc * 64, tl.h, krow);
          ++vn;
        }
      }
      if (*abort) {
        // let the loads in flight land before the CTA exits (bounded)
        int dummy = 0;
        for (uint32_t s = 0; s < (uint32_t)C::NK && s < kn; ++s) {
          const uint32_t last = kn - 1 - ((kn - 1 - s) % C::NK);
          mbar_wait(&bar.k_full[s], (last / C::NK) & 1, &dummy, 100000000ull);
        }
        for (uint32_t s = 0; s < (uint32_t)C::NV && s < vn; ++s) {
          const uint32_t last = vn - 1 - ((vn - 1 - s) % C::NV);
          mbar_wait(&bar.v_full[s], (last / C::NV) & 1, &dummy, 100000000ull);
        }
        if (tiles > 0) mbar_wait(&bar.q_full, (tiles - 1) & 1, &dummy, 100000000ull);
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      // One thread issues every MMA straight through.  Per kv step g the pipe
      // runs S_{g+1}, dP_{g+1}, dQ += dS_g K_g: the next step's products are
      // computed while the compute warps build dS_g.  S_{g+2} reuses the TMEM
      // buffer of S_g / dS_g and is issued after dQ_g: tcgen05 MMAs of one
      // thread execute in issue order, so it overwrites dS_g only after the
      // dQ product has read it.
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);  // S, dP
      constexpr uint32_t kIdQ = idesc_bf16_f32(128, D, false, true);     // dQ (dS from TMEM, K as MN-major B)
      const uint32_t qA = sw128_desc_lo(smem_addr(q_smem), 16);
      const uint32_t doA = sw128_desc_lo(smem_addr(do_smem), 16);
      const uint32_t kB = sw128_desc_lo(smem_addr(k_ring), 16);           // K slot 0, K-major
      const uint32_t vB = sw128_desc_lo(smem_addr(v_ring), 16);           // V slot 0, K-major
      const uint32_t kBm = sw128_desc_lo(smem_addr(k_ring), C::CHUNK);    // K slot 0, MN-major
      SegCursor c;
      cursor_init<kTileM>(c, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order);
      uint32_t tiles = 0, g = 0;
      bool ok = true;

      // Waits for kv step gg's K and clears its rows of a partial last 16-row
      // k-step past the segment end (dQ contracts over them; dS is 0 there,
      // and 0 * NaN must not occur).  nk = the k-steps of dQ.
      auto k_ready = [&](uint32_t gg, int32_t jt, int& nk) -> bool {
        const uint32_t slot = gg % C::NK;
        if (!mbar_wait(&bar.k_full[slot], (gg / C::NK) & 1, abort)) return false;
        const int32_t valid = min(kTileN, c.olen - jt * kTileN);
        nk = (valid + 15) >> 4;
        if (valid < kTileN) {
          uint8_t* kt = k_ring + slot * C::TILE;
          const int to = min(kTileN, nk * 16);
          for (int cc = 0; cc < C::NC; ++cc) {
            uint4* base = reinterpret_cast<uint4*>(kt + cc * C::CHUNK + valid * 128);
            for (int u = 0; u < (to - valid) * 8; ++u) base[u] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        return true;
      };
      auto issue_s = [&](uint32_t gg) {
        const uint32_t so = ((gg % C::NK) * C::TILE) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          mma_ss_lo(tmem + C::S_COL + (gg & 1) * 128, qA + o, kB + so + o, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar.s_full[gg & 1]);
      };
      // dP_gg = dO V^T; V's slot is free once this product is done
      auto issue_dp = [&](uint32_t gg) {
        const uint32_t so = ((gg % C::NV) * C::TILE) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          mma_ss_lo(tmem + C::DP_COL, doA + o, vB + so + o, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar.dp_full);
        mma_commit(&bar.v_empty[gg % C::NV]);
      };
      // dQ += dS_gg (bf16 in TMEM: kv columns [0, 64) at the buffer's columns
      // [0, 32), [64, 128) at [64, 96)) K_gg (MN-major B) over nk kv k-steps
      // (a whole tile takes a loop without a branch: a branch per MMA slows
      // the single issuing thread enough to leave the tensor core waiting)
      auto issue_dq = [&](uint32_t gg, int nk, bool acc0) {
        const uint32_t so = ((gg % C::NK) * C::TILE) >> 4;
        const uint32_t sbuf = tmem + C::S_COL + (gg & 1) * 128;
        const uint32_t a0 = acc0 ? 1u : 0u;
        if (nk == kTileN / 16) {
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            mma_ts_lo(tmem + C::DQ_COL, sbuf + (kk >> 2) * 64 + (kk & 3) * 8, kBm + so + ((kk * 2048) >> 4), kIdQ,
                      kk > 0 ? 1u : a0);
        } else {
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            if (kk < nk)
              mma_ts_lo(tmem + C::DQ_COL, sbuf + (kk >> 2) * 64 + (kk & 3) * 8, kBm + so + ((kk * 2048) >> 4),
                        kIdQ, kk > 0 ? 1u : a0);
        }
        mma_commit(&bar.k_empty[gg % C::NK]);
      };
      auto v_ready = [&](uint32_t gg) -> bool {
        return mbar_wait(&bar.v_full[gg % C::NV], (gg / C::NV) & 1, abort);
      };

      for (int64_t t = blockIdx.x; ok && cursor_seek<kTileM>(c, t, p.num_heads, p.cu_q, p.cu_k, p.batch,
                                                                p.total_q, p.total_k, order);
           t += G) {
        const Tile tl = cursor_tile(c, t);
        int32_t j_lo;
        const int32_t nkv = dq_kv_tiles<MASKED>(c, tl.m, p, j_lo);
        if (nkv == 0) continue;
        if (!mbar_wait(&bar.q_full, tiles & 1, abort)) break;
        // prologue: S and dP of the tile's first kv step
        int nk = 0, nk_next = 0;
        if (!k_ready(g, j_lo, nk)) break;
        tc_fence_after();
        issue_s(g);
        if (!v_ready(g)) break;
        if (g >= 1 && !mbar_wait(&bar.dp_free, (g - 1) & 1, abort)) break;
        tc_fence_after();
        issue_dp(g);
        if (nkv == 1) mma_commit(&bar.q_empty);
        for (int32_t i = 0; i < nkv; ++i) {
          const uint32_t gg = g + i;
          if (i + 1 < nkv) {
            const uint32_t g1 = gg + 1;
            if (!k_ready(g1, j_lo + i + 1, nk_next)) { ok = false; break; }
            tc_fence_after();
            issue_s(g1);
            if (!v_ready(g1)) { ok = false; break; }
            if (!mbar_wait(&bar.dp_free, gg & 1, abort)) { ok = false; break; }
            tc_fence_after();
            issue_dp(g1);
            if (i + 2 == nkv) mma_commit(&bar.q_empty);  // the tile's last S and dP are issued
          }
          if (!mbar_wait(&bar.ds_ready, gg & 1, abort)) { ok = false; break; }
          if (i == 0 && tiles > 0 && !mbar_wait(&bar.dq_free, (tiles - 1) & 1, abort)) { ok = false; break; }
          tc_fence_after();
          issue_dq(gg, nk, i > 0);
          nk = nk_next;
        }
        if (!ok) break;
        mma_commit(&bar.dq_full);
        g += nkv;
        ++tiles;
      }
      // every MMA this thread issued completes before TMEM is freed
      mma_commit(&bar.mma_done);
      int dummy = 0;
      mbar_wait(&bar.mma_done, 0, &dummy);
    }
  } else {
    warpgroup_set_regs<kDqRegsCompute, kDqRegsLaunch>();
    // ------------------------------------------------------------ compute
    const int half = (warp >> 2) - 1;            // kv columns [64 half, 64 half + 64)
    const int quad = warp & 3;                   // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;            // q row within the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c2 = p.scale_log2;
    constexpr int DH = D / 2;                    // dQ columns written by each warpgroup
    SegCursor c;
    cursor_init<kTileM>(c, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order);
    uint32_t tiles = 0, g = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; ok && cursor_seek<kTileM>(c, t, p.num_heads, p.cu_q, p.cu_k, p.batch,
                                                              p.total_q, p.total_k, order);
         t += G) {
      const Tile tl = cursor_tile(c, t);
      int32_t j_lo;
      const int32_t nkv = dq_kv_tiles<MASKED>(c, tl.m, p, j_lo);
      const int32_t r_seg = tl.m * kTileM + row;
      const bool row_valid = r_seg < c.len;
      __nv_bfloat16* dqrow = p.dq + ((int64_t)c.r0 + r_seg) * p.dq_rs + (int64_t)tl.h * p.dq_hs;
      if (nkv == 0) {
        if (row_valid)
          for (int d = half * DH; d < (half + 1) * DH; d += 8)
            if (in_span(p.dq_span, dqrow + d, 16, p.err)) *reinterpret_cast<uint4*>(dqrow + d) = make_uint4(0, 0, 0, 0);
        continue;
      }
      if (!mbar_wait(&bar.q_full, tiles & 1, abort)) break;
      const float lse2 = lse_rows[row];
      const float dlt = delta_rows[row];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.q_empty);  // this warp has its rows' lse2 / delta
      // keys [key_lo, key_hi) this row sees: all Sk, or with a mask its band
      int32_t key_lo = 0, key_hi = c.olen;
      if (MASKED) band_keys(r_seg, r_seg, c.len, c.olen, p.win_left, p.win_right, &key_lo, &key_hi);
      for (int32_t i = 0; i < nkv; ++i) {
        const uint32_t gg = g + i;
        const int32_t col0 = (j_lo + i) * kTileN + half * 64;  // key index of this thread's first column
        const int32_t lim_lo = key_lo - col0, lim_hi = key_hi - col0;  // columns [lim_lo, lim_hi) are visible
        const bool all_vis = !__any_sync(0xffffffffu, lim_lo > 0 || lim_hi < 64);  // no select needed
        // ---- P = exp2(S c - lse2) on this thread's 64 columns
        if (!mbar_wait(&bar.s_full[gg & 1], (gg >> 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        float pv[64];
        const uint32_t sa = tmem + lane_off + C::S_COL + (gg & 1) * 128 + half * 64;  // this thread's S columns
        {
          uint32_t sv[64];
          tmem_ld32(sa, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
          tmem_ld32(sa + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
          tmem_wait_ld();
          const float2 cc2 = make_float2(c2, c2), nl = make_float2(-lse2, -lse2);
#pragma unroll
          for (int k = 0; k < 64; k += 2) {
            const float2 x = ffma2(make_float2(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])), cc2, nl);
            pv[k] = ex2(x.x);
            pv[k + 1] = ex2(x.y);
          }
          // columns outside the row's band or past the segment end: P = 0 (by select)
          if (!all_vis) {
#pragma unroll
            for (int k = 0; k < 64; ++k) pv[k] = (k >= lim_lo && k < lim_hi) ? pv[k] : 0.f;
          }
        }
        // ---- dS = P (dP - delta), bf16
        if (!mbar_wait(&bar.dp_full, gg & 1, abort)) { ok = false; break; }
        tc_fence_after();
        uint32_t ds2[32];
        {
          uint32_t dv[64];
          const uint32_t da = tmem + lane_off + C::DP_COL + half * 64;
          tmem_ld32(da, *reinterpret_cast<uint32_t(*)[32]>(&dv[0]));
          tmem_ld32(da + 32, *reinterpret_cast<uint32_t(*)[32]>(&dv[32]));
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar.dp_free);
          const float2 nd = make_float2(-dlt, -dlt);
#pragma unroll
          for (int k = 0; k < 64; k += 2) {
            const float2 a = fmul2(make_float2(pv[k], pv[k + 1]),
                                   fadd2(make_float2(__uint_as_float(dv[k]), __uint_as_float(dv[k + 1])), nd));
            // select, not multiply: dP past the segment end may hold NaN
            if (all_vis)
              ds2[k / 2] = pack_bf16x2(a.x, a.y);
            else
              ds2[k / 2] = pack_bf16x2(k >= lim_lo && k < lim_hi ? a.x : 0.f,
                                       k + 1 >= lim_lo && k + 1 < lim_hi ? a.y : 0.f);
          }
        }
        // ---- dS into TMEM over the first 32 of this thread's S columns (read above)
        tmem_st32(sa, ds2);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.ds_ready);
      }
      if (!ok) break;
      // ---- epilogue: bf16(scale * dQ), this warpgroup's half of the columns
      if (!mbar_wait(&bar.dq_full, tiles & 1, abort)) break;
      tc_fence_after();
#pragma unroll
      for (int d0 = half * DH; d0 < (half + 1) * DH; d0 += 16) {
        uint32_t a[16];
        tmem_ld16(tmem + lane_off + C::DQ_COL + d0, a);
        tmem_wait_ld();
        if (row_valid) {
          uint32_t w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            w[k] = pack_bf16x2(__uint_as_float(a[2 * k]) * p.scale, __uint_as_float(a[2 * k + 1]) * p.scale);
          uint4* dst = reinterpret_cast<uint4*>(dqrow + d0);
          if (in_span(p.dq_span, dst, 16, p.err)) dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          if (in_span(p.dq_span, dst + 1, 16, p.err)) dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.dq_free);
      g += nkv;
      ++tiles;
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

template <int D, bool MASKED>
static cudaError_t launch_dq_d(const BwdLaunch& L, cudaStream_t stream) {
  using C = DqCfg<D>;
  auto kern = varlen_bwd_dq_kernel<D, MASKED>;
  // The warpgroup register split assumes the compiled per-thread count;
  // refuse to launch a build that came out differently.
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != (int)kDqRegsLaunch) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, 384, C::SMEM_BYTES, stream>>>(L.tm_q, L.tm_k, L.tm_v, L.tm_do, L.p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdLaunch& L, cudaStream_t stream) {
  switch (L.head_dim) {
    case 64: return L.p.masked ? launch_dq_d<64, true>(L, stream) : launch_dq_d<64, false>(L, stream);
    case 96: return L.p.masked ? launch_dq_d<96, true>(L, stream) : launch_dq_d<96, false>(L, stream);
    case 128: return L.p.masked ? launch_dq_d<128, true>(L, stream) : launch_dq_d<128, false>(L, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace varlen
