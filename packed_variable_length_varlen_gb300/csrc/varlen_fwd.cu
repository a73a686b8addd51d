// varlen_fwd.cu -- forward kernel of packed variable-length attention on
// sm_103a: persistent exact tile scheduler, TMA-fed Q tiles and K/V ring,
// tcgen05 MMAs with TMEM accumulators, warp-specialised online softmax.
//
// One scheduled unit is 256 q rows of one (segment, head): two 128-row
// halves A and B that share every K/V tile.  Per CTA (384 threads, one CTA
// per SM):
//   warp 0       TMA producer: Q_A, Q_B, then K_j, V_j tiles into a ring of
//                shared-memory slots (mbarrier full/empty per slot).
//   warp 1       MMA issuer (one lane), per kv step j:
//                  O_A += P_A V_j, S_A = Q_A K_{j+1}^T, O_B += P_B V_j,
//                  S_B = Q_B K_{j+1}^T
//                with S and P of each half in one 128-column TMEM region (P
//                is written over S as bf16 and read by the MMA from TMEM).
//                The next S of a half is issued right after that half's P V
//                product: tcgen05 MMAs of one thread execute in issue order,
//                so the new S overwrites P only after the product has read
//                it.  While half A's softmax runs, the tensor core works on
//                half B and the other way round.  Owns the TMEM allocation.
//   warps 4..7   softmax / correction / epilogue of half A; warps 8..11 of
//                half B.  Warp w reads TMEM lanes 32*(w % 4) .. +31, so each
//                warpgroup covers all 128 rows; thread = one q row.
//   warps 2,3    idle (they complete warpgroup 0 for the register split).
//                Masks key columns past the segment end, keeps the running
//                max m and sum l, writes P = exp2(S*c - m) into TMEM as
//                bf16, rescales O in TMEM when m grows by more than 2^8
//                (exact: O and l carry the same factor), and finally writes
//                O / l (bf16) and LSE.
//
// Semantics: O = softmax(scale * Q_b K_b^T) V_b per segment b, with the
// natural-log LSE per row -- the varlen attention called on the
// "[FA4][SM120] flash_attn_varlen_func ... >=4 varlen segments" issue (section
// "Bug 2 details").  Differences from the kernels on the pages: the tile
// count is exact (no tail blocks), no global load is issued before a tile is
// known to exist, and all row offsets are 64-bit.
#include "sm103_ptx.cuh"
#include "varlen_internal.h"
#include "varlen_sched.cuh"

namespace varlen {

constexpr int kFwdUnit = 2 * kTileM;  // q rows per scheduled unit (two halves)

// kv tiles [j_lo, j_lo + n) a unit (256 q rows of one segment and head)
// works through, n returned.  With a mask (the band of FwdParams) only the
// tiles holding keys that some row of the unit sees; 0 means no row of the
// unit sees a key (O = 0, LSE = -inf).  The cursor's scheduled side is q.
template <bool MASKED>
__device__ __forceinline__ int32_t fwd_kv_tiles(const SegCursor& c, int32_t unit, const FwdParams& p,
                                                int32_t& j_lo) {
  j_lo = 0;
  int32_t nkv = (c.olen + kTileN - 1) / kTileN;
  if (MASKED) {
    const int64_t q0 = (int64_t)unit * kFwdUnit;
    const int64_t q1 = min((int64_t)c.len, q0 + kFwdUnit) - 1;
    int32_t lo, hi;
    band_keys(q0, q1, c.len, c.olen, p.win_left, p.win_right, &lo, &hi);
    if (hi <= lo) return 0;
    j_lo = lo / kTileN;
    nkv = (hi + kTileN - 1) / kTileN - j_lo;
  }
  return nkv;
}

template <int D>
struct FwdCfg {
  static constexpr int NC = (D + 63) / 64;              // 64-column chunks of a tile
  static constexpr int CHUNK = 128 * 128;               // 128 rows x 128 bytes
  static constexpr int TILE = NC * CHUNK;               // one Q / K / V tile
  static constexpr int NSLOT = (NC == 1) ? 8 : 4;       // K/V ring slots
  static constexpr int O_COL = 256;                     // TMEM column of O_A (O_B at +128)
  static constexpr int TMEM_COLS = 512;
  static constexpr int ORDER_OFF = 1024 + TILE * (2 + NSLOT);         // LPT order table
  static constexpr int SMEM_BYTES = ORDER_OFF + 2 * kLptCapWide;
  static constexpr int KSTEPS = D / 16;                 // K-steps of S = Q K^T
};

struct FwdBarriers {
  uint64_t q_full, q_empty;
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t mma_done;
  uint64_t kv_full[10], kv_empty[10];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(FwdBarriers) <= 1024, "barrier block too large");

// Registers: the block launches 384 threads at 168 registers (64,512).
// Warpgroup 0 (producer, MMA, two idle warps) drops to 120 and the two
// softmax warpgroups rise to 192: 120*128 + 2*192*128 = 64,512, the launch
// allocation, and each SM sub-partition holds one warp of each group:
// (120+192+192)*32 <= 16K.
constexpr uint32_t kFwdRegsLaunch = 168, kFwdRegsCtl = 120, kFwdRegsSoftmax = 192;
static_assert(kFwdRegsCtl + 2 * kFwdRegsSoftmax <= 3 * kFwdRegsLaunch,
              "warpgroup register split exceeds the launch allocation");
static_assert(kFwdRegsLaunch * 384 <= 65536, "launch register count too large for 384 threads");

template <int D, bool MASKED>
__global__ void __launch_bounds__(384, 1)
    varlen_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D>;
  // The 128-byte swizzled tiles need 1024-byte alignment; the declaration
  // asks for it and the kernel refuses to run without it.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_addr(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(p.err, kErrBounds);
    return;
  }
  uint8_t* smem = smem_raw;
  FwdBarriers& bar = *reinterpret_cast<FwdBarriers*>(smem);
  uint8_t* q_smem = smem + 1024;           // Q_A then Q_B
  uint8_t* ring = q_smem + 2 * C::TILE;
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
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(&bar.kv_full[i], 1);
      mbar_init(&bar.kv_empty[i], 1);
    }
    bar.abort = 0;
    fence_barrier_init();
  }
  const WalkOrder order{reinterpret_cast<const uint16_t*>(smem_raw + C::ORDER_OFF), kLptCapWide};
  build_lpt_order(order, p.cu_k, p.batch, p.total_k);
  if (warp == 1) tmem_alloc(&bar.tmem_base, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;

  const int64_t G = gridDim.x;

  if (warp < 4) {
    warpgroup_set_regs<kFwdRegsCtl, kFwdRegsLaunch>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      SegCursor c;
      cursor_init<kFwdUnit>(c, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order);
      uint32_t q_loads = 0;
      uint32_t ring_pos = 0;  // loads issued into the ring so far
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && cursor_seek<kFwdUnit>(c, t, p.num_heads, p.cu_q, p.cu_k, p.batch,
                                                                 p.total_q, p.total_k, order);
           t += G) {
        const Tile tl = cursor_tile(c, t);
        int32_t j_lo;
        const int32_t nkv = fwd_kv_tiles<MASKED>(c, tl.m, p, j_lo);
        if (nkv == 0) continue;  // no visible keys: the softmax role writes O = 0, LSE = -inf
        const int32_t qrow = c.r0 + tl.m * kFwdUnit;
        if (q_loads > 0 && !mbar_wait(&bar.q_empty, (q_loads - 1) & 1, abort)) break;
        mbar_arrive_expect_tx(&bar.q_full, 2 * C::TILE);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int cc = 0; cc < C::NC; ++cc)
            tma_load_3d(q_smem + hf * C::TILE + cc * C::CHUNK, &tm_q, &bar.q_full, cc * 64, tl.h,
                        qrow + hf * kTileM);
        ++q_loads;
        for (int32_t j = 0; ok && j < nkv; ++j) {
          const int32_t krow = c.o0 + (j_lo + j) * kTileN;
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            const uint32_t slot = ring_pos % C::NSLOT;
            const uint32_t phase = (ring_pos / C::NSLOT) & 1;
            if (!mbar_wait(&bar.kv_empty[slot], phase ^ 1, abort)) {
              ok = false;
              break;
            }
            // (failure test: CTA 0 leaves one load out; its consumer's bounded
            // wait then gives up and the kernel unwinds, reporting a timeout)
            if (!(blockIdx.x == 0 && (int64_t)ring_pos == (int64_t)p.debug_skip_load)) {
              mbar_arrive_expect_tx(&bar.kv_full[slot], C::TILE);
              uint8_t* dst = ring + slot * C::TILE;
              const CUtensorMap* m = which ? &tm_v : &tm_k;
#pragma unroll
              for (int cc = 0; cc < C::NC; ++cc)
                tma_load_3d(dst + cc * C::CHUNK, m, &bar.kv_full[slot], cc * 64, tl.h, krow);
            }
            ++ring_pos;
          }
        }
      }
      if (*abort) {
        // Let every copy already issued land before the CTA's shared memory
        // can be released (bounded).
        for (uint32_t s = 0; s < C::NSLOT && s < ring_pos; ++s) {
          const uint32_t last = ring_pos - 1 - ((ring_pos - 1 - s) % C::NSLOT);
          int dummy = 0;
          mbar_wait(&bar.kv_full[s], (last / C::NSLOT) & 1, &dummy, 100000000ull);
        }
        if (q_loads > 0) {
          int dummy = 0;
          mbar_wait(&bar.q_full, (q_loads - 1) & 1, &dummy, 100000000ull);
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues every MMA straight through (the warp's other lanes
    // wait at the end), with descriptors kept as 32-bit low words: a warp
    // that rejoins between MMA groups, or spends many integer instructions
    // per MMA, leaves the tensor pipe idle.
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);
    SegCursor c;
    cursor_init<kFwdUnit>(c, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order);
    uint32_t tiles = 0, g = 0, ring0 = 0;
    bool ok = true;
    const uint32_t qlo = sw128_desc_lo(smem_addr(q_smem), 16);        // Q_A (Q_B at +TILE), K-major A
    const uint32_t rK = sw128_desc_lo(smem_addr(ring), 16);           // ring slot 0 as K-major B
    const uint32_t rV = sw128_desc_lo(smem_addr(ring), C::CHUNK);     // ring slot 0 as MN-major B
    auto issue_s = [&](int hf, uint32_t kslot) {
#pragma unroll
      for (int kk = 0; kk < C::KSTEPS; ++kk) {
        const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
        mma_ss_lo(tmem + hf * 128, qlo + ((hf * C::TILE) >> 4) + off, rK + ((kslot * C::TILE) >> 4) + off, kIdescS,
                  kk > 0 ? 1u : 0u);
      }
      mma_commit(&bar.s_full[hf]);
    };
    // O += P V over nk 16-row k-steps of kv (k-steps past the segment end are skipped)
    auto issue_pv = [&](int hf, uint32_t vslot, bool first, int nk) {
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        if (kk < nk)
          mma_ts_lo(tmem + C::O_COL + hf * 128, tmem + hf * 128 + kk * 8, rV + ((vslot * C::TILE + kk * 2048) >> 4),
                    kIdescO, (!first || kk > 0) ? 1u : 0u);
      mma_commit(&bar.pv_done[hf]);
    };
    for (int64_t t = blockIdx.x;
         ok && cursor_seek<kFwdUnit>(c, t, p.num_heads, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order); t += G) {
      int32_t j_lo;
      const int32_t nkv = fwd_kv_tiles<MASKED>(c, cursor_tile(c, t).m, p, j_lo);
      if (nkv == 0) continue;
      if (!mbar_wait(&bar.q_full, tiles & 1, abort)) break;
      ++tiles;
      // prologue: S_A and S_B of kv step 0
      {
        const uint32_t kslot = ring0 % C::NSLOT;
        if (!mbar_wait(&bar.kv_full[kslot], (ring0 / C::NSLOT) & 1, abort)) break;
        tc_fence_after();
        issue_s(0, kslot);
        issue_s(1, kslot);
        mma_commit(&bar.kv_empty[kslot]);
        if (nkv == 1) mma_commit(&bar.q_empty);
      }
      for (int32_t j = 0; j < nkv; ++j) {
        const uint32_t gj = g + j;
        const uint32_t vpos = ring0 + 2 * j + 1;
        const uint32_t vslot = vpos % C::NSLOT;
        const bool more = j + 1 < nkv;
        const uint32_t kpos = vpos + 1;
        const uint32_t kslot = kpos % C::NSLOT;
        if (!mbar_wait(&bar.kv_full[vslot], (vpos / C::NSLOT) & 1, abort)) { ok = false; break; }
        const int32_t kv_valid = min(kTileN, c.olen - (j_lo + j) * kTileN);
        const int nk = (kv_valid + 15) >> 4;
        if (kv_valid < kTileN) {
          // Rows past the segment end hold the next segment's values (or
          // TMA zero fill).  P is 0 there, but 0 * NaN would still poison
          // O: k-steps wholly past the end are skipped, and the rows of the
          // last partial one are cleared before the MMA reads them.
          uint8_t* vtile = ring + vslot * C::TILE;
#pragma unroll
          for (int cc = 0; cc < C::NC; ++cc) {
            uint4* base = reinterpret_cast<uint4*>(vtile + cc * C::CHUNK + kv_valid * 128);
            for (int u = 0; u < (min(kTileN, nk * 16) - kv_valid) * 8; ++u) base[u] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        if (more && !mbar_wait(&bar.kv_full[kslot], (kpos / C::NSLOT) & 1, abort)) { ok = false; break; }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (!mbar_wait(&bar.p_full[hf], gj & 1, abort)) { ok = false; break; }
          tc_fence_after();
          issue_pv(hf, vslot, j == 0, nk);
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
    // Drain: every MMA this thread issued completes before TMEM is freed.
    mma_commit(&bar.mma_done);
    int dummy = 0;
    mbar_wait(&bar.mma_done, 0, &dummy);
  }
  } else {
    warpgroup_set_regs<kFwdRegsSoftmax, kFwdRegsLaunch>();
    // ------------------------------------------------------------ softmax
    const int hf = (warp - 4) >> 2;                    // 0: half A (warps 4..7), 1: half B (warps 8..11)
    const int quad = warp & 3;                         // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;                  // TMEM lane = row within the half
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_col = hf * 128, o_col = C::O_COL + hf * 128;
    const float c2 = p.scale_log2;
    SegCursor c;
    cursor_init<kFwdUnit>(c, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order);
    uint32_t g = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x;
         ok && cursor_seek<kFwdUnit>(c, t, p.num_heads, p.cu_q, p.cu_k, p.batch, p.total_q, p.total_k, order); t += G) {
      const Tile tl = cursor_tile(c, t);
      int32_t j_lo;
      const int32_t nkv = fwd_kv_tiles<MASKED>(c, tl.m, p, j_lo);
      if (nkv == 0) {
        const int32_t r_in_seg = tl.m * kFwdUnit + hf * kTileM + row;
        const int64_t grow = (int64_t)c.r0 + r_in_seg;
        __nv_bfloat16* orow = p.out + grow * p.o_rs + (int64_t)tl.h * p.o_hs;
        float* lse_out = p.lse + (int64_t)tl.h * p.total_q + grow;
        if (r_in_seg < c.len) {
#pragma unroll
          for (int d = 0; d < D; d += 8)
            if (in_span(p.out_span, orow + d, 16, p.err)) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0, 0, 0, 0);
          if (in_span(p.lse_span, lse_out, 4, p.err)) *lse_out = -INFINITY;
        }
        continue;
      }
      // keys [key_lo, key_hi) this row sees: all Sk, or with a mask its band
      const int32_t r_seg = tl.m * kFwdUnit + hf * kTileM + row;
      int32_t key_lo = 0, key_hi = c.olen;
      if (MASKED) band_keys(r_seg, r_seg, c.len, c.olen, p.win_left, p.win_right, &key_lo, &key_hi);
      float m_use = -INFINITY, l = 0.f;
      for (int32_t j = 0; j < nkv; ++j) {
        const uint32_t gj = g + j;
        if (!mbar_wait(&bar.s_full[hf], gj & 1, abort)) { ok = false; break; }
        tc_fence_after();
        uint32_t s[128];
        {
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
        }
        float x[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) x[i] = __uint_as_float(s[i]);
        // columns outside the row's visible keys (past the segment end, or
        // outside the mask's band) are set to -inf by select
        const int32_t lim = key_hi - (j_lo + j) * kTileN;  // per thread
        const int32_t lim_lo = key_lo - (j_lo + j) * kTileN;
        if (MASKED && __any_sync(0xffffffffu, lim_lo > 0)) {  // the band's left edge crosses this tile
#pragma unroll
          for (int i = 0; i < 128; ++i) x[i] = (i < lim && i >= lim_lo) ? x[i] : -INFINITY;
        } else if (__any_sync(0xffffffffu, lim < kTileN)) {
#pragma unroll
          for (int i = 0; i < 128; ++i) x[i] = (i < lim) ? x[i] : -INFINITY;
        }
        // row max: four independent chains of 3-input max
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int i = 0; i < 128; i += 8) {
          m0 = fmax3(m0, x[i], x[i + 1]);
          m1 = fmax3(m1, x[i + 2], x[i + 3]);
          m2 = fmax3(m2, x[i + 4], x[i + 5]);
          m3 = fmax3(m3, x[i + 6], x[i + 7]);
        }
        const float mx = fmaxf(fmax3(m0, m1, m2), m3);
        const float m_new = fmaxf(m_use, mx * c2);
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_use = m_new;
        } else if (m_new > m_use + 8.0f) {
          alpha = ex2(m_use - m_new);
          m_use = m_new;
          rescale = true;
        }
        // P = exp2(S*c - m) two lanes at a time; row sum of the fp32 P.
        // P goes to TMEM in two 32-column halves as it is produced, which
        // keeps the live register set small.  Half h writes P columns
        // [32h, 32h+32), whose S values were consumed already.
        // a row that has seen no key yet keeps m = -inf; subtracting 0 then
        // gives P = exp2(-inf) = 0 instead of NaN
        const float m_sub = (MASKED && m_use == -INFINITY) ? 0.f : m_use;
        const float2 cc2 = make_float2(c2, c2), negm = make_float2(-m_sub, -m_sub);
        float2 rs2a = make_float2(0.f, 0.f), rs2b = make_float2(0.f, 0.f);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int e = hh * 64 + 2 * i;
            float2 t2 = ffma2(make_float2(x[e], x[e + 1]), cc2, negm);
            t2.x = ex2(t2.x);
            t2.y = ex2(t2.y);
            pk[i] = pack_bf16x2(t2.x, t2.y);
            if (i & 1) rs2b = fadd2(rs2b, t2); else rs2a = fadd2(rs2a, t2);
          }
          tmem_st32(tmem + lane_off + s_col + hh * 32, pk);
        }
        const float rs = (rs2a.x + rs2a.y) + (rs2b.x + rs2b.y);
        l = fmaf(l, alpha, rs);
        if (__any_sync(0xffffffffu, rescale)) {
          // S_j was issued after O += P_{j-1} V_{j-1} of this half, in MMA
          // issue order, so O is complete here.
#pragma unroll
          for (int d0 = 0; d0 < D; d0 += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + o_col + d0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tmem + lane_off + o_col + d0, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar.p_full[hf]);
      }
      if (!ok) break;
      // epilogue: wait for the last O += P V of this half, then O / l and LSE
      const int32_t r_in_seg = r_seg;
      const bool row_valid = r_in_seg < c.len;
      const int64_t grow = (int64_t)c.r0 + r_in_seg;
      __nv_bfloat16* orow = p.out + grow * p.o_rs + (int64_t)tl.h * p.o_hs;
      float* lse_out = p.lse + (int64_t)tl.h * p.total_q + grow;
      const uint32_t gl = g + nkv - 1;
      if (!mbar_wait(&bar.pv_done[hf], gl & 1, abort)) break;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;  // l = 0: the row saw no key (masked): O = 0
#pragma unroll
      for (int d0 = 0; d0 < D; d0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + o_col + d0, o);
        tmem_wait_ld();
        if (row_valid) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
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
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && bar.abort) record_error(p.err, kErrTimeout);
}

template <int D, bool MASKED>
static cudaError_t launch_fwd_d(const FwdLaunch& L, cudaStream_t stream) {
  using C = FwdCfg<D>;
  auto kern = varlen_fwd_kernel<D, MASKED>;
  // The warpgroup register split assumes the compiled per-thread count;
  // refuse to launch a build that came out differently.
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != (int)kFwdRegsLaunch) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, 384, C::SMEM_BYTES, stream>>>(L.tm_q, L.tm_k, L.tm_v, L.p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdLaunch& L, cudaStream_t stream) {
  switch (L.head_dim) {
    case 64: return L.p.masked ? launch_fwd_d<64, true>(L, stream) : launch_fwd_d<64, false>(L, stream);
    case 96: return L.p.masked ? launch_fwd_d<96, true>(L, stream) : launch_fwd_d<96, false>(L, stream);
    case 128: return L.p.masked ? launch_fwd_d<128, true>(L, stream) : launch_fwd_d<128, false>(L, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace varlen
