// varlen_bwd.cu -- backward of packed variable-length attention on sm_103a.
//
// Three kernels on the caller's stream:
//
//  1. varlen_bwd_prep_kernel (HBM-bound): for every q row i and head h,
//       delta[h,i] = sum_d dO[i,h,d] * O[i,h,d]      (fp32, from bf16)
//       lse2[h,i]  = LSE[h,i] * log2(e)
//     and zero the fp32 dQ accumulator.  dO and O are read through their own
//     row / head strides with 64-bit offsets: the preprocess is where the
//     "[FA4] cute varlen backward: int32 overflow in _bwd_preprocess" issue
//     (sections "Summary", "Root cause") wrapped cu_seqlens[b]*stride past
//     2^31.
//
//  2. varlen_bwd_main_kernel (tensor-bound), persistent over kv tiles
//     (segment b, 128 kv rows, head h) of an exact varlen schedule.  K and V
//     stay in shared memory; for each 64-row q step of the segment it issues
//     five tcgen05 MMAs (TMEM accumulators):
//         S^T  = K Q^T          (128 x 64, K = D)
//         dP^T = V dO^T         (128 x 64, K = D)
//         dV  += P^T dO         (128 x D,  K = 64)
//         dK  += dS^T Q         (128 x D,  K = 64)
//         dQ^T = K^T dS^T       (128(d) x 64, K = 128)
//     where P^T = exp2(S^T * scale*log2e - lse2) and dS^T = P^T (dP^T - delta)
//     are computed by eight compute warps (thread = kv row, half of the q
//     columns) and written to shared memory as bf16.  dQ^T is added into the
//     fp32 accumulator by TMA bulk reduce-add: each compute warp stages its
//     32 x 32 block and issues one reduction, which the L2 performs while
//     the warp moves on.  At the end of a kv tile, dK * scale and dV go to
//     their strided outputs; a segment without queries writes zeros.
//
//  3. varlen_bwd_post_kernel (HBM-bound): dq = bf16(scale * dq_acc), strided.
//
// The gradient formulas are the standard ones for O = softmax(scale QK^T) V:
// dP = dO V^T, dS = P (dP - rowsum(dO o O)), dQ = scale dS K,
// dK = scale dS^T Q, dV = P^T dO.
#include "sm103_ptx.cuh"
#include "varlen_internal.h"
#include "varlen_sched.cuh"

namespace varlen {

// ------------------------------------------------------------------ prep

__global__ void __launch_bounds__(256) varlen_bwd_prep_kernel(const PrepParams p) {
  const int32_t B = p.batch;
  const int32_t lo = clamp_row(__ldg(p.cu_q), p.total_q);
  const int32_t hi = clamp_row(__ldg(p.cu_q + B), p.total_q);
  if (hi <= lo) return;
  const int H = p.num_heads, D = p.head_dim;
  const int64_t n = (int64_t)(hi - lo) * H;
  const float kLog2e = 1.4426950408889634f;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = lo + t / H;
    const int h = (int)(t % H);
    const __nv_bfloat16* o = p.out + row * p.o_rs + (int64_t)h * p.o_hs;
    const __nv_bfloat16* g = p.dout + row * p.do_rs + (int64_t)h * p.do_hs;
    float acc = 0.f;
    for (int d = 0; d < D; d += 8) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + d));
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(g + d));
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(a2[i]);
        const float2 y = __bfloat1622float2(b2[i]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
    const int64_t hi_idx = (int64_t)h * p.total_q + row;
    p.delta[hi_idx] = acc;
    p.lse2[hi_idx] = p.lse[hi_idx] * kLog2e;
    float4* z = reinterpret_cast<float4*>(p.dq_acc + (row * H + h) * D);
    for (int d = 0; d < D; d += 4) *z++ = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ------------------------------------------------------------------ post

__global__ void __launch_bounds__(256) varlen_bwd_post_kernel(const PostParams p) {
  const int32_t B = p.batch;
  const int32_t lo = clamp_row(__ldg(p.cu_q), p.total_q);
  const int32_t hi = clamp_row(__ldg(p.cu_q + B), p.total_q);
  if (hi <= lo) return;
  const int H = p.num_heads, D = p.head_dim, V = D / 8;
  const int64_t n = (int64_t)(hi - lo) * H * V;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t rh = t / V;
    const int v = (int)(t - rh * V);
    const int64_t row = lo + rh / H;
    const int h = (int)(rh % H);
    const float4* s = reinterpret_cast<const float4*>(p.dq_acc + (row * H + h) * D + v * 8);
    const float4 a = s[0], b = s[1];
    uint4 w;
    w.x = pack_bf16x2(a.x * p.scale, a.y * p.scale);
    w.y = pack_bf16x2(a.z * p.scale, a.w * p.scale);
    w.z = pack_bf16x2(b.x * p.scale, b.y * p.scale);
    w.w = pack_bf16x2(b.z * p.scale, b.w * p.scale);
    *reinterpret_cast<uint4*>(p.dq + row * p.dq_rs + (int64_t)h * p.dq_hs + v * 8) = w;
  }
}

// ------------------------------------------------------------------ main

template <int D>
struct BwdCfg {
  static constexpr int NC = (D + 63) / 64;       // 64-column chunks of Q / dO / V
  static constexpr int KCH = 2;                  // K tile always holds 128 columns (dQ^T uses M = 128)
  static constexpr int KV_CHUNK = 128 * 128;     // 128 kv rows x 128 B
  static constexpr int Q_CHUNK = 64 * 128;       // 64 q rows x 128 B
  static constexpr int K_BYTES = KCH * KV_CHUNK;
  static constexpr int V_BYTES = NC * KV_CHUNK;
  static constexpr int Q_BYTES = NC * Q_CHUNK;   // one Q or dO tile
  static constexpr int NSTAGE = 3;               // Q / dO ring depth
  static constexpr int PS_BYTES = 128 * 128;     // P^T or dS^T: 128 kv rows x 64 q (bf16)
  static constexpr int STG_BYTES = 8 * 32 * 32 * 4;  // dQ staging: one 32 x 32 fp32 block per compute warp
  static constexpr int SMEM_BYTES = 1024 + 1024 + K_BYTES + V_BYTES + NSTAGE * 2 * Q_BYTES + 2 * PS_BYTES + STG_BYTES;
  static_assert(SMEM_BYTES <= 227 * 1024, "backward tile does not fit one CTA's shared memory");
  // TMEM columns: two S^T buffers, dP^T, dQ^T, dV, dK
  static constexpr int S_COL = 0, DP_COL = 128, DQ_COL = 192, DV_COL = 256, DK_COL = 384;
  static constexpr int TMEM_COLS = 512;
};

struct BwdBarriers {
  uint64_t kv_full, kv_empty;
  uint64_t qd_full[4], qd_empty[4];
  uint64_t s_full[2], dp_full, dp_free, ds_ready, step_done, mma_done;
  uint32_t tmem_base;
  int abort;
};

// Clears rows [row_from, row_to) of a tile made of `chunks` chunks of
// 128-byte rows; the warp's lanes store consecutive 16-byte units.
__device__ __forceinline__ void zero_rows(uint8_t* tile, int chunks, int chunk_bytes, int row_from, int row_to,
                                          int lane) {
  const int units = (row_to - row_from) * 8;
  for (int cc = 0; cc < chunks; ++cc) {
    uint4* base = reinterpret_cast<uint4*>(tile + cc * chunk_bytes + row_from * 128);
    for (int u = lane; u < units; u += 32) base[u] = make_uint4(0, 0, 0, 0);
  }
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    varlen_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                           const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBarriers& bar = *reinterpret_cast<BwdBarriers*>(smem);
  uint8_t* k_smem = smem + 1024;
  uint8_t* v_smem = k_smem + C::K_BYTES;
  uint8_t* qd_smem = v_smem + C::V_BYTES;                 // [stage][Q, dO]
  uint8_t* pt_smem = qd_smem + C::NSTAGE * 2 * C::Q_BYTES;
  uint8_t* dst_smem = pt_smem + C::PS_BYTES;
  uint8_t* stg_smem = dst_smem + C::PS_BYTES;
  volatile int* abort = &bar.abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bar.kv_full, 1);
    mbar_init(&bar.kv_empty, 1);
    for (int i = 0; i < C::NSTAGE; ++i) {
      mbar_init(&bar.qd_full[i], 1);
      mbar_init(&bar.qd_empty[i], 1);
    }
    mbar_init(&bar.s_full[0], 1);
    mbar_init(&bar.s_full[1], 1);
    mbar_init(&bar.dp_full, 1);
    mbar_init(&bar.dp_free, 256);
    mbar_init(&bar.ds_ready, 256);
    mbar_init(&bar.step_done, 1);
    mbar_init(&bar.mma_done, 1);
    bar.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&bar.tmem_base, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  const int64_t G = gridDim.x;
  constexpr int QT = kBwdTileQ;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      SegCursor c;
      cursor_init<kTileM>(c, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q);
      uint32_t tiles = 0, gs = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x;
           ok && cursor_seek<kTileM>(c, t, p.num_heads, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q); t += G) {
        if (c.olen == 0) continue;  // no queries: dK = dV = 0, written by the compute warps
        const Tile tl = cursor_tile(c, t);
        const int32_t krow = c.r0 + tl.m * kTileM;
        if (tiles > 0 && !mbar_wait(&bar.kv_empty, (tiles - 1) & 1, abort)) break;
        mbar_arrive_expect_tx(&bar.kv_full, C::K_BYTES + C::V_BYTES);
#pragma unroll
        for (int cc = 0; cc < C::KCH; ++cc)
          tma_load_3d(k_smem + cc * C::KV_CHUNK, &tm_k, &bar.kv_full, cc * 64, tl.h, krow);
#pragma unroll
        for (int cc = 0; cc < C::NC; ++cc)
          tma_load_3d(v_smem + cc * C::KV_CHUNK, &tm_v, &bar.kv_full, cc * 64, tl.h, krow);
        ++tiles;
        const int32_t nq = (c.olen + QT - 1) / QT;
        for (int32_t j = 0; j < nq; ++j, ++gs) {
          const uint32_t st = gs % C::NSTAGE;
          if (!mbar_wait(&bar.qd_empty[st], ((gs / C::NSTAGE) & 1) ^ 1, abort)) { ok = false; break; }
          mbar_arrive_expect_tx(&bar.qd_full[st], 2 * C::Q_BYTES);
          uint8_t* qs = qd_smem + st * 2 * C::Q_BYTES;
          const int32_t qrow = c.o0 + j * QT;
#pragma unroll
          for (int cc = 0; cc < C::NC; ++cc) {
            tma_load_3d(qs + cc * C::Q_CHUNK, &tm_q, &bar.qd_full[st], cc * 64, tl.h, qrow);
            tma_load_3d(qs + C::Q_BYTES + cc * C::Q_CHUNK, &tm_do, &bar.qd_full[st], cc * 64, tl.h, qrow);
          }
        }
      }
      if (*abort) {
        int dummy = 0;
        if (tiles > 0) mbar_wait(&bar.kv_full, (tiles - 1) & 1, &dummy, 100000000ull);
        for (uint32_t s = 0; s < C::NSTAGE && s < gs; ++s) {
          const uint32_t last = gs - 1 - ((gs - 1 - s) % C::NSTAGE);
          mbar_wait(&bar.qd_full[s], (last / C::NSTAGE) & 1, &dummy, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per q step j the tensor pipe runs  S^T_{j+1}, dV_j, dK_j, dQ^T_j, dP^T_{j+1}
    // so that S^T of the next step is ready while the compute warps finish
    // step j, and P of step j+1 can be built while dV/dK/dQ^T of step j run.
    constexpr uint32_t kIdS = idesc_bf16_f32(128, QT, false, false);   // S^T, dP^T
    constexpr uint32_t kIdG = idesc_bf16_f32(128, D, false, true);     // dV, dK
    constexpr uint32_t kIdQ = idesc_bf16_f32(128, QT, true, true);     // dQ^T
    SegCursor c;
    cursor_init<kTileM>(c, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q);
    uint32_t tiles = 0, gs = 0;
    const uint32_t k_base = smem_addr(k_smem), v_base = smem_addr(v_smem);
    const uint32_t pt_base = smem_addr(pt_smem), dst_base = smem_addr(dst_smem);
    bool ok = true;

    // Waits for the Q / dO tiles of global step g (tile-local step j), clears
    // rows past the segment end; returns the stage's Q base address.
    auto ready_q = [&](uint32_t g, int32_t j, uint32_t& q_base) -> bool {
      const uint32_t st = g % C::NSTAGE;
      if (!mbar_wait(&bar.qd_full[st], (g / C::NSTAGE) & 1, abort)) return false;
      uint8_t* qs = qd_smem + st * 2 * C::Q_BYTES;
      const int32_t q_valid = c.olen - j * QT;
      if (q_valid < QT) {
        // Q / dO rows past the segment end meet P^T = dS^T = 0 in dK / dV.
        zero_rows(qs, 2 * C::NC, C::Q_CHUNK, q_valid, QT, lane);
        fence_proxy_async_smem();
      }
      __syncwarp();
      q_base = smem_addr(qs);
      return true;
    };
    // Base descriptors, built once; each k-step adds a constant offset.
    const uint64_t dK_kmaj = sw128_desc(k_base, 16, 1024);             // K as K-major A
    const uint64_t dV_kmaj = sw128_desc(v_base, 16, 1024);             // V as K-major A
    const uint64_t dK_mn = sw128_desc(k_base, C::KV_CHUNK, 1024);      // K^T as MN-major A
    const uint64_t dPT = sw128_desc(pt_base, 16, 1024);                // P^T, K-major A
    const uint64_t dST_k = sw128_desc(dst_base, 16, 1024);             // dS^T, K-major A
    const uint64_t dST_mn = sw128_desc(dst_base, C::PS_BYTES, 1024);   // dS^T, MN-major B
    auto issue_s = [&](uint32_t g, uint32_t q_base) {
      const uint32_t sc = C::S_COL + (g & 1) * 64;
      const uint64_t dq_k = sw128_desc(q_base, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
        const uint32_t qo = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32;
        mma_ss(tmem + sc, desc_at(dK_kmaj, ko), desc_at(dq_k, qo), kIdS, kk > 0);
      }
      mma_commit(&bar.s_full[g & 1]);
    };
    auto issue_dp = [&](uint32_t do_base) {
      const uint64_t ddo_k = sw128_desc(do_base, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
        const uint32_t qo = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32;
        mma_ss(tmem + C::DP_COL, desc_at(dV_kmaj, ko), desc_at(ddo_k, qo), kIdS, kk > 0);
      }
      mma_commit(&bar.dp_full);
    };

    // Per step g the pipe runs  dP^T_{g+1}, dV_g, dK_g, dQ^T_g, S^T_{g+2}:
    // dP^T_{g+1} goes in as soon as the compute warps have read dP^T_g, so
    // both S^T and dP^T of the next step are ready when they get to it.
    uint32_t q_addr[3] = {0, 0, 0};  // Q stage address of steps g, g+1, g+2
    for (int64_t t = blockIdx.x;
         ok && cursor_seek<kTileM>(c, t, p.num_heads, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q); t += G) {
      if (c.olen == 0) continue;
      const Tile tl = cursor_tile(c, t);
      if (!mbar_wait(&bar.kv_full, tiles & 1, abort)) break;
      ++tiles;
      const int32_t kv_valid = c.len - tl.m * kTileM;
      if (kv_valid < kTileM) {
        // K rows past the segment end would meet dS^T = 0 in dQ^T = K^T dS^T;
        // clear them so that 0 * NaN cannot occur.
        zero_rows(k_smem, C::KCH, C::KV_CHUNK, kv_valid, kTileM, lane);
        fence_proxy_async_smem();
      }
      __syncwarp();
      const int32_t nq = (c.olen + QT - 1) / QT;
      // prologue: S^T_0, dP^T_0, S^T_1.  Both TMEM score buffers and the dP^T
      // buffer were last read before the previous step's dp_free arrival.
      if (gs > 0 && !mbar_wait(&bar.dp_free, (gs - 1) & 1, abort)) break;
      if (!ready_q(gs, 0, q_addr[0])) break;
      if (nq > 1 && !ready_q(gs + 1, 1, q_addr[1])) break;
      tc_fence_after();
      if (lane == 0) {
        issue_s(gs, q_addr[0]);
        issue_dp(q_addr[0] + C::Q_BYTES);
        if (nq > 1) issue_s(gs + 1, q_addr[1]);
      }
      __syncwarp();
      for (int32_t j = 0; j < nq; ++j, ++gs) {
        const bool more = j + 1 < nq;
        if (more) {
          // dP^T_{g+1} as soon as dP^T_g has been read
          if (!mbar_wait(&bar.dp_free, gs & 1, abort)) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) issue_dp(q_addr[1] + C::Q_BYTES);
          __syncwarp();
        }
        if (!mbar_wait(&bar.ds_ready, gs & 1, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t q_cur = q_addr[0];
        if (lane == 0) {
          const uint64_t ddo_mn = sw128_desc(q_cur + C::Q_BYTES, C::Q_CHUNK, 1024);  // dO as MN-major B
          const uint64_t dq_mn = sw128_desc(q_cur, C::Q_CHUNK, 1024);                // Q as MN-major B
#pragma unroll
          for (int kk = 0; kk < QT / 16; ++kk) {
            mma_ss(tmem + C::DV_COL, desc_at(dPT, kk * 32), desc_at(ddo_mn, kk * 2048), kIdG,
                   (j > 0 || kk > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < QT / 16; ++kk) {
            mma_ss(tmem + C::DK_COL, desc_at(dST_k, kk * 32), desc_at(dq_mn, kk * 2048), kIdG,
                   (j > 0 || kk > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk) {
            mma_ss(tmem + C::DQ_COL, desc_at(dK_mn, kk * 2048), desc_at(dST_mn, kk * 2048), kIdQ,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(&bar.qd_empty[gs % C::NSTAGE]);
          mma_commit(&bar.step_done);
          if (!more) mma_commit(&bar.kv_empty);
        }
        __syncwarp();
        if (j + 2 < nq) {
          // S^T_{g+2} into the score buffer S^T_g used (read before dp_free_g)
          if (!ready_q(gs + 2, j + 2, q_addr[2])) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) issue_s(gs + 2, q_addr[2]);
          __syncwarp();
        }
        q_addr[0] = q_addr[1];
        q_addr[1] = q_addr[2];
      }
    }
    if (lane == 0) {
      mma_commit(&bar.mma_done);
      int dummy = 0;
      mbar_wait(&bar.mma_done, 0, &dummy);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute
    const int quad = warp & 3;
    const int half = (warp - 4) >> 2;              // which 32 q columns (and half of D in the epilogue)
    const int r = quad * 32 + lane;                // kv row in the tile / d index for dQ^T
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c2 = p.scale_log2;
    const int H = p.num_heads;
    SegCursor c;
    cursor_init<kTileM>(c, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q);
    uint32_t gs = 0;
    bool ok = true;

    // dQ^T of global step g (tile-local step j): wait for it, then add this
    // warp's 32 (d) x 32 (q) block into dq_acc.  A block whose 32 q rows all
    // lie in the segment is staged row-major [q][d] in the warp's own 4 KB
    // of shared memory and added with one bulk reduce-add.  The segment's
    // last, partial block is added row by row with reductions instead: its
    // columns past the segment end are 0 * K, which is NaN when K is, and
    // must not reach the next segment's rows.
    float* stg = reinterpret_cast<float*>(stg_smem) + (warp - 4) * 32 * 32;
    const bool drains = quad * 32 < D;             // warp-uniform: d block inside head_dim
    auto drain_dq = [&](uint32_t g, int32_t j, int32_t h) -> bool {
      if (!mbar_wait(&bar.step_done, g & 1, abort)) return false;
      tc_fence_after();
      uint32_t q32[32];
      tmem_ld32(tmem + lane_off + C::DQ_COL + half * 32, q32);
      tmem_wait_ld();
      const int32_t qs0 = j * QT + half * 32;  // first q column of this warp, in the segment
      if (drains && qs0 + 32 <= c.olen) {
        if (lane == 0) bulk_wait_read_all();   // the previous reduce has read the staging
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 32; ++i) stg[i * 32 + lane] = __uint_as_float(q32[i]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(stg, &tm_dq, quad * 32, h, c.o0 + qs0);
          bulk_commit();
        }
      } else if (drains && qs0 < c.olen) {
        float* dst = p.dq_acc + (((int64_t)c.o0 + qs0) * H + h) * D + quad * 32 + lane;
        const int64_t step = (int64_t)H * D;
        const int32_t n = c.olen - qs0;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i < n) atomicAdd(dst + i * step, __uint_as_float(q32[i]));
      }
      return true;
    };

    for (int64_t t = blockIdx.x;
         ok && cursor_seek<kTileM>(c, t, p.num_heads, p.cu_k, p.cu_q, p.batch, p.total_k, p.total_q); t += G) {
      const Tile tl = cursor_tile(c, t);
      const int32_t kv_valid = c.len - tl.m * kTileM;
      const bool row_valid = r < kv_valid;
      const int64_t krow = (int64_t)c.r0 + tl.m * kTileM + r;
      const int32_t nq = (c.olen + QT - 1) / QT;
      const float* lse2 = p.lse2 + (int64_t)tl.h * p.total_q + c.o0;
      const float* delta = p.delta + (int64_t)tl.h * p.total_q + c.o0;
      for (int32_t j = 0; j < nq; ++j, ++gs) {
        const int32_t qc0 = j * QT + half * 32;              // first q column (in the segment)
        const int32_t ncol = min(32, c.olen - qc0);          // valid columns of this thread (may be <= 0)
        // lane i fetches column i's lse2 / delta; broadcast below
        float my_l2 = 0.f, my_dl = 0.f;
        if (lane < ncol) {
          my_l2 = __ldg(lse2 + qc0 + lane);
          my_dl = __ldg(delta + qc0 + lane);
        }
        const int32_t nvalid = row_valid ? max(0, ncol) : 0;
        // ---- P^T = exp2(S^T c - lse2) as soon as S^T_j is ready
        if (!mbar_wait(&bar.s_full[gs & 1], (gs >> 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[32];
        tmem_ld32(tmem + lane_off + C::S_COL + (gs & 1) * 64 + half * 32, sv);
        tmem_wait_ld();
        float pv[32];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 l2 = make_float2(__shfl_sync(0xffffffffu, my_l2, i), __shfl_sync(0xffffffffu, my_l2, i + 1));
          float2 t2 = ffma2(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), make_float2(c2, c2),
                            make_float2(-l2.x, -l2.y));
          pv[i] = (i < nvalid) ? ex2(t2.x) : 0.f;
          pv[i + 1] = (i + 1 < nvalid) ? ex2(t2.y) : 0.f;
        }
        // ---- dS^T = P^T (dP^T - delta); dP^T_g is released right after it is read
        if (!mbar_wait(&bar.dp_full, gs & 1, abort)) { ok = false; break; }
        tc_fence_after();
        uint32_t dpv[32];
        tmem_ld32(tmem + lane_off + C::DP_COL + half * 32, dpv);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bar.dp_free);
        uint32_t pk[16], dk2[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 dl = make_float2(__shfl_sync(0xffffffffu, my_dl, i), __shfl_sync(0xffffffffu, my_dl, i + 1));
          const float2 ds = fmul2(make_float2(pv[i], pv[i + 1]),
                                  fadd2(make_float2(__uint_as_float(dpv[i]), __uint_as_float(dpv[i + 1])),
                                        make_float2(-dl.x, -dl.y)));
          // select, not multiply: dP^T rows past the segment end may hold NaN
          pk[i / 2] = pack_bf16x2(pv[i], pv[i + 1]);
          dk2[i / 2] = pack_bf16x2(i < nvalid ? ds.x : 0.f, i + 1 < nvalid ? ds.y : 0.f);
        }
        // ---- dQ^T of the previous step; its completion also means the
        // previous step's MMAs are done reading the P^T / dS^T buffers
        if (j > 0 && !drain_dq(gs - 1, j - 1, tl.h)) { ok = false; break; }
        // write this thread's 64 bytes of the P^T and dS^T rows (128-byte
        // swizzle: 16-byte unit u of row r sits at unit u ^ (r % 8))
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (half * 4 + u) ^ (r & 7);
          *reinterpret_cast<uint4*>(pt_smem + r * 128 + unit * 16) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          *reinterpret_cast<uint4*>(dst_smem + r * 128 + unit * 16) =
              make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar.ds_ready);
      }
      if (!ok) break;
      if (nq > 0 && !drain_dq(gs - 1, nq - 1, tl.h)) break;
      // ---- epilogue: dV and dK * scale of this kv tile (zeros if no queries)
      if (row_valid && nq == 0) {
        __nv_bfloat16* dvrow = p.dv + krow * p.dv_rs + (int64_t)tl.h * p.dv_hs;
        __nv_bfloat16* dkrow = p.dk + krow * p.dk_rs + (int64_t)tl.h * p.dk_hs;
        for (int d = half * (D / 2); d < (half + 1) * (D / 2); d += 8) {
          *reinterpret_cast<uint4*>(dvrow + d) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(dkrow + d) = make_uint4(0, 0, 0, 0);
        }
      }
      if (nq > 0) {
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
            dv4[0] = make_uint4(wa[0], wa[1], wa[2], wa[3]);
            dv4[1] = make_uint4(wa[4], wa[5], wa[6], wa[7]);
            dk4[0] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
            dk4[1] = make_uint4(wb[4], wb[5], wb[6], wb[7]);
          }
        }
        tc_fence_before();
      }
    }
    if (lane == 0) bulk_wait_all();  // this warp's dQ reductions have completed
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && bar.abort) record_error(p.err, kErrTimeout);
}

template <int D>
static cudaError_t launch_bwd_d(const BwdLaunch& L, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const int elem_grid = L.grid * 8;
  auto mark = [&](int i) {
    if (L.phase_events[i] != nullptr) cudaEventRecord(L.phase_events[i], stream);
  };
  auto kern = varlen_bwd_main_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  mark(0);
  varlen_bwd_prep_kernel<<<elem_grid, 256, 0, stream>>>(L.prep);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mark(1);
  kern<<<L.grid, 384, C::SMEM_BYTES, stream>>>(L.tm_q, L.tm_k, L.tm_v, L.tm_do, L.tm_dq, L.p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mark(2);
  varlen_bwd_post_kernel<<<elem_grid, 256, 0, stream>>>(L.post);
  e = cudaGetLastError();
  mark(3);
  return e;
}

cudaError_t launch_bwd(const BwdLaunch& L, cudaStream_t stream) {
  switch (L.head_dim) {
    case 64: return launch_bwd_d<64>(L, stream);
    case 96: return launch_bwd_d<96>(L, stream);
    case 128: return launch_bwd_d<128>(L, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace varlen
