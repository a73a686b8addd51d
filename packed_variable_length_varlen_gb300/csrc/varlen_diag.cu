// varlen_diag.cu -- diagnostic kernels: the tile scheduler run on its own
// (so tests can check that every tile is visited exactly once and that no
// cu_seqlens entry past `batch` is read), a failure-detection self test
// whose bounded wait is never satisfied, and a tcgen05 issue-rate probe.
#include "sm103_ptx.cuh"
#include "varlen_internal.h"
#include "varlen_sched.cuh"

namespace varlen {

template <int TILE>
__global__ void debug_schedule_kernel(const int32_t* cu, int32_t batch, int32_t total, int32_t num_heads,
                                      int32_t* out, int64_t max_records) {
  __shared__ uint16_t order_tab[kLptCapWide];
  const CuView v{cu, 0};
  const WalkOrder order{order_tab, kLptCapWide};
  build_lpt_order(order, v, batch, total);
  __syncthreads();
  if (threadIdx.x != 0) return;
  SegCursor c;
  cursor_init<TILE>(c, v, v, batch, total, total, order);
  for (int64_t t = blockIdx.x; cursor_seek<TILE>(c, t, num_heads, v, v, batch, total, total, order); t += gridDim.x) {
    const Tile tl = cursor_tile(c, t);
    if (t < max_records) {
      int4 rec = make_int4(tl.b, tl.m, tl.h, (int)blockIdx.x);
      *reinterpret_cast<int4*>(out + 4 * t) = rec;
    }
  }
}

cudaError_t launch_debug_schedule(const int32_t* cu, int32_t batch, int32_t total, int32_t num_heads, int32_t tile,
                                  int32_t grid, int32_t* out, int64_t max_records, cudaStream_t stream) {
  if (tile == 256)
    debug_schedule_kernel<256><<<grid, 32, 0, stream>>>(cu, batch, total, num_heads, out, max_records);
  else if (tile == 128)
    debug_schedule_kernel<128><<<grid, 32, 0, stream>>>(cu, batch, total, num_heads, out, max_records);
  else
    debug_schedule_kernel<64><<<grid, 32, 0, stream>>>(cu, batch, total, num_heads, out, max_records);
  return cudaGetLastError();
}

// One CTA waits on an mbarrier that nothing arrives at; the bounded wait must
// give up after budget_ns, record kErrTimeout and let the kernel return.
__global__ void selftest_timeout_kernel(uint64_t budget_ns, unsigned int* err) {
  __shared__ uint64_t never;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&never, 0, &abort_flag, budget_ns);
  __syncthreads();
  if (threadIdx.x == 0 && abort_flag) record_error(err, kErrTimeout);
}

cudaError_t launch_selftest_timeout(uint64_t budget_ns, unsigned int* err, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(budget_ns, err);
  return cudaGetLastError();
}

// tcgen05 issue-rate probe: one thread issues n_mma MMAs of M = 128, N =
// n_cols, K = 16 (bf16 x bf16 -> fp32) into one TMEM accumulator, on zero
// operands, and the kernel reports the issuing thread's clock64 cycles from
// the first issue to the completion of the last (tcgen05.commit on an
// mbarrier, bounded wait).  mode 0: A and B from shared memory, descriptors
// as the kernels keep them (a constant high word, the low word advanced by
// an immediate per k-step); mode 1: A from TMEM; mode 2: as mode 0, but each
// MMA's two 64-bit descriptors are rebuilt from the shared-memory address.
// Modes 3 and 4 time TMEM <-> register traffic instead: each of the four
// warps loads (3) or stores (4) its 32 lanes x 32 columns (4 KB) n_mma
// times, waiting for each before the next (n_cols unused).  Mode 5: as mode
// 1 with B MN-major (the layout of V in O += P V: rows of 64 N elements,
// one per K index, 64-element N blocks 16 KB apart; n_cols at most 128).
// Mode 6: as mode 1 while four more warps keep loading TMEM columns the
// MMAs do not touch (tcgen05.ld 32 lanes x 32 columns and a wait, over and
// over), as a softmax does beside the tensor core.  Mode 7: as mode 1 while
// four more warps keep storing 16-byte words into a separate 16 KB of
// shared memory (shared-memory writes beside the operand reads, as K/V tile
// loads arrive during the products).
constexpr int kMmaProbeA = 16384, kMmaProbeB = 32768;  // A: 128 x 64 bf16; B: 256 x 64 bf16
constexpr int kMmaProbeW = 16384;  // mode 7's write target
constexpr int kMmaProbeSmem = 1024 + kMmaProbeA + kMmaProbeB + kMmaProbeW;

template <int MODE>
__global__ void __launch_bounds__(256, 1) mma_rate_kernel(int32_t n_mma, int32_t n_cols,
                                                          unsigned long long* cycles, unsigned int* err) {
  constexpr int mode = MODE;  // a template parameter: no branch in the issue loop
  extern __shared__ __align__(1024) uint8_t probe_smem[];
  __shared__ uint64_t done;
  __shared__ uint32_t tbase;
  __shared__ int abort_flag;
  __shared__ int stop;  // mode 6: the MMAs have completed
  uint8_t* base = probe_smem + ((1024u - (smem_addr(probe_smem) & 1023u)) & 1023u);  // 1024-byte aligned
  uint8_t* a_s = base;
  uint8_t* b_s = base + kMmaProbeA;
  for (int i = threadIdx.x; i < (kMmaProbeA + kMmaProbeB) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(base)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&done, 1);
    abort_flag = 0;
    stop = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < 32) tmem_alloc(&tbase, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tbase;
  if (threadIdx.x >= 128) {  // modes 6, 7: TMEM loads / shared-memory stores beside the MMAs, until they complete
    if constexpr (mode == 7) {
      uint4* wbuf = reinterpret_cast<uint4*>(base + kMmaProbeA + kMmaProbeB);
      const int t = threadIdx.x - 128;
      uint4 v = make_uint4(t, 1, 2, 3);
      for (int32_t i = 0; i < 256 * n_mma && !*reinterpret_cast<volatile int*>(&stop); ++i) {
        wbuf[(t + 128 * (i & 7)) & (kMmaProbeW / 16 - 1)] = v;
        v.x += 1;
      }
    }
    if constexpr (mode == 6) {
      const uint32_t lane_off = (uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16;
      uint32_t r[32];
      for (int32_t i = 0; i < 64 * n_mma && !*reinterpret_cast<volatile int*>(&stop); ++i) {
        tmem_ld32(tmem + lane_off + 384 + (uint32_t)(i & 3) * 32, r);
        tmem_wait_ld();
      }
      (void)r;
    }
  } else if constexpr (mode >= 3 && mode <= 4) {
    const uint32_t lane_off = (uint32_t)((threadIdx.x >> 5) * 32) << 16;
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = i;
    __syncthreads();
    const long long t0 = clock64();
    for (int32_t i = 0; i < n_mma; ++i) {
      const uint32_t col = (uint32_t)(i & 7) * 32;
      if constexpr (mode == 3) {
        tmem_ld32(tmem + lane_off + col, r);
        tmem_wait_ld();
      } else {
        tmem_st32(tmem + lane_off + col, r);
        tmem_wait_st();
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) cycles[0] = (unsigned long long)(clock64() - t0) + (r[0] & 0u);
  } else if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, n_cols, false, mode == 5);
    const uint32_t alo = sw128_desc_lo(smem_addr(a_s), 16);
    const uint32_t blo = sw128_desc_lo(smem_addr(b_s), mode == 5 ? 16384u : 16u);
    const long long t0 = clock64();
    for (int32_t i = 0; i < n_mma; i += 4) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {  // the four 16-wide k-steps of a 64-column chunk
        const uint32_t acc = (i + kk) > 0 ? 1u : 0u;
        if constexpr (mode == 1 || mode == 6 || mode == 7) {
          mma_ts_lo(tmem, tmem + 256 + kk * 8, blo + ((kk * 32) >> 4), idesc, acc);
        } else if constexpr (mode == 5) {
          mma_ts_lo(tmem, tmem + 256 + kk * 8, blo + ((kk * 2048) >> 4), idesc, acc);
        } else if constexpr (mode == 2) {
          const uint64_t ad = sw128_desc(smem_addr(a_s) + kk * 32, 16, 1024);
          const uint64_t bd = sw128_desc(smem_addr(b_s) + kk * 32, 16, 1024);
          mma_ss(tmem, ad, bd, idesc, acc);
        } else {
          mma_ss_lo(tmem, alo + ((kk * 32) >> 4), blo + ((kk * 32) >> 4), idesc, acc);
        }
      }
    }
    mma_commit(&done);
    mbar_wait(&done, 0, &abort_flag);
    cycles[0] = (unsigned long long)(clock64() - t0);
    *reinterpret_cast<volatile int*>(&stop) = 1;
    if (abort_flag) record_error(err, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int MODE>
static cudaError_t launch_mma_rate(int32_t n_mma, int32_t n_cols, unsigned long long* cycles, unsigned int* err,
                                   cudaStream_t stream) {
  cudaError_t e =
      cudaFuncSetAttribute(mma_rate_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaProbeSmem);
  if (e != cudaSuccess) return e;
  mma_rate_kernel<MODE><<<1, MODE >= 6 ? 256 : 128, kMmaProbeSmem, stream>>>(n_mma, n_cols, cycles, err);
  return cudaGetLastError();
}

cudaError_t launch_debug_mma_rate(int32_t n_mma, int32_t n_cols, int32_t mode, unsigned long long* cycles,
                                  unsigned int* err, cudaStream_t stream) {
  switch (mode) {
    case 0: return launch_mma_rate<0>(n_mma, n_cols, cycles, err, stream);
    case 1: return launch_mma_rate<1>(n_mma, n_cols, cycles, err, stream);
    case 2: return launch_mma_rate<2>(n_mma, n_cols, cycles, err, stream);
    case 3: return launch_mma_rate<3>(n_mma, n_cols, cycles, err, stream);
    case 4: return launch_mma_rate<4>(n_mma, n_cols, cycles, err, stream);
    case 5: return launch_mma_rate<5>(n_mma, n_cols, cycles, err, stream);
    case 6: return launch_mma_rate<6>(n_mma, n_cols, cycles, err, stream);
    case 7: return launch_mma_rate<7>(n_mma, n_cols, cycles, err, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace varlen
