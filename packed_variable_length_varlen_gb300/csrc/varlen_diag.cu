// varlen_diag.cu -- diagnostic kernels: the tile scheduler run on its own
// (so tests can check that every tile is visited exactly once and that no
// cu_seqlens entry past `batch` is read), and a failure-detection self test
// whose bounded wait is never satisfied.
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

}  // namespace varlen
