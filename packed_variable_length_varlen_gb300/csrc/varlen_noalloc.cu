// varlen_noalloc.cu -- varlen_attn_bwd_noalloc: the backward with its
// scratch memory in a fixed, library-owned device array instead of a
// caller-provided workspace.
//
// Some callers cannot allocate device memory: code that runs inside a host
// framework that owns every device allocation (a plugin or an inference
// runtime whose memory planner must not be bypassed), or code on a path
// where calling cudaMalloc is not allowed (a real-time loop, or a region
// whose allocator is locked).  This entry point lets them run the backward
// with only their inputs and outputs.
//
// The scratch array is a file-scope __device__ array of
// VARLEN_NOALLOC_SCRATCH_BYTES bytes; every GPU that loads the library keeps
// it until the process exits.  Its device address belongs to the CUDA
// context it was looked up in: it is looked up (cudaGetSymbolAddress, with
// the device current) on the first call in each context -- the first call
// on a device, and the first one after the caller reset the device or made
// another context current -- so that first call should come before any
// stream capture.  All calls share the one array and it keeps the last
// call's contents -- the backward's preprocess kernel rewrites every part of
// it whose value reaches a result (it zeroes the dQ accumulator and writes
// each segment's delta / LSE entries; padding entries between segments are
// read but masked out), so stale contents never matter -- but calls whose
// work overlaps on the GPU (different streams with no ordering between
// them) race on it.
#include <mutex>

#include "varlen_attn.h"
#include "varlen_internal.h"

namespace varlen {
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[VARLEN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
struct ScratchEntry {
  void* addr;
  unsigned long long ctx_id;  // context the address was looked up in
};
ScratchEntry g_scratch[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch in the context current on this
// thread, looked up again whenever that context is not the one of the
// cached address.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDev) return cuda_fail(cudaErrorInvalidDevice);
  unsigned long long ctx = 0;
  int st = current_context_id(&ctx);
  if (st != VARLEN_OK) return st;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& ent = g_scratch[dev];
  if (ent.addr == nullptr || ctx == 0 || ent.ctx_id != ctx) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess) return cuda_fail(e);
    if (p == nullptr) return cuda_fail(cudaErrorInvalidSymbol);
    if ((st = current_context_id(&ctx)) != VARLEN_OK) return st;
    ent.addr = p;
    ent.ctx_id = ctx;
  }
  *out = ent.addr;
  return VARLEN_OK;
}

}  // namespace
}  // namespace varlen

extern "C" int varlen_attn_bwd_noalloc(const void* q, varlen_stride sq, const void* k, varlen_stride sk,
                                       const void* v, varlen_stride sv, const void* out, varlen_stride so,
                                       const void* dout, varlen_stride sdo, const float* lse,
                                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                                       int32_t total_q, int32_t total_k, int32_t num_heads, int32_t head_dim,
                                       int32_t max_seqlen_q, int32_t max_seqlen_k, float scale, void* dq,
                                       varlen_stride sdq, void* dk, varlen_stride sdk, void* dv, varlen_stride sdv,
                                       void* stream) {
  // Size first: a problem that does not fit the fixed array is refused
  // before anything else is looked at or enqueued.
  if (batch < 1 || total_q < 0 || num_heads < 1 || head_dim < 1) return VARLEN_ERR_SHAPE;
  const size_t need = varlen_attn_bwd_workspace_size(batch, total_q, num_heads, head_dim);
  if (need > (size_t)VARLEN_NOALLOC_SCRATCH_BYTES) return VARLEN_ERR_WORKSPACE;
  // The device is checked before the lookup: on a GPU that is not sm_103
  // the call fails like varlen_attn_bwd does (VARLEN_ERR_ARCH).
  int st = varlen::device_ready();
  if (st != VARLEN_OK) return st;
  void* scratch = nullptr;
  if ((st = varlen::scratch_address(&scratch)) != VARLEN_OK) return st;
  return varlen_attn_bwd(q, sq, k, sk, v, sv, out, so, dout, sdo, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q,
                         total_k, num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, dq, sdq, dk, sdk, dv, sdv,
                         scratch, (size_t)VARLEN_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" size_t varlen_attn_bwd_noalloc_scratch_bytes(void) { return (size_t)VARLEN_NOALLOC_SCRATCH_BYTES; }

extern "C" int varlen_attn_debug_noalloc_scratch(void** addr, unsigned long long* ctx_id) {
  if (addr == nullptr || ctx_id == nullptr) return VARLEN_ERR_NULL;
  int st = varlen::device_ready();
  if (st != VARLEN_OK) return st;
  if ((st = varlen::scratch_address(addr)) != VARLEN_OK) return st;
  return varlen::current_context_id(ctx_id);
}
