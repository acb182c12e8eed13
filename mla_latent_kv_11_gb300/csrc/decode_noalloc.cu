// mla_decode_noalloc: the split-KV decode for callers that cannot allocate
// device memory.
//
// Some callers have no allocator to hand: code that runs inside another
// framework's memory pool without access to it, plugins whose host forbids
// cudaMalloc on its hot path (cudaMalloc synchronises the device and can fail
// under memory pressure), or embedded runtimes that reserve all device memory
// up front. mla_decode needs a caller-provided workspace for its schedule and
// chunk partials; this variant keeps that scratch in a fixed array of this
// module instead, so the caller passes only inputs and outputs.
//
// The array is MLA_DECODE_NOALLOC_SCRATCH_BYTES (40 MiB) of device memory
// that every GPU which loads the library holds until the process exits.
// Requests whose scratch would not fit are rejected with MLA_ERR_UNSUPPORTED.
// Nothing in the scratch needs to start at zero: every call rewrites the
// schedule before reading it and reads only the partial slots it wrote.
// All calls share the one array, so calls whose kernels overlap on the GPU
// (two streams, or two host threads) race on it and must be serialised by
// the caller.
#include <cstdint>
#include <mutex>
#include <vector>

#include "mla_internal.h"

namespace mla {

// The decode scratch (schedule + chunk partials + their LSE). In host code
// this name is only a stand-in for the device array; its device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[MLA_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The driver's cuCtxGetCurrent, found once through the runtime (the library links only the runtime).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

struct ScratchAddr {
  int dev;
  CUcontext ctx;
  void* ptr;
};
std::mutex g_scratch_mu;
std::vector<ScratchAddr> g_scratch_ptr;  // device address of the scratch, per (device, context)

// Device address of the scratch for the current device and context, looked up once per pair: the
// first call on a device (and the first after a reset of it, which makes a new context) does this
// set-up, so that call should come before any stream capture.
mla_status scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return report_status(MLA_ERR_CUDA, "mla_decode_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  CtxGetCurrentFn get = ctx_get_current();
  auto current_ctx = [get]() {
    CUcontext c = nullptr;
    if (get == nullptr || get(&c) != CUDA_SUCCESS) c = nullptr;
    return c;
  };
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  CUcontext ctx = current_ctx();
  if (ctx != nullptr)
    for (const ScratchAddr& a : g_scratch_ptr)
      if (a.dev == dev && a.ctx == ctx) {
        *out = a.ptr;
        return MLA_OK;
      }
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_decode_noalloc_scratch);   // also makes the device's context current
  if (e != cudaSuccess || ptr == nullptr)
    return report_status(MLA_ERR_CUDA, "mla_decode_noalloc: cudaGetSymbolAddress of the scratch: %s",
                         cudaGetErrorString(e));
  if (ctx == nullptr) ctx = current_ctx();
  g_scratch_ptr.push_back(ScratchAddr{dev, ctx, ptr});
  *out = ptr;
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status mla_decode_noalloc(mla_dtype dtype, mla_tensor o_lat_out, float* lse_out,
                                         mla_tensor q_cat, mla_tensor cache,
                                         const int32_t* block_table, int64_t block_table_stride,
                                         int32_t max_blocks, const int32_t* seq_lens,
                                         int32_t kv_lora_rank, int32_t rope_dim, float softmax_scale,
                                         int32_t num_splits, void* stream) {
  report_status(MLA_OK, nullptr);
  // the same checks, codes and messages as mla_decode
  DecodeCall dc;
  mla_status ms = check_decode_args(dtype, o_lat_out, q_cat, cache, block_table, block_table_stride, max_blocks,
                                    seq_lens, kv_lora_rank, rope_dim, softmax_scale, num_splits, &dc);
  if (ms != MLA_OK || dc.empty) return ms;
  const DecodeWsLayout lay = decode_ws_layout(dc.B, dc.H, dc.L, dc.units);
  if (lay.total > (size_t)MLA_DECODE_NOALLOC_SCRATCH_BYTES)
    return report_status(MLA_ERR_UNSUPPORTED,
                         "mla_decode_noalloc: this batch needs %zu bytes of scratch but the static "
                         "scratch holds %zu; use mla_decode with a workspace",
                         lay.total, (size_t)MLA_DECODE_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  ms = scratch_on_current_device(&scratch);
  if (ms != MLA_OK) return ms;
  return run_decode(dtype, dc, lse_out, block_table, block_table_stride, max_blocks, seq_lens, softmax_scale, scratch,
                    lay, (cudaStream_t)stream);
}
