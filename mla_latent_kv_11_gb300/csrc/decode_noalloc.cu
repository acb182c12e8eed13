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

std::mutex g_scratch_mu;
std::vector<void*> g_scratch_ptr;  // device address of the scratch, per device

// Device address of the scratch on the current device, looked up once per
// device (the first call on a device does this set-up).
mla_status scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return report_status(MLA_ERR_CUDA, "mla_decode_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if ((int)g_scratch_ptr.size() <= dev) g_scratch_ptr.resize(dev + 1, nullptr);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return report_status(MLA_ERR_CUDA, "mla_decode_noalloc: cudaGetSymbolAddress of the scratch: %s",
                           cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MLA_OK;
}

bool well_formed(const mla_tensor& t, int rank) {
  if (t.rank != rank) return false;
  int64_t n = 1;
  for (int i = 0; i < rank; ++i) {
    if (t.shape[i] < 0) return false;
    n *= t.shape[i];
  }
  if (n == 0) return true;
  if (t.data == nullptr || t.stride[rank - 1] != 1) return false;
  for (int i = 0; i < rank - 1; ++i)
    if (t.stride[i] < 0) return false;
  return true;
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
  if (dtype != MLA_F32 && dtype != MLA_BF16)
    return report_status(MLA_ERR_INVALID_ARG, "mla_decode_noalloc: unknown dtype %d", (int)dtype);
  if (!well_formed(q_cat, 3) || !well_formed(o_lat_out, 3) || !well_formed(cache, 3))
    return report_status(MLA_ERR_INVALID_ARG,
                         "mla_decode_noalloc: q_cat, o_lat_out and cache must be rank-3 views with "
                         "innermost stride 1");
  const int64_t B = q_cat.shape[0], H = q_cat.shape[1], L = kv_lora_rank, R = rope_dim;
  if (L <= 0 || R < 0 || q_cat.shape[2] != L + R || cache.shape[2] != L + R)
    return report_status(MLA_ERR_INVALID_ARG, "mla_decode_noalloc: widths must be L + R");
  if (o_lat_out.shape[0] != B || o_lat_out.shape[1] != H || o_lat_out.shape[2] != L)
    return report_status(MLA_ERR_INVALID_ARG, "mla_decode_noalloc: o_lat_out must be [B,H,L]");
  if (cache.shape[0] <= 0 || cache.shape[1] <= 0 || cache.shape[0] > INT32_MAX || cache.shape[1] > INT32_MAX)
    return report_status(MLA_ERR_INVALID_ARG, "mla_decode_noalloc: bad cache shape");
  if (num_splits < 0) return report_status(MLA_ERR_INVALID_ARG, "mla_decode_noalloc: num_splits < 0");
  if (B == 0 || H == 0) return MLA_OK;
  if (B > INT32_MAX / 2 || H > 4096 || L > 512 || L + R > 1024)
    return report_status(MLA_ERR_UNSUPPORTED, "mla_decode_noalloc: shape beyond the kernels' limits");
  if (block_table == nullptr || seq_lens == nullptr)
    return report_status(MLA_ERR_INVALID_ARG, "mla_decode_noalloc: block_table and seq_lens must be non-null");
  if (max_blocks <= 0 || block_table_stride < max_blocks)
    return report_status(MLA_ERR_INVALID_ARG, "mla_decode_noalloc: need 0 < max_blocks <= block_table_stride");

  const CacheView cv{cache.data, cache.stride[0], cache.stride[1], (int32_t)cache.shape[0],
                     (int32_t)cache.shape[1], (int32_t)cache.shape[2]};
  const View3 qv = view3(q_cat), ov = view3(o_lat_out);
  const bool tc = softmax_scale > 0.f && tc_attention_supported(dtype, (int)H, (int)L, (int)R, true, cv, qv, ov);
  const int32_t units = tc ? tc_decode_units(num_splits)
                           : (num_splits > 0 ? num_splits : 2 * device_sm_count());
  const DecodeWsLayout lay = decode_ws_layout(B, H, L, units);
  if (lay.total > (size_t)MLA_DECODE_NOALLOC_SCRATCH_BYTES)
    return report_status(MLA_ERR_UNSUPPORTED,
                         "mla_decode_noalloc: this batch needs %zu bytes of scratch but the static "
                         "scratch holds %zu; use mla_decode with a workspace",
                         lay.total, (size_t)MLA_DECODE_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  mla_status ms = scratch_on_current_device(&scratch);
  if (ms != MLA_OK) return ms;
  const DecodeSched s = decode_sched_from_ws(scratch, lay, (int32_t)B, units);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = launch_decode_schedule(seq_lens, (int32_t)B, max_blocks, cv.page, s, st);
  if (e == cudaSuccess)
    e = tc ? launch_decode_tc(ov, lse_out, qv, cv, block_table, block_table_stride, max_blocks, seq_lens,
                              (int32_t)B, (int32_t)H, (int32_t)L, (int32_t)R, softmax_scale, s, st)
           : launch_decode_simt(dtype, ov, lse_out, qv, cv, block_table, block_table_stride, max_blocks,
                                seq_lens, (int32_t)B, (int32_t)H, (int32_t)L, (int32_t)R, softmax_scale,
                                s, st);
  if (e == cudaSuccess)
    e = launch_decode_combine(dtype, ov, lse_out, seq_lens, (int32_t)B, (int32_t)H, (int32_t)L, s, st);
  if (e != cudaSuccess)
    return report_status(MLA_ERR_CUDA, "mla_decode_noalloc: %s", cudaGetErrorString(e));
  return MLA_OK;
}
