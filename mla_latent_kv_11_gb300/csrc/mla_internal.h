// Internal declarations shared by the translation units of libmla.so.
// Nothing here is part of the C ABI (include/mla.h is).
#pragma once

#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "mla.h"

namespace mla {

// Bits of the per-module device error words.
constexpr unsigned kErrDeviceData = 1u;  // slot / block id / length out of range
constexpr unsigned kErrTimeout = 2u;     // a bounded wait gave up

// Keys per schedule tile of the split-KV decode (one page of 64 rows at page 64).
constexpr int kTile = 64;

// The fp8 ds_mla cache entry: e4m3 latent codes, then float32 scales (one per group of
// latent columns), then bf16 rope values.
constexpr int kDsMlaLatent = 512;
constexpr int kDsMlaGroup = 128;
constexpr int kDsMlaRope = 64;
constexpr int kDsMlaRopeByte = kDsMlaLatent + 4 * (kDsMlaLatent / kDsMlaGroup);   // 528
constexpr int kDsMlaEntry = kDsMlaRopeByte + 2 * kDsMlaRope;                       // 656
static_assert(kDsMlaEntry == MLA_DS_MLA_ENTRY_BYTES, "ds_mla entry layout");

// A ds_mla cache view: entry (blk, row) at data + blk*s_blk + row*s_row bytes.
struct DsMlaCache {
  const void* data;
  int64_t s_blk, s_row;
  int32_t num_blocks, page;
};

// A rank-3 strided view in ELEMENTS (data already includes the storage offset).
struct View3 {
  void* data;
  int64_t n0, n1, n2;
  int64_t s0, s1, s2;
};

// Programmatic dependent launch. Every kernel of the library is launched with programmatic
// stream serialization, so its launch and prologue overlap the end of the kernel before it in
// the stream. Each kernel calls pdl_enter() before it touches memory an earlier kernel may
// write: griddepcontrol.wait returns once the preceding grid has completed and its writes are
// visible (at once if the preceding stream work was not a programmatic launch), and
// launch_dependents then lets the next kernel start launching.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_allow_dependents();
}
#endif

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline View3 view3(const mla_tensor& t) {
  return View3{t.data, t.shape[0], t.shape[1], t.shape[2], t.stride[0], t.stride[1], t.stride[2]};
}

// The paged cache as the kernels see it.
struct CacheView {
  const void* data;  // element (blk, row, e) at data + blk*s_blk + row*s_row + e
  int64_t s_blk, s_row;
  int32_t num_blocks, page, entry;
};

// Decode schedule kept in the caller's workspace (all device pointers).
struct DecodeSched {
  int32_t* tile_prefix;  // [B+1] prefix sum of ceil(len_b / kTile)
  int32_t* first_unit;   // [B]   work unit holding the first tile of b
  int32_t* npieces;      // [B]   work units touching b (0 for an empty sequence)
  int32_t* piece_base;   // [B]   first partial slot of b (if npieces[b] > 1)
  int32_t* unit_tile;    // [units+1] first global tile of each work unit (the last entry: total)
  int32_t* unit_seq;     // [units]   first sequence of each unit's range (B for an empty unit)
  int4* seqinfo;         // [B] {tile_prefix[b], clamped length, npieces[b], piece_base[b] - first_unit[b]}
  float* part_o;         // [max_pieces, H, L] normalised partial outputs
  float* part_lse;       // [max_pieces, H]    their natural-log LSE
  int32_t units;         // number of work units W
  int32_t max_pieces;    // B + W
};

// Workspace layout of mla_decode for (B, H, L, units).
struct DecodeWsLayout {
  size_t off_prefix, off_first, off_np, off_base, off_unit, off_useq, off_seqinfo, off_part_o, off_part_lse,
      total;
};
DecodeWsLayout decode_ws_layout(int64_t B, int64_t H, int64_t L, int64_t units);
DecodeSched decode_sched_from_ws(void* ws, const DecodeWsLayout& lay, int32_t B, int32_t units);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// A 3-D TMA map (dims innermost first, strides of dims 1 and 2 in bytes, box b0 x b1 x b2) of
// bf16 elements, or of another element type.
bool make_map3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle swz,
                CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
// True once the driver's tensor-map encoder has been found.
bool tensor_maps_available();

// ---- launchers (return cudaSuccess or the launch error) -------------------
cudaError_t launch_concat_q(mla_dtype dt, const View3& out, const View3& nope, const View3& rope,
                            cudaStream_t st);
cudaError_t launch_cache_write(mla_dtype dt, const View3& cache, const View3& kv_c,
                               const View3& k_pe, int64_t L, int64_t R, const int64_t* slots,
                               int64_t T, cudaStream_t st);
cudaError_t launch_bmm_simt(mla_dtype dt, const View3& out, const View3& a, const View3& b,
                            cudaStream_t st);
// Tensor-core bmm (bmm_tc.cu): bf16, K % 64 == 0, N % 128 == 0, 16-byte aligned views.
bool bmm_tc_supported(mla_dtype dt, const View3& out, const View3& a, const View3& b);
cudaError_t launch_bmm_tc(const View3& out, const View3& a, const View3& b, cudaStream_t st);

// Row tiles per prefill sequence, prefix-summed into out[0..B] (one block).
cudaError_t launch_prefill_items(const int32_t* cu_q, int32_t B, int32_t tpt, int32_t* out, cudaStream_t st);
cudaError_t launch_decode_schedule(const int32_t* seq_lens, int32_t B, int32_t max_blocks,
                                   int32_t page, const DecodeSched& s, cudaStream_t st);
// fp8_cache: the cache holds e4m3 codes (one byte each), read as value * (*descale_k) with the
// query scaled by *descale_q (null pointers read as 1).
cudaError_t launch_decode_simt(mla_dtype dt, const View3& o_lat, float* lse, const View3& q,
                               const CacheView& cache, const int32_t* block_table,
                               int64_t bt_stride, int32_t max_blocks, const int32_t* seq_lens, int32_t B, int32_t H,
                               int32_t L, int32_t R, float scale, const DecodeSched& s,
                               cudaStream_t st, bool fp8_cache = false, const float* descale_q = nullptr,
                               const float* descale_k = nullptr);
// Sparse top-k decode over a ds_mla cache (split kernel only: schedule and combine as above,
// the schedule run with null lengths and cap = topk).
cudaError_t launch_decode_sparse_simt(mla_dtype dt, const View3& o_lat, float* lse, const View3& q,
                                      const DsMlaCache& cache, const int32_t* indices, int64_t idx_stride,
                                      int32_t topk, int32_t B, int32_t H, float scale, const DecodeSched& s,
                                      cudaStream_t st);
// The LSE combine and the W_UV un-projection in one kernel (combine_vup.cu): bf16, L = 512,
// V a multiple of 128, v-contiguous out and W_UV views, W_UV 16-byte aligned.
bool combine_vup_supported(mla_dtype dt, int L, int V, const View3& out, const View3& w_uv);
// out[b, h, :] = combine(o_lat rows / partials of (b, h)) @ w_uv[h], o_lat rounded to bf16 first.
cudaError_t launch_combine_vup(const View3& out, const View3& o_lat, float* lse, const View3& w_uv, int32_t B,
                               int32_t H, int32_t V, const DecodeSched& s, cudaStream_t st);
// The valid slots of each sparse query in listed order ([B, topk], compacted) and their counts.
cudaError_t launch_sparse_compact(const int32_t* indices, int64_t idx_stride, int32_t topk, int32_t B,
                                  int64_t num_rows, int32_t* out, int32_t* counts, cudaStream_t st);
// Tensor-core decode over gathered e4m3 rows (attn_tc.cu): bf16 queries, 64 or 128 heads, a
// 16-byte aligned cache with 16-byte strides, 16-byte aligned query and output views.
bool tc_gather_supported(mla_dtype dt, int H, const void* cache, int64_t s_blk_bytes, int64_t s_row_bytes,
                         const View3& q, const View3& o);
// An e4m3 paged cache (rope 0 or 64, L = 512).
cudaError_t launch_decode_tc_fp8(const View3& o_lat, float* lse, const View3& q, const CacheView& cache,
                                 const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                 int32_t B, int32_t H, int32_t R, float scale, const float* descale_q,
                                 const float* descale_k, const DecodeSched& s, cudaStream_t st);
// A ds_mla cache at compacted slots (the schedule ran on their counts, cap topk).
cudaError_t launch_decode_tc_dsmla(const View3& o_lat, float* lse, const View3& q, const DsMlaCache& cache,
                                   const int32_t* slots, int64_t slot_stride, int32_t topk, int32_t B, int32_t H,
                                   float scale, const DecodeSched& s, cudaStream_t st);
// e4m3 cache write: codes of x / (*scale) (float32, correctly rounded), round to nearest even,
// saturating; src_dt is kv_c's and k_pe's element type.
cudaError_t launch_cache_write_fp8(mla_dtype src_dt, const View3& cache, const View3& kv_c, const View3& k_pe,
                                   int64_t L, int64_t R, const int64_t* slots, int64_t T, const float* scale,
                                   cudaStream_t st);
cudaError_t launch_decode_combine(mla_dtype dt, const View3& o_lat, float* lse,
                                  const int32_t* seq_lens, int32_t B, int32_t H, int32_t L,
                                  const DecodeSched& s, cudaStream_t st);
cudaError_t launch_prefill_simt(mla_dtype dt, const View3& o_lat, float* lse, const View3& q,
                                const CacheView& cache, const int32_t* block_table,
                                int64_t bt_stride, int32_t max_blocks, const int32_t* cu_q,
                                const int32_t* kv_lens, int32_t B, int32_t T, int32_t H,
                                int32_t L, int32_t R, float scale, cudaStream_t st);

// Tensor-core attention (attn_tc.cu): bf16, L = 512, R in {0, 64}, H in {64, 128}, 16-byte
// aligned views.
bool tc_attention_supported(mla_dtype dt, int H, int L, int R, bool decode, const CacheView& cv,
                            const View3& q, const View3& o);
int tc_decode_units(int num_splits);
cudaError_t launch_decode_tc(const View3& o_lat, float* lse, const View3& q, const CacheView& cache,
                             const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t B, int32_t H, int32_t L, int32_t R,
                             float scale, const DecodeSched& s, cudaStream_t st);
cudaError_t launch_prefill_tc(const View3& o_lat, float* lse, const View3& q, const CacheView& cache,
                              const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                              const int32_t* cu_q, const int32_t* kv_lens, int32_t B, int32_t H,
                              int32_t L, int32_t R, float scale, int32_t* item_prefix,
                              cudaStream_t st);

// Validated views of a q concat and of a cache write (mla_api.cu).
struct ConcatPlan {
  bool empty = true;
  View3 out{}, nope{}, rope{};
};
struct WritePlan {
  bool empty = true;
  int64_t L = 0, R = 0;
  View3 cache{}, kv_c{}, k_pe{};
};
mla_status plan_concat(mla_dtype dtype, const mla_tensor& q_cat_out, const mla_tensor& nope,
                       const mla_tensor& rope, ConcatPlan* out);
mla_status plan_cache_write(mla_dtype dtype, const mla_tensor& cache, const mla_tensor& kv_c,
                            const mla_tensor& k_pe, const int64_t* slot_mapping, int64_t num_tokens,
                            WritePlan* out);
// The q concat and the cache write in one launch when both take 16-byte words, else two.
// `alongside`: the launch directly follows a kernel of the same call that writes none of this
// one's inputs or outputs and waits for its own predecessors before it lets dependents launch
// (the absorb into q_cat's latent columns); the copies then run alongside it and wait for it
// only before this kernel ends, so whatever follows still sees both complete.
cudaError_t launch_concat_cache(mla_dtype dt, const View3& out, const View3& nope, const View3& rope,
                                const View3& cache, const View3& kv_c, const View3& k_pe, int64_t L, int64_t R,
                                const int64_t* slots, int64_t T, cudaStream_t st,
                                bool alongside = false);

// Work units of the general (CUDA-core) split-KV decode: num_splits, or two per SM.
int32_t decode_units(int32_t num_splits);

// A decode call after validation: the views the kernels take, the path and its work units.
struct DecodeCall {
  int64_t B = 0, H = 0, L = 0, R = 0;
  bool empty = true;   // nothing to do (B or H is 0)
  CacheView cv{};
  View3 qv{}, ov{};
  bool tc = false;     // tensor-core path
  int32_t units = 0;
};
// The argument checks of mla_decode (every decode entry point uses them, so they report the same
// codes and messages); fills *out on MLA_OK.
mla_status check_decode_args(mla_dtype dtype, const mla_tensor& o_lat_out, const mla_tensor& q_cat,
                             const mla_tensor& cache, const int32_t* block_table, int64_t block_table_stride,
                             int32_t max_blocks, const int32_t* seq_lens, int32_t kv_lora_rank, int32_t rope_dim,
                             float softmax_scale, int32_t num_splits, DecodeCall* out);
// Schedule, split kernel and combine of a validated decode, with its scratch laid out by `lay`.
// fp8_cache: the cache holds e4m3 codes read as value * (*descale_k), the query scaled by *descale_q.
mla_status run_decode(mla_dtype dtype, const DecodeCall& dc, float* lse_out, const int32_t* block_table,
                      int64_t block_table_stride, int32_t max_blocks, const int32_t* seq_lens, float softmax_scale,
                      void* scratch, const DecodeWsLayout& lay, cudaStream_t st, bool fp8_cache = false,
                      const float* descale_q = nullptr, const float* descale_k = nullptr, bool combine = true);

// Set (or clear, with MLA_OK) the calling thread's mla_last_error() message.
mla_status report_status(mla_status st, const char* fmt, ...);

// Per-module error words: read and clear (after the stream was synchronised).
unsigned copy_errors_read_clear();
unsigned attn_simt_errors_read_clear();
unsigned attn_tc_errors_read_clear();
unsigned combine_vup_errors_read_clear();
unsigned bmm_tc_errors_read_clear();
cudaError_t launch_wait_check(uint32_t limit_us, cudaStream_t st);

}  // namespace mla
