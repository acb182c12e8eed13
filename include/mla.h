/*
 * mla.h - C ABI of the weight-absorbed Multi-head Latent Attention (MLA) hot
 * path over a paged latent KV cache, for NVIDIA GB300 (sm_103a).
 *
 * One decode step is five calls, all asynchronous on the caller's stream:
 *
 *   mla_absorb_q    q_lat[h,b,:] = q_nope[h,b,:] @ W_UK[h]        (step 1)
 *   mla_concat_q    q_cat[t,h,:] = [q_lat[t,h,:] | q_pe[t,h,:]]    (step 2)
 *   mla_cache_write cache[slot]  = [kv_c | k_pe]                   (step 3)
 *   mla_decode      o_lat = softmax(scale * q_cat . cache) c_kv    (step 4)
 *   mla_v_up        out[h,b,:]   = o_lat[h,b,:] @ W_UV[h]          (step 5)
 *
 * and mla_prefill is step 4 for many causal queries per sequence. Fused forms:
 * mla_concat_q_cache_write (steps 2 and 3 in one launch), mla_absorb_concat_cache_write
 * (steps 1 to 3 in one call, the copies alongside the absorb) and mla_decode_v_up (step 4
 * with step 5 in its combine).
 *
 * Sources of the operations (web pages):
 *   [vt]    vllm.cpp, tests/vt/test_ops_mla_absorb.cpp (BatchedMatmul and
 *           ConcatMlaNopeRope test cases; strided views Contig/View3).
 *   [memra] memra-engine 0.124.1, tests/mla_gpu_forward.rs (absorbed and naive
 *           oracles; cache rows [c_kv | k_pe]; causal prefill and stepwise decode).
 *   [vllm]  vLLM, tests/kernels/attention/test_mla_cross_layer_kernel_equivalence.py
 *           (concat_and_cache_mla into a unified-slot layer view; paged dense
 *           decode with a block table and cache_seqlens).
 *
 * Conventions shared by every call
 *   - Ownership: the caller allocates and owns every buffer. Unless a call says
 *     otherwise the library allocates no device memory; it keeps a host-side
 *     cache of TMA tensor maps and a few bytes of static device state (an
 *     error word per kernel module).
 *   - Pointers: every data pointer is a DEVICE pointer of the current CUDA
 *     device. `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Execution: asynchronous; no call synchronises the stream or the device.
 *   - Views: an mla_tensor is {data, rank, shape, stride}; strides count
 *     ELEMENTS and `data` already includes any storage offset ([vt] View3).
 *     The innermost stride must be 1 on every tensor ([vt] "rejects malformed
 *     shapes/strides rather than mis-computing").
 *   - Validation: shapes, strides, dtypes, null pointers and alignment are
 *     checked on the host before any launch. A failed check returns
 *     MLA_ERR_INVALID_ARG (malformed) or MLA_ERR_UNSUPPORTED (well formed but
 *     outside what the kernels handle) and launches nothing.
 *   - Device-resident values (slots, block ids, sequence lengths) cannot be
 *     checked on the host. The kernels check them: an access that would leave
 *     the cache view is skipped and recorded; mla_device_error() reports it.
 *   - Empty work (zero tokens, zero sequences) returns MLA_OK and launches
 *     nothing ([memra]: "never a zero-extent launch").
 *   - Errors: mla_last_error() returns a message for the calling thread's
 *     last failed call. Launch failures return MLA_ERR_CUDA.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_ABI_VERSION 1

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,  /* malformed shape, stride, dtype or pointer   */
  MLA_ERR_UNSUPPORTED = 2,  /* well formed, but not handled by the kernels  */
  MLA_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed         */
  MLA_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up           */
  MLA_ERR_DEVICE_DATA = 5   /* a device-resident index was out of range     */
} mla_status;

typedef enum {
  MLA_F32 = 0,   /* IEEE binary32 */
  MLA_BF16 = 1   /* bfloat16; results rounded to nearest even */
} mla_dtype;

/* A strided view: element (i0,..,i_{rank-1}) lives at
 * data + sum_k i_k * stride[k] elements. rank <= 4; unused entries ignored. */
typedef struct {
  void* data;
  int32_t rank;
  int64_t shape[4];
  int64_t stride[4];
} mla_tensor;

/* ABI version of the loaded library (MLA_ABI_VERSION at build time). */
int mla_abi_version(void);

/* Message for the calling thread's last failed call ("" if none). The string
 * stays valid until the thread's next call into the library. */
const char* mla_last_error(void);

/* Static name of a status code. */
const char* mla_status_string(mla_status status);

/* Step 1 - W_UK absorption ([vt] BatchedMatmul, q-side fold: a (B,N,P) -> (N,B,P)
 * transposed view times W_UK_T [N,P,L]; [memra] mla_absorb_q).
 *   q_lat_out [H,B,L] (written), q_nope [H,B,P], w_uk [H,P,L]; any strides with
 *   innermost 1 (q_nope is usually the transpose of a [B,H,P] buffer and
 *   q_lat_out the transpose of a [B,H,L] buffer).
 *   q_lat[h,b,l] = sum_p q_nope[h,b,p] * w_uk[h,p,l], accumulated in fp32 and
 *   stored in `dtype`. All three tensors have `dtype`. */
mla_status mla_absorb_q(mla_dtype dtype, mla_tensor q_lat_out, mla_tensor q_nope,
                        mla_tensor w_uk, void* stream);

/* Step 2 - q concat ([vt] ConcatMlaNopeRope: a pure copy, bit for bit, that must
 * follow the strides of a transposed nope operand; a rope operand with one head
 * is broadcast to every head, as for _concat_k_nope_k_pe).
 *   q_cat_out [T,H,L+R] (written), nope [T,H,L], rope [T,H,R] or [T,1,R]
 *   (a rope stride(1) of 0 also broadcasts). Bits are copied unchanged,
 *   including NaN payloads and signed zeros. R may be 0.
 *   nope may be q_cat_out's own first L columns (the same data pointer and
 *   strides: mla_absorb_q can write q_lat straight into q_cat_out); then only
 *   the rope columns are copied. Any other overlap of q_cat_out with an input
 *   is undefined. */
mla_status mla_concat_q(mla_dtype dtype, mla_tensor q_cat_out, mla_tensor nope,
                        mla_tensor rope, void* stream);

/* Step 3 - paged latent cache write ([vllm] concat_and_cache_mla with kv_cache_dtype
 * "auto"; [memra] mla_append_latent).
 *   cache [num_blocks, page, L+R] view (written): any stride(0) and storage
 *   offset, e.g. one layer of a block-major unified slot; kv_c [T,L], k_pe [T,R];
 *   slot_mapping: device int64 [num_tokens].
 *   For token i with s = slot_mapping[i] >= 0:
 *     cache[s / page, s % page, 0:L]   = kv_c[i]
 *     cache[s / page, s % page, L:L+R] = k_pe[i]
 *   bit for bit. Negative slots are padding and write nothing. Slots at or beyond
 *   num_blocks*page write nothing and set MLA_ERR_DEVICE_DATA in mla_device_error.
 *   No element outside the addressed rows is written. Duplicate slots: the
 *   surviving row is unspecified. */
mla_status mla_cache_write(mla_dtype dtype, mla_tensor cache, mla_tensor kv_c, mla_tensor k_pe,
                           const int64_t* slot_mapping, int64_t num_tokens, void* stream);

/* Step 4 - paged split-KV decode ([vllm] flash_mla_with_kvcache / FlashInfer MLA
 * decode over a strided cache view; [memra] mla_attn_absorbed with t_q = 1).
 *   o_lat_out [B,H,L] (written; `dtype`), lse_out: device float [B,H] contiguous
 *   or NULL; q_cat [B,H,L+R]; cache as in mla_cache_write;
 *   block_table: device int32 [B, max_blocks] with row stride block_table_stride;
 *   seq_lens: device int32 [B].
 *   For every sequence b and head h, over rows t < seq_lens[b] of the cache
 *   (row t at block block_table[b, t / page], offset t % page):
 *     s_t = softmax_scale * (q_cat[b,h,0:L] . c_kv_t + q_cat[b,h,L:] . k_pe_t)
 *     o_lat[b,h,:] = sum_t softmax(s)_t * c_kv_t,  lse[b,h] = ln sum_t e^{s_t}
 *   with fp32 softmax and accumulation. seq_lens[b] == 0 gives o = 0 and
 *   lse = -inf. The context is cut into chunks processed in parallel and merged
 *   by their LSE; num_splits > 0 sets the number of chunks processed in
 *   parallel over the whole batch (0 = chosen from the SM count). For fixed
 *   (seq_lens, num_splits, device) the result is bit-identical from run to run
 *   and does not depend on the cache strides.
 *   workspace: device scratch of at least mla_decode_workspace_size(...) bytes,
 *   256-byte aligned, owned by the caller, not used by concurrent calls. */
mla_status mla_decode(mla_dtype dtype, mla_tensor o_lat_out, float* lse_out, mla_tensor q_cat,
                      mla_tensor cache, const int32_t* block_table, int64_t block_table_stride,
                      int32_t max_blocks, const int32_t* seq_lens, int32_t kv_lora_rank,
                      int32_t rope_dim, float softmax_scale, int32_t num_splits,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace mla_decode needs for `batch` sequences of `num_heads` heads
 * with latent width `kv_lora_rank` and the given num_splits (0 = automatic) on
 * the current device. */
size_t mla_decode_workspace_size(int32_t batch, int32_t num_heads, int32_t kv_lora_rank,
                                 int32_t num_splits);

/* Steps 2 and 3 in one launch - the q concat and the cache write of the same
 * decode step (the fused pre-attention of the vllm.cpp and memra pages' step
 * order: the new rows' [c_kv | k_pe] go into the cache while the query's rope
 * columns join q_cat).
 *   Arguments: those of mla_concat_q followed by those of mla_cache_write (one
 *   dtype for all tensors). Results, errors and the in-place nope case are
 *   exactly theirs; when either part cannot move 16-byte words the two run as
 *   two launches. */
mla_status mla_concat_q_cache_write(mla_dtype dtype, mla_tensor q_cat_out, mla_tensor nope,
                                    mla_tensor rope, mla_tensor cache, mla_tensor kv_c,
                                    mla_tensor k_pe, const int64_t* slot_mapping,
                                    int64_t num_tokens, void* stream);

/* Steps 1, 2 and 3 of a decode step in one call - the absorb straight into q_cat, the
 * rope columns of q_cat and the cache write of the new rows (the fused pre-attention of the
 * vllm.cpp and memra pages' step order, absorb -> q_cat included).
 *   q_cat [T,H,L+R] (written), q_nope [H,T,P] (any strides with innermost 1: usually the
 *   transpose of a [T,H,P] buffer), w_uk [H,P,L], q_pe [T,H,R] or [T,1,R]; cache, kv_c,
 *   k_pe, slot_mapping and num_tokens as for mla_cache_write. One dtype for all tensors.
 *   Results are exactly those of mla_absorb_q(q_cat's first L columns seen as [H,T,L],
 *   q_nope, w_uk) followed by mla_concat_q_cache_write(q_cat, q_cat's own first L columns,
 *   q_pe, cache, kv_c, k_pe, slot_mapping, num_tokens), and so are the errors (a w_uk wider
 *   than q_cat, or shapes that do not match, return MLA_ERR_INVALID_ARG). The copies touch
 *   only q_cat's rope columns and the cache, none of the absorb's operands or output, so on
 *   the GPU they run alongside the absorb instead of after it; the call's work is complete,
 *   as a whole, before anything queued after it on the stream starts reading it. q_cat,
 *   q_nope, w_uk, q_pe, the cache, kv_c and k_pe must not overlap one another. */
mla_status mla_absorb_concat_cache_write(mla_dtype dtype, mla_tensor q_cat, mla_tensor q_nope,
                                         mla_tensor w_uk, mla_tensor q_pe, mla_tensor cache,
                                         mla_tensor kv_c, mla_tensor k_pe,
                                         const int64_t* slot_mapping, int64_t num_tokens,
                                         void* stream);

/* Step 3, fp8 cache - the cache write into an e4m3 cache ([vllm] concat_and_cache_mla
 * with a quantized cache dtype and its scale).
 *   cache [num_blocks, page, L+R] view of e4m3 codes, one byte per element (strides
 *   count bytes), any stride(0) and storage offset; kv_c [T,L] and k_pe [T,R] in
 *   src_dtype (MLA_F32 or MLA_BF16); slot_mapping: device int64 [num_tokens];
 *   scale: device float [1], the cache scale.
 *   For token i with s = slot_mapping[i] >= 0 the row s becomes the e4m3 codes of
 *   float32(x) / scale (the division correctly rounded), rounded to nearest with
 *   ties to even; finite values beyond 448 saturate to +-448, NaN stays NaN.
 *   Padding slots, out-of-range slots and the untouched rows: as mla_cache_write. */
mla_status mla_cache_write_fp8(mla_dtype src_dtype, mla_tensor cache, mla_tensor kv_c,
                               mla_tensor k_pe, const int64_t* slot_mapping, int64_t num_tokens,
                               const float* scale, void* stream);

/* Step 4, fp8 cache - paged split-KV decode over an e4m3 cache ([vllm]
 * flash_mla_with_kvcache_fp8 with descale_q and descale_k).
 *   Arguments as mla_decode, except: cache holds e4m3 codes (one byte per element,
 *   strides in bytes); every cache value is its code's value times *descale_k and
 *   the query is q_cat times *descale_q (device floats [1]; NULL reads as 1).
 *   o_lat_out and q_cat have `dtype`; the workspace is mla_decode's
 *   (mla_decode_workspace_size). Results: as mla_decode over the dequantised
 *   values. */
mla_status mla_decode_fp8(mla_dtype dtype, mla_tensor o_lat_out, float* lse_out, mla_tensor q_cat,
                          mla_tensor cache, const int32_t* block_table, int64_t block_table_stride,
                          int32_t max_blocks, const int32_t* seq_lens, int32_t kv_lora_rank,
                          int32_t rope_dim, float softmax_scale, const float* descale_q,
                          const float* descale_k, int32_t num_splits, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Bytes of one fp8 ds_mla cache entry: 512 e4m3 latent codes, four float32
 * scales (scale g covers latent columns 128g .. 128g+127), 64 bf16 rope values. */
#define MLA_DS_MLA_ENTRY_BYTES 656

/* Step 4, sparse fp8 - top-k decode over an fp8 ds_mla cache ([vllm]
 * flash_mla_with_kvcache with is_fp8_kvcache and indices, the DeepSeek sparse
 * attention path; the indexer that picks the slots is not part of this library).
 *   o_lat_out [B,H,512] (written), lse_out device float [B,H] or NULL,
 *   q_cat [B,H,576] (latent 512 | rope 64), both in `dtype`;
 *   cache [num_blocks, page, 656] byte view (strides in bytes, any stride(0) and
 *   storage offset: one layer of a unified-slot buffer), data and strides 16-byte
 *   aligned; indices: device int32 [B, topk] with row stride indices_stride
 *   (>= topk); slot = block * page + row; negative entries are padding.
 *   Query b attends the rows at its listed slots (each once per listing, in any
 *   order): key [c_kv | k_pe], value c_kv, c_kv[i] = e4m3 value * scale[i / 128]
 *   and k_pe the bf16 rope values; the softmax and outputs as mla_decode. A query
 *   with no valid slot gets o = 0, lse = -inf. A slot past the cache is skipped and
 *   reported by mla_device_error (MLA_ERR_DEVICE_DATA).
 *   num_splits: as mla_decode; workspace: device scratch of at least
 *   mla_decode_sparse_workspace_size(B, H, topk, num_splits) bytes, 256-byte
 *   aligned, caller-owned. */
/* Bytes of workspace mla_decode_sparse_fp8 needs. */
size_t mla_decode_sparse_workspace_size(int32_t batch, int32_t num_heads, int32_t topk, int32_t num_splits);

mla_status mla_decode_sparse_fp8(mla_dtype dtype, mla_tensor o_lat_out, float* lse_out, mla_tensor q_cat,
                                 mla_tensor cache, const int32_t* indices, int64_t indices_stride,
                                 int32_t topk, float softmax_scale, int32_t num_splits, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Step 4, prefill - causal attention of many queries per sequence over the same
 * paged cache ([memra] gate 1: pure prefill t_q == t_kv and the chunked shape
 * where the queries are a suffix of an already populated cache).
 *   o_lat_out [T,H,L] (written), lse_out device float [T,H] or NULL,
 *   q_cat [T,H,L+R] with the queries of sequence b in rows
 *   cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 (device int32 [batch+1]);
 *   seq_lens_kv: device int32 [batch], rows of sequence b already in the cache
 *   (including its own queries' rows).
 *   Query i of sequence b sits at position p = seq_lens_kv[b] - q_len_b + i and
 *   attends rows 0..p (bottom-right causal alignment); otherwise as mla_decode.
 *   max_q_len bounds q_len_b. workspace: device scratch of at least
 *   mla_prefill_workspace_size(batch) bytes, 256-byte aligned, caller-owned. */
mla_status mla_prefill(mla_dtype dtype, mla_tensor o_lat_out, float* lse_out, mla_tensor q_cat,
                       mla_tensor cache, const int32_t* block_table, int64_t block_table_stride,
                       int32_t max_blocks, const int32_t* cu_seqlens_q, const int32_t* seq_lens_kv,
                       int32_t batch, int32_t max_q_len, int32_t kv_lora_rank, int32_t rope_dim,
                       float softmax_scale, void* workspace, size_t workspace_bytes,
                       void* stream);

/* Bytes of workspace mla_prefill needs for `batch` sequences. */
size_t mla_prefill_workspace_size(int32_t batch);

/* Step 5 - W_UV un-projection ([vt] BatchedMatmul at the _v_up_proj call site: a
 * (B,N,L) -> (N,B,L) transposed input, output written into a transposed (B,N,V);
 * [memra] mla_decompress_v).
 *   out [H,B,V] (written), o_lat [H,B,L], w_uv [H,L,V].
 *   out[h,b,v] = sum_l o_lat[h,b,l] * w_uv[h,l,v], fp32 accumulation. */
mla_status mla_v_up(mla_dtype dtype, mla_tensor out, mla_tensor o_lat, mla_tensor w_uv,
                    void* stream);

/* Steps 4 and 5 as one call - split-KV paged decode whose output goes straight
 * through the W_UV un-projection ([vt] _v_up_proj at the end of the absorbed
 * decode; [memra] mla_attn_absorbed -> mla_decompress_v): the LSE combine of the
 * split sequences and the un-projection run as one kernel, so o_lat is never
 * written out.
 *   out [B,H,V] (written; any strides with unit v stride), lse_out device float
 *   [B,H] or NULL, q_cat, cache, block table, lengths, kv_lora_rank, rope_dim,
 *   softmax_scale, num_splits: as mla_decode; w_uv [H,L,V] as mla_v_up.
 *   out[b,h,:] = o_lat[b,h,:] @ w_uv[h] with o_lat the decode's output rounded to
 *   `dtype` (as mla_decode followed by mla_v_up computes it).
 *   workspace: device scratch of at least
 *   mla_decode_v_up_workspace_size(B, H, L, num_splits) bytes, 256-byte aligned,
 *   caller-owned (it also holds o_lat). Errors: as mla_decode and mla_v_up. */
mla_status mla_decode_v_up(mla_dtype dtype, mla_tensor out, float* lse_out, mla_tensor q_cat, mla_tensor cache,
                           const int32_t* block_table, int64_t block_table_stride, int32_t max_blocks,
                           const int32_t* seq_lens, int32_t kv_lora_rank, int32_t rope_dim, float softmax_scale,
                           mla_tensor w_uv, int32_t num_splits, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Bytes of workspace mla_decode_v_up needs. */
size_t mla_decode_v_up_workspace_size(int32_t batch, int32_t num_heads, int32_t kv_lora_rank,
                                      int32_t num_splits);

/* Bytes of the static scratch behind mla_decode_noalloc (40 MiB). */
#define MLA_DECODE_NOALLOC_SCRATCH_BYTES (40u * 1024u * 1024u)

/* mla_decode without a workspace, for callers that cannot allocate device
 * memory: code running inside another framework's memory pool, plugins whose
 * host forbids cudaMalloc on the hot path (it synchronises the device and can
 * fail under memory pressure), runtimes that reserve all device memory up
 * front. The source pages have no counterpart of this call.
 *   Arguments, results and errors are those of mla_decode minus the workspace.
 *   The split-KV scratch lives in a static device array of
 *   MLA_DECODE_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds
 *   until the process exits; a batch whose scratch would not fit (about
 *   (B + work units) * H * L * 4 bytes) returns MLA_ERR_UNSUPPORTED. The call
 *   allocates nothing. Its first call on a device looks up the array's device
 *   address (once per device and context: again after a reset of the device);
 *   make that first call before any stream capture.
 *   All calls share the array: calls whose kernels overlap on the GPU race and
 *   must be serialised by the caller. */
mla_status mla_decode_noalloc(mla_dtype dtype, mla_tensor o_lat_out, float* lse_out,
                              mla_tensor q_cat, mla_tensor cache, const int32_t* block_table,
                              int64_t block_table_stride, int32_t max_blocks,
                              const int32_t* seq_lens, int32_t kv_lora_rank, int32_t rope_dim,
                              float softmax_scale, int32_t num_splits, void* stream);

/* Synchronises `stream`, then reports and clears the device-side error words the
 * kernels set (out-of-range slot, block id or length: MLA_ERR_DEVICE_DATA; a
 * bounded wait that gave up: MLA_ERR_TIMEOUT). MLA_OK if none was set. */
mla_status mla_device_error(void* stream);

/* Self-check of failure detection. Every wait in the library's kernels is
 * bounded in time: a wait that gives up records MLA_ERR_TIMEOUT for
 * mla_device_error and the kernel winds down, so a stuck pipeline never hangs
 * the GPU. This call launches one warp that runs that same bounded wait on an
 * mbarrier nothing ever arrives on, with a limit of limit_us microseconds
 * (1 .. 1000000) instead of the kernels' 2 s; afterwards mla_device_error on
 * the same stream reports MLA_ERR_TIMEOUT (and clears it) while the context
 * stays usable. Returns MLA_ERR_INVALID_ARG for a limit out of range. The
 * source pages have no counterpart of this call. */
mla_status mla_check_bounded_wait(uint32_t limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
