// Host side of the C ABI: argument validation, dispatch, error reporting.
// Nothing in this file touches device memory except through the launchers.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "mla_internal.h"

namespace mla {

namespace {
thread_local char g_msg[512] = "";

mla_status fail(mla_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

mla_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MLA_OK;
  return fail(MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int64_t numel(const mla_tensor& t) {
  int64_t n = 1;
  for (int i = 0; i < t.rank; ++i) n *= t.shape[i];
  return n;
}

// Well-formedness of one view: rank, non-negative sizes, non-null data when
// non-empty, innermost stride 1 (the one layout rule the source tests assert).
mla_status check_view(const mla_tensor& t, int rank, const char* name) {
  if (t.rank != rank) return fail(MLA_ERR_INVALID_ARG, "%s: rank %d, expected %d", name, t.rank, rank);
  for (int i = 0; i < rank; ++i)
    if (t.shape[i] < 0) return fail(MLA_ERR_INVALID_ARG, "%s: negative shape[%d]", name, i);
  if (numel(t) == 0) return MLA_OK;
  if (t.data == nullptr) return fail(MLA_ERR_INVALID_ARG, "%s: null data", name);
  if (t.stride[rank - 1] != 1)
    return fail(MLA_ERR_INVALID_ARG, "%s: innermost stride %lld, must be 1", name,
                (long long)t.stride[rank - 1]);
  for (int i = 0; i < rank - 1; ++i)
    if (t.stride[i] < 0) return fail(MLA_ERR_INVALID_ARG, "%s: negative stride[%d]", name, i);
  return MLA_OK;
}

#define MLA_TRY(expr)                 \
  do {                                \
    mla_status s__ = (expr);          \
    if (s__ != MLA_OK) return s__;    \
  } while (0)

mla_status check_dtype(mla_dtype dt) {
  if (dt != MLA_F32 && dt != MLA_BF16) return fail(MLA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  return MLA_OK;
}

// Shared validation of the three bmm operands: out [G,M,N] = a [G,M,K] @ b [G,K,N].
mla_status check_bmm(const mla_tensor& out, const mla_tensor& a, const mla_tensor& b,
                     const char* on, const char* an, const char* bn) {
  MLA_TRY(check_view(out, 3, on));
  MLA_TRY(check_view(a, 3, an));
  MLA_TRY(check_view(b, 3, bn));
  if (a.shape[0] != b.shape[0] || out.shape[0] != a.shape[0])
    return fail(MLA_ERR_INVALID_ARG, "batch (head) mismatch: %s %lld, %s %lld, %s %lld", an,
                (long long)a.shape[0], bn, (long long)b.shape[0], on, (long long)out.shape[0]);
  if (a.shape[2] != b.shape[1])
    return fail(MLA_ERR_INVALID_ARG, "inner dimension mismatch: %s K=%lld, %s K=%lld", an,
                (long long)a.shape[2], bn, (long long)b.shape[1]);
  if (out.shape[1] != a.shape[1] || out.shape[2] != b.shape[2])
    return fail(MLA_ERR_INVALID_ARG, "%s shape [%lld,%lld,%lld] does not match the product", on,
                (long long)out.shape[0], (long long)out.shape[1], (long long)out.shape[2]);
  if (a.shape[2] > 4096) return fail(MLA_ERR_UNSUPPORTED, "inner dimension %lld > 4096", (long long)a.shape[2]);
  if (a.shape[0] > 65535 || a.shape[1] > 65535LL * 8 || b.shape[2] > INT32_MAX / 2)
    return fail(MLA_ERR_UNSUPPORTED, "bmm shape beyond the launch limits");
  return MLA_OK;
}

mla_status check_cache(const mla_tensor& cache, int64_t E, const char* name) {
  MLA_TRY(check_view(cache, 3, name));
  if (cache.shape[2] != E)
    return fail(MLA_ERR_INVALID_ARG, "%s: entry width %lld, expected L+R = %lld", name,
                (long long)cache.shape[2], (long long)E);
  if (cache.shape[1] <= 0 || cache.shape[0] <= 0)
    return fail(MLA_ERR_INVALID_ARG, "%s: empty cache", name);
  if (cache.shape[0] > INT32_MAX || cache.shape[1] > INT32_MAX)
    return fail(MLA_ERR_UNSUPPORTED, "%s: too many blocks or rows per block", name);
  return MLA_OK;
}

}  // namespace

mla_status report_status(mla_status st, const char* fmt, ...) {
  if (st == MLA_OK || fmt == nullptr) {
    g_msg[0] = 0;
    return st;
  }
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

DecodeWsLayout decode_ws_layout(int64_t B, int64_t H, int64_t L, int64_t units) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  DecodeWsLayout l{};
  size_t off = 0;
  l.off_prefix = off; off = up(off + sizeof(int32_t) * (B + 1));
  l.off_first = off;  off = up(off + sizeof(int32_t) * B);
  l.off_np = off;     off = up(off + sizeof(int32_t) * B);
  l.off_base = off;   off = up(off + sizeof(int32_t) * B);
  l.off_unit = off;   off = up(off + sizeof(int32_t) * (units + 1));
  l.off_useq = off;   off = up(off + sizeof(int32_t) * units);
  l.off_seqinfo = off; off = up(off + sizeof(int4) * B);
  const int64_t pieces = B + units;
  l.off_part_o = off;   off = up(off + sizeof(float) * pieces * H * L);
  l.off_part_lse = off; off = up(off + sizeof(float) * pieces * H);
  l.total = off;
  return l;
}

DecodeSched decode_sched_from_ws(void* ws, const DecodeWsLayout& lay, int32_t B, int32_t units) {
  char* p = static_cast<char*>(ws);
  DecodeSched s;
  s.tile_prefix = reinterpret_cast<int32_t*>(p + lay.off_prefix);
  s.first_unit = reinterpret_cast<int32_t*>(p + lay.off_first);
  s.npieces = reinterpret_cast<int32_t*>(p + lay.off_np);
  s.piece_base = reinterpret_cast<int32_t*>(p + lay.off_base);
  s.unit_tile = reinterpret_cast<int32_t*>(p + lay.off_unit);
  s.unit_seq = reinterpret_cast<int32_t*>(p + lay.off_useq);
  s.seqinfo = reinterpret_cast<int4*>(p + lay.off_seqinfo);
  s.part_o = reinterpret_cast<float*>(p + lay.off_part_o);
  s.part_lse = reinterpret_cast<float*>(p + lay.off_part_lse);
  s.units = units;
  s.max_pieces = B + units;
  return s;
}

int device_sm_count() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> g(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// bmm on the tensor cores when the shape and layout allow, else on CUDA cores.
static cudaError_t launch_bmm(mla_dtype dt, const View3& out, const View3& a, const View3& b, cudaStream_t st) {
  if (bmm_tc_supported(dt, out, a, b)) return launch_bmm_tc(out, a, b, st);
  return launch_bmm_simt(dt, out, a, b, st);
}

// Work units of the general split-KV decode: explicit, or two per SM.
int32_t decode_units(int32_t num_splits) {
  if (num_splits > 0) return num_splits;
  return 2 * device_sm_count();
}

// The argument checks of the q concat; on MLA_OK *out holds the views to copy (when nope is
// q_cat_out's own first L columns, only the rope columns remain to move).
mla_status plan_concat(mla_dtype dtype, const mla_tensor& q_cat_out, const mla_tensor& nope,
                       const mla_tensor& rope, ConcatPlan* out) {
  MLA_TRY(check_dtype(dtype));
  MLA_TRY(check_view(q_cat_out, 3, "q_cat_out"));
  MLA_TRY(check_view(nope, 3, "nope"));
  MLA_TRY(check_view(rope, 3, "rope"));
  const int64_t T = q_cat_out.shape[0], H = q_cat_out.shape[1];
  if (nope.shape[0] != T || nope.shape[1] != H)
    return fail(MLA_ERR_INVALID_ARG, "nope [%lld,%lld,.] does not match q_cat_out [%lld,%lld,.]",
                (long long)nope.shape[0], (long long)nope.shape[1], (long long)T, (long long)H);
  if (rope.shape[0] != T || (rope.shape[1] != H && rope.shape[1] != 1))
    return fail(MLA_ERR_INVALID_ARG, "rope must be [T,H,R] or [T,1,R]");
  if (nope.shape[2] + rope.shape[2] != q_cat_out.shape[2])
    return fail(MLA_ERR_INVALID_ARG, "q_cat_out width %lld != L + R = %lld",
                (long long)q_cat_out.shape[2], (long long)(nope.shape[2] + rope.shape[2]));
  out->empty = numel(q_cat_out) == 0;
  if (out->empty) return MLA_OK;
  View3 r = view3(rope);
  if (rope.shape[1] == 1) r.s1 = 0;  // one rope head broadcast to every head
  r.n1 = H;
  View3 o = view3(q_cat_out), nv = view3(nope);
  if (nope.data == q_cat_out.data && nope.stride[0] == q_cat_out.stride[0] &&
      nope.stride[1] == q_cat_out.stride[1] && nope.stride[2] == q_cat_out.stride[2]) {
    // nope is q_cat_out's own first L columns (the absorb wrote q_lat in place): they are
    // already there, only the rope columns move
    const size_t es = dtype == MLA_F32 ? 4 : 2;
    o.data = static_cast<char*>(o.data) + es * (size_t)nope.shape[2];
    o.n2 = rope.shape[2];
    nv.n2 = 0;
    if (rope.shape[2] == 0) out->empty = true;
  }
  out->out = o;
  out->nope = nv;
  out->rope = r;
  return MLA_OK;
}

// The argument checks of the cache write; on MLA_OK *out holds the views.
mla_status plan_cache_write(mla_dtype dtype, const mla_tensor& cache, const mla_tensor& kv_c,
                            const mla_tensor& k_pe, const int64_t* slot_mapping, int64_t num_tokens,
                            WritePlan* out) {
  MLA_TRY(check_dtype(dtype));
  if (num_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "num_tokens < 0");
  MLA_TRY(check_view(kv_c, 2, "kv_c"));
  MLA_TRY(check_view(k_pe, 2, "k_pe"));
  const int64_t L = kv_c.shape[1], R = k_pe.shape[1];
  MLA_TRY(check_cache(cache, L + R, "cache"));
  if (kv_c.shape[0] != num_tokens || k_pe.shape[0] != num_tokens)
    return fail(MLA_ERR_INVALID_ARG, "kv_c/k_pe rows (%lld/%lld) != num_tokens %lld",
                (long long)kv_c.shape[0], (long long)k_pe.shape[0], (long long)num_tokens);
  out->empty = num_tokens == 0;
  if (out->empty) return MLA_OK;
  if (slot_mapping == nullptr) return fail(MLA_ERR_INVALID_ARG, "slot_mapping is null");
  out->L = L;
  out->R = R;
  out->cache = view3(cache);
  out->kv_c = View3{kv_c.data, kv_c.shape[0], 1, kv_c.shape[1], kv_c.stride[0], 0, 1};
  out->k_pe = View3{k_pe.data, k_pe.shape[0], 1, k_pe.shape[1], k_pe.stride[0], 0, 1};
  return MLA_OK;
}

mla_status check_decode_args(mla_dtype dtype, const mla_tensor& o_lat_out, const mla_tensor& q_cat,
                             const mla_tensor& cache, const int32_t* block_table, int64_t block_table_stride,
                             int32_t max_blocks, const int32_t* seq_lens, int32_t kv_lora_rank, int32_t rope_dim,
                             float softmax_scale, int32_t num_splits, DecodeCall* out) {
  MLA_TRY(check_dtype(dtype));
  MLA_TRY(check_view(q_cat, 3, "q_cat"));
  MLA_TRY(check_view(o_lat_out, 3, "o_lat_out"));
  const int64_t B = q_cat.shape[0], H = q_cat.shape[1];
  const int64_t L = kv_lora_rank, R = rope_dim;
  if (L <= 0 || R < 0) return fail(MLA_ERR_INVALID_ARG, "kv_lora_rank must be > 0 and rope_dim >= 0");
  if (q_cat.shape[2] != L + R)
    return fail(MLA_ERR_INVALID_ARG, "q_cat width %lld != L + R = %lld", (long long)q_cat.shape[2],
                (long long)(L + R));
  if (o_lat_out.shape[0] != B || o_lat_out.shape[1] != H || o_lat_out.shape[2] != L)
    return fail(MLA_ERR_INVALID_ARG, "o_lat_out must be [B,H,L] = [%lld,%lld,%lld]", (long long)B,
                (long long)H, (long long)L);
  MLA_TRY(check_cache(cache, L + R, "cache"));
  if (num_splits < 0) return fail(MLA_ERR_INVALID_ARG, "num_splits < 0");
  out->B = B;
  out->H = H;
  out->L = L;
  out->R = R;
  out->empty = B == 0 || H == 0;
  if (out->empty) return MLA_OK;
  if (B > INT32_MAX / 2 || H > 4096) return fail(MLA_ERR_UNSUPPORTED, "batch or head count too large");
  if (block_table == nullptr || seq_lens == nullptr)
    return fail(MLA_ERR_INVALID_ARG, "block_table and seq_lens must be non-null");
  if (max_blocks <= 0 || block_table_stride < max_blocks)
    return fail(MLA_ERR_INVALID_ARG, "need 0 < max_blocks <= block_table_stride");
  if (L > 512) return fail(MLA_ERR_UNSUPPORTED, "kv_lora_rank %lld > 512", (long long)L);
  if (L + R > 1024) return fail(MLA_ERR_UNSUPPORTED, "entry width %lld > 1024", (long long)(L + R));
  out->cv = CacheView{cache.data, cache.stride[0], cache.stride[1], (int32_t)cache.shape[0],
                      (int32_t)cache.shape[1], (int32_t)cache.shape[2]};
  out->qv = view3(q_cat);
  out->ov = view3(o_lat_out);
  out->tc = softmax_scale > 0.f &&
            tc_attention_supported(dtype, (int)H, (int)L, (int)R, true, out->cv, out->qv, out->ov);
  // work units: one per 2-CTA cluster on the tensor-core path, else from num_splits
  out->units = out->tc ? tc_decode_units(num_splits) : decode_units(num_splits);
  return MLA_OK;
}

mla_status run_decode(mla_dtype dtype, const DecodeCall& dc, float* lse_out, const int32_t* block_table,
                      int64_t block_table_stride, int32_t max_blocks, const int32_t* seq_lens, float softmax_scale,
                      void* scratch, const DecodeWsLayout& lay, cudaStream_t st, bool fp8_cache,
                      const float* descale_q, const float* descale_k, bool combine) {
  const DecodeSched s = decode_sched_from_ws(scratch, lay, (int32_t)dc.B, dc.units);
  const int32_t B = (int32_t)dc.B, H = (int32_t)dc.H, L = (int32_t)dc.L, R = (int32_t)dc.R;
  MLA_TRY(cuda_status(launch_decode_schedule(seq_lens, B, max_blocks, dc.cv.page, s, st), "mla_decode schedule"));
  if (dc.tc && fp8_cache) {
    MLA_TRY(cuda_status(launch_decode_tc_fp8(dc.ov, lse_out, dc.qv, dc.cv, block_table, block_table_stride,
                                             max_blocks, B, H, R, softmax_scale, descale_q, descale_k, s, st),
                        "mla_decode split kernel (tensor cores, e4m3 cache)"));
  } else if (dc.tc) {
    MLA_TRY(cuda_status(launch_decode_tc(dc.ov, lse_out, dc.qv, dc.cv, block_table, block_table_stride,
                                         max_blocks, seq_lens, B, H, L, R, softmax_scale, s, st),
                        "mla_decode split kernel (tensor cores)"));
  } else {
    MLA_TRY(cuda_status(launch_decode_simt(dtype, dc.ov, lse_out, dc.qv, dc.cv, block_table, block_table_stride,
                                           max_blocks, seq_lens, B, H, L, R, softmax_scale, s, st, fp8_cache,
                                           descale_q, descale_k),
                        "mla_decode split kernel"));
  }
  if (!combine) return MLA_OK;
  return cuda_status(launch_decode_combine(dtype, dc.ov, lse_out, seq_lens, B, H, L, s, st), "mla_decode combine");
}

}  // namespace mla

using namespace mla;

extern "C" {

int mla_abi_version(void) { return MLA_ABI_VERSION; }

const char* mla_last_error(void) { return g_msg; }

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_DEVICE_DATA: return "MLA_ERR_DEVICE_DATA";
  }
  return "MLA_ERR_UNKNOWN";
}

mla_status mla_absorb_q(mla_dtype dtype, mla_tensor q_lat_out, mla_tensor q_nope, mla_tensor w_uk,
                        void* stream) {
  g_msg[0] = 0;
  MLA_TRY(check_dtype(dtype));
  MLA_TRY(check_bmm(q_lat_out, q_nope, w_uk, "q_lat_out", "q_nope", "w_uk"));
  if (numel(q_lat_out) == 0) return MLA_OK;
  return cuda_status(launch_bmm(dtype, view3(q_lat_out), view3(q_nope), view3(w_uk), (cudaStream_t)stream),
                     "mla_absorb_q");
}

mla_status mla_v_up(mla_dtype dtype, mla_tensor out, mla_tensor o_lat, mla_tensor w_uv,
                    void* stream) {
  g_msg[0] = 0;
  MLA_TRY(check_dtype(dtype));
  MLA_TRY(check_bmm(out, o_lat, w_uv, "out", "o_lat", "w_uv"));
  if (numel(out) == 0) return MLA_OK;
  return cuda_status(launch_bmm(dtype, view3(out), view3(o_lat), view3(w_uv), (cudaStream_t)stream),
                     "mla_v_up");
}

mla_status mla_concat_q(mla_dtype dtype, mla_tensor q_cat_out, mla_tensor nope, mla_tensor rope,
                        void* stream) {
  g_msg[0] = 0;
  ConcatPlan cp;
  MLA_TRY(plan_concat(dtype, q_cat_out, nope, rope, &cp));
  if (cp.empty) return MLA_OK;
  return cuda_status(launch_concat_q(dtype, cp.out, cp.nope, cp.rope, (cudaStream_t)stream), "mla_concat_q");
}

mla_status mla_cache_write(mla_dtype dtype, mla_tensor cache, mla_tensor kv_c, mla_tensor k_pe,
                           const int64_t* slot_mapping, int64_t num_tokens, void* stream) {
  g_msg[0] = 0;
  WritePlan wp;
  MLA_TRY(plan_cache_write(dtype, cache, kv_c, k_pe, slot_mapping, num_tokens, &wp));
  if (wp.empty) return MLA_OK;
  return cuda_status(launch_cache_write(dtype, wp.cache, wp.kv_c, wp.k_pe, wp.L, wp.R, slot_mapping, num_tokens,
                                        (cudaStream_t)stream), "mla_cache_write");
}

mla_status mla_concat_q_cache_write(mla_dtype dtype, mla_tensor q_cat_out, mla_tensor nope, mla_tensor rope,
                                    mla_tensor cache, mla_tensor kv_c, mla_tensor k_pe,
                                    const int64_t* slot_mapping, int64_t num_tokens, void* stream) {
  g_msg[0] = 0;
  ConcatPlan cp;
  MLA_TRY(plan_concat(dtype, q_cat_out, nope, rope, &cp));
  WritePlan wp;
  MLA_TRY(plan_cache_write(dtype, cache, kv_c, k_pe, slot_mapping, num_tokens, &wp));
  if (cp.empty && wp.empty) return MLA_OK;
  View3 out = cp.out, nv = cp.nope, rv = cp.rope;
  if (cp.empty) {   // nothing to concatenate: an empty q part
    out.n0 = 0;
    nv.n2 = 0;
    rv.n2 = 0;
  }
  return cuda_status(launch_concat_cache(dtype, out, nv, rv, wp.cache, wp.kv_c, wp.k_pe, wp.L, wp.R, slot_mapping,
                                         wp.empty ? 0 : num_tokens, (cudaStream_t)stream),
                     "mla_concat_q_cache_write");
}

mla_status mla_absorb_concat_cache_write(mla_dtype dtype, mla_tensor q_cat, mla_tensor q_nope, mla_tensor w_uk,
                                         mla_tensor q_pe, mla_tensor cache, mla_tensor kv_c, mla_tensor k_pe,
                                         const int64_t* slot_mapping, int64_t num_tokens, void* stream) {
  g_msg[0] = 0;
  MLA_TRY(check_dtype(dtype));
  MLA_TRY(check_view(q_cat, 3, "q_cat"));
  MLA_TRY(check_view(w_uk, 3, "w_uk"));
  const int64_t L = w_uk.shape[2];
  if (L > q_cat.shape[2])
    return fail(MLA_ERR_INVALID_ARG, "w_uk's latent width %lld exceeds q_cat's width %lld", (long long)L,
                (long long)q_cat.shape[2]);
  // the absorb writes q_cat's first L columns, seen as [H, T, L]
  mla_tensor lat = q_cat;
  lat.shape[0] = q_cat.shape[1];
  lat.shape[1] = q_cat.shape[0];
  lat.shape[2] = L;
  lat.stride[0] = q_cat.stride[1];
  lat.stride[1] = q_cat.stride[0];
  MLA_TRY(check_bmm(lat, q_nope, w_uk, "q_cat", "q_nope", "w_uk"));
  // the concat with q_cat's own first L columns as its nope operand: only the rope moves
  mla_tensor nope = q_cat;
  nope.shape[2] = L;
  ConcatPlan cp;
  MLA_TRY(plan_concat(dtype, q_cat, nope, q_pe, &cp));
  WritePlan wp;
  MLA_TRY(plan_cache_write(dtype, cache, kv_c, k_pe, slot_mapping, num_tokens, &wp));
  const cudaStream_t st = (cudaStream_t)stream;
  const bool absorb = numel(lat) > 0;
  if (absorb) MLA_TRY(cuda_status(launch_bmm(dtype, view3(lat), view3(q_nope), view3(w_uk), st),
                                  "mla_absorb_concat_cache_write absorb"));
  if (cp.empty && wp.empty) return MLA_OK;
  View3 out = cp.out, nv = cp.nope, rv = cp.rope;
  if (cp.empty) {   // nothing to concatenate: an empty q part
    out.n0 = 0;
    nv.n2 = 0;
    rv.n2 = 0;
  }
  // the copies touch q_cat's rope columns and the cache, none of the absorb's operands or its
  // output: they run alongside it
  return cuda_status(launch_concat_cache(dtype, out, nv, rv, wp.cache, wp.kv_c, wp.k_pe, wp.L, wp.R, slot_mapping,
                                         wp.empty ? 0 : num_tokens, st, absorb),
                     "mla_absorb_concat_cache_write copies");
}

size_t mla_decode_workspace_size(int32_t batch, int32_t num_heads, int32_t kv_lora_rank,
                                 int32_t num_splits) {
  if (batch < 0 || num_heads < 0 || kv_lora_rank < 0 || num_splits < 0) return 0;
  return decode_ws_layout(batch, num_heads, kv_lora_rank, decode_units(num_splits)).total;
}

mla_status mla_decode(mla_dtype dtype, mla_tensor o_lat_out, float* lse_out, mla_tensor q_cat,
                      mla_tensor cache, const int32_t* block_table, int64_t block_table_stride,
                      int32_t max_blocks, const int32_t* seq_lens, int32_t kv_lora_rank,
                      int32_t rope_dim, float softmax_scale, int32_t num_splits, void* workspace,
                      size_t workspace_bytes, void* stream) {
  g_msg[0] = 0;
  DecodeCall dc;
  MLA_TRY(check_decode_args(dtype, o_lat_out, q_cat, cache, block_table, block_table_stride, max_blocks,
                            seq_lens, kv_lora_rank, rope_dim, softmax_scale, num_splits, &dc));
  if (dc.empty) return MLA_OK;
  // the workspace is sized for the general work-unit count, which covers the tensor-core one
  const DecodeWsLayout lay = decode_ws_layout(dc.B, dc.H, dc.L, decode_units(num_splits));
  if (workspace == nullptr || workspace_bytes < lay.total)
    return fail(MLA_ERR_INVALID_ARG, "workspace too small: %zu bytes, need %zu", workspace_bytes,
                lay.total);
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(MLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  return run_decode(dtype, dc, lse_out, block_table, block_table_stride, max_blocks, seq_lens, softmax_scale,
                    workspace, lay, (cudaStream_t)stream);
}

mla_status mla_cache_write_fp8(mla_dtype src_dtype, mla_tensor cache, mla_tensor kv_c, mla_tensor k_pe,
                               const int64_t* slot_mapping, int64_t num_tokens, const float* scale,
                               void* stream) {
  g_msg[0] = 0;
  MLA_TRY(check_dtype(src_dtype));
  if (num_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "num_tokens < 0");
  MLA_TRY(check_view(kv_c, 2, "kv_c"));
  MLA_TRY(check_view(k_pe, 2, "k_pe"));
  const int64_t L = kv_c.shape[1], R = k_pe.shape[1];
  MLA_TRY(check_cache(cache, L + R, "cache"));
  if (kv_c.shape[0] != num_tokens || k_pe.shape[0] != num_tokens)
    return fail(MLA_ERR_INVALID_ARG, "kv_c/k_pe rows (%lld/%lld) != num_tokens %lld",
                (long long)kv_c.shape[0], (long long)k_pe.shape[0], (long long)num_tokens);
  if (num_tokens == 0) return MLA_OK;
  if (slot_mapping == nullptr || scale == nullptr)
    return fail(MLA_ERR_INVALID_ARG, "slot_mapping and scale must be non-null");
  View3 kc{kv_c.data, kv_c.shape[0], 1, kv_c.shape[1], kv_c.stride[0], 0, 1};
  View3 kp{k_pe.data, k_pe.shape[0], 1, k_pe.shape[1], k_pe.stride[0], 0, 1};
  return cuda_status(launch_cache_write_fp8(src_dtype, view3(cache), kc, kp, L, R, slot_mapping, num_tokens, scale,
                                            (cudaStream_t)stream),
                     "mla_cache_write_fp8");
}

mla_status mla_decode_fp8(mla_dtype dtype, mla_tensor o_lat_out, float* lse_out, mla_tensor q_cat,
                          mla_tensor cache, const int32_t* block_table, int64_t block_table_stride,
                          int32_t max_blocks, const int32_t* seq_lens, int32_t kv_lora_rank, int32_t rope_dim,
                          float softmax_scale, const float* descale_q, const float* descale_k,
                          int32_t num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  g_msg[0] = 0;
  DecodeCall dc;
  MLA_TRY(check_decode_args(dtype, o_lat_out, q_cat, cache, block_table, block_table_stride, max_blocks,
                            seq_lens, kv_lora_rank, rope_dim, softmax_scale, num_splits, &dc));
  if (dc.empty) return MLA_OK;
  // the tensor-core kernel gathers e4m3 rows with 16-byte copies and converts them to bf16
  dc.tc = softmax_scale > 0.f && dc.L == 512 && (dc.R == 0 || dc.R == 64) &&
          tc_gather_supported(dtype, (int)dc.H, dc.cv.data, dc.cv.s_blk, dc.cv.s_row, dc.qv, dc.ov);
  dc.units = dc.tc ? tc_decode_units(num_splits) : decode_units(num_splits);
  const DecodeWsLayout lay = decode_ws_layout(dc.B, dc.H, dc.L, decode_units(num_splits));
  if (workspace == nullptr || workspace_bytes < lay.total)
    return fail(MLA_ERR_INVALID_ARG, "workspace too small: %zu bytes, need %zu", workspace_bytes,
                lay.total);
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(MLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  return run_decode(dtype, dc, lse_out, block_table, block_table_stride, max_blocks, seq_lens, softmax_scale,
                    workspace, lay, (cudaStream_t)stream, true, descale_q, descale_k);
}

namespace {
// The sparse decode's workspace: mla_decode's layout, then the compacted slots [B, topk] and
// their counts [B].
struct SparseWs {
  DecodeWsLayout lay;
  size_t off_slots, off_counts, total;
};
SparseWs sparse_ws(int64_t B, int64_t H, int64_t topk, int32_t units) {
  SparseWs w;
  w.lay = decode_ws_layout(B, H, kDsMlaLatent, units);
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  w.off_slots = up(w.lay.total);
  w.off_counts = up(w.off_slots + (size_t)B * (size_t)topk * 4);
  w.total = up(w.off_counts + (size_t)B * 4);
  return w;
}
}  // namespace

size_t mla_decode_sparse_workspace_size(int32_t batch, int32_t num_heads, int32_t topk, int32_t num_splits) {
  if (batch < 0 || num_heads < 0 || topk < 0 || num_splits < 0) return 0;
  return sparse_ws(batch, num_heads, topk, decode_units(num_splits)).total;
}

mla_status mla_decode_sparse_fp8(mla_dtype dtype, mla_tensor o_lat_out, float* lse_out, mla_tensor q_cat,
                                 mla_tensor cache, const int32_t* indices, int64_t indices_stride,
                                 int32_t topk, float softmax_scale, int32_t num_splits, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  g_msg[0] = 0;
  MLA_TRY(check_dtype(dtype));
  MLA_TRY(check_view(q_cat, 3, "q_cat"));
  MLA_TRY(check_view(o_lat_out, 3, "o_lat_out"));
  const int64_t B = q_cat.shape[0], H = q_cat.shape[1];
  if (q_cat.shape[2] != kDsMlaLatent + kDsMlaRope)
    return fail(MLA_ERR_INVALID_ARG, "q_cat width %lld, a ds_mla query is 576 wide", (long long)q_cat.shape[2]);
  if (o_lat_out.shape[0] != B || o_lat_out.shape[1] != H || o_lat_out.shape[2] != kDsMlaLatent)
    return fail(MLA_ERR_INVALID_ARG, "o_lat_out must be [B,H,512] = [%lld,%lld,512]", (long long)B, (long long)H);
  MLA_TRY(check_cache(cache, kDsMlaEntry, "cache"));
  if (reinterpret_cast<uintptr_t>(cache.data) % 16 != 0 || cache.stride[0] % 16 != 0 || cache.stride[1] % 16 != 0)
    return fail(MLA_ERR_INVALID_ARG, "cache: data and strides must be 16-byte aligned");
  if (cache.shape[0] * cache.shape[1] > INT32_MAX)
    return fail(MLA_ERR_UNSUPPORTED, "cache: more slots than an int32 index can name");
  if (topk < 0) return fail(MLA_ERR_INVALID_ARG, "topk < 0");
  if (num_splits < 0) return fail(MLA_ERR_INVALID_ARG, "num_splits < 0");
  if (B == 0 || H == 0) return MLA_OK;
  if (B > INT32_MAX / 2 || H > 4096) return fail(MLA_ERR_UNSUPPORTED, "batch or head count too large");
  if (topk > 0 && (indices == nullptr || indices_stride < topk))
    return fail(MLA_ERR_INVALID_ARG, "indices must be non-null with a row stride >= topk");
  const SparseWs ws = sparse_ws(B, H, topk, decode_units(num_splits));
  if (workspace == nullptr || workspace_bytes < ws.total)
    return fail(MLA_ERR_INVALID_ARG, "workspace too small: %zu bytes, need %zu", workspace_bytes, ws.total);
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(MLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const cudaStream_t st = (cudaStream_t)stream;
  const DsMlaCache cv{cache.data, cache.stride[0], cache.stride[1], (int32_t)cache.shape[0], (int32_t)cache.shape[1]};
  const View3 ov = view3(o_lat_out), qv = view3(q_cat);
  const bool tc = softmax_scale > 0.f && topk > 0 &&
                  tc_gather_supported(dtype, (int)H, cache.data, cache.stride[0], cache.stride[1], qv, ov);
  const int32_t units = tc ? tc_decode_units(num_splits) : decode_units(num_splits);
  const DecodeSched s = decode_sched_from_ws(workspace, ws.lay, (int32_t)B, units);
  if (tc) {
    // the tensor-core kernel takes each query's valid slots, compacted, as a sequence of
    // count rows
    int32_t* slots = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + ws.off_slots);
    int32_t* counts = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + ws.off_counts);
    MLA_TRY(cuda_status(launch_sparse_compact(indices, indices_stride, topk, (int32_t)B,
                                              (int64_t)cv.num_blocks * cv.page, slots, counts, st),
                        "mla_decode_sparse_fp8 slot compaction"));
    MLA_TRY(cuda_status(launch_decode_schedule(counts, (int32_t)B, topk, 1, s, st), "mla_decode_sparse_fp8 schedule"));
    MLA_TRY(cuda_status(launch_decode_tc_dsmla(ov, lse_out, qv, cv, slots, topk, topk, (int32_t)B, (int32_t)H,
                                               softmax_scale, s, st),
                        "mla_decode_sparse_fp8 split kernel (tensor cores)"));
  } else {
    // every query has topk listed rows: the schedule's lengths are all topk (cap topk, page 1)
    MLA_TRY(cuda_status(launch_decode_schedule(nullptr, (int32_t)B, topk, 1, s, st), "mla_decode_sparse_fp8 schedule"));
    MLA_TRY(cuda_status(launch_decode_sparse_simt(dtype, ov, lse_out, qv, cv, indices, indices_stride, topk,
                                                  (int32_t)B, (int32_t)H, softmax_scale, s, st),
                        "mla_decode_sparse_fp8 split kernel"));
  }
  return cuda_status(launch_decode_combine(dtype, ov, lse_out, nullptr, (int32_t)B, (int32_t)H, kDsMlaLatent, s, st),
                     "mla_decode_sparse_fp8 combine");
}

namespace {
// mla_decode_v_up's workspace: mla_decode's layout, then o_lat [B, H, L] (4 bytes an element
// covers both dtypes).
struct VupWs {
  DecodeWsLayout lay;
  size_t off_olat, total;
};
VupWs vup_ws(int64_t B, int64_t H, int64_t L, int32_t units) {
  VupWs w;
  w.lay = decode_ws_layout(B, H, L, units);
  w.off_olat = (w.lay.total + 255) & ~size_t(255);
  w.total = (w.off_olat + (size_t)B * (size_t)H * (size_t)L * 4 + 255) & ~size_t(255);
  return w;
}
}  // namespace

size_t mla_decode_v_up_workspace_size(int32_t batch, int32_t num_heads, int32_t kv_lora_rank, int32_t num_splits) {
  if (batch < 0 || num_heads < 0 || kv_lora_rank < 0 || num_splits < 0) return 0;
  return vup_ws(batch, num_heads, kv_lora_rank, decode_units(num_splits)).total;
}

mla_status mla_decode_v_up(mla_dtype dtype, mla_tensor out, float* lse_out, mla_tensor q_cat, mla_tensor cache,
                           const int32_t* block_table, int64_t block_table_stride, int32_t max_blocks,
                           const int32_t* seq_lens, int32_t kv_lora_rank, int32_t rope_dim, float softmax_scale,
                           mla_tensor w_uv, int32_t num_splits, void* workspace, size_t workspace_bytes,
                           void* stream) {
  g_msg[0] = 0;
  MLA_TRY(check_dtype(dtype));
  MLA_TRY(check_view(q_cat, 3, "q_cat"));
  MLA_TRY(check_view(out, 3, "out"));
  MLA_TRY(check_view(w_uv, 3, "w_uv"));
  const int64_t B = q_cat.shape[0], H = q_cat.shape[1], L = kv_lora_rank, V = out.shape[2];
  if (L <= 0 || rope_dim < 0) return fail(MLA_ERR_INVALID_ARG, "kv_lora_rank must be > 0 and rope_dim >= 0");
  if (num_splits < 0) return fail(MLA_ERR_INVALID_ARG, "num_splits < 0");
  if (out.shape[0] != B || out.shape[1] != H)
    return fail(MLA_ERR_INVALID_ARG, "out must be [B,H,V] = [%lld,%lld,.]", (long long)B, (long long)H);
  if (w_uv.shape[0] != H || w_uv.shape[1] != L || w_uv.shape[2] != V)
    return fail(MLA_ERR_INVALID_ARG, "w_uv must be [H,L,V] = [%lld,%lld,%lld]", (long long)H, (long long)L,
                (long long)V);
  if (B == 0 || H == 0 || V == 0) return MLA_OK;
  const VupWs ws = vup_ws(B, H, L, decode_units(num_splits));
  if (workspace == nullptr || workspace_bytes < ws.total)
    return fail(MLA_ERR_INVALID_ARG, "workspace too small: %zu bytes, need %zu", workspace_bytes, ws.total);
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(MLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  // o_lat, the intermediate, lives in the workspace: [B, H, L] contiguous in dtype
  mla_tensor o_lat{};
  o_lat.data = static_cast<char*>(workspace) + ws.off_olat;
  o_lat.rank = 3;
  o_lat.shape[0] = B;
  o_lat.shape[1] = H;
  o_lat.shape[2] = L;
  o_lat.stride[0] = H * L;
  o_lat.stride[1] = L;
  o_lat.stride[2] = 1;
  DecodeCall dc;
  MLA_TRY(check_decode_args(dtype, o_lat, q_cat, cache, block_table, block_table_stride, max_blocks, seq_lens,
                            kv_lora_rank, rope_dim, softmax_scale, num_splits, &dc));
  const cudaStream_t st = (cudaStream_t)stream;
  MLA_TRY(run_decode(dtype, dc, lse_out, block_table, block_table_stride, max_blocks, seq_lens, softmax_scale,
                     workspace, ws.lay, st, false, nullptr, nullptr, /*combine=*/false));
  const DecodeSched s = decode_sched_from_ws(workspace, ws.lay, (int32_t)B, dc.units);
  const View3 ov = view3(out), wv = view3(w_uv);
  if (combine_vup_supported(dtype, (int)L, (int)V, ov, wv))
    return cuda_status(launch_combine_vup(ov, dc.ov, lse_out, wv, (int32_t)B, (int32_t)H, (int32_t)V, s, st),
                       "mla_decode_v_up combine + v_up");
  // otherwise the two steps as separate kernels: the combine into o_lat, then the bmm
  MLA_TRY(cuda_status(launch_decode_combine(dtype, dc.ov, lse_out, seq_lens, (int32_t)B, (int32_t)H, (int32_t)L, s, st),
                      "mla_decode_v_up combine"));
  const View3 out_hbv{out.data, H, B, V, out.stride[1], out.stride[0], out.stride[2]};
  const View3 o_hbl{dc.ov.data, H, B, L, dc.ov.s1, dc.ov.s0, 1};
  return cuda_status(launch_bmm(dtype, out_hbv, o_hbl, wv, st), "mla_decode_v_up v_up");
}

size_t mla_prefill_workspace_size(int32_t batch) {
  if (batch < 0) return 0;
  return ((size_t)(batch + 1) * sizeof(int32_t) + 255) & ~size_t(255);
}

mla_status mla_prefill(mla_dtype dtype, mla_tensor o_lat_out, float* lse_out, mla_tensor q_cat,
                       mla_tensor cache, const int32_t* block_table, int64_t block_table_stride,
                       int32_t max_blocks, const int32_t* cu_seqlens_q, const int32_t* seq_lens_kv,
                       int32_t batch, int32_t max_q_len, int32_t kv_lora_rank, int32_t rope_dim,
                       float softmax_scale, void* workspace, size_t workspace_bytes,
                       void* stream) {
  g_msg[0] = 0;
  MLA_TRY(check_dtype(dtype));
  MLA_TRY(check_view(q_cat, 3, "q_cat"));
  MLA_TRY(check_view(o_lat_out, 3, "o_lat_out"));
  const int64_t T = q_cat.shape[0], H = q_cat.shape[1];
  const int64_t L = kv_lora_rank, R = rope_dim;
  if (L <= 0 || R < 0) return fail(MLA_ERR_INVALID_ARG, "kv_lora_rank must be > 0 and rope_dim >= 0");
  if (q_cat.shape[2] != L + R) return fail(MLA_ERR_INVALID_ARG, "q_cat width != L + R");
  if (o_lat_out.shape[0] != T || o_lat_out.shape[1] != H || o_lat_out.shape[2] != L)
    return fail(MLA_ERR_INVALID_ARG, "o_lat_out must be [T,H,L]");
  MLA_TRY(check_cache(cache, L + R, "cache"));
  if (batch < 0 || max_q_len < 0) return fail(MLA_ERR_INVALID_ARG, "batch and max_q_len must be >= 0");
  if (T == 0 || H == 0 || batch == 0) return MLA_OK;
  if (T > INT32_MAX / 2 || H > 4096) return fail(MLA_ERR_UNSUPPORTED, "token or head count too large");
  if (block_table == nullptr || cu_seqlens_q == nullptr || seq_lens_kv == nullptr)
    return fail(MLA_ERR_INVALID_ARG, "block_table, cu_seqlens_q and seq_lens_kv must be non-null");
  if (max_blocks <= 0 || block_table_stride < max_blocks)
    return fail(MLA_ERR_INVALID_ARG, "need 0 < max_blocks <= block_table_stride");
  if (L > 512) return fail(MLA_ERR_UNSUPPORTED, "kv_lora_rank %lld > 512", (long long)L);
  if (L + R > 1024) return fail(MLA_ERR_UNSUPPORTED, "entry width > 1024");
  if (workspace == nullptr || workspace_bytes < mla_prefill_workspace_size(batch))
    return fail(MLA_ERR_INVALID_ARG, "workspace too small: %zu bytes, need %zu", workspace_bytes,
                mla_prefill_workspace_size(batch));
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(MLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const CacheView cv{cache.data, cache.stride[0], cache.stride[1], (int32_t)cache.shape[0],
                     (int32_t)cache.shape[1], (int32_t)cache.shape[2]};
  const View3 qv = view3(q_cat), ov = view3(o_lat_out);
  cudaStream_t st = (cudaStream_t)stream;
  if (softmax_scale > 0.f && tc_attention_supported(dtype, (int)H, (int)L, (int)R, false, cv, qv, ov))
    return cuda_status(launch_prefill_tc(ov, lse_out, qv, cv, block_table, block_table_stride,
                                         max_blocks, cu_seqlens_q, seq_lens_kv, batch, (int32_t)H,
                                         (int32_t)L, (int32_t)R, softmax_scale,
                                         static_cast<int32_t*>(workspace), st),
                       "mla_prefill (tensor cores)");
  return cuda_status(launch_prefill_simt(dtype, ov, lse_out, qv, cv, block_table, block_table_stride,
                                         max_blocks, cu_seqlens_q, seq_lens_kv, batch, (int32_t)T,
                                         (int32_t)H, (int32_t)L, (int32_t)R, softmax_scale, st),
                     "mla_prefill");
}

mla_status mla_check_bounded_wait(uint32_t limit_us, void* stream) {
  g_msg[0] = 0;
  if (limit_us == 0 || limit_us > 1000000u)
    return fail(MLA_ERR_INVALID_ARG, "limit_us must be in [1, 1000000], got %u", limit_us);
  return cuda_status(launch_wait_check(limit_us, (cudaStream_t)stream), "mla_check_bounded_wait");
}

mla_status mla_device_error(void* stream) {
  g_msg[0] = 0;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "mla_device_error: stream synchronize");
  unsigned bits = copy_errors_read_clear() | attn_simt_errors_read_clear() | attn_tc_errors_read_clear() |
                  bmm_tc_errors_read_clear() | combine_vup_errors_read_clear();
  if (bits & kErrTimeout) return fail(MLA_ERR_TIMEOUT, "a bounded device-side wait gave up");
  if (bits & kErrDeviceData)
    return fail(MLA_ERR_DEVICE_DATA, "a slot, block id or sequence length was out of range");
  return MLA_OK;
}

}  // extern "C"
