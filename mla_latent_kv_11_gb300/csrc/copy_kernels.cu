// Step 2 (q concat) and step 3 (paged latent cache write): pure bit copies; and the
// cache write into an fp8 (e4m3) cache, which converts instead of copying.
//
// Both move whole rows. When every row start and row length is a multiple of
// 16 bytes the copy goes in 16-byte vectors (uint4), consecutive lanes on
// consecutive vectors of a row; otherwise it falls back to element copies of
// the same order. The element type never matters: bits are moved as integers, so NaN
// payloads and signed zeros survive unchanged.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "mla_internal.h"

namespace mla {
namespace {

__device__ unsigned g_copy_err = 0;

template <int BYTES> struct Word;
template <> struct Word<16> { using T = uint4; };
template <> struct Word<4> { using T = uint32_t; };
template <> struct Word<2> { using T = uint16_t; };

// Rows are spread over groups of G lanes (G a power of two, 8..32, at least the row's word
// count when that is below 32): a group handles one row, its lanes stride over the row's
// words, so a row's index arithmetic (a 32-bit divide, a slot lookup) is done once per row,
// not once per word, and short rows (the 8 words of the rope columns alone) still fill the
// warp.
struct RowSplit {
  int G;        // lanes per row group
  int shift;    // log2(G)
};

__device__ __forceinline__ void row_lane(const RowSplit rs, int64_t& first_row, int64_t& row_step, int& c0) {
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int per_warp = 32 >> rs.shift;
  first_row = gwarp * per_warp + (lane >> rs.shift);
  row_step = nwarps * per_warp;
  c0 = lane & (rs.G - 1);
}

// One row: words [0, La) from a, [La, E) from b (b already offset by -La), lanes c0, c0 + G,
// ... of a row group. A lane loads up to four words before it stores any, so a row costs one
// memory latency instead of one per word.
template <typename W>
__device__ __forceinline__ void copy_row(W* __restrict__ o, const W* __restrict__ a, const W* __restrict__ b,
                                         int La, int E, int c0, int G) {
  for (int c = c0; c < E; c += 4 * G) {
    W v[4] = {};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int cc = c + u * G;
      if (cc < E) v[u] = cc < La ? a[cc] : b[cc];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int cc = c + u * G;
      if (cc < E) o[cc] = v[u];
    }
  }
}

// q_cat[t,h,0:L] = nope[t,h,:]; q_cat[t,h,L:L+R] = rope[t,h,:] (rope s1 may be 0).
// Counts and strides are in units of W (the copy word); L and R are multiples
// of the word on the vector path. rows = T * H < 2^31.
template <typename W>
__global__ void __launch_bounds__(256) concat_q_kernel(
    W* __restrict__ out, int64_t o_s0, int64_t o_s1, const W* __restrict__ nope, int64_t n_s0,
    int64_t n_s1, const W* __restrict__ rope, int64_t r_s0, int64_t r_s1, int32_t H, int32_t Lw,
    int32_t Rw, int32_t rows, RowSplit rs) {
  pdl_enter();
  const int Ew = Lw + Rw;
  int64_t r, step;
  int c0;
  row_lane(rs, r, step, c0);
  for (; r < rows; r += step) {
    const int t = (int)r / H, h = (int)r - t * H;
    W* o = out + t * o_s0 + h * o_s1;
    const W* nr = nope + t * n_s0 + h * n_s1;
    const W* rr = rope + t * r_s0 + h * r_s1 - Lw;
    copy_row(o, nr, rr, Lw, Ew, c0, rs.G);
  }
}

// cache[s/page, s%page, :] = [kv_c[i] | k_pe[i]] for every token i with slot s >= 0.
template <typename W>
__global__ void __launch_bounds__(256) cache_write_kernel(
    W* __restrict__ cache, int64_t c_blk, int64_t c_row, int64_t num_rows, int32_t page,
    const W* __restrict__ kv_c, int64_t k_s0, const W* __restrict__ k_pe, int64_t p_s0,
    const int64_t* __restrict__ slots, int32_t Lw, int32_t Rw, int64_t T, RowSplit rs) {
  pdl_enter();
  const int Ew = Lw + Rw;
  int64_t tok, step;
  int c0;
  row_lane(rs, tok, step, c0);
  for (; tok < T; tok += step) {
    const int64_t s = slots[tok];
    if (s < 0) continue;  // padding
    if (s >= num_rows) {  // would land outside the view: skip and record
      if (c0 == 0) atomicOr(&g_copy_err, kErrDeviceData);
      continue;
    }
    const int64_t blk = s / page, r = s - blk * page;
    W* o = cache + blk * c_blk + r * c_row;
    const W* kr = kv_c + tok * k_s0;
    const W* pr = k_pe + tok * p_s0 - Lw;
    copy_row(o, kr, pr, Lw, Ew, c0, rs.G);
  }
}

// e4m3 code of x / scale: the division correctly rounded in float32, then round to nearest
// (ties to even), finite values beyond 448 saturating to +-448, NaN to NaN.
__device__ __forceinline__ uint8_t e4m3_of(float x, float scale) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(x, scale), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

// Eight consecutive source values as floats (16-byte aligned: one 16-byte load for bf16, two for fp32).
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// cache[s/page, s%page, :] = e4m3([kv_c[i] | k_pe[i]] / scale) for every token with slot s >= 0.
// Element strides (cache strides count bytes). vec8: every row start and L, R are multiples of 8
// elements with the sources 16-byte and the cache rows 8-byte aligned, so a lane converts eight
// values and stores them at once.
template <typename T>
__global__ void __launch_bounds__(256) cache_write_fp8_kernel(
    uint8_t* __restrict__ cache, int64_t c_blk, int64_t c_row, int64_t num_rows, int32_t page,
    const T* __restrict__ kv_c, int64_t k_s0, const T* __restrict__ k_pe, int64_t p_s0,
    const int64_t* __restrict__ slots, int32_t L, int32_t R, int64_t T_, const float* __restrict__ scale_p,
    RowSplit rs, int vec8) {
  pdl_enter();
  const float scale = *scale_p;
  const int E = L + R;
  int64_t tok, step;
  int c0;
  row_lane(rs, tok, step, c0);
  for (; tok < T_; tok += step) {
    const int64_t s = slots[tok];
    if (s < 0) continue;  // padding
    if (s >= num_rows) {  // would land outside the view: skip and record
      if (c0 == 0) atomicOr(&g_copy_err, kErrDeviceData);
      continue;
    }
    const int64_t blk = s / page, r = s - blk * page;
    uint8_t* o = cache + blk * c_blk + r * c_row;
    const T* kr = kv_c + tok * k_s0;
    const T* pr = k_pe + tok * p_s0 - L;
    if (vec8) {
      for (int c = c0 * 8; c < E; c += rs.G * 8) {
        float x[8];
        load8(c < L ? kr + c : pr + c, x);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          lo |= (uint32_t)e4m3_of(x[i], scale) << (8 * i);
          hi |= (uint32_t)e4m3_of(x[4 + i], scale) << (8 * i);
        }
        *reinterpret_cast<uint2*>(o + c) = make_uint2(lo, hi);
      }
    } else {
      for (int c = c0; c < E; c += rs.G) o[c] = e4m3_of(to_f(c < L ? kr[c] : pr[c]), scale);
    }
  }
}

RowSplit row_split(int64_t words) {
  RowSplit rs{32, 5};
  while (rs.G > 8 && rs.G / 2 >= words) {
    rs.G /= 2;
    rs.shift -= 1;
  }
  return rs;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The q concat and the cache write of the same step in one launch: blocks [0, q_blocks) run
// the concat over q rows, the remaining blocks the cache write over tokens, each part with its
// own lane-group split and striding over its own block range. Both parts move 16-byte words.
struct ConcatArgs {
  uint4* out;
  int64_t o_s0, o_s1;
  const uint4* nope;
  int64_t n_s0, n_s1;
  const uint4* rope;
  int64_t r_s0, r_s1;
  int32_t H, Lw, Rw, rows;
  RowSplit rs;
};
struct CacheArgs {
  uint4* cache;
  int64_t c_blk, c_row, num_rows;
  int32_t page;
  const uint4* kv_c;
  int64_t k_s0;
  const uint4* k_pe;
  int64_t p_s0;
  const int64_t* slots;
  int32_t Lw, Rw;
  int64_t T;
  RowSplit rs;
};

template <bool kAlongside>
__global__ void __launch_bounds__(256) concat_cache_kernel(ConcatArgs a, CacheArgs c, int q_blocks) {
  if (kAlongside)
    pdl_allow_dependents();   // the kernel before writes nothing this one touches (see the launcher)
  else
    pdl_enter();
  const bool q_part = (int)blockIdx.x < q_blocks;
  const int part_block = q_part ? blockIdx.x : blockIdx.x - q_blocks;
  const int part_blocks = q_part ? q_blocks : gridDim.x - q_blocks;
  const RowSplit rs = q_part ? a.rs : c.rs;
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = (part_block * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)part_blocks * blockDim.x) >> 5;
  const int per_warp = 32 >> rs.shift;
  const int c0 = lane & (rs.G - 1);
  const int64_t step = nwarps * per_warp;
  int64_t r = gwarp * per_warp + (lane >> rs.shift);
  if (q_part) {
    const int Ew = a.Lw + a.Rw;
    for (; r < a.rows; r += step) {
      const int t = (int)r / a.H, h = (int)r - t * a.H;
      uint4* o = a.out + t * a.o_s0 + h * a.o_s1;
      const uint4* nr = a.nope + t * a.n_s0 + h * a.n_s1;
      const uint4* rr = a.rope + t * a.r_s0 + h * a.r_s1 - a.Lw;
      copy_row(o, nr, rr, a.Lw, Ew, c0, rs.G);
    }
  } else {
    const int Ew = c.Lw + c.Rw;
    for (; r < c.T; r += step) {
      const int64_t sl = c.slots[r];
      if (sl < 0) continue;
      if (sl >= c.num_rows) {
        if (c0 == 0) atomicOr(&g_copy_err, kErrDeviceData);
        continue;
      }
      const int64_t blk = sl / c.page, row = sl - blk * c.page;
      uint4* o = c.cache + blk * c.c_blk + row * c.c_row;
      const uint4* kr = c.kv_c + r * c.k_s0;
      const uint4* pr = c.k_pe + r * c.p_s0 - c.Lw;
      copy_row(o, kr, pr, c.Lw, Ew, c0, rs.G);
    }
  }
  // alongside: complete only once the kernel before is, so the next kernel's wait covers both
  if (kAlongside) pdl_wait();
}



// Enough 256-thread blocks for one row group per row, capped at 16 blocks per SM (the
// kernels stride over the rest).
int grid_for(int64_t rows, const RowSplit& rs) {
  const int64_t rows_per_block = 256 / rs.G;
  const int64_t want = (rows + rows_per_block - 1) / rows_per_block;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_concat_q(mla_dtype dt, const View3& out, const View3& nope, const View3& rope,
                            cudaStream_t st) {
  const int64_t es = dt == MLA_F32 ? 4 : 2;
  const int64_t T = out.n0, H = out.n1, L = nope.n2, R = rope.n2;
  const int64_t rows = T * H;
  if (rows >= INT32_MAX || L + R >= INT32_MAX / 4) return cudaErrorInvalidValue;
  const int64_t per = 16 / es;  // elements per 16-byte word
  bool vec = aligned16(out.data) && aligned16(nope.data) && (R == 0 || aligned16(rope.data)) &&
             L % per == 0 && R % per == 0 && out.s0 % per == 0 && out.s1 % per == 0 &&
             nope.s0 % per == 0 && nope.s1 % per == 0 &&
             (R == 0 || (rope.s0 % per == 0 && rope.s1 % per == 0));
  const void* rp = R == 0 ? nope.data : rope.data;  // never read when R == 0
  if (vec) {
    const RowSplit rs = row_split((L + R) / per);
    return launch_k(concat_q_kernel<uint4>, grid_for(rows, rs), 256, 0, st,
        (uint4*)out.data, out.s0 / per, out.s1 / per, (const uint4*)nope.data, nope.s0 / per,
        nope.s1 / per, (const uint4*)rp, rope.s0 / per, rope.s1 / per, (int32_t)H, (int32_t)(L / per),
        (int32_t)(R / per), (int32_t)rows, rs);
  }
  const RowSplit rs = row_split(L + R);
  if (es == 4)
    return launch_k(concat_q_kernel<uint32_t>, grid_for(rows, rs), 256, 0, st,
        (uint32_t*)out.data, out.s0, out.s1, (const uint32_t*)nope.data, nope.s0, nope.s1,
        (const uint32_t*)rp, rope.s0, rope.s1, (int32_t)H, (int32_t)L, (int32_t)R, (int32_t)rows, rs);
  return launch_k(concat_q_kernel<uint16_t>, grid_for(rows, rs), 256, 0, st,
      (uint16_t*)out.data, out.s0, out.s1, (const uint16_t*)nope.data, nope.s0, nope.s1,
      (const uint16_t*)rp, rope.s0, rope.s1, (int32_t)H, (int32_t)L, (int32_t)R, (int32_t)rows, rs);
}

cudaError_t launch_cache_write(mla_dtype dt, const View3& cache, const View3& kv_c,
                               const View3& k_pe, int64_t L, int64_t R, const int64_t* slots,
                               int64_t T, cudaStream_t st) {
  const int64_t es = dt == MLA_F32 ? 4 : 2;
  const int64_t per = 16 / es;
  const int64_t rows = cache.n0 * cache.n1;
  const int32_t page = (int32_t)cache.n1;
  if (L + R >= INT32_MAX / 4) return cudaErrorInvalidValue;
  bool vec = aligned16(cache.data) && aligned16(kv_c.data) && (R == 0 || aligned16(k_pe.data)) &&
             L % per == 0 && R % per == 0 && cache.s0 % per == 0 && cache.s1 % per == 0 &&
             kv_c.s0 % per == 0 && (R == 0 || k_pe.s0 % per == 0);
  const void* kp = R == 0 ? kv_c.data : k_pe.data;
  if (vec) {
    const RowSplit rs = row_split((L + R) / per);
    return launch_k(cache_write_kernel<uint4>, grid_for(T, rs), 256, 0, st,
        (uint4*)cache.data, cache.s0 / per, cache.s1 / per, rows, page, (const uint4*)kv_c.data,
        kv_c.s0 / per, (const uint4*)kp, k_pe.s0 / per, slots, (int32_t)(L / per), (int32_t)(R / per), T, rs);
  }
  const RowSplit rs = row_split(L + R);
  if (es == 4)
    return launch_k(cache_write_kernel<uint32_t>, grid_for(T, rs), 256, 0, st,
        (uint32_t*)cache.data, cache.s0, cache.s1, rows, page, (const uint32_t*)kv_c.data,
        kv_c.s0, (const uint32_t*)kp, k_pe.s0, slots, (int32_t)L, (int32_t)R, T, rs);
  return launch_k(cache_write_kernel<uint16_t>, grid_for(T, rs), 256, 0, st,
      (uint16_t*)cache.data, cache.s0, cache.s1, rows, page, (const uint16_t*)kv_c.data,
      kv_c.s0, (const uint16_t*)kp, k_pe.s0, slots, (int32_t)L, (int32_t)R, T, rs);
}

cudaError_t launch_cache_write_fp8(mla_dtype src_dt, const View3& cache, const View3& kv_c, const View3& k_pe,
                                   int64_t L, int64_t R, const int64_t* slots, int64_t T, const float* scale,
                                   cudaStream_t st) {
  const int64_t rows = cache.n0 * cache.n1;
  const int32_t page = (int32_t)cache.n1;
  if (L + R >= INT32_MAX / 4) return cudaErrorInvalidValue;
  auto al = [](const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
  const bool vec8 = L % 8 == 0 && R % 8 == 0 && al(cache.data, 8) && cache.s0 % 8 == 0 && cache.s1 % 8 == 0 &&
                    al(kv_c.data, 16) && (R == 0 || al(k_pe.data, 16)) &&
                    (kv_c.s0 * (src_dt == MLA_F32 ? 4 : 2)) % 16 == 0 &&
                    (R == 0 || (k_pe.s0 * (src_dt == MLA_F32 ? 4 : 2)) % 16 == 0);
  const RowSplit rs = row_split(vec8 ? (L + R) / 8 : L + R);
  const void* kp = R == 0 ? kv_c.data : k_pe.data;
  if (src_dt == MLA_F32)
    return launch_k(cache_write_fp8_kernel<float>, grid_for(T, rs), 256, 0, st, (uint8_t*)cache.data, cache.s0,
                    cache.s1, rows, page, (const float*)kv_c.data, kv_c.s0, (const float*)kp, k_pe.s0, slots,
                    (int32_t)L, (int32_t)R, T, scale, rs, vec8 ? 1 : 0);
  return launch_k(cache_write_fp8_kernel<__nv_bfloat16>, grid_for(T, rs), 256, 0, st, (uint8_t*)cache.data,
                  cache.s0, cache.s1, rows, page, (const __nv_bfloat16*)kv_c.data, kv_c.s0,
                  (const __nv_bfloat16*)kp, k_pe.s0, slots, (int32_t)L, (int32_t)R, T, scale, rs, vec8 ? 1 : 0);
}

cudaError_t launch_concat_cache(mla_dtype dt, const View3& out, const View3& nope, const View3& rope,
                                const View3& cache, const View3& kv_c, const View3& k_pe, int64_t L, int64_t R,
                                const int64_t* slots, int64_t T, cudaStream_t st, bool alongside) {
  const int64_t es = dt == MLA_F32 ? 4 : 2;
  const int64_t per = 16 / es;
  const int64_t Tq = out.n0, H = out.n1, Lq = nope.n2, Rq = rope.n2;
  const int64_t qrows = Tq * H;
  const bool q_vec = aligned16(out.data) && (Lq == 0 || aligned16(nope.data)) && (Rq == 0 || aligned16(rope.data)) &&
                     Lq % per == 0 && Rq % per == 0 && out.s0 % per == 0 && out.s1 % per == 0 &&
                     nope.s0 % per == 0 && nope.s1 % per == 0 && (Rq == 0 || (rope.s0 % per == 0 && rope.s1 % per == 0));
  const bool c_vec = aligned16(cache.data) && aligned16(kv_c.data) && (R == 0 || aligned16(k_pe.data)) &&
                     L % per == 0 && R % per == 0 && cache.s0 % per == 0 && cache.s1 % per == 0 &&
                     kv_c.s0 % per == 0 && (R == 0 || k_pe.s0 % per == 0);
  if (!q_vec || !c_vec || qrows >= INT32_MAX || qrows == 0 || T == 0) {
    // one of the two cannot take 16-byte words (or is empty): two launches, same results
    cudaError_t e = cudaSuccess;
    if (qrows > 0) e = launch_concat_q(dt, out, nope, rope, st);
    if (e == cudaSuccess && T > 0) e = launch_cache_write(dt, cache, kv_c, k_pe, L, R, slots, T, st);
    return e;
  }
  ConcatArgs a;
  a.out = (uint4*)out.data;
  a.o_s0 = out.s0 / per;
  a.o_s1 = out.s1 / per;
  a.nope = (const uint4*)(Lq == 0 ? out.data : nope.data);
  a.n_s0 = nope.s0 / per;
  a.n_s1 = nope.s1 / per;
  a.rope = (const uint4*)(Rq == 0 ? out.data : rope.data);
  a.r_s0 = rope.s0 / per;
  a.r_s1 = rope.s1 / per;
  a.H = (int32_t)H;
  a.Lw = (int32_t)(Lq / per);
  a.Rw = (int32_t)(Rq / per);
  a.rows = (int32_t)qrows;
  a.rs = row_split((Lq + Rq) / per);
  CacheArgs c;
  c.cache = (uint4*)cache.data;
  c.c_blk = cache.s0 / per;
  c.c_row = cache.s1 / per;
  c.num_rows = cache.n0 * cache.n1;
  c.page = (int32_t)cache.n1;
  c.kv_c = (const uint4*)kv_c.data;
  c.k_s0 = kv_c.s0 / per;
  c.k_pe = (const uint4*)(R == 0 ? kv_c.data : k_pe.data);
  c.p_s0 = k_pe.s0 / per;
  c.slots = slots;
  c.Lw = (int32_t)(L / per);
  c.Rw = (int32_t)(R / per);
  c.T = T;
  c.rs = row_split((L + R) / per);
  const int qb = grid_for(qrows, a.rs), cb = grid_for(T, c.rs);
  return launch_k(alongside ? concat_cache_kernel<true> : concat_cache_kernel<false>, qb + cb, 256, 0, st, a, c, qb);
}

unsigned copy_errors_read_clear() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_copy_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_copy_err, &zero, sizeof(zero));
  return v;
}

}  // namespace mla
