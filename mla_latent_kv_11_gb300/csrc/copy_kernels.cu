// Step 2 (q concat) and step 3 (paged latent cache write): pure bit copies.
//
// Both move whole rows. When every row start and row length is a multiple of
// 16 bytes the copy goes in 16-byte vectors (uint4), one vector per thread,
// consecutive threads on consecutive vectors of a row, so a warp moves 512
// contiguous bytes; otherwise it falls back to element copies of the same
// order. The element type never matters: bits are moved as integers, so NaN
// payloads and signed zeros survive unchanged.
#include <cstdint>

#include "mla_internal.h"

namespace mla {
namespace {

__device__ unsigned g_copy_err = 0;

template <int BYTES> struct Word;
template <> struct Word<16> { using T = uint4; };
template <> struct Word<4> { using T = uint32_t; };
template <> struct Word<2> { using T = uint16_t; };

// q_cat[t,h,0:L] = nope[t,h,:]; q_cat[t,h,L:L+R] = rope[t,h,:] (rope s1 may be 0).
// Counts and strides are in units of W (the copy word); L and R are multiples
// of the word on the vector path.
template <typename W>
__global__ void __launch_bounds__(256) concat_q_kernel(
    W* __restrict__ out, int64_t o_s0, int64_t o_s1, const W* __restrict__ nope, int64_t n_s0,
    int64_t n_s1, const W* __restrict__ rope, int64_t r_s0, int64_t r_s1, int64_t H, int64_t Lw,
    int64_t Rw, int64_t total) {
  pdl_enter();
  const int64_t Ew = Lw + Rw;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / Ew;
    const int64_t c = i - row * Ew;
    const int64_t t = row / H, h = row - t * H;
    W v;
    if (c < Lw)
      v = nope[t * n_s0 + h * n_s1 + c];
    else
      v = rope[t * r_s0 + h * r_s1 + (c - Lw)];
    out[t * o_s0 + h * o_s1 + c] = v;
  }
}

// cache[s/page, s%page, :] = [kv_c[i] | k_pe[i]] for every token i with slot s >= 0.
template <typename W>
__global__ void __launch_bounds__(256) cache_write_kernel(
    W* __restrict__ cache, int64_t c_blk, int64_t c_row, int64_t num_rows, int32_t page,
    const W* __restrict__ kv_c, int64_t k_s0, const W* __restrict__ k_pe, int64_t p_s0,
    const int64_t* __restrict__ slots, int64_t Lw, int64_t Rw, int64_t total) {
  pdl_enter();
  const int64_t Ew = Lw + Rw;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = i / Ew;
    const int64_t c = i - tok * Ew;
    const int64_t s = slots[tok];
    if (s < 0) continue;  // padding
    if (s >= num_rows) {  // would land outside the view: skip and record
      if (c == 0) atomicOr(&g_copy_err, kErrDeviceData);
      continue;
    }
    const int64_t blk = s / page, r = s - blk * page;
    const W v = c < Lw ? kv_c[tok * k_s0 + c] : k_pe[tok * p_s0 + (c - Lw)];
    cache[blk * c_blk + r * c_row + c] = v;
  }
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int grid_for(int64_t total) {
  const int64_t want = (total + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_concat_q(mla_dtype dt, const View3& out, const View3& nope, const View3& rope,
                            cudaStream_t st) {
  const int64_t es = dt == MLA_F32 ? 4 : 2;
  const int64_t T = out.n0, H = out.n1, L = nope.n2, R = rope.n2;
  const int64_t per = 16 / es;  // elements per 16-byte word
  bool vec = aligned16(out.data) && aligned16(nope.data) && (R == 0 || aligned16(rope.data)) &&
             L % per == 0 && R % per == 0 && out.s0 % per == 0 && out.s1 % per == 0 &&
             nope.s0 % per == 0 && nope.s1 % per == 0 &&
             (R == 0 || (rope.s0 % per == 0 && rope.s1 % per == 0));
  const void* rp = R == 0 ? nope.data : rope.data;  // never read when R == 0
  if (vec) {
    const int64_t total = T * H * (L + R) / per;
    return launch_k(concat_q_kernel<uint4>, grid_for(total), 256, 0, st,
        (uint4*)out.data, out.s0 / per, out.s1 / per, (const uint4*)nope.data, nope.s0 / per,
        nope.s1 / per, (const uint4*)rp, rope.s0 / per, rope.s1 / per, H, L / per, R / per, total);
  } else {
    const int64_t total = T * H * (L + R);
    if (es == 4)
      return launch_k(concat_q_kernel<uint32_t>, grid_for(total), 256, 0, st,
          (uint32_t*)out.data, out.s0, out.s1, (const uint32_t*)nope.data, nope.s0, nope.s1,
          (const uint32_t*)rp, rope.s0, rope.s1, H, L, R, total);
    else
      return launch_k(concat_q_kernel<uint16_t>, grid_for(total), 256, 0, st,
          (uint16_t*)out.data, out.s0, out.s1, (const uint16_t*)nope.data, nope.s0, nope.s1,
          (const uint16_t*)rp, rope.s0, rope.s1, H, L, R, total);
  }
  return cudaGetLastError();
}

cudaError_t launch_cache_write(mla_dtype dt, const View3& cache, const View3& kv_c,
                               const View3& k_pe, int64_t L, int64_t R, const int64_t* slots,
                               int64_t T, cudaStream_t st) {
  const int64_t es = dt == MLA_F32 ? 4 : 2;
  const int64_t per = 16 / es;
  const int64_t rows = cache.n0 * cache.n1;
  const int32_t page = (int32_t)cache.n1;
  bool vec = aligned16(cache.data) && aligned16(kv_c.data) && (R == 0 || aligned16(k_pe.data)) &&
             L % per == 0 && R % per == 0 && cache.s0 % per == 0 && cache.s1 % per == 0 &&
             kv_c.s0 % per == 0 && (R == 0 || k_pe.s0 % per == 0);
  const void* kp = R == 0 ? kv_c.data : k_pe.data;
  if (vec) {
    const int64_t total = T * (L + R) / per;
    return launch_k(cache_write_kernel<uint4>, grid_for(total), 256, 0, st,
        (uint4*)cache.data, cache.s0 / per, cache.s1 / per, rows, page, (const uint4*)kv_c.data,
        kv_c.s0 / per, (const uint4*)kp, k_pe.s0 / per, slots, L / per, R / per, total);
  } else {
    const int64_t total = T * (L + R);
    if (es == 4)
      return launch_k(cache_write_kernel<uint32_t>, grid_for(total), 256, 0, st,
          (uint32_t*)cache.data, cache.s0, cache.s1, rows, page, (const uint32_t*)kv_c.data,
          kv_c.s0, (const uint32_t*)kp, k_pe.s0, slots, L, R, total);
    else
      return launch_k(cache_write_kernel<uint16_t>, grid_for(total), 256, 0, st,
          (uint16_t*)cache.data, cache.s0, cache.s1, rows, page, (const uint16_t*)kv_c.data,
          kv_c.s0, (const uint16_t*)kp, k_pe.s0, slots, L, R, total);
  }
  return cudaGetLastError();
}

unsigned copy_errors_read_clear() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_copy_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_copy_err, &zero, sizeof(zero));
  return v;
}

}  // namespace mla
