// Steps 4b and 5 in one kernel: the LSE combine of the split-KV partials and the W_UV
// un-projection, so o_lat never makes a round trip through HBM between them.
//
// One CTA owns head h, a 128-wide tile of v_head columns and a chunk of 64 sequences. It
// TMA-loads W_UV[h][:, v-tile] (512 x 128 bf16, 128 KB) before waiting on the kernels
// before it (the weight is not written by them), then builds the chunk's o_lat rows for
// head h in shared memory as bf16: a sequence held whole by one work unit is copied from
// the row the attention kernel wrote, a split one is merged from its fp32 partials by their
// LSE weights (the combine kernel's arithmetic), an empty one is zero. One tcgen05 MMA chain
// then computes out^T = W_UV[h]^T (M = 128 v, K = 512, an MN-major operand straight from the
// TMA boxes) times o_lat^T (N = 64 sequences, K-major), fp32 in TMEM, and the epilogue
// writes out[b, h, v-tile] in bf16 with one TMA store. The o_lat rows are rounded to bf16
// before the MMA, as the separate combine and v_up do.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "mla_internal.h"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

__device__ unsigned g_cvu_err = 0;

constexpr int kThreads = 384;
constexpr int kWarps = kThreads / 32;
constexpr int kSeqs = 64;                  // sequences per CTA: the MMA's N
constexpr int kVT = 128;                   // v columns per CTA: the MMA's M
constexpr int kL = 512;                    // latent width: the MMA's K
constexpr int kWBox = 64 * 128;            // one [64 l x 64 v] bf16 box, 128-byte rows (8 KB)
constexpr int kWBytes = (kL / 64) * 2 * kWBox;   // 128 KB
constexpr int kOBox = kSeqs * 128;         // one [64 seq x 64 l] bf16 box (8 KB)
constexpr int kOBytes = (kL / 64) * kOBox; // 64 KB
constexpr int kOffBar = kWBytes + kOBytes;
constexpr int kSmemAlloc = kOffBar + 64 + 2 * kSeqs * 4 + 1024;   // + barriers, per-sequence words
constexpr uint32_t kTmemCols = 64;

struct CvuParams {
  const __nv_bfloat16* o_lat;    // [B, H, L] rows of sequences held whole by one unit
  int64_t o_s0, o_s1;
  float* lse;                    // [B, H] or null
  int B, H, V;
  DecodeSched s;
};

__global__ void __launch_bounds__(kThreads, 1)
    combine_vup_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap omap,
                       const CvuParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~uintptr_t(1023));
  unsigned char* sW = smem;
  unsigned char* sO = smem + kWBytes;
  uint64_t* w_full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* mma_done = w_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, vt = blockIdx.y, b0 = blockIdx.z * kSeqs;

  if (tid == 0) {
    mbar_init(w_full, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort = abort_flag;
  if (tid == 0) {
    // the weight tile: box (kc, vg) holds l in [64 kc, 64 kc + 64) x v in [64 vg, 64 vg + 64)
    tma_prefetch_desc(&wmap);
    mbar_arrive_expect_tx(w_full, kWBytes);
    for (int kc = 0; kc < kL / 64; ++kc)
      for (int vg = 0; vg < 2; ++vg)
        tma_load_3d(sW + (kc * 2 + vg) * kWBox, &wmap, w_full, vt * kVT + 64 * vg, 64 * kc, h);
  }
  // Each sequence's piece count and first partial slot come from the schedule kernel two
  // launches back, which had completed before this kernel could launch: the split kernel in
  // between waits for it (griddepcontrol.wait) before it lets this kernel launch. They are
  // read before this kernel's own wait; the o_lat rows and partials, the split kernel's
  // output, only after it.
  int* s_np = reinterpret_cast<int*>(abort_flag + 1);   // [kSeqs] pieces of each sequence
  int* s_base = s_np + kSeqs;                              // [kSeqs] its first partial slot
  if (tid < kSeqs) {
    const int b = b0 + tid;
    s_np[tid] = b < p.B ? p.s.npieces[b] : 0;
    s_base[tid] = b < p.B ? p.s.piece_base[b] : 0;
  }
  pdl_enter();   // o_lat rows and partials come from the split kernel before
  __syncthreads();

  // ---- o_lat rows of the chunk for head h, bf16, as K-major [64 seq x 64 l] boxes with
  // 128-byte swizzle; lane owns columns lane*4 + 128k (k = 0..3). The loads are batched so a
  // warp waits about one memory latency per phase, not one per sequence.
  auto store_row = [&](int n, const uint32_t (&w2)[4][2]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int l = lane * 4 + 128 * k;
      const int chunk = (l & 63) >> 3;
      *reinterpret_cast<uint2*>(sO + (l >> 6) * kOBox + n * 128 + ((chunk ^ (n & 7)) << 4) + (lane & 1) * 8) =
          make_uint2(w2[k][0], w2[k][1]);
    }
  };
  constexpr int kPerWarp = (kSeqs + kWarps - 1) / kWarps;   // sequences a warp: n = warp + kWarps j
  // phase 1: sequences held whole by one unit (the attention kernel wrote their bf16 row) and
  // empty ones, all of a warp's loads issued before any is used
  {
    uint2 v[kPerWarp][4];
#pragma unroll
    for (int j = 0; j < kPerWarp; ++j) {
      const int n = warp + kWarps * j;
      const __nv_bfloat16* row = p.o_lat + (int64_t)(b0 + n) * p.o_s0 + (int64_t)h * p.o_s1;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        v[j][k] = n < kSeqs && s_np[n] == 1 ? *reinterpret_cast<const uint2*>(row + lane * 4 + 128 * k)
                                            : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kPerWarp; ++j) {
      const int n = warp + kWarps * j;
      if (n >= kSeqs || s_np[n] > 1) continue;
      uint32_t w2[4][2];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w2[k][0] = v[j][k].x;
        w2[k][1] = v[j][k].y;
      }
      store_row(n, w2);
      if (s_np[n] == 0 && b0 + n < p.B && lane == 0 && vt == 0 && p.lse)
        p.lse[(int64_t)(b0 + n) * p.H + h] = -CUDART_INF_F;   // an empty sequence
    }
  }
  // phase 2: sequences cut across units, merged from their fp32 partials by their LSE
  // weights; the maxima and rows of up to four pieces are loaded together
  const int64_t pstride = (int64_t)p.H * kL;
  for (int n = warp; n < kSeqs; n += kWarps) {
    const int np = s_np[n];
    if (np <= 1) continue;
    const int b = b0 + n;
    const float* lse_p = p.s.part_lse + (int64_t)s_base[n] * p.H + h;
    const float* part = p.s.part_o + ((int64_t)s_base[n] * p.H + h) * kL;
    float m = -CUDART_INF_F, tot = 0.f;
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < np; i0 += 4) {
      float li[4];
      float4 v[4][4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const int i = i0 + ii;
        li[ii] = i < np ? lse_p[(int64_t)i * p.H] : -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[ii][k] = i < np ? *reinterpret_cast<const float4*>(part + i * pstride + lane * 4 + 128 * k)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      // online merge: rescale what came before when a group raises the maximum
      float gm = m;
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) gm = fmaxf(gm, li[ii]);
      const float r = (m == -CUDART_INF_F || gm == -CUDART_INF_F) ? 0.f : __expf(m - gm);
      tot *= r;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[k].x *= r;
        acc[k].y *= r;
        acc[k].z *= r;
        acc[k].w *= r;
      }
      m = gm;
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const float wi = li[ii] == -CUDART_INF_F ? 0.f : __expf(li[ii] - m);
        tot += wi;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[k].x = fmaf(wi, v[ii][k].x, acc[k].x);
          acc[k].y = fmaf(wi, v[ii][k].y, acc[k].y);
          acc[k].z = fmaf(wi, v[ii][k].z, acc[k].z);
          acc[k].w = fmaf(wi, v[ii][k].w, acc[k].w);
        }
      }
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    uint32_t w2[4][2];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __nv_bfloat162 a = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
      const __nv_bfloat162 c = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
      w2[k][0] = *reinterpret_cast<const uint32_t*>(&a);
      w2[k][1] = *reinterpret_cast<const uint32_t*>(&c);
    }
    store_row(n, w2);
    if (lane == 0 && vt == 0 && p.lse) p.lse[(int64_t)b * p.H + h] = tot > 0.f ? m + logf(tot) : -CUDART_INF_F;
  }
  fence_proxy_async_smem();   // the tensor core reads the rows through the async proxy
  __syncthreads();

  if (warp == 1) {
    // ---- out^T = W^T o_lat^T: 32 MMAs of K = 16, issued by one elected lane of the warp
    bool ok = __all_sync(0xffffffffu, mbar_wait(w_full, 0, abort));
    if (ok) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16(kVT, kSeqs, true, false);
      const uint32_t wb = smem_u32(sW), ob = smem_u32(sO);
#pragma unroll
      for (int kc = 0; kc < kL / 64; ++kc)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_elect(tmem, sdesc_sw128(wb + kc * 2 * kWBox + kk * 16 * 128, kWBox, 1024),
                          sdesc_sw128(ob + kc * kOBox + kk * 32, 16, 1024), idesc, (kc | kk) ? 1u : 0u);
    }
    umma_commit_elect(mma_done);   // also when nothing was issued: the epilogue never waits forever
    if (!ok && lane == 0) atomicOr(&g_cvu_err, kErrTimeout);
  }
  if (warp < 4) {
    // ---- epilogue: TMEM lane = v row of the tile, column = sequence of the chunk. The tile is
    // staged as [64 sequences x 128 v] bf16 in the o_lat buffer (the MMA has read it) and goes
    // out in one TMA store, which drops sequences past B
    const bool ok = mbar_wait(mma_done, 0, abort) && *abort == 0;   // no MMA ran if the weight never landed
    tc_fence_after();
    if (ok) {
      const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
      __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(sO);
      const int vl = warp * 32 + lane;
      for (int c = 0; c < kSeqs; c += 32) {
        float d[32];
        tmem_ld32(tmem + lane_addr + c, d);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) stage[(c + i) * kVT + vl] = __float2bfloat16_rn(d[i]);
      }
      fence_proxy_async_smem();   // the TMA store reads the stage through the async proxy
    }
    const bool all_ok = named_bar_and(1, 128, ok);
    if (tid == 0) {
      if (all_ok) {
        tma_store_3d(&omap, sO, vt * kVT, h, b0);
        bulk_commit_group();
        bulk_wait_read_all();
      } else {
        atomicOr(&g_cvu_err, kErrTimeout);
      }
    }
  }
  if (tid == 0 && *abort) {
    // never leave with the weight's copies in flight: wait for them once more, with a limit
    volatile int dummy = 0;
    mbar_wait(w_full, 0, &dummy);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool combine_vup_supported(mla_dtype dt, int L, int V, const View3& out, const View3& w_uv) {
  if (dt != MLA_BF16 || L != kL || V % kVT != 0 || !tensor_maps_available()) return false;
  if (out.s2 != 1 || w_uv.s2 != 1) return false;
  auto al16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  // both go through tensor maps: 16-byte aligned bases and strides
  return al16(w_uv.data) && w_uv.s0 % 8 == 0 && w_uv.s1 % 8 == 0 && al16(out.data) && out.s0 % 8 == 0 &&
         out.s1 % 8 == 0;
}

cudaError_t launch_combine_vup(const View3& out, const View3& o_lat, float* lse, const View3& w_uv, int32_t B,
                               int32_t H, int32_t V, const DecodeSched& s, cudaStream_t st) {
  CUtensorMap wmap;
  // W_UV[h] as [H, L, V]: dims (V, L, H), box 64 v x 64 l, 128-byte swizzle
  if (!make_map3d(&wmap, w_uv.data, (uint64_t)V, kL, (uint64_t)H, (uint64_t)w_uv.s1 * 2, (uint64_t)w_uv.s0 * 2, 64,
                  64, 1, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  CUtensorMap omap;
  // out as [B, H, V]: dims (V, H, B), box 128 v x 1 head x 64 sequences, no swizzle
  if (!make_map3d(&omap, out.data, (uint64_t)V, (uint64_t)H, (uint64_t)B, (uint64_t)out.s1 * 2, (uint64_t)out.s0 * 2,
                  kVT, 1, kSeqs, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  CvuParams p;
  p.o_lat = static_cast<const __nv_bfloat16*>(o_lat.data);
  p.o_s0 = o_lat.s0;
  p.o_s1 = o_lat.s1;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.V = V;
  p.s = s;
  cudaError_t e = cudaFuncSetAttribute(combine_vup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)H, (unsigned)(V / kVT), (unsigned)((B + kSeqs - 1) / kSeqs));
  return launch_k(combine_vup_kernel, grid, dim3(kThreads), kSmemAlloc, st, wmap, omap, p);
}

unsigned combine_vup_errors_read_clear() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_cvu_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_cvu_err, &zero, sizeof(zero));
  return v;
}

}  // namespace mla
