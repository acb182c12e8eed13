// Steps 1 and 5 on the tensor cores: out[g,m,n] = sum_k a[g,m,k] * b[g,k,n] in
// bf16 with fp32 accumulation (tcgen05 + TMEM + TMA), for K a multiple of 64
// and N a multiple of 128.
//
// One CTA computes a 128 x BN tile of one head g: BN = 512 when N is a
// multiple of 512 and one tile per head fits in a single wave of CTAs (the
// decode absorb: 128 heads x 64 tokens x 512), else 256, else 128. A 512-wide
// tile accumulates in all 512 TMEM columns through two N=256 MMAs per k-step. TMA 3-D tensor maps read the operands straight from
// their strided views (the usual transposed [H,B,P] operand and [H,B,L]
// output cost nothing extra): A tiles are K-major [128 rows x 64 k] boxes,
// B tiles are [64 k x 64 n] boxes used as an MN-major operand. A 4-stage ring
// of k-steps feeds one issuing warp; the fp32 accumulator sits in TMEM. The
// epilogue converts to bf16 through a 128-byte-swizzled staging tile and
// writes it with TMA stores, which clip rows past M (the decode batch, padded
// to 128 rows by the loads' zero fill).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "mla_internal.h"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

__device__ unsigned g_bmm_err = 0;

constexpr int kThreads = 128;
constexpr int kBM = 128, kBK = 64;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kBBox = kBK * 64 * 2;      // 8 KB: 64 k-rows x 64 n

template <int kBN>
struct BmmCfg {
  static constexpr int kStages = kBN > 256 ? 2 : 4;
  static constexpr int kNHalf = kBN > 256 ? 256 : kBN;      // N of one MMA
  static constexpr uint32_t kTmemCols = kBN > 256 ? 512 : 256;
  static constexpr int kBBytes = (kBN / 64) * kBBox;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kSmem = kBarOff + 256 + 1024;  // + barriers + alignment slack
};

template <int kBN>
__global__ void __launch_bounds__(kThreads, 1)
    bmm_tc_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                  const __grid_constant__ CUtensorMap cmap, int K) {
  using C = BmmCfg<kBN>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + C::kStages;
  uint64_t* done = empty + C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM, g = blockIdx.z;
  const int ksteps = K / kBK;

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort = abort_flag;
  pdl_enter();   // the operands may come from the kernel before: everything below reads them

  if (warp == 0 && lane == 0) {
    // producer
    tma_prefetch_desc(&amap);
    tma_prefetch_desc(&bmap);
    int issued[C::kStages] = {};
    for (int ks = 0; ks < ksteps; ++ks) {
      const int s = ks % C::kStages;
      if (!mbar_wait(&empty[s], ((ks / C::kStages) & 1) ^ 1, abort)) break;
      unsigned char* st = smem + s * C::kStageBytes;
      mbar_arrive_expect_tx(&full[s], C::kStageBytes);
      tma_load_3d(st, &amap, &full[s], ks * kBK, m0, g);
      for (int j = 0; j < kBN / 64; ++j) tma_load_3d(st + kABytes + j * kBBox, &bmap, &full[s], n0 + 64 * j, ks * kBK, g);
      ++issued[s];
    }
    volatile int dummy = 0;
    for (int s = 0; s < C::kStages; ++s)
      if (issued[s] > 0 && !mbar_wait(&full[s], (issued[s] - 1) & 1, &dummy)) atomicOr(&g_bmm_err, kErrTimeout);
  } else if (warp == 1) {
    // MMA issuer: the converged warp walks the k-steps, one elected lane issues
    constexpr uint32_t idesc = idesc_bf16(kBM, C::kNHalf, false, true);
    bool ok = true;
    for (int ks = 0; ks < ksteps && ok; ++ks) {
      const int s = ks % C::kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (ks / C::kStages) & 1, abort));
      if (!ok) break;
      tc_fence_after();
      const uint32_t a = smem_u32(smem + s * C::kStageBytes), b = a + kABytes;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
#pragma unroll
        for (int h = 0; h < kBN / C::kNHalf; ++h)   // N halves: accumulators at columns 0 and 256
          umma_bf16_elect(tmem + h * C::kNHalf, sdesc_sw128(a + kk * 32, 16, 1024),
                          sdesc_sw128(b + h * (C::kNHalf / 64) * kBBox + kk * 16 * 128, kBBox, 1024), idesc,
                          (ks | kk) ? 1u : 0u);
      umma_commit_elect(&empty[s]);
    }
    umma_commit_elect(done);
    volatile int dummy = 0;
    if (!mbar_wait(done, 0, &dummy) && lane == 0) atomicOr(&g_bmm_err, kErrTimeout);
  }
  __syncwarp();
  // epilogue: every thread owns one row (TMEM lane) of the tile
  const bool ok = mbar_wait(done, 0, abort);
  tc_fence_after();
  __syncthreads();   // the pipeline stages are free: reuse them as the staging tile
  if (ok) {
    const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
    for (int c = 0; c < kBN; c += 32) {
      float v[32];
      tmem_ld32(tmem + lane_addr + c, v);
      tmem_ld_wait();
      unsigned char* box = smem + (c / 64) * (kBM * 128);
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        uint4 w;
        __nv_bfloat162 h0 = __floats2bfloat162_rn(v[i], v[i + 1]);
        __nv_bfloat162 h1 = __floats2bfloat162_rn(v[i + 2], v[i + 3]);
        __nv_bfloat162 h2 = __floats2bfloat162_rn(v[i + 4], v[i + 5]);
        __nv_bfloat162 h3 = __floats2bfloat162_rn(v[i + 6], v[i + 7]);
        w.x = *reinterpret_cast<uint32_t*>(&h0);
        w.y = *reinterpret_cast<uint32_t*>(&h1);
        w.z = *reinterpret_cast<uint32_t*>(&h2);
        w.w = *reinterpret_cast<uint32_t*>(&h3);
        const int chunk = ((c % 64) + i) / 8;   // 16-byte chunk within the 128-byte row
        *reinterpret_cast<uint4*>(box + tid * 128 + ((chunk ^ (tid & 7)) << 4)) = w;
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    if (ok) {
      for (int j = 0; j < kBN / 64; ++j) tma_store_3d(&cmap, smem + j * (kBM * 128), n0 + 64 * j, m0, g);
      bulk_commit_group();
      bulk_wait_read_all();
    } else {
      atomicOr(&g_bmm_err, kErrTimeout);
    }
  }
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over a [n2, n1, n0] view with element strides (s2, s1, 1), box (b0, b1, 1).
bool map3(CUtensorMap* m, const void* base, int64_t n0, int64_t n1, int64_t n2, int64_t s1, int64_t s2, uint32_t b0,
          uint32_t b1) {
  auto fn = encode();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)n0, (cuuint64_t)n1, (cuuint64_t)n2};
  cuuint64_t strides[2] = {(cuuint64_t)s1 * 2, (cuuint64_t)s2 * 2};
  cuuint32_t box[3] = {b0, b1, 1}, es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kBN>
cudaError_t launch(const CUtensorMap& am, const CUtensorMap& bm, const CUtensorMap& cm, int G, int M, int N, int K,
                   cudaStream_t st) {
  using C = BmmCfg<kBN>;
  cudaError_t e = cudaFuncSetAttribute(bmm_tc_kernel<kBN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid(N / kBN, (M + kBM - 1) / kBM, G);
  return launch_k(bmm_tc_kernel<kBN>, grid, kThreads, C::kSmem, st, am, bm, cm, K);
}

}  // namespace

bool bmm_tc_supported(mla_dtype dt, const View3& out, const View3& a, const View3& b) {
  if (dt != MLA_BF16 || !encode()) return false;
  const int64_t K = a.n2, N = b.n2;
  if (K % 64 != 0 || N % 128 != 0 || a.n1 < 1) return false;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!al16(out.data) || !al16(a.data) || !al16(b.data)) return false;
  if (a.s0 % 8 || a.s1 % 8 || b.s0 % 8 || b.s1 % 8 || out.s0 % 8 || out.s1 % 8) return false;
  if (a.n0 > 65535 || a.n1 > 65535LL * kBM) return false;
  return true;
}

cudaError_t launch_bmm_tc(const View3& out, const View3& a, const View3& b, cudaStream_t st) {
  const int G = (int)a.n0, M = (int)a.n1, K = (int)a.n2, N = (int)b.n2;
  const int tiles_per_head_m = (M + kBM - 1) / kBM;
  const int bn = (N % 512 == 0 && (long long)G * tiles_per_head_m <= device_sm_count()) ? 512
                 : N % 256 == 0                                                  ? 256
                                                                                 : 128;
  CUtensorMap am, bm, cm;
  if (!map3(&am, a.data, K, M, G, a.s1, a.s0, 64, kBM) || !map3(&bm, b.data, N, K, G, b.s1, b.s0, 64, kBK) ||
      !map3(&cm, out.data, N, M, G, out.s1, out.s0, 64, kBM))
    return cudaErrorInvalidValue;
  if (bn == 512) return launch<512>(am, bm, cm, G, M, N, K, st);
  return bn == 256 ? launch<256>(am, bm, cm, G, M, N, K, st) : launch<128>(am, bm, cm, G, M, N, K, st);
}

namespace {
// One warp waits, with the bounded wait every kernel of the library uses, on an mbarrier that
// nothing arrives on; when the wait gives up it records kErrTimeout like any kernel would.
__global__ void wait_check_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  pdl_enter();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = mbar_wait(&bar, 0, &abort_flag, limit_ns);
  if (!ok && threadIdx.x == 0) atomicOr(&g_bmm_err, kErrTimeout);
}
}  // namespace

cudaError_t launch_wait_check(uint32_t limit_us, cudaStream_t st) {
  return launch_k(wait_check_kernel, 1, 32, 0, st, (uint64_t)limit_us * 1000ull);
}

unsigned bmm_tc_errors_read_clear() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_bmm_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_bmm_err, &zero, sizeof(zero));
  return v;
}

}  // namespace mla
