// Steps 1 and 5 on CUDA cores: out[g,m,n] = sum_k a[g,m,k] * b[g,k,n].
//
// The general path for any shape, stride and dtype (and the fp32 path, where
// tensor-core tf32 would not meet an fp32 bound). One CTA owns 8 rows of `a`
// (staged in shared memory as fp32) and 256 columns of one head's weight; each
// thread keeps 8 x 2 fp32 accumulators and walks k, reading the weight row k
// coalesced across the warp. Weights are read once per 8 rows.
#include <cuda_bf16.h>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kRows = 8;
constexpr int kThreads = 128;
constexpr int kCols = 2 * kThreads;

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float v) { *p = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T>
__global__ void __launch_bounds__(kThreads) bmm_simt_kernel(
    T* __restrict__ out, int64_t o_s0, int64_t o_s1, const T* __restrict__ a, int64_t a_s0,
    int64_t a_s1, const T* __restrict__ b, int64_t b_s0, int64_t b_s1, int M, int K, int N) {
  extern __shared__ float a_sm[];  // [kRows][K]
  pdl_enter();
  const int g = blockIdx.y;
  const int m0 = blockIdx.z * kRows;
  const int n0 = blockIdx.x * kCols;
  const int rows = min(kRows, M - m0);
  for (int i = threadIdx.x; i < kRows * K; i += kThreads) {
    const int r = i / K, k = i - r * K;
    a_sm[i] = r < rows ? ld(a + g * a_s0 + (int64_t)(m0 + r) * a_s1 + k) : 0.f;
  }
  __syncthreads();
  const int c0 = n0 + threadIdx.x, c1 = c0 + kThreads;
  const bool v0 = c0 < N, v1 = c1 < N;
  float acc[kRows][2];
#pragma unroll
  for (int r = 0; r < kRows; ++r) acc[r][0] = acc[r][1] = 0.f;
  const T* bg = b + g * b_s0;
  for (int k = 0; k < K; ++k) {
    const float w0 = v0 ? ld(bg + (int64_t)k * b_s1 + c0) : 0.f;
    const float w1 = v1 ? ld(bg + (int64_t)k * b_s1 + c1) : 0.f;
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const float x = a_sm[r * K + k];
      acc[r][0] = fmaf(x, w0, acc[r][0]);
      acc[r][1] = fmaf(x, w1, acc[r][1]);
    }
  }
  for (int r = 0; r < rows; ++r) {
    T* o = out + g * o_s0 + (int64_t)(m0 + r) * o_s1;
    if (v0) st(o + c0, acc[r][0]);
    if (v1) st(o + c1, acc[r][1]);
  }
}

}  // namespace

cudaError_t launch_bmm_simt(mla_dtype dt, const View3& out, const View3& a, const View3& b,
                            cudaStream_t st) {
  const int G = (int)a.n0, M = (int)a.n1, K = (int)a.n2, N = (int)b.n2;
  dim3 grid((N + kCols - 1) / kCols, G, (M + kRows - 1) / kRows);
  const size_t smem = sizeof(float) * kRows * K;
  if (dt == MLA_F32) {
    auto k = bmm_simt_kernel<float>;
    if (smem > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_k(k, grid, kThreads, smem, st, (float*)out.data, out.s0, out.s1, (const float*)a.data, a.s0,
                    a.s1, (const float*)b.data, b.s0, b.s1, M, K, N);
  } else {
    auto k = bmm_simt_kernel<__nv_bfloat16>;
    if (smem > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_k(k, grid, kThreads, smem, st, (__nv_bfloat16*)out.data, out.s0, out.s1,
                    (const __nv_bfloat16*)a.data, a.s0, a.s1, (const __nv_bfloat16*)b.data, b.s0, b.s1, M, K, N);
  }
  return cudaGetLastError();
}

}  // namespace mla
