// Step 4 on CUDA cores: the split-KV schedule, the LSE combine, and the general
// (any head count, any dtype) decode and prefill kernels.
//
// Schedule. The batch's context is cut into tiles of kTile rows; sequence b
// owns ceil(len_b / kTile) tiles and tile_prefix is their prefix sum. The W
// work units take contiguous global tile ranges [unit_tile[w], unit_tile[w+1])
// of equal cost, where a sequence costs its tiles plus kSeqCost for its start
// (starting a sequence drains and refills the attention pipeline: about as
// long as kSeqCost tiles), so units that hold many short sequences get fewer
// tiles; a unit may get none. A unit that covers a whole sequence writes the
// final output; a sequence cut across n > 1 units gets n partial slots
// (normalised o and LSE), merged afterwards by the combine kernel. The
// schedule depends only on the lengths and W: results are run-to-run
// bit-identical and do not depend on the cache strides.
//
// SIMT attention. One CTA holds the queries of a group of up to 16 heads of one
// token in shared memory (fp32), streams the key rows of its range in tiles of
// 32 (through the block table), computes the 16 x 32 scores, runs the online
// softmax per head with warp shuffles and accumulates o_lat (each thread owns
// 2 latent columns of every head of the group).
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <math_constants.h>

#include <algorithm>

#include "mla_internal.h"

namespace mla {
namespace {

__device__ unsigned g_attn_err = 0;

constexpr int kHeads = 16;    // heads per CTA
constexpr int kKeys = 32;     // keys per inner tile
constexpr int kThreads = 256;

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
// an fp8 cache holds e4m3 codes; their values are exact in float
__device__ __forceinline__ float ld(const uint8_t* p) {
  __nv_fp8_e4m3 v;
  v.__x = *p;
  return static_cast<float>(v);
}
__device__ __forceinline__ void st(float* p, float v) { *p = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// ---------------------------------------------------------------------------
// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32, at most 1024).
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  const int nwarps = blockDim.x >> 5;
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
  *total = warp_tot[nwarps - 1];
  __syncthreads();
  return before;
}

// A null length array gives every sequence cap rows (a sparse query's index list).
__device__ __forceinline__ int clamp_len(const int32_t* seq_lens, int b, int cap) {
  if (seq_lens == nullptr) return cap;
  int n = seq_lens[b];
  if (n < 0 || n > cap) {
    atomicOr(&g_attn_err, kErrDeviceData);
    n = n < 0 ? 0 : cap;
  }
  return n;
}

constexpr int kSeqCost = 6;   // cost of starting a sequence, in tiles (measured)

// The unit whose range holds global tile t: the last w with unit_tile[w] <= t (units with
// empty ranges sit only at sequence starts, so this is never an empty unit).
__device__ __forceinline__ int unit_of(const int32_t* unit_tile, int W, int t) {
  int lo = 0, hi = W - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (unit_tile[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The prefix arrays live in shared memory while the batch fits (the binary searches then cost
// no global round trips); larger batches work on the workspace arrays directly.
constexpr int kSchedSmemSeqs = 2048;
constexpr int kSchedSmemUnits = 1024;

__global__ void __launch_bounds__(1024) decode_schedule_kernel(const int32_t* __restrict__ seq_lens,
                                                               int B, int cap, DecodeSched s) {
  __shared__ int warp_tot[32];
  __shared__ int carry_sh, starts_sh;
  __shared__ int pre_sh[kSchedSmemSeqs + 1], nz_sh[kSchedSmemSeqs + 1], ut_sh[kSchedSmemUnits + 1];
  __shared__ int len_sh[kSchedSmemSeqs];   // clamped lengths, read from global memory once
  pdl_enter();
  const int W = s.units;
  const bool seqs_in_smem = B <= kSchedSmemSeqs, units_in_smem = W <= kSchedSmemUnits;
  int* pre = seqs_in_smem ? pre_sh : s.tile_prefix;   // tile prefix
  int* nzb = seqs_in_smem ? nz_sh : s.first_unit;     // sequences with tiles before b
  int* ut = units_in_smem ? ut_sh : s.unit_tile;      // unit boundaries
  if (threadIdx.x == 0) {
    carry_sh = 0;
    starts_sh = 0;
  }
  __syncthreads();
  // pass 1: tile prefix
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    const int len = b < B ? clamp_len(seq_lens, b, cap) : 0;
    if (seqs_in_smem && b < B) len_sh[b] = len;
    const int n = (len + kTile - 1) / kTile;
    int tot;
    const int ex = block_exclusive_scan(n, warp_tot, &tot);
    const int carry = carry_sh;
    if (b < B) pre[b] = carry + ex;
    __syncthreads();
    if (threadIdx.x == 0) carry_sh = carry + tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) pre[B] = carry_sh;
  __syncthreads();
  const int total = carry_sh;
  // the number of sequences with tiles before each b
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    const int nz = b < B && pre[b + 1] > pre[b] ? 1 : 0;
    int tot;
    const int ex = block_exclusive_scan(nz, warp_tot, &tot);
    const int carry = starts_sh;
    if (b < B) nzb[b] = carry + ex;
    __syncthreads();
    if (threadIdx.x == 0) starts_sh = carry + tot;
    __syncthreads();
  }
  const int starts = starts_sh;
  // unit boundaries: unit w < We = min(W, total) starts at cost floor(w * C / We),
  // C = total + kSeqCost * starts; sequence b spans costs [cost_b, cost_b + (kSeqCost if it
  // has tiles) + tiles_b) with cost_b = tile_prefix[b] + kSeqCost * (sequences with tiles
  // before b). C >= We, so boundaries inside a sequence's tiles are distinct; units from We
  // on get empty ranges at the end
  const long long C = (long long)total + (long long)kSeqCost * starts;
  const int We = min(W, total);
  for (int w = threadIdx.x; w <= W; w += blockDim.x) {
    if (w >= We) {
      ut[w] = total;
      continue;
    }
    const long long x = ((long long)w * C) / We;
    int lo = 0, hi = B;   // the last b with cost_b <= x (cost_B = C)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      const long long cm = pre[mid] + (long long)kSeqCost * (mid < B ? nzb[mid] : starts);
      if (cm <= x) lo = mid; else hi = mid - 1;
    }
    int t = total;
    if (lo < B) {
      const int tiles = pre[lo + 1] - pre[lo];
      const long long into = x - (pre[lo] + (long long)kSeqCost * nzb[lo]) - (tiles > 0 ? kSeqCost : 0);
      t = pre[lo] + (int)(into < 0 ? 0 : (into > tiles ? tiles : into));
    }
    ut[w] = t;
  }
  __syncthreads();
  // the first sequence of each unit's range: the b with pre[b] <= unit_tile[w] < pre[b + 1]
  for (int w = threadIdx.x; w < W; w += blockDim.x) {
    const int t0 = ut[w];
    int bw = B;
    if (t0 < total && t0 < ut[w + 1]) {
      int lo = 0, hi = B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= t0) lo = mid; else hi = mid - 1;
      }
      bw = lo;
    }
    s.unit_seq[w] = bw;
  }
  if (threadIdx.x == 0) carry_sh = 0;
  __syncthreads();
  // pass 2: units touching each sequence, and partial-slot bases
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int np = 0, fu = 0;
    if (b < B) {
      const int t0 = pre[b], t1 = pre[b + 1];
      if (t1 > t0) {
        fu = unit_of(ut, W, t0);
        np = unit_of(ut, W, t1 - 1) - fu + 1;
      }
    }
    // every thread has read nzb (which may alias first_unit) before any first_unit is written
    __syncthreads();
    if (b < B) {
      s.first_unit[b] = fu;
      s.npieces[b] = np;
    }
    int tot;
    const int ex = block_exclusive_scan(np > 1 ? np : 0, warp_tot, &tot);
    const int carry = carry_sh;
    if (b < B) {
      s.piece_base[b] = carry + ex;
      // everything a tensor-core walker needs about b in one 16-byte load
      const int len = seqs_in_smem ? len_sh[b] : (seq_lens == nullptr ? cap : min(max(seq_lens[b], 0), cap));
      s.seqinfo[b] = make_int4(pre[b], len, np, carry + ex - fu);
    }
    __syncthreads();
    if (threadIdx.x == 0) carry_sh = carry + tot;
    __syncthreads();
  }
  // the staged arrays out to the workspace
  if (seqs_in_smem)
    for (int b = threadIdx.x; b <= B; b += blockDim.x) s.tile_prefix[b] = pre_sh[b];
  if (units_in_smem)
    for (int w = threadIdx.x; w <= W; w += blockDim.x) s.unit_tile[w] = ut_sh[w];
}

// ---------------------------------------------------------------------------
// Attention of one query token (heads [h0, h0+hn)) over cache rows [k0, k1).
// Returns per thread the unnormalised accumulators, and in shared memory the
// running max m_sh and denominator l_sh of each head.
// Shared memory of the SIMT attention: q [kHeads][E+1] and k [kKeys][E+1] fp32
// (odd pitch: a warp reading one column of 32 rows hits 32 banks), then the
// probabilities and the per-head softmax state.
struct SimtSmem {
  int64_t* kbase;   // [kKeys] offset of each staged key row's first element (-1: not attended)
  float* q;
  float* k;
  float (*p)[kKeys];
  float* m;
  float* l;
  float* alpha;
  int pitch;
};

__host__ __device__ inline size_t simt_smem_bytes(int E) {
  const int pitch = E + 1;
  return sizeof(int64_t) * kKeys +
         sizeof(float) * ((size_t)(kHeads + kKeys) * pitch + kHeads * kKeys + 3 * kHeads);
}

__device__ inline SimtSmem simt_smem(unsigned char* raw, int E) {
  SimtSmem s;
  s.pitch = E + 1;
  s.kbase = reinterpret_cast<int64_t*>(raw);
  float* f = reinterpret_cast<float*>(s.kbase + kKeys);
  s.q = f;
  s.k = s.q + kHeads * s.pitch;
  s.p = reinterpret_cast<float(*)[kKeys]>(s.k + kKeys * s.pitch);
  s.m = reinterpret_cast<float*>(s.p + kHeads);
  s.l = s.m + kHeads;
  s.alpha = s.l + kHeads;
  return s;
}

// Where the key rows of one query come from. row(t) gives the element offset of the query's
// t-th row (-1 if that row is not attended; a bad block id or slot is reported too) and
// at(base, e) the value of its element e.
//
// Paged rows of a sequence: row t sits in block bt_row[t / page] at row t % page; K is the
// cache's element type (T, or e4m3 codes read as value * dk).
template <typename K>
struct PagedRows {
  const K* cache;
  CacheView cv;
  const int32_t* bt_row;
  float dk;
  __device__ int64_t row(int t) const {
    const int blk = bt_row[t / cv.page];
    if (blk < 0 || blk >= cv.num_blocks) {
      atomicOr(&g_attn_err, kErrDeviceData);
      return -1;
    }
    return (int64_t)blk * cv.s_blk + (int64_t)(t % cv.page) * cv.s_row;
  }
  __device__ float at(int64_t base, int e) const { return ld(cache + base + e) * dk; }
};

// The listed slots of a sparse query over a ds_mla cache (656-byte entries: 512 e4m3 latent
// codes, four float32 scales each covering 128 latent columns, 64 bf16 rope values): row t is
// slot idx_row[t] (block slot / page, row slot % page); negative slots are padding.
struct DsMlaRows {
  const uint8_t* cache;   // byte addressed
  int64_t s_blk, s_row;   // bytes
  int32_t page;
  int64_t num_rows;
  const int32_t* idx_row;
  __device__ int64_t row(int t) const {
    const int slot = idx_row[t];
    if (slot < 0) return -1;
    if (slot >= num_rows) {
      atomicOr(&g_attn_err, kErrDeviceData);
      return -1;
    }
    return (int64_t)(slot / page) * s_blk + (int64_t)(slot % page) * s_row;
  }
  __device__ float at(int64_t base, int e) const {
    const uint8_t* p = cache + base;
    if (e < kDsMlaLatent)
      return ld(p + e) * *reinterpret_cast<const float*>(p + kDsMlaLatent + 4 * (e / kDsMlaGroup));
    return ld(reinterpret_cast<const __nv_bfloat16*>(p + kDsMlaRopeByte) + (e - kDsMlaLatent));
  }
};

// Rows [k0, k1) of one query through the row source; the query is multiplied by dq as it is
// staged (the dequantisation of an fp8 query scale; 1 else).
template <typename T, typename Rows>
__device__ void attend_rows(const SimtSmem& sm, const T* __restrict__ q_row, int64_t q_s_head,
                            int h0, int hn, int E, int L, const Rows& rows, int k0, int k1, float scale,
                            float (&acc)[kHeads][2], float dq = 1.f) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = sm.pitch;
  __syncthreads();  // the previous segment's epilogue may still read m and l
  for (int i = tid; i < kHeads * E; i += kThreads) {
    const int h = i / E, e = i - h * E;
    sm.q[h * P + e] = h < hn ? ld(q_row + (int64_t)(h0 + h) * q_s_head + e) * dq : 0.f;
  }
  if (tid < kHeads) {
    sm.m[tid] = -CUDART_INF_F;
    sm.l[tid] = 0.f;
  }
#pragma unroll
  for (int h = 0; h < kHeads; ++h) acc[h][0] = acc[h][1] = 0.f;
  for (int kt = k0; kt < k1; kt += kKeys) {
    __syncthreads();
    // where key rows kt .. kt+31 live (rows past k1 and unattended rows: -1, zero and masked)
    if (tid < kKeys) sm.kbase[tid] = kt + tid < k1 ? rows.row(kt + tid) : -1;
    __syncthreads();
    for (int i = tid; i < kKeys * E; i += kThreads) {
      const int j = i / E, e = i - j * E;
      const int64_t base = sm.kbase[j];
      sm.k[j * P + e] = base >= 0 ? rows.at(base, e) : 0.f;
    }
    __syncthreads();
    // scores: warp w owns heads 2w, 2w+1; lane owns key kt + lane
    for (int hh = 0; hh < 2; ++hh) {
      const int h = 2 * warp + hh;
      float s = 0.f;
      for (int e = 0; e < E; ++e) s = fmaf(sm.q[h * P + e], sm.k[lane * P + e], s);
      s = sm.kbase[lane] >= 0 ? s * scale : -CUDART_INF_F;
      float mx = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_old = sm.m[h];
      const float m_new = fmaxf(m_old, mx);
      const float p = (s == -CUDART_INF_F) ? 0.f : __expf(s - m_new);
      float sum = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      sm.p[h][lane] = p;
      __syncwarp();
      if (lane == 0) {
        const float a = (m_old == -CUDART_INF_F) ? 0.f : __expf(m_old - m_new);
        sm.alpha[h] = a;
        sm.l[h] = sm.l[h] * a + sum;
        sm.m[h] = m_new;
      }
    }
    __syncthreads();
    // o_lat accumulators: thread owns latent columns tid and tid + 256 of every head
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int l = tid + c * kThreads;
      if (l < L) {
        float kv[kKeys];
#pragma unroll
        for (int j = 0; j < kKeys; ++j) kv[j] = sm.k[j * P + l];
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          float a = acc[h][c] * sm.alpha[h];
#pragma unroll
          for (int j = 0; j < kKeys; ++j) a = fmaf(sm.p[h][j], kv[j], a);
          acc[h][c] = a;
        }
      }
    }
  }
  __syncthreads();
}

// The row sources of the split kernel, one per query: a paged sequence through its block-table
// row, or a sparse query's index list.
template <typename K>
struct PagedSource {
  CacheView cv;
  const int32_t* block_table;
  int64_t bt_stride;
  const float* descale_k;
  __device__ PagedRows<K> rows(int b) const {
    return PagedRows<K>{static_cast<const K*>(cv.data), cv, block_table + (int64_t)b * bt_stride,
                        descale_k != nullptr ? *descale_k : 1.f};
  }
};

struct DsMlaSource {
  const uint8_t* cache;
  int64_t s_blk, s_row;
  int32_t page;
  int64_t num_rows;
  const int32_t* indices;
  int64_t idx_stride;
  __device__ DsMlaRows rows(int b) const {
    return DsMlaRows{cache, s_blk, s_row, page, num_rows, indices + (int64_t)b * idx_stride};
  }
};

// One work unit's tile range: every sequence segment in it is attended by attend_rows and
// written whole (o_lat, lse) or as a partial slot for the combine. A null seq_lens gives every
// query cap rows.
template <typename T, typename Source>
__global__ void __launch_bounds__(kThreads) decode_split_simt_kernel(
    T* __restrict__ o_lat, int64_t o_s0, int64_t o_s1, float* __restrict__ lse_out,
    const T* __restrict__ q, int64_t q_s0, int64_t q_s1, Source src,
    const int32_t* __restrict__ seq_lens, int cap, int B, int H, int L, int R, float scale,
    DecodeSched s, const float* __restrict__ descale_q) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  pdl_enter();
  const float dq = descale_q != nullptr ? *descale_q : 1.f;
  const SimtSmem sm = simt_smem(smem_raw, L + R);
  const int w = blockIdx.x;
  const int t0 = s.unit_tile[w], t1 = s.unit_tile[w + 1];
  if (t0 >= t1) return;
  const int h0 = blockIdx.y * kHeads, hn = min(kHeads, H - h0);
  const int E = L + R;
  // first sequence: the last b with tile_prefix[b] <= t0
  int lo = 0, hi = B;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.tile_prefix[mid] <= t0) lo = mid; else hi = mid - 1;
  }
  int b = lo;
  float acc[kHeads][2];
  for (int t = t0; t < t1;) {
    while (s.tile_prefix[b + 1] <= t) ++b;
    const int seg_end = min(t1, s.tile_prefix[b + 1]);
    const int len = seq_lens == nullptr ? cap : min(max(seq_lens[b], 0), cap);
    const int k0 = (t - s.tile_prefix[b]) * kTile;
    const int k1 = min((seg_end - s.tile_prefix[b]) * kTile, len);
    attend_rows(sm, q + (int64_t)b * q_s0, q_s1, h0, hn, E, L, src.rows(b), k0, k1, scale, acc, dq);
    const bool whole = s.npieces[b] == 1;
    const int slot = whole ? 0 : s.piece_base[b] + (w - s.first_unit[b]);
    for (int h = 0; h < hn; ++h) {
      const float l = sm.l[h];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? sm.m[h] + logf(l) : -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col = threadIdx.x + c * kThreads;
        if (col < L) {
          const float v = acc[h][c] * inv;
          if (whole)
            st(o_lat + (int64_t)b * o_s0 + (int64_t)(h0 + h) * o_s1 + col, v);
          else
            s.part_o[((int64_t)slot * H + h0 + h) * L + col] = v;
        }
      }
      if (threadIdx.x == 0) {
        if (whole) {
          if (lse_out) lse_out[(int64_t)b * H + h0 + h] = lse;
        } else {
          s.part_lse[(int64_t)slot * H + h0 + h] = lse;
        }
      }
    }
    t = seg_end;
  }
}

// Merge the partials of every sequence cut across several units; write o = 0
// and lse = -inf for empty sequences. One warp per (sequence, head); each lane
// combines 16-byte chunks of the rows with weights e^(lse_i - max).
template <typename T>
__device__ __forceinline__ void store4(T* o, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* o, float4 v) {
  *reinterpret_cast<float4*>(o) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* o, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&a);
  w.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(o) = w;
}

template <typename T>
__global__ void __launch_bounds__(128) decode_combine_kernel(
    T* __restrict__ o_lat, int64_t o_s0, int64_t o_s1, float* __restrict__ lse_out,
    int B, int H, int L, DecodeSched s) {
  const int b = blockIdx.x;
  const int h = blockIdx.y * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (h >= H) return;
  // a sequence's piece count and first slot come from the schedule kernel two launches back,
  // complete before this kernel can launch (the split kernel between waits for it before it
  // lets dependents launch): read before this kernel's wait; the partials only after it
  const int np = s.npieces[b];
  const int base = s.piece_base[b];   // loaded beside np: one memory latency for both
  if (np == 1) return;
  pdl_enter();
  T* o = o_lat + (int64_t)b * o_s0 + (int64_t)h * o_s1;
  if (np == 0) {
    for (int c = lane; c < L; c += 32) st(o + c, 0.f);
    if (lane == 0 && lse_out) lse_out[(int64_t)b * H + h] = -CUDART_INF_F;
    return;
  }
  const float* lse_p = s.part_lse + (int64_t)base * H + h;
  const int64_t pstride = (int64_t)H * L;
  const bool vec = (L % 4 == 0) && ((o_s0 | o_s1) % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(o_lat) % (4 * sizeof(T)) == 0);
  if (vec && L == 512 && np <= 4) {
    // up to four pieces: their maxima and their rows are loaded together, so the warp waits
    // one memory latency in all; the arithmetic is the general path's, in the same order
    const float* part = s.part_o + ((int64_t)base * H + h) * L;
    float li[4];
    float4 v[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      li[i] = i < np ? lse_p[(int64_t)i * H] : -CUDART_INF_F;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        v[i][k] = i < np ? *reinterpret_cast<const float4*>(part + i * pstride + lane * 4 + k * 128)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float m = -CUDART_INF_F;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i < np) m = fmaxf(m, li[i]);
    float wi[4], tot = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      wi[i] = li[i] == -CUDART_INF_F ? 0.f : __expf(li[i] - m);
      if (i < np) tot += wi[i];
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[k].x = fmaf(wi[i], v[i][k].x, acc[k].x);
        acc[k].y = fmaf(wi[i], v[i][k].y, acc[k].y);
        acc[k].z = fmaf(wi[i], v[i][k].z, acc[k].z);
        acc[k].w = fmaf(wi[i], v[i][k].w, acc[k].w);
      }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      store4<T>(o + lane * 4 + k * 128, make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv));
    if (lane == 0 && lse_out) lse_out[(int64_t)b * H + h] = tot > 0.f ? m + logf(tot) : -CUDART_INF_F;
    return;
  }
  float m = -CUDART_INF_F;
  for (int i = 0; i < np; ++i) m = fmaxf(m, lse_p[(int64_t)i * H]);
  float tot = 0.f;
  for (int i = 0; i < np; ++i) {
    const float li = lse_p[(int64_t)i * H];
    tot += li == -CUDART_INF_F ? 0.f : __expf(li - m);
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  const float* part = s.part_o + ((int64_t)base * H + h) * L;
  if (vec && L == 512) {
    // each lane owns four 16-byte chunks of the row; every load of a group of up to four
    // pieces is issued before any of them is used, so the warp waits one memory latency
    // per group instead of one per piece and chunk
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < np; i0 += 4) {
      float4 v[4][4];
      float wi[4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const int i = i0 + ii;
        const float li = i < np ? lse_p[(int64_t)i * H] : -CUDART_INF_F;
        wi[ii] = li == -CUDART_INF_F ? 0.f : __expf(li - m);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[ii][k] = i < np ? *reinterpret_cast<const float4*>(part + i * pstride + lane * 4 + k * 128)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[k].x = fmaf(wi[ii], v[ii][k].x, acc[k].x);
          acc[k].y = fmaf(wi[ii], v[ii][k].y, acc[k].y);
          acc[k].z = fmaf(wi[ii], v[ii][k].z, acc[k].z);
          acc[k].w = fmaf(wi[ii], v[ii][k].w, acc[k].w);
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      store4<T>(o + lane * 4 + k * 128, make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv));
  } else if (vec) {
    for (int c = lane * 4; c < L; c += 128) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = 0; i < np; ++i) {
        const float li = lse_p[(int64_t)i * H];
        const float wi = li == -CUDART_INF_F ? 0.f : __expf(li - m);
        const float4 v = *reinterpret_cast<const float4*>(part + i * pstride + c);
        acc.x = fmaf(wi, v.x, acc.x);
        acc.y = fmaf(wi, v.y, acc.y);
        acc.z = fmaf(wi, v.z, acc.z);
        acc.w = fmaf(wi, v.w, acc.w);
      }
      store4<T>(o + c, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    }
  } else {
    for (int c = lane; c < L; c += 32) {
      float acc = 0.f;
      for (int i = 0; i < np; ++i) {
        const float li = lse_p[(int64_t)i * H];
        const float wi = li == -CUDART_INF_F ? 0.f : __expf(li - m);
        acc = fmaf(wi, part[i * pstride + c], acc);
      }
      st(o + c, acc * inv);
    }
  }
  if (lane == 0 && lse_out) lse_out[(int64_t)b * H + h] = tot > 0.f ? m + logf(tot) : -CUDART_INF_F;
}

// Causal prefill: one CTA per (query row, head group), no split.
template <typename T>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(
    T* __restrict__ o_lat, int64_t o_s0, int64_t o_s1, float* __restrict__ lse_out,
    const T* __restrict__ q, int64_t q_s0, int64_t q_s1, CacheView cv,
    const int32_t* __restrict__ block_table, int64_t bt_stride, int max_blocks,
    const int32_t* __restrict__ cu_q, const int32_t* __restrict__ kv_lens, int B, int H, int L,
    int R, float scale) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  pdl_enter();
  const SimtSmem sm = simt_smem(smem_raw, L + R);
  const int r = blockIdx.x;
  const int h0 = blockIdx.y * kHeads, hn = min(kHeads, H - h0);
  // the sequence holding global query row r: last b with cu_q[b] <= r
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_q[mid] <= r) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int q_len = cu_q[b + 1] - cu_q[b];
  const int i = r - cu_q[b];
  const int kv = clamp_len(kv_lens, b, max_blocks * cv.page);
  int end = 0;
  if (i >= 0 && i < q_len) end = min(kv, max(0, kv - q_len + i + 1));
  float acc[kHeads][2];
  const PagedRows<T> rows{static_cast<const T*>(cv.data), cv, block_table + (int64_t)b * bt_stride, 1.f};
  attend_rows(sm, q + (int64_t)r * q_s0, q_s1, h0, hn, L + R, L, rows, 0, end, scale, acc);
  for (int h = 0; h < hn; ++h) {
    const float l = sm.l[h];
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col = threadIdx.x + c * kThreads;
      if (col < L) st(o_lat + (int64_t)r * o_s0 + (int64_t)(h0 + h) * o_s1 + col, acc[h][c] * inv);
    }
    if (threadIdx.x == 0 && lse_out)
      lse_out[(int64_t)r * H + h0 + h] = l > 0.f ? sm.m[h] + logf(l) : -CUDART_INF_F;
  }
}

// A sparse query's index list, compacted: its valid slots (0 <= slot < num_rows) in listed
// order and their count; a slot past the cache is dropped and reported. One block a query:
// each thread loads up to kPer consecutive entries at once, and a block-wide exclusive scan of
// the per-thread counts places them, so a list costs one load round and one scan per
// blockDim * kPer entries.
constexpr int kCompactThreads = 256;
constexpr int kCompactPer = 8;
__global__ void __launch_bounds__(kCompactThreads) sparse_compact_kernel(const int32_t* __restrict__ idx,
                                                                         int64_t idx_stride, int topk, int B,
                                                                         int64_t num_rows, int32_t* __restrict__ out,
                                                                         int32_t* __restrict__ counts) {
  __shared__ int warp_tot[32];
  pdl_enter();
  const int q = blockIdx.x;
  if (q >= B) return;   // the whole block
  const int32_t* row = idx + (int64_t)q * idx_stride;
  int32_t* o = out + (int64_t)q * topk;
  int carry = 0;
  for (int base = 0; base < topk; base += kCompactThreads * kCompactPer) {
    const int t0 = base + threadIdx.x * kCompactPer;
    int v[kCompactPer];
    int n = 0;
#pragma unroll
    for (int i = 0; i < kCompactPer; ++i) {
      int slot = t0 + i < topk ? row[t0 + i] : -1;
      if (slot >= num_rows) {
        atomicOr(&g_attn_err, kErrDeviceData);
        slot = -1;
      }
      v[i] = slot;
      n += slot >= 0;
    }
    int tot;
    const int ex = block_exclusive_scan(n, warp_tot, &tot);
    int at = carry + ex;
#pragma unroll
    for (int i = 0; i < kCompactPer; ++i)
      if (v[i] >= 0) o[at++] = v[i];
    carry += tot;
  }
  if (threadIdx.x == 0) counts[q] = carry;
}

template <typename K>
void allow_smem(K k, size_t bytes) {
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

namespace {
// Row tiles per sequence of a prefill (ceil(query tokens / tpt), none for an empty one),
// prefix-summed into out[0..B]: one block, a block scan per blockDim sequences.
__global__ void __launch_bounds__(1024) prefill_items_kernel(const int32_t* __restrict__ cu_q, int B, int tpt,
                                                             int32_t* __restrict__ out) {
  __shared__ int warp_tot[32];
  pdl_enter();
  int carry = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int n = 0;
    if (b < B) {
      const int q = cu_q[b + 1] - cu_q[b];
      n = q > 0 ? (q + tpt - 1) / tpt : 0;
    }
    int tot;
    const int ex = block_exclusive_scan(n, warp_tot, &tot);
    if (b < B) out[b] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) out[B] = carry;
}
}  // namespace

cudaError_t launch_prefill_items(const int32_t* cu_q, int32_t B, int32_t tpt, int32_t* out, cudaStream_t st) {
  const int threads = std::min(1024, std::max(32, (B + 31) / 32 * 32));
  return launch_k(prefill_items_kernel, 1, threads, 0, st, cu_q, (int)B, (int)tpt, out);
}

cudaError_t launch_decode_schedule(const int32_t* seq_lens, int32_t B, int32_t max_blocks,
                                   int32_t page, const DecodeSched& s, cudaStream_t st) {
  const long long cap = (long long)max_blocks * page;
  // one thread per sequence or unit boundary, in whole warps: a small batch waits on few warps
  // at each of the kernel's barriers
  const int need = (int)std::max<int64_t>(B, (int64_t)s.units + 1);
  const int threads = std::min(1024, std::max(32, (need + 31) / 32 * 32));
  return launch_k(decode_schedule_kernel, 1, threads, 0, st, seq_lens, B, (int)(cap > INT32_MAX ? INT32_MAX : cap), s);
}

namespace {
template <typename T, typename Source>
cudaError_t launch_split_simt(const View3& o_lat, float* lse, const View3& q, const Source& src,
                              const int32_t* seq_lens, int cap, int32_t B, int32_t H, int32_t L, int32_t R,
                              float scale, const DecodeSched& s, const float* descale_q, cudaStream_t st) {
  const dim3 grid(s.units, (H + kHeads - 1) / kHeads);
  const size_t sm = simt_smem_bytes(L + R);
  allow_smem(decode_split_simt_kernel<T, Source>, sm);
  return launch_k(decode_split_simt_kernel<T, Source>, grid, kThreads, sm, st, (T*)o_lat.data, o_lat.s0,
                  o_lat.s1, lse, (const T*)q.data, q.s0, q.s1, src, seq_lens, cap, B, H, L, R, scale, s,
                  descale_q);
}

template <typename T>
cudaError_t launch_paged_simt(const View3& o_lat, float* lse, const View3& q, const CacheView& cache,
                              const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens, int cap,
                              int32_t B, int32_t H, int32_t L, int32_t R, float scale, const DecodeSched& s,
                              cudaStream_t st, bool fp8_cache, const float* descale_q, const float* descale_k) {
  if (fp8_cache)
    return launch_split_simt<T>(o_lat, lse, q, PagedSource<uint8_t>{cache, block_table, bt_stride, descale_k},
                                seq_lens, cap, B, H, L, R, scale, s, descale_q, st);
  return launch_split_simt<T>(o_lat, lse, q, PagedSource<T>{cache, block_table, bt_stride, descale_k}, seq_lens,
                              cap, B, H, L, R, scale, s, descale_q, st);
}
}  // namespace

cudaError_t launch_decode_simt(mla_dtype dt, const View3& o_lat, float* lse, const View3& q,
                               const CacheView& cache, const int32_t* block_table,
                               int64_t bt_stride, int32_t max_blocks, const int32_t* seq_lens, int32_t B, int32_t H,
                               int32_t L, int32_t R, float scale, const DecodeSched& s,
                               cudaStream_t st, bool fp8_cache, const float* descale_q, const float* descale_k) {
  const long long cap_ll = (long long)max_blocks * cache.page;
  const int cap = (int)(cap_ll > INT32_MAX ? INT32_MAX : cap_ll);
  if (dt == MLA_F32)
    return launch_paged_simt<float>(o_lat, lse, q, cache, block_table, bt_stride, seq_lens, cap, B, H, L, R, scale,
                                    s, st, fp8_cache, descale_q, descale_k);
  return launch_paged_simt<__nv_bfloat16>(o_lat, lse, q, cache, block_table, bt_stride, seq_lens, cap, B, H, L, R,
                                          scale, s, st, fp8_cache, descale_q, descale_k);
}

cudaError_t launch_decode_sparse_simt(mla_dtype dt, const View3& o_lat, float* lse, const View3& q,
                                      const DsMlaCache& cache, const int32_t* indices, int64_t idx_stride,
                                      int32_t topk, int32_t B, int32_t H, float scale, const DecodeSched& s,
                                      cudaStream_t st) {
  const DsMlaSource src{static_cast<const uint8_t*>(cache.data), cache.s_blk, cache.s_row, cache.page,
                        (int64_t)cache.num_blocks * cache.page, indices, idx_stride};
  if (dt == MLA_F32)
    return launch_split_simt<float>(o_lat, lse, q, src, nullptr, topk, B, H, kDsMlaLatent, kDsMlaRope, scale, s,
                                    nullptr, st);
  return launch_split_simt<__nv_bfloat16>(o_lat, lse, q, src, nullptr, topk, B, H, kDsMlaLatent, kDsMlaRope, scale,
                                          s, nullptr, st);
}

cudaError_t launch_decode_combine(mla_dtype dt, const View3& o_lat, float* lse,
                                  const int32_t* seq_lens, int32_t B, int32_t H, int32_t L,
                                  const DecodeSched& s, cudaStream_t st) {
  (void)seq_lens;
  const dim3 grid(B, (H + 3) / 4);
  if (dt == MLA_F32)
    return launch_k(decode_combine_kernel<float>, grid, 128, 0, st, (float*)o_lat.data, o_lat.s0, o_lat.s1, lse,
                    B, H, L, s);
  return launch_k(decode_combine_kernel<__nv_bfloat16>, grid, 128, 0, st, (__nv_bfloat16*)o_lat.data, o_lat.s0,
                  o_lat.s1, lse, B, H, L, s);
}

cudaError_t launch_prefill_simt(mla_dtype dt, const View3& o_lat, float* lse, const View3& q,
                                const CacheView& cache, const int32_t* block_table,
                                int64_t bt_stride, int32_t max_blocks, const int32_t* cu_q,
                                const int32_t* kv_lens, int32_t B, int32_t T, int32_t H,
                                int32_t L, int32_t R, float scale, cudaStream_t st) {
  const dim3 grid(T, (H + kHeads - 1) / kHeads);
  const size_t sm = simt_smem_bytes(L + R);
  if (dt == MLA_F32) {
    allow_smem(prefill_simt_kernel<float>, sm);
    return launch_k(prefill_simt_kernel<float>, grid, kThreads, sm, st,
        (float*)o_lat.data, o_lat.s0, o_lat.s1, lse, (const float*)q.data, q.s0, q.s1, cache,
        block_table, bt_stride, max_blocks, cu_q, kv_lens, B, H, L, R, scale);
  } else {
    allow_smem(prefill_simt_kernel<__nv_bfloat16>, sm);
    return launch_k(prefill_simt_kernel<__nv_bfloat16>, grid, kThreads, sm, st,
        (__nv_bfloat16*)o_lat.data, o_lat.s0, o_lat.s1, lse, (const __nv_bfloat16*)q.data, q.s0,
        q.s1, cache, block_table, bt_stride, max_blocks, cu_q, kv_lens, B, H, L, R, scale);
  }
  return cudaGetLastError();
}

cudaError_t launch_sparse_compact(const int32_t* indices, int64_t idx_stride, int32_t topk, int32_t B,
                                  int64_t num_rows, int32_t* out, int32_t* counts, cudaStream_t st) {
  return launch_k(sparse_compact_kernel, (int)B, kCompactThreads, 0, st, indices, idx_stride, (int)topk, (int)B,
                  num_rows, out, counts);
}

unsigned attn_simt_errors_read_clear() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_attn_err, &zero, sizeof(zero));
  return v;
}

}  // namespace mla
