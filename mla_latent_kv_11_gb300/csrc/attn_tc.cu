// Step 4 on the tensor cores (tcgen05 + TMEM + TMA): paged split-KV decode and
// causal prefill of the weight-absorbed MLA over the latent cache, bf16 in,
// fp32 accumulation, for kv_lora_rank 512 and rope 64 or 0.
//
// Tile shape. A row tile is 128 query rows = (128 / H) tokens x H heads, the
// M dimension of every MMA; keys come in tiles of 64 cache rows. The output
// accumulator O is 128 x 512 fp32, which alone would fill a CTA's 512 TMEM
// columns, so a cluster of two CTAs shares each row tile:
//   CTA 0 owns latent columns   0..255            (Q, K and V boxes 0..3)
//   CTA 1 owns latent columns 256..511 + the rope (Q, K and V boxes 4..7, 8)
// Each CTA loads only its columns of every cache row (the row is read from
// HBM once per pair), computes its partial scores S_r = Q_r K_r^T (M=128,
// N=64), hands them to the peer through distributed shared memory, and both
// form S = S_0 + S_1 in the same order, so both run the identical online
// softmax. Each CTA then accumulates its own half O_r += P V_r (M=128, N=256,
// K=64) in TMEM: no MMA is duplicated and no cache byte is read twice.
//
// Roles (256 threads per CTA): warp 0 issues TMA loads, warp 1 issues MMAs,
// warp 2 owns the TMEM allocation, warps 4..7 run the softmax, the O rescale
// and the epilogue, one thread per query row (TMEM lane). Stages are tracked
// with mbarriers; every wait is bounded in time and a timeout winds the
// kernel down and reports MLA_ERR_TIMEOUT instead of hanging.
//
// Softmax is evaluated in base 2 with the scale folded in. The running max is
// updated lazily: O and the denominator are only rescaled when the max grows
// by more than 2^8, so exponentials stay below 256 and the result is exact
// up to rounding. P is rounded to bf16 for the PV MMA and the denominator sums
// the rounded values.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <cstdlib>
#include <mutex>
#include <vector>

#include "mla_internal.h"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

__device__ unsigned g_tc_err = 0;

constexpr int kRows = 128;          // M: query rows per tile
constexpr int kKeysT = 64;          // keys per tile
constexpr int kBoxBytesQ = kRows * 128;   // one 64-column box of the row tile (16 KB)
constexpr int kBoxBytesK = kKeysT * 128;  // one 64-column box of a key tile (8 KB)
constexpr int kThreads = 256;
constexpr int kSoftmaxWarp0 = 4;
constexpr float kLazyRescale = 8.0f;      // log2 units
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;            // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;          // S buffers: [256, 320) and [320, 384)

template <int kRope>
struct Cfg {
  static constexpr int kBoxes = 4 + kRope / 64;      // boxes per CTA (max over ranks)
  static constexpr int kStages = kRope ? 2 : 3;
  static constexpr int kQBytes = kBoxes * kBoxBytesQ;
  static constexpr int kStageBytes = kBoxes * kBoxBytesK;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQBytes;
  static constexpr int kOffP = kOffKV + kStages * kStageBytes;
  static constexpr int kOffX = kOffP + 2 * kRows * 128;
  static constexpr int kOffBar = kOffX + kRows * kKeysT * 4;
  static constexpr int kBarBytes = 1024;
  static constexpr int kSmem = kOffBar + kBarBytes;
  static constexpr int kSmemAlloc = kSmem + 1024;    // slack for 1 KB alignment
};

struct Bars {
  uint64_t q_full, seg_done, o_empty, mma_final;
  uint64_t kv_full[3], kv_empty[3];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], pv_done[2];
  uint64_t x_full, x_empty;
  uint32_t tmem_base;
  int abort_flag;
};

struct Seg {
  int b;      // sequence
  int tok0;   // first query token (row of q_cat / o_lat)
  int ntok;   // tokens of this tile that are real
  int k0, k1; // key range
  int pos0;   // causal position of token 0 (keys <= pos0 + t are visible to token t)
  int slot;   // partial slot, or -1 for a final output
};

struct TcParams {
  int mode;          // 0 decode, 1 prefill
  int H, tpt;        // heads, tokens per row tile (128 / H)
  int L, R;
  float scale_log2;
  // output
  __nv_bfloat16* o_lat;
  int64_t o_s0, o_s1;
  float* lse;
  // cache
  int page, num_blocks;
  const int32_t* block_table;
  int64_t bt_stride;
  int cap;           // max_blocks * page
  // decode
  const int32_t* seq_lens;
  int B;
  DecodeSched sched;
  // prefill
  const int32_t* cu_q;
  const int32_t* kv_lens;
  const int32_t* item_prefix;  // [B+1] row tiles per sequence, prefix-summed
};

// ------------------------------------------------------------------ segments
// Every role of both CTAs walks the same segment list.
struct Walker {
  int unit, nunits;
  int t, t1, b;      // decode: tile cursor, end, sequence
  int g;             // prefill: next item
  bool active;

  __device__ void init(const TcParams& p, int unit_, int nunits_) {
    unit = unit_;
    nunits = nunits_;
    active = true;
    if (p.mode == 0) {
      const int total = p.sched.tile_prefix[p.B];
      const int W = min(p.sched.units, total);
      if (unit >= W) {
        active = false;
        return;
      }
      t = (int)(((long long)unit * total) / W);
      t1 = (int)(((long long)(unit + 1) * total) / W);
      int lo = 0, hi = p.B;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.sched.tile_prefix[mid] <= t) lo = mid; else hi = mid - 1;
      }
      b = lo;
    } else {
      const int total = p.item_prefix[p.B];
      g = total - 1 - unit;
    }
  }

  __device__ bool next(const TcParams& p, Seg& s) {
    if (!active) return false;
    if (p.mode == 0) {
      if (t >= t1) return false;
      while (p.sched.tile_prefix[b + 1] <= t) ++b;
      const int pre = p.sched.tile_prefix[b];
      const int seg_end = min(t1, p.sched.tile_prefix[b + 1]);
      const int len = min(max(p.seq_lens[b], 0), p.cap);
      s.b = b;
      s.tok0 = b;
      s.ntok = 1;
      s.k0 = (t - pre) * kKeysT;
      s.k1 = min((seg_end - pre) * kKeysT, len);
      s.pos0 = 0x3fffffff;
      s.slot = p.sched.npieces[b] == 1 ? -1 : p.sched.piece_base[b] + (unit - p.sched.first_unit[b]);
      t = seg_end;
      return true;
    }
    if (g < 0) return false;
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.item_prefix[mid] <= g) lo = mid; else hi = mid - 1;
    }
    const int bb = lo;
    const int i0 = (g - p.item_prefix[bb]) * p.tpt;
    const int q0 = p.cu_q[bb];
    const int q_len = p.cu_q[bb + 1] - q0;
    int kv = p.kv_lens[bb];
    kv = min(max(kv, 0), p.cap);
    s.b = bb;
    s.tok0 = q0 + i0;
    s.ntok = min(p.tpt, q_len - i0);
    s.pos0 = kv - q_len + i0;
    s.k0 = 0;
    s.k1 = max(0, min(kv, s.pos0 + s.ntok));
    s.slot = -1;
    g -= nunits;
    return true;
  }
};

__device__ __forceinline__ int ntiles(const Seg& s) { return (s.k1 - s.k0 + kKeysT - 1) / kKeysT; }

__device__ __forceinline__ void set_abort(Bars& bars, uint32_t peer) {
  bars.abort_flag = 1;
  // tell the peer too, so it stops waiting for this CTA
  const uint32_t remote = map_to_rank(&bars.abort_flag, peer);
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(1) : "memory");
}

// 16-byte chunk `c` of row `r` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

template <int kRope>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kvmap,
                       const TcParams p) {
  using C = Cfg<kRope>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~uintptr_t(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + C::kOffBar);
  unsigned char* sQ = smem + C::kOffQ;
  unsigned char* sKV = smem + C::kOffKV;
  unsigned char* sP = smem + C::kOffP;
  float* sX = reinterpret_cast<float*>(smem + C::kOffX);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int unit = (int)cluster_id_x(), nunits = (int)nclusters_x();
  // columns of this CTA: latent [256*rank, +256) and, on rank 1, the rope
  const int nbox = rank == 0 ? 4 : 4 + kRope / 64;
  const int col0 = rank == 0 ? 0 : 256;

  if (tid == 0) {
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.seg_done, 1);
    mbar_init(&bars.o_empty, 128);
    mbar_init(&bars.mma_final, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_empty[i], 128);
      mbar_init(&bars.p_full[i], 128);
      mbar_init(&bars.pv_done[i], 1);
    }
    mbar_init(&bars.x_full, 128);
    mbar_init(&bars.x_empty, 128);
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&bars.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kvmap);
  }
  tc_fence_before();
  cluster_sync();   // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort = &bars.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    Walker wk;
    wk.init(p, unit, nunits);
    Seg sg;
    int gt = 0, seg_i = 0;
    int issued_q = 0;
    int issued[3] = {0, 0, 0};
    bool ok = true;
    const int rows_box = min(p.page, kKeysT);
    const int subs = kKeysT / rows_box;
    while (ok && wk.next(p, sg)) {
      if (lane == 0) {
        if (seg_i > 0) ok = mbar_wait(&bars.seg_done, (seg_i - 1) & 1, abort);
        if (ok) {
          mbar_arrive_expect_tx(&bars.q_full, nbox * kBoxBytesQ);
          for (int c = 0; c < nbox; ++c)
            tma_load_3d(sQ + c * kBoxBytesQ, &qmap, &bars.q_full, col0 + 64 * c, 0, sg.tok0);
          ++issued_q;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      const int nt = ntiles(sg);
      const int32_t* bt = p.block_table + (int64_t)sg.b * p.bt_stride;
      for (int j0 = 0; ok && j0 < nt; j0 += 32) {
        // lanes prefetch the block ids of the next 32 tiles (pages of >= 64 rows)
        int my_blk = 0;
        if (subs == 1 && j0 + lane < nt) my_blk = bt[(sg.k0 + (j0 + lane) * kKeysT) / p.page];
        const int n = min(32, nt - j0);
        for (int jj = 0; jj < n; ++jj) {
          const int blk1 = __shfl_sync(0xffffffffu, my_blk, jj);
          if (lane == 0 && ok) {
            const int s = gt % C::kStages;
            ok = mbar_wait(&bars.kv_empty[s], ((gt / C::kStages) & 1) ^ 1, abort);
            if (ok) {
              const int kt = sg.k0 + (j0 + jj) * kKeysT;
              unsigned char* dst = sKV + s * C::kStageBytes;
              // gather the (block, row) pieces of this tile that hold rows < k1
              int blks[8], rows0[8], nsub = 0;
              if (subs == 1) {
                blks[0] = blk1;
                rows0[0] = kt % p.page;
                nsub = 1;
              } else {
                for (int i = 0; i < subs; ++i) {
                  const int key = kt + i * rows_box;
                  if (key >= sg.k1) break;
                  blks[nsub] = bt[key / p.page];
                  rows0[nsub] = 0;
                  ++nsub;
                }
              }
              uint32_t bytes = 0;
              for (int i = 0; i < nsub; ++i) {
                if (blks[i] < 0 || blks[i] >= p.num_blocks) {
                  atomicOr(&g_tc_err, kErrDeviceData);
                  blks[i] = -1;
                } else {
                  bytes += (uint32_t)(nbox * rows_box * 128);
                }
              }
              mbar_arrive_expect_tx(&bars.kv_full[s], bytes);
              for (int i = 0; i < nsub; ++i) {
                if (blks[i] < 0) continue;
                for (int c = 0; c < nbox; ++c)
                  tma_load_3d(dst + c * kBoxBytesK + i * rows_box * 128, &kvmap, &bars.kv_full[s],
                              col0 + 64 * c, rows0[i], blks[i]);
              }
              ++issued[s];
            }
          }
          ++gt;
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
      }
      ++seg_i;
    }
    if (!ok && lane == 0) set_abort(bars, peer);
    // never leave with copies in flight: wait for the last phase of every barrier we loaded into
    if (lane == 0) {
      volatile int dummy = 0;
      if (issued_q > 0) mbar_wait(&bars.q_full, (issued_q - 1) & 1, &dummy);
      for (int s = 0; s < C::kStages; ++s)
        if (issued[s] > 0) mbar_wait(&bars.kv_full[s], (issued[s] - 1) & 1, &dummy);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      Walker wk;
      wk.init(p, unit, nunits);
      Seg sg;
      int gt = 0, seg_i = 0;
      bool ok = true;
      const uint32_t id_qk = idesc_bf16(kRows, kKeysT, false, false);
      const uint32_t id_pv = idesc_bf16(kRows, 256, false, true);
      const uint32_t q_base = smem_u32(sQ), kv_base = smem_u32(sKV), p_base = smem_u32(sP);
      auto issue_pv = [&](int g, bool first) -> bool {
        const int pb = g & 1;
        if (!mbar_wait(&bars.p_full[pb], (g >> 1) & 1, abort)) return false;
        tc_fence_after();
        const int s = g % C::kStages;
        const uint32_t vb = kv_base + s * C::kStageBytes;
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t a = sdesc_sw128(p_base + pb * kRows * 128 + kk * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(vb + kk * 16 * 128, kBoxBytesK, 1024);
          umma_bf16(tmem + kTmemO, a, b, id_pv, (first && kk == 0) ? 0u : 1u);
        }
        umma_commit(&bars.kv_empty[s]);
        umma_commit(&bars.pv_done[pb]);
        return true;
      };
      while (ok && wk.next(p, sg)) {
        ok = mbar_wait(&bars.q_full, seg_i & 1, abort);
        const int nt = ntiles(sg);
        for (int j = 0; ok && j < nt; ++j) {
          const int g = gt + j;
          const int s = g % C::kStages, sb = g & 1;
          ok = mbar_wait(&bars.kv_full[s], (g / C::kStages) & 1, abort) &&
               mbar_wait(&bars.s_empty[sb], ((g >> 1) & 1) ^ 1, abort);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kb = kv_base + s * C::kStageBytes;
          for (int c = 0; c < nbox; ++c)
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = sdesc_sw128(q_base + c * kBoxBytesQ + kk * 32, 16, 1024);
              const uint64_t b = sdesc_sw128(kb + c * kBoxBytesK + kk * 32, 16, 1024);
              umma_bf16(tmem + kTmemS + sb * kKeysT, a, b, id_qk, (c | kk) ? 1u : 0u);
            }
          umma_commit(&bars.s_full[sb]);
          if (j > 0) {
            if (j == 1 && seg_i > 0) ok = mbar_wait(&bars.o_empty, (seg_i - 1) & 1, abort);
            ok = ok && issue_pv(g - 1, j == 1);
          }
        }
        if (ok && nt > 0) {
          if (nt == 1 && seg_i > 0) ok = mbar_wait(&bars.o_empty, (seg_i - 1) & 1, abort);
          ok = ok && issue_pv(gt + nt - 1, nt == 1);
        }
        if (!ok) break;
        umma_commit(&bars.seg_done);
        gt += nt;
        ++seg_i;
      }
      if (!ok) set_abort(bars, peer);
      // every MMA this thread issued is complete before the TMEM is released
      umma_commit(&bars.mma_final);
      volatile int dummy = 0;
      mbar_wait(&bars.mma_final, 0, &dummy);
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------ softmax / epilogue
    const int row = tid - kSoftmaxWarp0 * 32;               // 0..127 == TMEM lane
    const uint32_t lane_addr = (uint32_t)((warp - kSoftmaxWarp0) * 32) << 16;
    const int t_in_tile = row / p.H, head = row - t_in_tile * p.H;
    const uint32_t peer_x = map_to_rank(sX + row * kKeysT, peer);
    float* my_x = sX + row * kKeysT;
    Walker wk;
    wk.init(p, unit, nunits);
    Seg sg;
    int gt = 0, seg_i = 0;
    bool ok = true;
    while (ok && wk.next(p, sg)) {
      const int nt = ntiles(sg);
      const bool row_valid = row < p.H * p.tpt && t_in_tile < sg.ntok;
      const int limit = row_valid ? min(sg.k1, sg.pos0 + t_in_tile + 1) : 0;
      float m = -CUDART_INF_F, l = 0.f;
      for (int j = 0; ok && j < nt; ++j) {
        const int g = gt + j, sb = g & 1, pb = g & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[sb], (g >> 1) & 1, abort));
        if (!ok) break;
        tc_fence_after();
        float sp[64];
        tmem_ld32(tmem + lane_addr + kTmemS + sb * kKeysT, *reinterpret_cast<float(*)[32]>(sp));
        tmem_ld32(tmem + lane_addr + kTmemS + sb * kKeysT + 32, *reinterpret_cast<float(*)[32]>(sp + 32));
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bars.s_empty[sb]);
        // exchange partial scores with the peer
        ok = __all_sync(0xffffffffu, mbar_wait<true>(&bars.x_empty, (g & 1) ^ 1, abort));
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < 64; c += 4) st_cluster_v4(peer_x + c * 4, sp[c], sp[c + 1], sp[c + 2], sp[c + 3]);
        mbar_arrive_remote(&bars.x_full, peer);
        ok = __all_sync(0xffffffffu, mbar_wait<true>(&bars.x_full, g & 1, abort));
        if (!ok) break;
        const int kbase = sg.k0 + j * kKeysT;
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 o = *reinterpret_cast<const float4*>(my_x + c);
          // S = S_rank0 + S_rank1 in both CTAs
          const float x0 = rank == 0 ? sp[c] + o.x : o.x + sp[c];
          const float x1 = rank == 0 ? sp[c + 1] + o.y : o.y + sp[c + 1];
          const float x2 = rank == 0 ? sp[c + 2] + o.z : o.z + sp[c + 2];
          const float x3 = rank == 0 ? sp[c + 3] + o.w : o.w + sp[c + 3];
          sp[c] = kbase + c < limit ? x0 * p.scale_log2 : -CUDART_INF_F;
          sp[c + 1] = kbase + c + 1 < limit ? x1 * p.scale_log2 : -CUDART_INF_F;
          sp[c + 2] = kbase + c + 2 < limit ? x2 * p.scale_log2 : -CUDART_INF_F;
          sp[c + 3] = kbase + c + 3 < limit ? x3 * p.scale_log2 : -CUDART_INF_F;
          mx = fmaxf(mx, fmaxf(fmaxf(sp[c], sp[c + 1]), fmaxf(sp[c + 2], sp[c + 3])));
        }
        mbar_arrive_remote(&bars.x_empty, peer);   // my receive buffer is free again
        // lazy online softmax
        float alpha = 1.f;
        bool rescale_o = false;
        if (mx > m + kLazyRescale || (m == -CUDART_INF_F && mx > -CUDART_INF_F)) {
          alpha = m == -CUDART_INF_F ? 0.f : exp2f(m - mx);
          rescale_o = (m != -CUDART_INF_F) && j > 0;
          m = mx;
        }
        float sum = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float e0 = m == -CUDART_INF_F ? 0.f : exp2f(sp[c] - m);
          const float e1 = m == -CUDART_INF_F ? 0.f : exp2f(sp[c + 1] - m);
          const __nv_bfloat162 h = __floats2bfloat162_rn(e0, e1);
          const float2 hf = __bfloat1622float2(h);
          sum += hf.x + hf.y;
          pk[c >> 1] = *reinterpret_cast<const uint32_t*>(&h);
        }
        l = l * alpha + sum;
        // the P buffer was last read by PV(g - 2)
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.pv_done[pb], ((g >> 1) & 1) ^ 1, abort));
        if (!ok) break;
        unsigned char* prow = sP + pb * kRows * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(prow + sw128(row, c)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        // rows of a partial tile past the sequence: zero their V so garbage cannot reach O
        const int nvalid = sg.k1 - kbase;
        if (nvalid < kKeysT) {
          unsigned char* st = sKV + (g % C::kStages) * C::kStageBytes;
          const int nz = (kKeysT - nvalid) * 8 * 4;       // 16-byte chunks in 4 latent boxes
          for (int i = row; i < nz; i += 128) {
            const int box = i / ((kKeysT - nvalid) * 8);
            const int rem = i - box * ((kKeysT - nvalid) * 8);
            const int r = nvalid + rem / 8, c = rem & 7;
            *reinterpret_cast<uint4*>(st + box * kBoxBytesK + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        // tcgen05.ld/st are warp-collective: the whole warp rescales if any of its rows must
        if (__any_sync(0xffffffffu, rescale_o)) {
          const float f = rescale_o ? alpha : 1.f;
          // O must hold PV(g-1) before it is scaled
          ok = __all_sync(0xffffffffu, mbar_wait(&bars.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort));
          if (!ok) break;
          tc_fence_after();
          for (int c = 0; c < 256; c += 32) {
            float v[32];
            tmem_ld32(tmem + lane_addr + kTmemO + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= f;
            tmem_st32(tmem + lane_addr + kTmemO + c, v);
          }
          tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars.p_full[pb]);
      }
      if (!ok) break;
      // epilogue: O / l for this CTA's 256 columns
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.seg_done, seg_i & 1, abort));
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int tok = sg.tok0 + t_in_tile;
      for (int c = 0; c < 256; c += 32) {
        float v[32];
        if (nt > 0) {
          tmem_ld32(tmem + lane_addr + kTmemO + c, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        if (!row_valid) continue;
        if (sg.slot < 0) {
          __nv_bfloat16* o = p.o_lat + (int64_t)tok * p.o_s0 + (int64_t)head * p.o_s1 + col0 + c;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(v[i] * inv, v[i + 1] * inv);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(v[i + 2] * inv, v[i + 3] * inv);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(v[i + 4] * inv, v[i + 5] * inv);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(v[i + 6] * inv, v[i + 7] * inv);
            w.x = *reinterpret_cast<uint32_t*>(&h0);
            w.y = *reinterpret_cast<uint32_t*>(&h1);
            w.z = *reinterpret_cast<uint32_t*>(&h2);
            w.w = *reinterpret_cast<uint32_t*>(&h3);
            *reinterpret_cast<uint4*>(o + i) = w;
          }
        } else {
          float* o = p.sched.part_o + ((int64_t)sg.slot * p.H + head) * p.L + col0 + c;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(o + i) = make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
        }
      }
      if (row_valid && rank == 0) {
        const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
        if (sg.slot < 0) {
          if (p.lse) p.lse[(int64_t)tok * p.H + head] = lse;
        } else {
          p.sched.part_lse[(int64_t)sg.slot * p.H + head] = lse;
        }
      }
      tc_fence_before();
      mbar_arrive(&bars.o_empty);
      gt += nt;
      ++seg_i;
    }
    if (!ok) set_abort(bars, peer);
  }
  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && bars.abort_flag) atomicOr(&g_tc_err, kErrTimeout);
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();   // no CTA leaves while its peer may still touch its shared memory
}

// Row tiles per sequence (prefill), prefix-summed: one CTA.
__global__ void prefill_items_kernel(const int32_t* __restrict__ cu_q, int B, int tpt, int32_t* __restrict__ out) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      out[b] = acc;
      const int q = cu_q[b + 1] - cu_q[b];
      acc += q > 0 ? (q + tpt - 1) / tpt : 0;
    }
    out[B] = acc;
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool make_map3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kRope>
int max_clusters() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> g(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    using C = Cfg<kRope>;
    cudaFuncSetAttribute(mla_attn_tc_kernel<kRope>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * device_sm_count(), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemAlloc;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mla_attn_tc_kernel<kRope>, &cfg) != cudaSuccess || n <= 0)
      n = device_sm_count() / 2;
    cudaGetLastError();
    cache[dev] = n;
  }
  return cache[dev];
}

template <int kRope>
cudaError_t launch_tc(const TcParams& p, const CUtensorMap& qm, const CUtensorMap& km, int clusters,
                      cudaStream_t st) {
  using C = Cfg<kRope>;
  cudaError_t e = cudaFuncSetAttribute(mla_attn_tc_kernel<kRope>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemAlloc);
  if (e != cudaSuccess) return e;
  mla_attn_tc_kernel<kRope><<<dim3(2 * clusters), dim3(kThreads), C::kSmemAlloc, st>>>(qm, km, p);
  return cudaGetLastError();
}

}  // namespace

bool tc_attention_supported(mla_dtype dt, int H, int L, int R, bool decode, const CacheView& cv,
                            const View3& q, const View3& o) {
  if (getenv("MLA_DISABLE_TC") != nullptr) return false;
  if (dt != MLA_BF16 || L != 512 || (R != 0 && R != 64)) return false;
  if (decode ? H != 128 : (H != 128 && H != 64)) return false;
  const int page = cv.page;
  if (!(page % 64 == 0 || (64 % page == 0 && page % 8 == 0))) return false;
  auto al16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  if (!al16(cv.data) || cv.s_blk % 8 || cv.s_row % 8) return false;
  if (!al16(q.data) || q.s0 % 8 || q.s1 % 8) return false;
  if (!al16(o.data) || o.s0 % 8 || o.s1 % 8) return false;
  if (!encode_fn()) return false;
  return true;
}

int tc_decode_units(int num_splits) {
  return num_splits > 0 ? num_splits : max_clusters<64>();
}

static cudaError_t run_tc(mla_dtype, TcParams& p, const View3& q, const CacheView& cv, int clusters,
                          cudaStream_t st) {
  CUtensorMap qm, km;
  const int E = p.L + p.R;
  if (!make_map3d(&qm, q.data, E, p.H, q.n0, (uint64_t)q.s1 * 2, (uint64_t)q.s0 * 2, 64, p.H, p.tpt))
    return cudaErrorInvalidValue;
  if (!make_map3d(&km, cv.data, E, cv.page, cv.num_blocks, (uint64_t)cv.s_row * 2, (uint64_t)cv.s_blk * 2, 64,
                  cv.page < 64 ? cv.page : 64, 1))
    return cudaErrorInvalidValue;
  return p.R == 64 ? launch_tc<64>(p, qm, km, clusters, st) : launch_tc<0>(p, qm, km, clusters, st);
}

cudaError_t launch_decode_tc(const View3& o_lat, float* lse, const View3& q, const CacheView& cache,
                             const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t B, int32_t H, int32_t L, int32_t R, float scale,
                             const DecodeSched& s, cudaStream_t st) {
  TcParams p{};
  p.mode = 0;
  p.H = H;
  p.tpt = kRows / H;
  p.L = L;
  p.R = R;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o_lat = static_cast<__nv_bfloat16*>(o_lat.data);
  p.o_s0 = o_lat.s0;
  p.o_s1 = o_lat.s1;
  p.lse = lse;
  p.page = cache.page;
  p.num_blocks = cache.num_blocks;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  const long long cap = (long long)max_blocks * cache.page;
  p.cap = (int)(cap > 0x3fffffff ? 0x3fffffff : cap);
  p.seq_lens = seq_lens;
  p.B = B;
  p.sched = s;
  return run_tc(MLA_BF16, p, q, cache, s.units, st);
}

cudaError_t launch_prefill_tc(const View3& o_lat, float* lse, const View3& q, const CacheView& cache,
                              const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                              const int32_t* cu_q, const int32_t* kv_lens, int32_t B, int32_t H, int32_t L,
                              int32_t R, float scale, int32_t* item_prefix, cudaStream_t st) {
  TcParams p{};
  p.mode = 1;
  p.H = H;
  p.tpt = kRows / H;
  p.L = L;
  p.R = R;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o_lat = static_cast<__nv_bfloat16*>(o_lat.data);
  p.o_s0 = o_lat.s0;
  p.o_s1 = o_lat.s1;
  p.lse = lse;
  p.page = cache.page;
  p.num_blocks = cache.num_blocks;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  const long long cap = (long long)max_blocks * cache.page;
  p.cap = (int)(cap > 0x3fffffff ? 0x3fffffff : cap);
  p.B = B;
  p.cu_q = cu_q;
  p.kv_lens = kv_lens;
  p.item_prefix = item_prefix;
  prefill_items_kernel<<<1, 32, 0, st>>>(cu_q, B, p.tpt, item_prefix);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int clusters = R == 64 ? max_clusters<64>() : max_clusters<0>();
  return run_tc(MLA_BF16, p, q, cache, clusters, st);
}

unsigned attn_tc_errors_read_clear() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_tc_err, &zero, sizeof(zero));
  return v;
}

}  // namespace mla
