// Step 4 on the tensor cores (tcgen05 + TMEM + TMA): paged split-KV decode and
// causal prefill of the weight-absorbed MLA over the latent cache, bf16 in,
// fp32 accumulation, for kv_lora_rank 512 and rope 64 or 0.
//
// Tile shape. A row tile is 128 query rows = (128 / H) tokens x H heads, the
// M dimension of every MMA; keys come in tiles of 64 cache rows. The output
// accumulator O is 128 x 512 fp32, which alone would fill a CTA's 512 TMEM
// columns, so a cluster of two CTAs shares each row tile:
//   CTA 0 owns latent columns   0..255 and rope columns 512..543
//   CTA 1 owns latent columns 256..511 and rope columns 544..575
// Each CTA TMA-loads only its columns of every cache row (a row crosses HBM
// once per pair), computes its partial scores S_r = Q_r K_r^T, and the pair
// swaps partials so both hold S = S_0 + S_1 (summed in the same order) and run
// the identical online softmax. Each CTA then accumulates its half
// O_r += P V_r. No MMA is duplicated and no cache byte is read twice.
//
// Memory plan per CTA. Tensor memory holds everything the MMAs reuse:
//   O half [0,256) fp32 | S [256,320) fp32 | P [320,352) bf16 pairs |
//   Q half [352, 480) latent, [480, 496) rope, bf16 pairs | l [496,512) fp32,
// where l, the row sums of P, comes from an N=16 MMA of P against a tile of
// ones issued with each PV (so the denominator sums exactly the bf16 P that O
// accumulates, and the softmax warps never add P up). Both MMAs take their A
// operand from TMEM; shared memory only streams the B operand (the cache
// tile): the latent columns in 64-column boxes with 128-byte swizzle, the 32
// rope columns in one box with 64-byte swizzle. Shared memory holds 5 cache
// stages (36 KB with rope, 32 KB without), the tile of ones, one outgoing
// exchange tile (two pieces) and a ring of three incoming pieces: 226 KB.
//
// Exchange. The SM-to-SM network moves about 19 bytes per clock each way, so
// the pair does not swap fp32 partial scores (32 KB per tile) but
// exponentials: each CTA takes its row maximum of x_r = s_r * scale * log2 e,
// rounded up to an integer c_r, and sends E_r = 2^(x_r - c_r) in bf16 with c_r,
// as two 8.5 KB pieces (keys 0..31 and 32..63): the first goes out as soon as
// its 32 exponentials are written, while the second is computed. Since
//   2^(x_0 + x_1 - m) = E_0 * E_1 * 2^(c_0 + c_1 - m),
// both CTAs form P = bf16(E_own * E_peer) * 2^(M - m), the same value in both
// (IEEE multiplication commutes); c_0 + c_1 bounds the row maximum from
// above, so nothing can overflow, and it is an integer, so every rescaling
// factor is an exact power of two. A dedicated exchange warpgroup reads S out
// of TMEM as soon as the MMA has produced it, computes c and E and pushes each
// piece with one bulk copy into the peer's incoming ring (completion counted in
// bytes on the peer's barrier); the softmax warpgroup takes its own tile at
// once and each peer piece as it lands.
//
// Roles (384 threads): warp 0 issues TMA loads, warp 1 issues MMAs (a polling
// state machine that issues whichever of QK(g+1) and PV(g) is ready; the warp
// runs it converged and an elected lane issues, which keeps the N=64 QK MMAs at
// the tensor core's rate instead of the issue rate of one thread), warp 2
// owns the TMEM allocation, warps 4..7 load Q into TMEM and run the exchange,
// warps 8..11 run the softmax, the O rescale and the epilogue, one thread per
// query row (TMEM lane) in each group; warp 3 forwards the softmax group's
// "incoming piece read" signals to the peer as relaxed remote arrives (the
// reads they answer for were completed by a bar.sync). For e4m3 caches warps 0
// and 2 convert staged tiles to bf16 instead, warp 3 issues the staging loads of
// whole pages, and the softmax group sends its slot releases itself. Every wait is bounded
// in time; a timeout winds the kernel down and reports MLA_ERR_TIMEOUT
// instead of hanging.
//
// The running reference maximum m is updated lazily: O and its denominator are
// rescaled only when the bound c_0 + c_1 exceeds m by more than 8, so P stays
// below 2^8.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
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

constexpr int kRows = 128;                // M: query rows per tile
constexpr int kKeysT = 64;                // keys per tile
static_assert(kKeysT == kTile, "a decode key tile is a schedule tile");
constexpr int kBoxBytesK = kKeysT * 128;  // one 64-column box of a key tile (8 KB)
constexpr int kRopeHalf = 32;             // rope columns per CTA
constexpr int kRopeBoxBytes = kKeysT * kRopeHalf * 2;   // 4 KB
constexpr int kHalfKeys = kKeysT / 2;             // keys per exchange piece
constexpr int kESlotBytes = kRows * kHalfKeys * 2; // E = 2^(x - c) of half a tile, bf16 (8 KB)
constexpr int kXSlot = kESlotBytes + kRows * 4;     // + the rows' maxima c (8.5 KB): one piece
constexpr int kInSlots = 3;                         // incoming pieces: a ring of three
constexpr int kThreads = 384;
constexpr int kXchgWarp0 = 4;             // exchange warpgroup: warps 4..7
constexpr int kSoftmaxWarp0 = 8;          // softmax warpgroup: warps 8..11
constexpr int kSoftmaxBar = 1;            // named barrier of the softmax warpgroup
constexpr int kXchgBar = 2;               // named barrier of the exchange warpgroup
constexpr int kLoadBar = 3;               // named barrier of the loader warps (e4m3 caches)
constexpr int kLoaders = 64;              // loader threads: warps 0 and 2
// Dense e4m3 caches: warp 3 issues the staging TMA loads instead of forwarding the softmax
// group's slot releases, which that group's first thread then sends to the peer itself.
constexpr int kIssuerWarp = 3;
constexpr float kLazyRescale = 8.0f;      // log2 units
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;
constexpr uint32_t kTmemP = 320;
constexpr uint32_t kTmemQ = 352;
constexpr uint32_t kTmemL = 496;          // row sums of P, accumulated by the tensor core (16 equal columns)
constexpr int kOnesBytes = 16 * kKeysT * 2;   // a 16 x 64 tile of bf16 ones: B operand of the row-sum MMA

// kSrc: where a CTA's key tile comes from. 0: bf16 cache rows, TMA-loaded as swizzled boxes.
// 1: e4m3 cache rows through the block table, 2: fp8 ds_mla entries at a query's (compacted)
// slots; both gathered by cp.async into a staging ring and converted to bf16 in the layout the
// TMA would have written.
template <int kRope, int kSrc>
struct Cfg {
  static constexpr int kStages = kSrc ? 3 : 5;
  static constexpr int kStageBytes = 4 * kBoxBytesK + (kRope ? kRopeBoxBytes : 0);
  // staged 16-byte granules of one row: 16 latent + 2 rope (e4m3), or 16 latent + the four
  // scales + 4 rope (ds_mla: the rope is bf16)
  static constexpr int kGran = kSrc == 1 ? 16 + (kRope ? 2 : 0) : kSrc == 2 ? 21 : 0;
  static constexpr int kStg = kSrc ? 3 : 0;
  static constexpr int kStgBytes = kKeysT * kGran * 16;
  static constexpr int kOffKV = 0;
  static constexpr int kOffOnes = kOffKV + kStages * kStageBytes;   // 1 KB aligned: stages are
  static constexpr int kOffXloc = kOffOnes + kOnesBytes;            // own E + c of a tile: 2 pieces
  static constexpr int kOffXrem = kOffXloc + 2 * kXSlot;            // the peer's pieces: a ring of 3
  static constexpr int kOffStg = kOffXrem + kInSlots * kXSlot;      // staging ring (16-byte aligned)
  static constexpr int kOffRowBase = kOffStg + kStg * kStgBytes;    // [2][64] row offsets of a tile
  static constexpr int kOffBar = (kOffRowBase + (kSrc ? 2 * kKeysT * 8 : 0) + 127) & ~127;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmem = kOffBar + kBarBytes;
  static constexpr int kSmemAlloc = kSmem + 1024;    // slack for 1 KB alignment
};

struct Bars {
  uint64_t kv_full[8], kv_empty[8];
  uint64_t s_full, s_empty, p_full, pv_done;
  uint64_t seg_done, o_empty, q_ready, mma_final;
  // Exchange. Half h of tile t (keys [32h, 32h + 32)) is piece q = 2t + h; the peer's
  // piece q lands in incoming slot q % 3 (those barriers complete a phase every three
  // pieces); the own tile sits in the outgoing slot (one phase per tile).
  uint64_t own_ready;          // own E and c of the tile are in the outgoing slot
  uint64_t xloc_free;          // the softmax group has read the outgoing slot
  uint64_t x_full[kInSlots];   // the peer's piece has landed in incoming slot i
  uint64_t x_empty[kInSlots];  // the peer has read its incoming slot i (arrived on by the peer)
  uint64_t xin_free[kInSlots]; // the softmax group has read incoming slot i
  // gathered (e4m3) tiles: staging slot u holds the raw bytes of a tile, and is free again
  uint64_t stg_full[3], stg_empty[3];
  uint32_t tmem_base;
  int abort_flag;
};

#ifdef MLA_TRACE
// Cycle stamps of pipeline events of work unit 0, for tuning builds only.
__device__ long long g_trace[2][8][512];
__device__ long long g_trace2[2][8][512];
// per CTA: SM id, start and end (globaltimer ns), tiles issued, start and end (clock64), cycles
// the MMA issuer had a QK allowed but waited only on the cache tile, and only on S being free,
// cycles spent issuing QK MMAs and PV MMAs
__device__ long long g_cta_time[512][10];
// the same stamps for every CTA, first 128 tiles of each
__device__ long long g_trace_all[2][304][8][128];
#define MLA_TRACE_AT(ev, g)                                                          \
  do {                                                                                \
    const long long now_ = clock64();                                                 \
    if (unit == 0 && (g) < 512) g_trace[rank][ev][(g)] = now_;                        \
    if (blockIdx.x < 304 && (g) < 128) g_trace_all[0][blockIdx.x][ev][(g)] = now_;    \
  } while (0)
// loader events of work unit 0 (e4m3 caches)
__device__ long long g_trace3[2][16][512];
#define MLA_TRACE3_AT(ev, g)                                                   \
  do {                                                                          \
    if (unit == 0 && lt == 0 && (g) < 512) g_trace3[rank][ev][(g)] = clock64(); \
  } while (0)
// the same for the issuer warp's first thread
#define MLA_TRACE3I_AT(ev, g)                                                     \
  do {                                                                             \
    if (unit == 0 && lane == 0 && (g) < 512) g_trace3[rank][ev][(g)] = clock64(); \
  } while (0)
// the same for the first thread of the second loader warp
#define MLA_TRACE3B_AT(ev, g)                                                   \
  do {                                                                           \
    if (unit == 0 && lt == 32 && (g) < 512) g_trace3[rank][ev][(g)] = clock64(); \
  } while (0)
// exchange group, unit 0, first row: segment transitions (indexed by segment)
__device__ long long g_trace4[2][4][64];
#define MLA_TRACE4_AT(ev, g)                                                    \
  do {                                                                           \
    if (unit == 0 && row == 0 && (g) < 64) g_trace4[rank][ev][(g)] = clock64(); \
  } while (0)
#define MLA_TRACE2_AT(ev, g)                                                                  \
  do {                                                                                         \
    const long long now_ = clock64();                                                          \
    if (unit == 0 && row == 0 && (g) < 512) g_trace2[rank][ev][(g)] = now_;                    \
    if (row == 0 && blockIdx.x < 304 && (g) < 128) g_trace_all[1][blockIdx.x][ev][(g)] = now_; \
  } while (0)
#else
#define MLA_TRACE_AT(ev, g) \
  do {                      \
  } while (0)
#define MLA_TRACE2_AT(ev, g) \
  do {                       \
  } while (0)
#define MLA_TRACE4_AT(ev, g) \
  do {                       \
  } while (0)
#define MLA_TRACE3_AT(ev, g) \
  do {                       \
  } while (0)
#define MLA_TRACE3B_AT(ev, g) \
  do {                        \
  } while (0)
#define MLA_TRACE3I_AT(ev, g) \
  do {                        \
  } while (0)
#endif

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
  // queries [tokens, H, L+R]
  const __nv_bfloat16* q;
  int64_t q_s0, q_s1;
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
  // e4m3 rows (byte strides): kSrc 1 through the block table with descale_q / descale_k
  // (null: 1) folded into the scores and the output; kSrc 2 at slots[b * slot_stride + t]
  const uint8_t* cache8;
  int64_t s_blk8, s_row8;
  const float* descale_q;
  const float* descale_k;
  const int32_t* slots;
  int64_t slot_stride;
  int fp8_tma;       // kSrc 1: whole pages of rows come as TMA boxes (else per-row gathers)
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
      t = p.sched.unit_tile[unit];
      t1 = p.sched.unit_tile[unit + 1];
      if (t >= t1) {
        active = false;
        return;
      }
      b = p.sched.unit_seq[unit];   // the schedule's first sequence of this unit
    } else {
      const int total = p.item_prefix[p.B];
      g = total - 1 - unit;
    }
  }

  __device__ bool next(const TcParams& p, Seg& s) {
    if (!active) return false;
    if (p.mode == 0) {
      if (t >= t1) return false;
      // {first tile, clamped length, pieces, slot base - first unit}: one 16-byte load a segment
      int4 si = p.sched.seqinfo[b];
      while (si.x + (si.y + kKeysT - 1) / kKeysT <= t) si = p.sched.seqinfo[++b];
      const int seg_end = min(t1, si.x + (si.y + kKeysT - 1) / kKeysT);
      s.b = b;
      s.tok0 = b;
      s.ntok = 1;
      s.k0 = (t - si.x) * kKeysT;
      s.k1 = min((seg_end - si.x) * kKeysT, si.y);
      s.pos0 = 0x3fffffff;
      s.slot = si.z == 1 ? -1 : si.w + unit;
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

// 2^d for an integer-valued d <= 127, exactly (built from the exponent bits); 0 below -126.
__device__ __forceinline__ float exp2_int(float d) {
  return d < -126.f ? 0.f : __int_as_float(((int)d + 127) << 23);
}

// e4m3 -> bf16 in shared memory. Two codes go to f16x2 in one hardware conversion (every e4m3
// value, the NaN codes included, is exact in f16), each half widens to fp32 exactly, and one
// pack rounds the pair to bf16x2: exact without a scale (e4m3 values are bf16 values), the
// scaled product rounded once with one. Bits [16k, 16k + 16) of x hold codes 2k (low byte) and
// 2k + 1.
template <bool kScaled>
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two, float sc) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
  float lo = __half2float(__ushort_as_half(h.x)), hi = __half2float(__ushort_as_half(h.y));
  if (kScaled) {
    lo *= sc;
    hi *= sc;
  }
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 16 codes (one 16-byte granule) -> 16 bf16 as two 16-byte chunks, low code first.
template <bool kScaled>
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 w, float sc, uint4& c0, uint4& c1) {
  c0 = make_uint4(e4m3x2_to_bf16x2<kScaled>(w.x, sc), e4m3x2_to_bf16x2<kScaled>(w.x >> 16, sc),
                  e4m3x2_to_bf16x2<kScaled>(w.y, sc), e4m3x2_to_bf16x2<kScaled>(w.y >> 16, sc));
  c1 = make_uint4(e4m3x2_to_bf16x2<kScaled>(w.z, sc), e4m3x2_to_bf16x2<kScaled>(w.z >> 16, sc),
                  e4m3x2_to_bf16x2<kScaled>(w.w, sc), e4m3x2_to_bf16x2<kScaled>(w.w >> 16, sc));
}

__device__ __forceinline__ int ntiles(const Seg& s) { return (s.k1 - s.k0 + kKeysT - 1) / kKeysT; }

__device__ __forceinline__ void set_abort(Bars& bars, uint32_t peer) {
  bars.abort_flag = 1;
  // tell the peer too, so it stops waiting for this CTA
  const uint32_t remote = map_to_rank(&bars.abort_flag, peer);
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(1) : "memory");
}

template <int kRope, int kSrc>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_attn_tc_kernel(const __grid_constant__ CUtensorMap kvmap, const __grid_constant__ CUtensorMap ropemap,
                       const TcParams p) {
  using C = Cfg<kRope, kSrc>;
  static_assert(kSrc == 0 || kSrc == 1 || (kSrc == 2 && kRope == 64), "a ds_mla entry has a 64-wide rope part");
  static_assert(sizeof(Bars) <= C::kBarBytes, "barrier block overflows its slot");
  static_assert(C::kSmemAlloc <= 232448, "shared memory beyond the 227 KB a CTA may hold");
  static_assert(C::kStages <= 8, "kv barrier arrays hold 8 stages");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~uintptr_t(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + C::kOffBar);
  unsigned char* sKV = smem + C::kOffKV;
  unsigned char* sXloc = smem + C::kOffXloc;   // 2 pieces x (E [128 rows x 64 B, chunk-rotated] | c [128])
  unsigned char* sXrem = smem + C::kOffXrem;   // same layout, written by the peer

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int unit = (int)cluster_id_x(), nunits = (int)nclusters_x();
  // columns of this CTA: latent [col0, col0 + 256) and rope [rope0, rope0 + 32)
  const int col0 = 256 * (int)rank;
  const int rope0 = p.L + kRopeHalf * (int)rank;

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars.kv_full[s], kSrc ? kLoaders : 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    for (int u = 0; u < C::kStg; ++u) {
      // TMA boxes: one expect-tx arrival; gathers: one cp.async arrival per loader thread
      mbar_init(&bars.stg_full[u], (kSrc == 1 && p.fp8_tma) ? 1 : 32);
      mbar_init(&bars.stg_empty[u], kLoaders);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.s_empty, 4);
    mbar_init(&bars.p_full, 4);
    mbar_init(&bars.pv_done, 1);
    mbar_init(&bars.seg_done, 1);
    mbar_init(&bars.o_empty, 4);
    mbar_init(&bars.q_ready, 4);
    mbar_init(&bars.mma_final, 1);
    mbar_init(&bars.own_ready, 4);
    mbar_init(&bars.xloc_free, 1);
    for (int i = 0; i < kInSlots; ++i) {
      mbar_init(&bars.x_full[i], 1);
      mbar_init(&bars.x_empty[i], 1);
      mbar_init(&bars.xin_free[i], 1);
    }
    bars.abort_flag = 0;
    fence_mbar_init();
    // every incoming slot is armed for its first piece before the peer can send
    for (int i = 0; i < kInSlots; ++i) mbar_arrive_expect_tx(&bars.x_full[i], kXSlot);
  }
  if (warp == 2) {
    tmem_alloc(&bars.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (kSrc == 0 && warp == 0 && lane == 0) {
    tma_prefetch_desc(&kvmap);
    if (kRope) tma_prefetch_desc(&ropemap);
  }
  for (int i = tid; i < kOnesBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + C::kOffOnes)[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  fence_proxy_async_smem();   // the ones tile is read by the tensor core (async proxy)
  tc_fence_before();
  cluster_sync();   // barriers of both CTAs initialised before any remote access
  tc_fence_after();
  pdl_enter();      // the queries, the cache and the schedule come from the kernels before
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort = &bars.abort_flag;

#ifdef MLA_TRACE
  if (tid == 0 && blockIdx.x < 512) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    g_cta_time[blockIdx.x][0] = smid;
    g_cta_time[blockIdx.x][1] = (long long)globaltimer_ns();
    g_cta_time[blockIdx.x][4] = clock64();
  }
#endif

  if (kSrc == 0 && warp == 0) {
    // ------------------------------------------------------------ TMA producer (cache tiles)
    Walker wk;
    wk.init(p, unit, nunits);
    Seg sg;
    int gt = 0;
    int issued[C::kStages] = {};
    bool ok = true;
    const int rows_box = min(p.page, kKeysT);
    const int subs = kKeysT / rows_box;
    while (ok && wk.next(p, sg)) {
      const int nt = ntiles(sg);
      const int32_t* bt = p.block_table + (int64_t)sg.b * p.bt_stride;
      if (p.mode == 1) {
        // prefill: the next row tile's queries (this CTA's 512 + 64 bytes of each of its rows)
        // into L2 while this one runs, so the exchange group's Q load at its start finds them
        // there; row tiles are short (about sixteen key tiles at 2048 tokens)
        Walker wn = wk;
        Seg sn;
        if (wn.next(p, sn)) {
          constexpr int kParts = kRope ? 5 : 4;   // 128-byte lines of a row's part
          for (int i = lane; i < kRows * kParts; i += 32) {
            const int r = i / kParts, part = i - r * kParts, t = r / p.H;
            if (r < p.H * p.tpt && t < sn.ntok)
              prefetch_l2(p.q + (int64_t)(sn.tok0 + t) * p.q_s0 + (int64_t)(r - t * p.H) * p.q_s1 +
                          (part < 4 ? col0 + 64 * part : rope0));
          }
        }
      }
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
            MLA_TRACE_AT(0, gt);
            if (ok) {
              const int kt = sg.k0 + (j0 + jj) * kKeysT;
              unsigned char* dst = sKV + s * C::kStageBytes;
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
                  bytes += (uint32_t)(rows_box * (4 * 128 + (kRope ? 2 * kRopeHalf : 0)));
                }
              }
              mbar_arrive_expect_tx(&bars.kv_full[s], bytes);
              for (int i = 0; i < nsub; ++i) {
                if (blks[i] < 0) continue;
                for (int c = 0; c < 4; ++c)
                  tma_load_3d(dst + c * kBoxBytesK + i * rows_box * 128, &kvmap, &bars.kv_full[s],
                              col0 + 64 * c, rows0[i], blks[i]);
                if (kRope)
                  tma_load_3d(dst + 4 * kBoxBytesK + i * rows_box * 2 * kRopeHalf, &ropemap, &bars.kv_full[s],
                              rope0, rows0[i], blks[i]);
              }
              ++issued[s];
            }
          }
          ++gt;
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
      }
    }
    if (!ok && lane == 0) set_abort(bars, peer);
    // never leave with copies in flight: wait for the last phase of every stage loaded
    if (lane == 0) {
      volatile int dummy = 0;
      for (int s = 0; s < C::kStages; ++s)
        if (issued[s] > 0 && !mbar_wait(&bars.kv_full[s], (issued[s] - 1) & 1, &dummy))
          atomicOr(&g_tc_err, kErrTimeout);   // a copy that never landed: report, never pass silently
    }
  } else if (kSrc != 0 && (warp == 0 || warp == 2)) {
    if constexpr (kSrc != 0) {
      // ------------------------------------------------------------ loader (e4m3 caches): 64
      // threads convert each tile that warp 3 has staged (up to kStg tiles ahead) to bf16 in the
      // swizzled layout of a TMA box once its bf16 stage is free
      const int lt = (warp == 0 ? 0 : 32) + lane;
      constexpr int G = C::kGran;
      auto group_all = [](bool v) { return named_bar_and(kLoadBar, kLoaders, v); };
      unsigned char* stg = smem + C::kOffStg;
      Walker wk;
      wk.init(p, unit, nunits);
      Seg sg;
      int nt = 0, j = 0;           // tiles of the current segment, next tile in it
      bool have = false;           // a segment is open
      int gi = 0, gc = 0;          // tiles issued, tiles converted
      bool ok = true, more = true;     // ok: the group's decision, the same in every loader thread
      while (ok) {
        // ---- the tiles warp 3 issues, up to kStg ahead of the conversion
        while (ok && more && gi < gc + C::kStg) {
          while (!have || j >= nt) {
            if (!wk.next(p, sg)) {
              more = false;
              break;
            }
            nt = ntiles(sg);
            j = 0;
            have = true;
          }
          if (!more) break;
          ++gi;   // warp 3 loads the tiles; the loaders only count them
          ++j;
        }
        if (!ok || gc == gi) break;
        // ---- convert tile gc: staging slot u -> bf16 stage s
        const int u = gc % C::kStg, s = gc % C::kStages;
        MLA_TRACE3_AT(3, gc);
        bool mine = mbar_wait(&bars.stg_full[u], (gc / C::kStg) & 1, abort);
        MLA_TRACE3_AT(4, gc);
        ok = group_all(mine && mbar_wait(&bars.kv_empty[s], ((gc / C::kStages) & 1) ^ 1, abort));
        MLA_TRACE3_AT(5, gc);
        MLA_TRACE3B_AT(10, gc);
        if (!ok) break;
        const unsigned char* src = stg + u * C::kStgBytes;
        unsigned char* dst = sKV + s * C::kStageBytes;
        // TMA'd pages sit as [64 rows x 256 B] latent then [64 rows x 32 B] rope; gathered rows as
        // rows of G granules. Rows at or past `keep` and rows of pages in `bad` are zeroed.
        const bool boxes = kSrc == 1 && p.fp8_tma;
        int keep = kKeysT, bad = 0, box_shift = 6;
        if (boxes) {
          const int* meta = reinterpret_cast<const int*>(smem + C::kOffRowBase);
          keep = meta[2 * u];
          bad = meta[2 * u + 1];
          box_shift = 31 - __clz(min(p.page, kKeysT));
        }
        auto dropped = [&](int r) { return r >= keep || ((bad >> (r >> box_shift)) & 1); };
        // latent: 16 codes per staged granule -> 16 bf16, two 16-byte chunks of box g / 4 (one
        // loop per part, so the lanes of a warp never split between the two). A warp converts
        // two rows at a time, each thread one fixed granule g of its row: lanes 4q..4q+3 take
        // granules 4q..4q+3 of the even row, lanes 4q+4..4q+7 granules 4(q^1).. of the odd one,
        // so every quarter-warp reads eight distinct 16-byte bank groups of a staged 256-byte
        // row and writes eight distinct chunks of the swizzled stage (even ones for the even
        // row, odd ones for the odd row)
        {
          const int l = lt & 31, half = (l >> 2) & 1;
          const int g = 4 * ((l >> 3) ^ half) + (l & 3);
          const int j0 = (g & 3) * 2;
          unsigned char* box = dst + (g >> 2) * kBoxBytesK;
#pragma unroll 4
          for (int r = 2 * (lt >> 5) + half; r < kKeysT; r += 4) {
            const unsigned char* row = src + r * G * 16;
            uint4 w = *reinterpret_cast<const uint4*>(boxes ? src + r * 256 + g * 16 : row + g * 16);
            if (boxes && dropped(r)) w = make_uint4(0u, 0u, 0u, 0u);
            uint4 c0, c1;
            if (kSrc == 1)
              e4m3x16_to_bf16<false>(w, 1.f, c0, c1);
            else
              e4m3x16_to_bf16<true>(w, reinterpret_cast<const float*>(row + 16 * 16)[2 * (int)rank + g / 8], c0, c1);
            unsigned char* bx = box + r * 128;
            *reinterpret_cast<uint4*>(bx + ((j0 ^ (r & 7)) << 4)) = c0;
            *reinterpret_cast<uint4*>(bx + (((j0 + 1) ^ (r & 7)) << 4)) = c1;
          }
        }
        MLA_TRACE3_AT(7, gc);
        MLA_TRACE3B_AT(8, gc);
        // rope: 64-byte rows of the rope box, 64-byte swizzle
        if (kRope) {
          constexpr int RG = kSrc == 1 ? 2 : 4;   // staged rope granules per row
          for (int f = lt; f < kKeysT * RG; f += kLoaders) {
            const int r = f / RG, g = f - r * RG;
            const unsigned char* row = src + r * G * 16;
            unsigned char* bx = dst + 4 * kBoxBytesK + r * 64;
            if (kSrc == 1) {
              uint4 w = *reinterpret_cast<const uint4*>(boxes ? src + kKeysT * 256 + r * 32 + g * 16
                                                              : row + (16 + g) * 16);
              if (boxes && dropped(r)) w = make_uint4(0u, 0u, 0u, 0u);
              uint4 c0, c1;
              e4m3x16_to_bf16<false>(w, 1.f, c0, c1);
              const int j0 = g * 2;
              *reinterpret_cast<uint4*>(bx + ((j0 ^ ((r >> 1) & 3)) << 4)) = c0;
              *reinterpret_cast<uint4*>(bx + (((j0 + 1) ^ ((r >> 1) & 3)) << 4)) = c1;
            } else {
              // bf16 already: one chunk, from staged granule 17 + g (16 holds the scales)
              *reinterpret_cast<uint4*>(bx + ((g ^ ((r >> 1) & 3)) << 4)) =
                  *reinterpret_cast<const uint4*>(row + (17 + g) * 16);
            }
          }
        }
        MLA_TRACE3_AT(9, gc);
        fence_proxy_async_smem();   // the tensor core reads the stage through the async proxy
        mbar_arrive(&bars.kv_full[s]);
        mbar_arrive(&bars.stg_empty[u]);
        MLA_TRACE3_AT(6, gc);
        MLA_TRACE3B_AT(11, gc);
        ++gc;
      }
      if (!ok) set_abort(bars, peer);
    }
  } else if (kSrc != 0 && warp == kIssuerWarp) {
    if constexpr (kSrc != 0) {
      // ------------------------------------------------------------ staging issuer (e4m3
      // caches). Whole pages: one thread loads this CTA's latent box (and rope box) of every
      // page a tile spans into the tile's staging slot once the loaders have freed it, with
      // the slot's metadata (rows kept, pages that did not load) for the conversion, which
      // zeroes the rest. With pages of 64 rows or more the lanes fetch the block ids of the
      // next 32 tiles of a segment at once. The same walk as the loaders': the same tiles in
      // the same slots.
      if (kSrc == 1 && p.fp8_tma) {
        unsigned char* stg = smem + C::kOffStg;
        int* meta = reinterpret_cast<int*>(smem + C::kOffRowBase);
        const int rows_box = min(p.page, kKeysT), subs = kKeysT / rows_box;
        Walker wk;
        wk.init(p, unit, nunits);
        Seg sg;
        int gi = 0;
        bool ok = true;
        while (ok && wk.next(p, sg)) {
          const int nt = ntiles(sg);
          int blk_pf = -1;
          for (int j = 0; ok && j < nt; ++j, ++gi) {
            const int u = gi % C::kStg;
            const int kt = sg.k0 + j * kKeysT;
            int blk_now = -1;
            if (subs == 1) {
              if ((j & 31) == 0) {
                const int jj = j + lane;
                blk_pf = jj < nt ? p.block_table[(int64_t)sg.b * p.bt_stride + (sg.k0 + jj * kKeysT) / p.page] : -1;
              }
              blk_now = __shfl_sync(0xffffffffu, blk_pf, j & 31);
            }
            if (lane == 0) {
              MLA_TRACE3I_AT(13, gi);
              ok = mbar_wait(&bars.stg_empty[u], ((gi / C::kStg) & 1) ^ 1, abort);
              MLA_TRACE3I_AT(14, gi);
              if (ok) {
                uint32_t bytes = 0;
                int bad = 0, blk0 = -1;
                for (int i = 0; i < subs; ++i) {   // pass 1: bytes and bad pages
                  const int key = kt + i * rows_box;
                  if (key >= sg.k1) continue;
                  const int blk = subs == 1 ? blk_now : p.block_table[(int64_t)sg.b * p.bt_stride + key / p.page];
                  if (blk < 0 || blk >= p.num_blocks) {
                    atomicOr(&g_tc_err, kErrDeviceData);
                    bad |= 1 << i;
                    continue;
                  }
                  if (i == 0) blk0 = blk;
                  bytes += (uint32_t)(rows_box * (256 + (kRope ? kRopeHalf : 0)));
                }
                meta[2 * u] = min(kKeysT, sg.k1 - kt);   // rows kept
                meta[2 * u + 1] = bad;                   // bit i: page i of the tile did not load
                mbar_arrive_expect_tx(&bars.stg_full[u], bytes);
                unsigned char* dst = stg + u * C::kStgBytes;
                const int row0 = subs == 1 ? kt % p.page : 0;
                for (int i = 0; i < subs; ++i) {   // pass 2: the loads (block ids re-read: cached)
                  const int key = kt + i * rows_box;
                  if (key >= sg.k1 || ((bad >> i) & 1)) continue;
                  const int blk = i == 0 ? blk0 : p.block_table[(int64_t)sg.b * p.bt_stride + key / p.page];
                  tma_load_3d(dst + i * rows_box * 256, &kvmap, &bars.stg_full[u], col0, row0, blk);
                  if (kRope)
                    tma_load_3d(dst + kKeysT * 256 + i * rows_box * kRopeHalf, &ropemap, &bars.stg_full[u],
                                512 + kRopeHalf * (int)rank, row0, blk);
                }
              }
              MLA_TRACE3I_AT(15, gi);
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          }
        }
        if (!ok && lane == 0) set_abort(bars, peer);
        // never leave with copies in flight: wait for the last phase issued to every slot
        if (lane == 0) {
          volatile int dummy = 0;
          for (int u = 0; u < C::kStg; ++u) {
            const int issued = gi / C::kStg + (u < gi % C::kStg ? 1 : 0);
            if (issued > 0 && !mbar_wait(&bars.stg_full[u], (issued - 1) & 1, &dummy))
              atomicOr(&g_tc_err, kErrTimeout);
          }
        }
      } else {
        // gathered rows (ds_mla slots; e4m3 pages a TMA box cannot take): the warp's 32 threads
        // copy this CTA's granules of every row of a tile with 16-byte cp.async into its
        // staging slot once the loaders have freed it (rows past the segment zero-filled by the
        // copy's source size), each thread's copies then counted on the slot's barrier
        constexpr int G = C::kGran;
        int64_t* rowbase = reinterpret_cast<int64_t*>(smem + C::kOffRowBase);
        unsigned char* stg = smem + C::kOffStg;
        Walker wk;
        wk.init(p, unit, nunits);
        Seg sg;
        int gi = 0;
        bool ok = true;
        while (ok && wk.next(p, sg)) {
          const int nt = ntiles(sg);
          // the block id (pages) or slot (ds_mla) of this lane's rows lane and lane + 32 of a
          // tile; the next tile's are loaded while this one's copies are issued
          auto fetch = [&](int jj, int (&raw)[2]) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int t = sg.k0 + jj * kKeysT + lane + 32 * k;
              raw[k] = t >= sg.k1 ? -1
                       : kSrc == 1 ? p.block_table[(int64_t)sg.b * p.bt_stride + t / p.page]
                                   : p.slots[(int64_t)sg.b * p.slot_stride + t];   // compacted: in range
            }
          };
          int raw[2], nxt[2] = {-1, -1};
          if (nt > 0) fetch(0, raw);
          for (int j = 0; ok && j < nt; ++j, ++gi) {
            const int u = gi % C::kStg;
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.stg_empty[u], ((gi / C::kStg) & 1) ^ 1, abort));
            if (!ok) break;
            if (j + 1 < nt) fetch(j + 1, nxt);
            // byte offset of each row of the tile (-1: past the segment or a bad block id)
            int64_t* rb = rowbase + (gi & 1) * kKeysT;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int r = lane + 32 * k, t = sg.k0 + j * kKeysT + r;
              int64_t off = -1;
              if (t < sg.k1) {
                if (kSrc == 1) {
                  const int blk = raw[k];
                  if (blk >= 0 && blk < p.num_blocks)
                    off = (int64_t)blk * p.s_blk8 + (int64_t)(t % p.page) * p.s_row8;
                  else
                    atomicOr(&g_tc_err, kErrDeviceData);
                } else {
                  const int slot = raw[k];
                  off = (int64_t)(slot / p.page) * p.s_blk8 + (int64_t)(slot % p.page) * p.s_row8;
                }
              }
              rb[r] = off;
            }
            raw[0] = nxt[0];
            raw[1] = nxt[1];
            __syncwarp();
            const uint32_t dst0 = smem_u32(stg + u * C::kStgBytes);
            // the 16 latent granules of every row, then the tail granules (rope; and the scales
            // of a ds_mla entry): one loop each, so no lane of the warp takes the other kind
#pragma unroll 4
            for (int f = lane; f < kKeysT * 16; f += 32) {
              const int r = f >> 4, g = f & 15;
              const int64_t off = rb[r];
              cp_async16(dst0 + (r * G + g) * 16, p.cache8 + (off < 0 ? 0 : off + col0 + 16 * g), off < 0 ? 0u : 16u);
            }
            constexpr int TG = G > 16 ? G - 16 : 1;   // tail granules per row (none without rope)
            for (int f = lane; f < kKeysT * (G - 16); f += 32) {
              const int r = f / TG, g = f - r * TG;
              const int64_t off = rb[r];
              const int byte = kSrc == 1 ? 512 + kRopeHalf * (int)rank + 16 * g
                                         : (g == 0 ? kDsMlaLatent : kDsMlaRopeByte + 64 * (int)rank + 16 * (g - 1));
              cp_async16(dst0 + (r * G + 16 + g) * 16, p.cache8 + (off < 0 ? 0 : off + byte), off < 0 ? 0u : 16u);
            }
            cp_async_commit();
            cp_async_arrive_noinc(&bars.stg_full[u]);
            __syncwarp();   // every lane has read this tile's offsets before the next tile's are written
          }
        }
        if (!ok && lane == 0) set_abort(bars, peer);
        cp_async_wait_all();   // never leave with copies in flight
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer. The whole
    // warp walks the state machine in lockstep (every decision is lane 0's, broadcast) and
    // one elected lane issues each MMA and commit.
    auto uni = [&](bool v) { return __shfl_sync(0xffffffffu, v ? 1 : 0, 0) != 0; };
    Walker wk;
    wk.init(p, unit, nunits);
    Seg sg;
    int gt = 0, seg_i = 0, full_i = 0;   // unit tile, segment, segment among those with tiles
    bool ok = true;
    constexpr uint32_t id_qk = idesc_bf16(kRows, kKeysT, false, false);
    constexpr uint32_t id_pv = idesc_bf16(kRows, 256, false, true);
    constexpr uint32_t id_sum = idesc_bf16(kRows, 16, false, false);
    const uint32_t kv_base = smem_u32(sKV);
    const uint32_t ones_base = smem_u32(smem + C::kOffOnes);
#ifdef MLA_TRACE
    long long tr_starve = 0, tr_sblock = 0, tr_t0 = 0, tr_qkiss = 0, tr_pviss = 0, tr_i0 = 0;
    int tr_state = 0;   // 0 none, 1 waiting on the tile only, 2 waiting on S only
#endif
    while (ok && wk.next(p, sg)) {
      const int nt = ntiles(sg);
      if (nt == 0) {
        // an empty segment completes once the epilogue has read the previous segment's O: one
        // completion per epilogue, so the softmax group's parity waits never fall two behind
        ok = __all_sync(0xffffffffu, seg_i == 0 || mbar_wait(&bars.o_empty, (seg_i - 1) & 1, abort));
        if (!ok) break;
        umma_commit_elect(&bars.seg_done);
        ++seg_i;
        continue;
      }
      // its Q is in TMEM (q_ready completes one phase per segment with tiles; the exchange
      // group loads the next Q only after consuming every S of this one, so no parity aliasing)
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.q_ready, full_i & 1, abort));
      int qk = 0, pv = 0;
      uint64_t last = globaltimer_ns();
      uint32_t spins = 0;
      while (ok && pv < nt) {
        bool did = false;
        if (qk < nt && qk <= pv + 2) {
          const int t = gt + qk, s = t % C::kStages;
          // S is single-buffered: QK(t) needs S(t-1) read out by the exchange group. At most two
          // QKs run ahead of the PVs: a third would hold up PV(t) behind its issue (measured)
          const bool kv_ok = mbar_poll(&bars.kv_full[s], (t / C::kStages) & 1);
          const bool s_ok = mbar_poll(&bars.s_empty, (t & 1) ^ 1);
#ifdef MLA_TRACE
          {
            const int st = (kv_ok && s_ok) ? 0 : (!kv_ok && s_ok) ? 1 : (kv_ok && !s_ok) ? 2 : 3;
            if (st != tr_state) {
              const long long now = clock64();
              if (tr_state == 1) tr_starve += now - tr_t0;
              if (tr_state == 2) tr_sblock += now - tr_t0;
              tr_state = st;
              tr_t0 = now;
            }
          }
#endif
          if (uni(kv_ok && s_ok)) {
            MLA_TRACE_AT(1, t);
#ifdef MLA_TRACE
            tr_i0 = clock64();
#endif
            tc_fence_after();
            const uint32_t kb = kv_base + s * C::kStageBytes;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_bf16_ta_elect(tmem + kTmemS, tmem + kTmemQ + c * 32 + kk * 8,
                                   sdesc_sw128(kb + c * kBoxBytesK + kk * 32, 16, 1024), id_qk, (c | kk) ? 1u : 0u);
            if (kRope) {
#pragma unroll
              for (int kk = 0; kk < 2; ++kk)
                umma_bf16_ta_elect(tmem + kTmemS, tmem + kTmemQ + 128 + kk * 8,
                                   sdesc_sw64(kb + 4 * kBoxBytesK + kk * 32, 16, 512), id_qk, 1u);
            }
            umma_commit_elect(&bars.s_full);
#ifdef MLA_TRACE
            tr_qkiss += clock64() - tr_i0;
#endif
            ++qk;
            did = true;
          }
        }
#ifdef MLA_TRACE
        else if (tr_state != 0) {
          const long long now = clock64();
          if (tr_state == 1) tr_starve += now - tr_t0;
          if (tr_state == 2) tr_sblock += now - tr_t0;
          tr_state = 0;
        }
#endif
        if (pv < qk) {
          const int t = gt + pv, s = t % C::kStages;
          const bool o_free = pv > 0 || seg_i == 0 || mbar_poll(&bars.o_empty, (seg_i - 1) & 1);
          if (uni(o_free && mbar_poll(&bars.p_full, t & 1))) {
            MLA_TRACE_AT(2, t);
#ifdef MLA_TRACE
            tr_i0 = clock64();
#endif
            tc_fence_after();
            const uint32_t vb = kv_base + s * C::kStageBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_ta_elect(tmem + kTmemO, tmem + kTmemP + kk * 8,
                                 sdesc_sw128(vb + kk * 16 * 128, kBoxBytesK, 1024), id_pv, (pv > 0 || kk > 0) ? 1u : 0u);
            // l += P * ones: the row sums of exactly the bf16 P that O accumulates
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_ta_elect(tmem + kTmemL, tmem + kTmemP + kk * 8, sdesc_sw128(ones_base + kk * 32, 16, 1024),
                                 id_sum, (pv > 0 || kk > 0) ? 1u : 0u);
            umma_commit_elect(&bars.kv_empty[s]);
            umma_commit_elect(&bars.pv_done);
            if (pv == nt - 1) umma_commit_elect(&bars.seg_done);
#ifdef MLA_TRACE
            tr_pviss += clock64() - tr_i0;
#endif
            ++pv;
            did = true;
          }
        }
        if (did) {
          spins = 0;
          last = globaltimer_ns();
        } else {
          __nanosleep(32);   // leave the issue slots to the softmax warps
          if ((++spins & 255u) == 0 && (*abort || globaltimer_ns() - last > kWaitLimitNs)) ok = false;
          ok = uni(ok);
        }
      }
      if (!ok) break;
      gt += nt;
      ++seg_i;
      ++full_i;
    }
    if (!ok && lane == 0) set_abort(bars, peer);
#ifdef MLA_TRACE
    if (lane == 0 && blockIdx.x < 512) {
      g_cta_time[blockIdx.x][3] = gt;
      g_cta_time[blockIdx.x][6] = tr_starve;
      g_cta_time[blockIdx.x][7] = tr_sblock;
      g_cta_time[blockIdx.x][8] = tr_qkiss;
      g_cta_time[blockIdx.x][9] = tr_pviss;
    }
#endif
    __syncwarp();
    // every MMA this warp issued is complete before the TMEM is released
    umma_commit_elect(&bars.mma_final);
    volatile int dummy = 0;
    if (!mbar_wait(&bars.mma_final, 0, &dummy) && lane == 0) atomicOr(&g_tc_err, kErrTimeout);
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ forwarder: releases the
    // incoming slots to the peer once the softmax group has read them (a relaxed arrive: the
    // reads it answers for were completed by the softmax group's barrier before it was asked)
    if (lane == 0) {
      Walker wk;
      wk.init(p, unit, nunits);
      Seg sg;
      int gt = 0;
      bool ok = true;
      while (ok && wk.next(p, sg)) {
        const int nt = ntiles(sg);
        for (int q = 2 * gt; ok && q < 2 * (gt + nt); ++q) {
          const int rs = q % kInSlots;
          ok = mbar_wait(&bars.xin_free[rs], (q / kInSlots) & 1, abort);
          if (ok) mbar_arrive_remote_relaxed(&bars.x_empty[rs], peer);
#ifdef MLA_TRACE
          if (unit == 0 && q < 1024 && (q & 1)) g_trace2[rank][4][q >> 1] = clock64();
#endif
        }
        gt += nt;
      }
      if (!ok) set_abort(bars, peer);
    }
  } else if (warp >= kXchgWarp0 && warp < kXchgWarp0 + 4) {
    // ------------------------------------------------------------ exchange group: Q load;
    // per tile: S out of TMEM, own row max c and E = 2^(s*scale - c) in bf16, pushed to the peer
    const int row = tid - kXchgWarp0 * 32;                  // 0..127 == TMEM lane
    const uint32_t lane_addr = (uint32_t)((warp - kXchgWarp0) * 32) << 16;
    const int t_in_tile = row / p.H, head = row - t_in_tile * p.H;
    const uint32_t peer_rem0 = map_to_rank(sXrem, peer);
    const uint32_t peer_xfull0 = map_to_rank(&bars.x_full[0], peer);
    // A named barrier has no timeout, so every decision is taken by all 128 threads.
    auto group_all = [](bool v) { return named_bar_and(kXchgBar, 128, v); };
    // Q rows at 32-byte aligned addresses (base and strides; the column offsets are): loaded
    // 32 bytes at a time. Only without a rope part (the prefill and the 64-head decode, 8% and
    // 3% faster): with one, the code this adds to the group measured 6% slower for the decode.
    const bool q_32B = kRope == 0 && (reinterpret_cast<uintptr_t>(p.q) & 31) == 0 && p.q_s0 % 16 == 0 &&
                       p.q_s1 % 16 == 0;
    auto prefetch_row = [&](const __nv_bfloat16* r) {   // this CTA's 512 + 64 bytes of a Q row
#pragma unroll
      for (int i = 0; i < 256; i += 64) prefetch_l2(r + col0 + i);
      if (kRope) prefetch_l2(r + rope0);
    };
    Walker wk;
    wk.init(p, unit, nunits);
    Seg sg;
    int gt = 0, seg_i = 0;
    bool ok = true;
    while (ok && wk.next(p, sg)) {
      const int nt = ntiles(sg);
      const bool row_valid = row < p.H * p.tpt && t_in_tile < sg.ntok;
      const int limit = row_valid ? min(sg.k1, sg.pos0 + t_in_tile + 1) : 0;
      // ---- this CTA's Q columns of the row tile into TMEM (two bf16 per column, the even
      // one low), for segments with tiles only (q_ready completes one phase per such segment).
      // The group has consumed every S so far, so every QK MMA that read the old Q is
      // complete: no wait for the old segment's PVs.
      tc_fence_after();
      MLA_TRACE4_AT(0, seg_i);
      if (nt > 0) {
        const __nv_bfloat16* qrow = p.q + (int64_t)(sg.tok0 + t_in_tile) * p.q_s0 + (int64_t)head * p.q_s1;
        // The row's parts are read in five dependent rounds below; prefetched into L2 first,
        // only the first round waits for DRAM
        if (row_valid) prefetch_row(qrow);
        // two rounds of loads: latent chunks 0 and 1, then chunks 2 and 3 with the rope part
        // (a chunk: 64 values, 32 columns). This CTA's 32 rope values fill exactly 16 columns;
        // the row-sum columns l follow them, and the softmax group may still be about to read
        // the current segment's l, so nothing beyond the rope's 16 columns may be written here.
#pragma unroll
        for (int c2 = 0; c2 < 4; c2 += 2) {
          uint32_t v[2][32];
          uint32_t vr[16];
          if (q_32B) {
            // 32-byte loads: each reads one whole sector of the row, half the requests
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const __nv_bfloat16* src = qrow + col0 + (c2 + cc) * 64;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                if (row_valid) ld_global_32B(src + i * 16, w);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[cc][8 * i + e] = w[e];
              }
            }
            if (kRope && c2 == 2) {
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                if (row_valid) ld_global_32B(qrow + rope0 + i * 16, w);
#pragma unroll
                for (int e = 0; e < 8; ++e) vr[8 * i + e] = w[e];
              }
            }
          } else {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const __nv_bfloat16* src = qrow + col0 + (c2 + cc) * 64;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                uint4 w = make_uint4(0, 0, 0, 0);
                if (row_valid) w = *reinterpret_cast<const uint4*>(src + i * 8);
                v[cc][4 * i] = w.x;
                v[cc][4 * i + 1] = w.y;
                v[cc][4 * i + 2] = w.z;
                v[cc][4 * i + 3] = w.w;
              }
            }
            if (kRope && c2 == 2) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint4 w = make_uint4(0, 0, 0, 0);
                if (row_valid) w = *reinterpret_cast<const uint4*>(qrow + rope0 + i * 8);
                vr[4 * i] = w.x;
                vr[4 * i + 1] = w.y;
                vr[4 * i + 2] = w.z;
                vr[4 * i + 3] = w.w;
              }
            }
          }
          if (c2 == 0) MLA_TRACE4_AT(1, seg_i);
          tmem_st32u(tmem + lane_addr + kTmemQ + c2 * 32, v[0]);
          tmem_st32u(tmem + lane_addr + kTmemQ + (c2 + 1) * 32, v[1]);
          if (kRope && c2 == 2) tmem_st16u(tmem + lane_addr + kTmemQ + 128, vr);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.q_ready);
        MLA_TRACE4_AT(2, seg_i);
      }
      bool sent = true;   // row 0: its last push went out
      for (int j = 0; ok && j < nt; ++j) {
        const int t = gt + j;
        // ---- one group decision per tile: S(t) is in TMEM, the outgoing slot is free (the
        // softmax group has read tile t-1 from it and both its pushes have left it) and row
        // 0's last push went out
        bool mine = mbar_wait(&bars.s_full, t & 1, abort) && mbar_wait(&bars.xloc_free, (t & 1) ^ 1, abort);
        if (row == 0) {
          mine = mine && sent;
          bulk_wait_read_all();
        }
        ok = group_all(mine);
        if (!ok) break;
        MLA_TRACE_AT(3, t);
        // ---- S(t) out of TMEM; the MMA may then compute S(t+1)
        tc_fence_after();
        float sv[64];
        tmem_ld32(tmem + lane_addr + kTmemS, *reinterpret_cast<float(*)[32]>(sv));
        tmem_ld32(tmem + lane_addr + kTmemS + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.s_empty);
        // ---- own row max c (base 2, scale folded in) and E = 2^(x - c) in bf16. The bf16 path's
        // scale is positive (checked on the host), so max(s) * scale is the maximum of x; an e4m3
        // cache's descales are device values of either sign, so there x is formed first
        float xs = p.scale_log2;
        if (kSrc == 1) {
          // an e4m3 cache's descales: the scores scale by descale_q * descale_k
          const float dq = p.descale_q != nullptr ? *p.descale_q : 1.f;
          const float dk = p.descale_k != nullptr ? *p.descale_k : 1.f;
          const float sl2 = p.scale_log2 * (dq * dk);
#pragma unroll
          for (int k = 0; k < 64; ++k) sv[k] *= sl2;
          xs = 1.f;
        }
        const int kbase = sg.k0 + j * kKeysT;
        if (!__all_sync(0xffffffffu, kbase + kKeysT <= limit)) {
#pragma unroll
          for (int k = 0; k < 64; ++k) sv[k] = kbase + k < limit ? sv[k] : -CUDART_INF_F;
        }
        float mx[8];   // eight running maxima and a tree: no 64-long dependency chain
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = sv[k];
#pragma unroll
        for (int k = 8; k < 64; ++k) mx[k & 7] = fmaxf(mx[k & 7], sv[k]);
        float c = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        // rounded up to an integer: still an upper bound, and it makes every factor
        // 2^(M - m) of the softmax an exact power of two
        c = c == -CUDART_INF_F ? -CUDART_INF_F : ceilf(c * xs);
        const float neg_c = c == -CUDART_INF_F ? 0.f : -c;
        // ---- each half: E of its 32 keys into its piece, then straight to the peer, so the
        // first piece is on its way while the second is computed
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t ek[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const __nv_bfloat162 hv = __floats2bfloat162_rn(ex2_approx(fmaf(sv[32 * h + k], xs, neg_c)),
                                                            ex2_approx(fmaf(sv[32 * h + k + 1], xs, neg_c)));
            ek[k >> 1] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          unsigned char* piece = sXloc + h * kXSlot;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
            *reinterpret_cast<uint4*>(piece + row * 64 + ((ch ^ ((row >> 1) & 3)) << 4)) =
                make_uint4(ek[4 * ch], ek[4 * ch + 1], ek[4 * ch + 2], ek[4 * ch + 3]);
          reinterpret_cast<float*>(piece + kESlotBytes)[row] = c;
          fence_proxy_async_smem();
          named_bar(kXchgBar, 128);
          if (h == 1) {
            MLA_TRACE_AT(4, t);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.own_ready);
          }
          if (row == 0 && sent) {
            // piece q goes to the peer's incoming slot q % 3, free once it has read piece q - 3
            const int q = 2 * t + h, rs = q % kInSlots;
            sent = mbar_wait<true>(&bars.x_empty[rs], ((q / kInSlots) & 1) ^ 1, abort);
            if (h == 0) MLA_TRACE2_AT(0, t);
            if (sent) {
              bulk_copy_to_peer(peer_rem0 + rs * kXSlot, piece, kXSlot, peer_xfull0 + rs * 8);
              bulk_commit_group();
            }
          }
        }
      }
      if (!ok) break;
      ok = group_all(sent);   // the segment's last push went out
      MLA_TRACE4_AT(3, seg_i);
      if (!ok) break;
      gt += nt;
      ++seg_i;
    }
    if (!ok) set_abort(bars, peer);
    if (row == 0) bulk_wait_read_all();
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------ softmax group: P, O rescale, epilogue
    const int row = tid - kSoftmaxWarp0 * 32;               // 0..127 == TMEM lane
    const uint32_t lane_addr = (uint32_t)((warp - kSoftmaxWarp0) * 32) << 16;
    const int t_in_tile = row / p.H, head = row - t_in_tile * p.H;
    auto group_all = [](bool v) { return named_bar_and(kSoftmaxBar, 128, v); };
    Walker wk;
    wk.init(p, unit, nunits);
    Seg sg;
    int gt = 0, seg_i = 0;
    bool ok = true;
    while (ok && wk.next(p, sg)) {
      const int nt = ntiles(sg);
      const bool row_valid = row < p.H * p.tpt && t_in_tile < sg.ntok;
      float m = -CUDART_INF_F;             // running reference max (base 2); the denominator is in TMEM
      for (int j = 0; ok && j < nt; ++j) {
        const int g = gt + j;
        // ---- the own tile: both pieces and c at once, which frees the outgoing slot early
        MLA_TRACE2_AT(1, g);
        ok = group_all(mbar_wait(&bars.own_ready, g & 1, abort));
        MLA_TRACE2_AT(2, g);
        if (!ok) break;
        uint4 eo[8];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
            eo[4 * h + ch] = *reinterpret_cast<const uint4*>(sXloc + h * kXSlot + row * 64 + ((ch ^ ((row >> 1) & 3)) << 4));
        const float c_own = reinterpret_cast<const float*>(sXloc + kESlotBytes)[row];
        float alpha = 1.f, factor = 0.f;
        bool rescale_o = false;
        uint32_t pk[32];
        // ---- the peer's pieces, each as soon as it lands
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = 2 * g + h, rs = q % kInSlots;
          ok = group_all(mbar_wait<true>(&bars.x_full[rs], (q / kInSlots) & 1, abort));
          if (h == 0) MLA_TRACE2_AT(3, g);
          if (!ok) break;
          const unsigned char* rem = sXrem + rs * kXSlot;
          uint4 er[4];
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
            er[ch] = *reinterpret_cast<const uint4*>(rem + row * 64 + ((ch ^ ((row >> 1) & 3)) << 4));
          const float c_rem = reinterpret_cast<const float*>(rem + kESlotBytes)[row];
          // read: re-arm the incoming slot and release it to the peer (through warp 3); after
          // the first piece the outgoing slot goes back to the exchange group
          named_bar(kSoftmaxBar, 128);
          if (row == 0) {
            mbar_arrive_expect_tx(&bars.x_full[rs], kXSlot);
            if (kSrc != 0)   // no forwarder: release the slot to the peer directly (relaxed: the
              mbar_arrive_remote_relaxed(&bars.x_empty[rs], peer);   // reads are behind the barrier)
            else
              mbar_arrive(&bars.xin_free[rs]);
            if (h == 0) mbar_arrive(&bars.xloc_free);
          }
          if (h == 0) {
            MLA_TRACE2_AT(5, g);
            // ---- tile upper bound M = c_0 + c_1; IEEE addition and multiplication commute, so
            // own-then-peer operands give both CTAs bit-identical M and P without knowing rank
            const float M = (c_own == -CUDART_INF_F || c_rem == -CUDART_INF_F) ? -CUDART_INF_F : c_own + c_rem;
            if (M > m + kLazyRescale || (m == -CUDART_INF_F && M > -CUDART_INF_F)) {
              alpha = m == -CUDART_INF_F ? 0.f : exp2_int(m - M);
              rescale_o = (m != -CUDART_INF_F) && j > 0;
              m = M;
            }
            factor = M == -CUDART_INF_F ? 0.f : exp2_int(M - m);
            MLA_TRACE2_AT(6, g);
          }
          // ---- P = (E_own * E_peer) * 2^(M - m): packed bf16 products rounded once (the
          // factor is an exact power of two), the same value in both CTAs
          const __nv_bfloat162 f2 = __float2bfloat162_rn(factor);
          const uint32_t* w0 = reinterpret_cast<const uint32_t*>(eo + 4 * h);
          const uint32_t* w1 = reinterpret_cast<const uint32_t*>(er);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const __nv_bfloat162 e = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&w0[k]),
                                             *reinterpret_cast<const __nv_bfloat162*>(&w1[k]));
            const __nv_bfloat162 pq = __hmul2(e, f2);
            pk[16 * h + k] = *reinterpret_cast<const uint32_t*>(&pq);
          }
        }
        if (!ok) break;
        MLA_TRACE_AT(7, g);
        // ---- P(g) replaces P(g-1) in TMEM once PV(g-1) is done; O is rescaled then too
        if (g > 0) {
          ok = group_all(mbar_wait(&bars.pv_done, (g - 1) & 1, abort));
          if (!ok) break;
        }
        MLA_TRACE_AT(5, g);
        tc_fence_after();
        // tcgen05.ld/st are warp-collective: the whole warp rescales if any of its rows must
        if (__any_sync(0xffffffffu, rescale_o)) {
          const float f = rescale_o ? alpha : 1.f;
          for (int c = 0; c < 256; c += 32) {
            float v[32];
            tmem_ld32(tmem + lane_addr + kTmemO + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= f;
            tmem_st32(tmem + lane_addr + kTmemO + c, v);
          }
          float lv[16];
          tmem_ld16(tmem + lane_addr + kTmemL, lv);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) lv[i] *= f;
          tmem_st16(tmem + lane_addr + kTmemL, lv);
        }
        tmem_st32u(tmem + lane_addr + kTmemP, pk);
        // rows of a partial tile past the sequence: zero their V so garbage cannot reach O
        const int kbase = sg.k0 + j * kKeysT;
        const int nvalid = sg.k1 - kbase;
        if (kSrc == 0 && nvalid < kKeysT) {   // gathered tiles were zero-filled past the segment
          unsigned char* st = sKV + (g % C::kStages) * C::kStageBytes;
          const int per_box = (kKeysT - nvalid) * 8;         // 16-byte chunks per latent box
          for (int i = row; i < 4 * per_box; i += 128) {
            const int box = i / per_box, rem_i = i - box * per_box;
            *reinterpret_cast<uint4*>(st + box * kBoxBytesK + (nvalid + rem_i / 8) * 128 + (rem_i & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tmem_st_wait();
        MLA_TRACE2_AT(7, g);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full);
        MLA_TRACE_AT(6, g);
      }
      if (!ok) break;
      // ---- epilogue: O / l for this CTA's 256 columns
      ok = group_all(mbar_wait(&bars.seg_done, seg_i & 1, abort));
      if (!ok) break;
      tc_fence_after();
      float l = 0.f;   // an empty segment issued no MMA: its sum columns hold stale data
      if (nt > 0) {
        float lv[16];
        tmem_ld16(tmem + lane_addr + kTmemL, lv);
        tmem_ld_wait();
        l = lv[0];
      }
      // an e4m3 cache's values scale by descale_k
      const float out_mul = kSrc == 1 && p.descale_k != nullptr ? *p.descale_k : 1.f;
      const float inv = l > 0.f ? out_mul / l : 0.f;
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
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.o_empty);
      gt += nt;
      ++seg_i;
    }
    if (!ok) set_abort(bars, peer);
  }
  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && bars.abort_flag) atomicOr(&g_tc_err, kErrTimeout);
#ifdef MLA_TRACE
  if (tid == 0 && blockIdx.x < 512) {
    g_cta_time[blockIdx.x][2] = (long long)globaltimer_ns();
    g_cta_time[blockIdx.x][5] = clock64();
  }
#endif
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();   // no CTA leaves while its peer may still touch its shared memory
}

template <int kRope, int kSrc = 0>
int max_clusters() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> g(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    using C = Cfg<kRope, kSrc>;
    cudaFuncSetAttribute(mla_attn_tc_kernel<kRope, kSrc>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         C::kSmemAlloc);
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
    if (cudaOccupancyMaxActiveClusters(&n, mla_attn_tc_kernel<kRope, kSrc>, &cfg) != cudaSuccess || n <= 0)
      n = device_sm_count() / 2;
    cudaGetLastError();
    cache[dev] = n;
  }
  return cache[dev];
}

template <int kRope, int kSrc>
cudaError_t launch_tc(const TcParams& p, const CUtensorMap& km, const CUtensorMap& rm, int clusters,
                      cudaStream_t st) {
  using C = Cfg<kRope, kSrc>;
  cudaError_t e = cudaFuncSetAttribute(mla_attn_tc_kernel<kRope, kSrc>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemAlloc);
  if (e != cudaSuccess) return e;
  return launch_k(mla_attn_tc_kernel<kRope, kSrc>, dim3(2 * clusters), dim3(kThreads), C::kSmemAlloc, st, km, rm,
                  p);
}

}  // namespace

// ------------------------------------------------------------------ host side
namespace {
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

}  // namespace

bool tensor_maps_available() { return encode_fn() != nullptr; }

bool make_map3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle swz,
                CUtensorMapDataType dt) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


bool tc_attention_supported(mla_dtype dt, int H, int L, int R, bool decode, const CacheView& cv,
                            const View3& q, const View3& o) {
  if (dt != MLA_BF16 || L != 512 || (R != 0 && R != 64)) return false;
  // 128 heads fill the 128-row tile; 64 heads use half of it in decode (one token per
  // sequence: the other rows are masked) and two tokens per tile in prefill
  (void)decode;
  if (H != 128 && H != 64) return false;
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
  return num_splits > 0 ? num_splits : max_clusters<64, 0>();
}

static cudaError_t run_tc(mla_dtype, TcParams& p, const View3& q, const CacheView& cv, int clusters,
                          cudaStream_t st) {
  CUtensorMap km, rm;
  const int E = p.L + p.R;
  const uint32_t rows_box = cv.page < 64 ? cv.page : 64;
  p.q = static_cast<const __nv_bfloat16*>(q.data);
  p.q_s0 = q.s0;
  p.q_s1 = q.s1;
  // latent boxes: 64 columns x rows_box rows, 128-byte swizzle; rope boxes: 32 columns, 64-byte swizzle
  if (!make_map3d(&km, cv.data, E, cv.page, cv.num_blocks, (uint64_t)cv.s_row * 2, (uint64_t)cv.s_blk * 2, 64,
                  rows_box, 1, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (p.R == 0) return launch_tc<0, 0>(p, km, km, clusters, st);
  if (!make_map3d(&rm, cv.data, E, cv.page, cv.num_blocks, (uint64_t)cv.s_row * 2, (uint64_t)cv.s_blk * 2,
                  kRopeHalf, rows_box, 1, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  return launch_tc<64, 0>(p, km, rm, clusters, st);
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

namespace {
TcParams decode_params(const View3& o_lat, float* lse, const View3& q, int32_t B, int32_t H, int32_t R, float scale,
                       const DecodeSched& s) {
  TcParams p{};
  p.mode = 0;
  p.H = H;
  p.tpt = kRows / H;
  p.L = 512;
  p.R = R;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q = static_cast<const __nv_bfloat16*>(q.data);
  p.q_s0 = q.s0;
  p.q_s1 = q.s1;
  p.o_lat = static_cast<__nv_bfloat16*>(o_lat.data);
  p.o_s0 = o_lat.s0;
  p.o_s1 = o_lat.s1;
  p.lse = lse;
  p.B = B;
  p.sched = s;
  return p;
}
}  // namespace

bool tc_gather_supported(mla_dtype dt, int H, const void* cache, int64_t s_blk_bytes, int64_t s_row_bytes,
                         const View3& q, const View3& o) {
  if (dt != MLA_BF16 || (H != 128 && H != 64)) return false;
  auto al16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  if (!al16(cache) || s_blk_bytes % 16 || s_row_bytes % 16) return false;
  if (!al16(q.data) || q.s0 % 8 || q.s1 % 8) return false;
  if (!al16(o.data) || o.s0 % 8 || o.s1 % 8) return false;
  return true;
}

cudaError_t launch_decode_tc_fp8(const View3& o_lat, float* lse, const View3& q, const CacheView& cache,
                                 const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                 int32_t B, int32_t H, int32_t R, float scale, const float* descale_q,
                                 const float* descale_k, const DecodeSched& s, cudaStream_t st) {
  TcParams p = decode_params(o_lat, lse, q, B, H, R, scale, s);
  p.page = cache.page;
  p.num_blocks = cache.num_blocks;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  const long long cap = (long long)max_blocks * cache.page;
  p.cap = (int)(cap > 0x3fffffff ? 0x3fffffff : cap);
  p.cache8 = static_cast<const uint8_t*>(cache.data);
  p.s_blk8 = cache.s_blk;
  p.s_row8 = cache.s_row;
  p.descale_q = descale_q;
  p.descale_k = descale_k;
  // pages of whole 64-row tiles (or tiles of whole pages) come as TMA boxes of bytes: this CTA's
  // 256 latent codes and 32 rope codes of every row; other page sizes are gathered row by row
  CUtensorMap km{}, rm{};
  const int page = cache.page;
  const uint32_t rows_box = page < 64 ? (uint32_t)page : 64u;
  const uint64_t E = 512 + (uint64_t)R;
  p.fp8_tma = (page % 64 == 0 || (64 % page == 0 && page % 8 == 0)) &&
              make_map3d(&km, cache.data, E, (uint64_t)page, (uint64_t)cache.num_blocks, (uint64_t)cache.s_row,
                         (uint64_t)cache.s_blk, 256, rows_box, 1, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_DATA_TYPE_UINT8) &&
              (R == 0 || make_map3d(&rm, cache.data, E, (uint64_t)page, (uint64_t)cache.num_blocks,
                                    (uint64_t)cache.s_row, (uint64_t)cache.s_blk, kRopeHalf, rows_box, 1,
                                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_DATA_TYPE_UINT8))
                  ? 1
                  : 0;
  if (R == 0) return launch_tc<0, 1>(p, km, km, s.units, st);
  return launch_tc<64, 1>(p, km, rm, s.units, st);
}

cudaError_t launch_decode_tc_dsmla(const View3& o_lat, float* lse, const View3& q, const DsMlaCache& cache,
                                   const int32_t* slots, int64_t slot_stride, int32_t topk, int32_t B, int32_t H,
                                   float scale, const DecodeSched& s, cudaStream_t st) {
  TcParams p = decode_params(o_lat, lse, q, B, H, kDsMlaRope, scale, s);
  p.page = cache.page;
  p.num_blocks = cache.num_blocks;
  p.cap = topk;
  p.cache8 = static_cast<const uint8_t*>(cache.data);
  p.s_blk8 = cache.s_blk;
  p.s_row8 = cache.s_row;
  p.slots = slots;
  p.slot_stride = slot_stride;
  CUtensorMap none{};
  return launch_tc<64, 2>(p, none, none, s.units, st);
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
  cudaError_t e = launch_prefill_items(cu_q, B, p.tpt, item_prefix, st);
  if (e != cudaSuccess) return e;
  const int clusters = R == 64 ? max_clusters<64, 0>() : max_clusters<0, 0>();
  return run_tc(MLA_BF16, p, q, cache, clusters, st);
}

#ifdef MLA_TRACE
extern "C" int mla_debug_trace(long long* host) {
  int e = (int)cudaMemcpyFromSymbol(host, g_trace, sizeof(g_trace));
  if (!e) e = (int)cudaMemcpyFromSymbol(host + 2 * 8 * 512, g_trace2, sizeof(g_trace2));
  if (!e) e = (int)cudaMemcpyFromSymbol(host + 4 * 8 * 512, g_cta_time, sizeof(g_cta_time));
  if (!e) e = (int)cudaMemcpyFromSymbol(host + 4 * 8 * 512 + 512 * 10, g_trace_all, sizeof(g_trace_all));
  if (!e)
    e = (int)cudaMemcpyFromSymbol(host + 4 * 8 * 512 + 512 * 10 + sizeof(g_trace_all) / 8, g_trace3,
                                  sizeof(g_trace3));
  if (!e)
    e = (int)cudaMemcpyFromSymbol(host + 4 * 8 * 512 + 512 * 10 + sizeof(g_trace_all) / 8 + sizeof(g_trace3) / 8,
                                  g_trace4, sizeof(g_trace4));
  return e;
}
#endif

unsigned attn_tc_errors_read_clear() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_tc_err, &zero, sizeof(zero));
  return v;
}

}  // namespace mla
