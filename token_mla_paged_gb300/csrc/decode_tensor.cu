// Tensor-core MLA decode kernel for sm_103a (tcgen05 pairs + TMEM + TMA gathers).
//
// All H*T query rows of a request share one stream of latent KV rows, so QK^T
// over 576 columns and PV over 512 are dense contractions.  A work item is 256
// query rows of one request (two 128-row halves) over one split of its KV
// entries, and runs on a cluster of four CTAs on four SMs:
//
//   ranks 0 and 1, the score pair: rank h holds query rows [128h, 128h+128) of
//     the item in TMEM (the A operand), gathered by TMA into the two KV stages
//     (exactly the 144 KB they hold) while they are free between items and moved
//     into TMEM by the row warps.  Each 128-entry KV tile is gathered
//     once per pair: rank h gathers entries [64h, 64h+64) of the tile, all 576
//     columns.  One cta_group::2 MMA per 16 columns (M = 256 rows, N = 128
//     entries, each CTA supplying half of N) writes S = Q K^T of the CTA's own
//     rows into its TMEM, so every gathered byte serves 256 query rows.  Eight
//     row warps per CTA run the masked online softmax (two threads per query
//     row, 64 entries each, exchanging the row max through shared memory) and
//     ship P (bf16) with the per-row rescale factor and running max/sums to the
//     output CTA of the same half with one bulk copy.
//   ranks 2 and 3, the output pair: O[256, 512] accumulates in fp32 TMEM, rank
//     2+h holding the rows of half h.  PV runs as cta_group::2 MMAs of M = 256,
//     N = 256: for latent columns [256c, 256c+256) rank 2 supplies V columns
//     [256c, 256c+128) and rank 3 [256c+128, 256c+256), so each output CTA
//     gathers half of the 512 latent columns of every entry.  Their row warps
//     (two per row, 256 columns each) rescale O when the score side raised its
//     reference max and write O / l and the log-sum-exp (or the split partial
//     and the fused split merge).
//
// KV tiles sit in shared memory as 64-column chunks in the 128-byte swizzled
// layout: the score CTAs read them as the K-major B operand of QK^T, the output
// CTAs as the MN-major B operand of PV.  A TMA gather op costs its issuing warp
// about a hundred cycles, so seven warps share a tile's ops.  fp8 e4m3 pools
// are gathered as bytes and converted to bf16 in registers by four warps
// (exact: e4m3 -> f16 by the hardware conversion, then the f16 bits are placed
// in a bf16 word, which scales every value by 2^-112; the factor is folded into
// the logit and output scales).  The MMA of a pair is issued by its even rank;
// the odd rank relays "my half of the tile is in place" to it through a
// cluster mbarrier.
//
// Sources: absorbed-latent MLA decode with one 576-wide latent row per KV entry
// ("[ROCm] Dspark MLA module", Details); page-size-1 index lists and the
// non-causal draft block ("[ROCm][Spec Decode] Add Aiter MLA decode support
// non-causal draft block", Purpose); causal mask on global positions over a
// round-robin shard with an LSE output ("Speculative decode + DCP on gfx1250",
// Problem); splits over the KV merged in-kernel ("[DSV4] Tuned ASM FP8 decode
// with split plans; HCA on aiter's persistent V4-NM kernel", Summary part 2).
#include <cuda.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "tc_primitives.cuh"

namespace mla {
namespace {

using namespace tc;

// 16 warps, 128 registers each:
//   0-7   row warps: TMEM lane quadrant warp & 3, column half warp >> 2
//   8     MMA issue (even rank) / relay (odd rank); owns TMEM
//   9-15  bf16: TMA gathers; fp8: 9, 14, 15 gather the raw rows, 10-13 convert
constexpr int kThreads = 512;
constexpr int kRowWarps = 8;
constexpr int kWarpMma = 8;
constexpr int kWarpAux0 = 9;
constexpr int kConvWarps = 4;
constexpr int kWarpConv0 = 10;
constexpr int kStages = 2;             // KV tile ring
constexpr int kPBufs = 2;              // P hand-off ring

constexpr int kTileN = kBlockN;        // 128 entries per tile
constexpr int kHalfN = kTileN / 2;     // entries gathered by one score CTA
constexpr int kHalfRows = kRows / 2;   // 128 query rows per CTA
static_assert(kTileN == 128 && kHalfRows == 128, "tile geometry");

constexpr int kSChunk = kHalfN * 128;          // score: [64 entries][64 bf16 columns] = 8 KB
constexpr int kStageBytes = 9 * kSChunk;       // score stage: 576 columns, 72 KB
constexpr int kOChunk = kTileN * 128;          // output: [128 entries][64 columns] = 16 KB
constexpr int kOStageUsed = 4 * kOChunk;       // output stage: 4 column chunks, 64 KB
// fp8 raw rows land in the upper part of a stage and are converted in place.
constexpr int kF8SOff = kStageBytes / 2;       // score: 64 rows x 576 B at 36 KB
constexpr int kF8SBlock = kHalfN * 192;        //   three [64][192 B] column blocks
constexpr int kF8OOff = kOStageUsed / 2;       // output: 128 rows x 2 x 128 B at 32 KB
constexpr int kF8OBlock = kTileN * 128;        //   two [128][128 B] column blocks
constexpr int kPChunk = kHalfRows * 128;       // P: [128 rows][64 entries bf16] = 16 KB
constexpr int kPBytes = 2 * kPChunk;           // 128 entries
constexpr int kPStatsOff = kPBytes;            // alpha[128], m[128], l[2][128] (per column half), flags[4]
constexpr int kPCopyBytes = kPBytes + 4 * 512 + 64;  // bytes handed over per tile, a multiple of 16
// Q of an item on the score side: 128 rows x 576 bf16 = nine 16 KB chunks of 64
// columns (128-byte swizzled, like K), staged in the two KV stages.
constexpr int kQChunk = kHalfRows * 128;
constexpr int kQIssuers = 7;                   // warps 9-15 gather Q (bf16: all gather warps; fp8: with the converters)
constexpr int kQBytes = 9 * kQChunk;
constexpr int kPBufBytes = 35 * 1024;          // buffer stride: each P buffer starts on a swizzle atom

// Shared-memory map (identical offsets in all four CTAs; barriers first).
constexpr int kOffBars = 0;
constexpr int kOffRed = 1024;                                     // score: row-max exchange [2][2][128] fp32
constexpr int kOffTiles = 3072;                                   // kStages x 72 KB
constexpr int kOffPBuf = kOffTiles + kStages * kStageBytes;       // kPBufs P buffers
constexpr int kSmemBytes = kOffPBuf + kPBufs * kPBufBytes;
constexpr int kSmemAlign = 1024;
// Output CTAs: epilogue staging (8 warps x 2 KB) and merge weights live in the
// last 8 KB of each stage, which their 64 KB of V never touches.
constexpr int kOffEpi0 = kOffTiles + kOStageUsed;
constexpr int kOffEpi1 = kOffTiles + kStageBytes + kOStageUsed;
static_assert(kStageBytes - kOStageUsed == 8192, "epilogue staging");
static_assert(kSmemBytes + kSmemAlign <= 232448, "shared memory");
static_assert(kQBytes == kStages * kStageBytes && kQChunk % 1024 == 0, "Q staging fills the two KV stages");
// Every operand the MMA reads through a 128-byte-swizzle descriptor starts on a
// 1024-byte boundary (the swizzle is a function of the address bits).
static_assert(kOffTiles % 1024 == 0 && kStageBytes % 1024 == 0 && kOffPBuf % 1024 == 0 &&
                  kPBufBytes % 1024 == 0 && kPChunk % 1024 == 0 && kPCopyBytes % 16 == 0 &&
                  kPCopyBytes <= kPBufBytes,
              "alignment");

// TMEM columns.
constexpr uint32_t kTmemQ = 0;         // score: Q as A operand, 288 columns
constexpr uint32_t kTmemS = 288;       // score: S, 128 columns
constexpr uint32_t kTmemO = 0;         // output: O, 512 columns

struct Bars {
  uint64_t full[kStages];     // this CTA's share of the tile is in place (TMA, or fp8 conversion)
  uint64_t peer[kStages];     // even rank: the odd rank's share is in place (relayed)
  uint64_t empty[kStages];    // the pair's MMA on this stage is done
  uint64_t full8[kStages];    // fp8: raw e4m3 rows landed (TMA)
  uint64_t cv_sync;           // fp8: the conversion warps finished reading the raw rows
  uint64_t q_full;            // score, even rank: Q of both CTAs written to TMEM
  uint64_t q_free;            // score: every QK^T of the item done
  uint64_t s_full;            // score: S computed
  uint64_t s_free;            // score, even rank: S read out by both CTAs
  uint64_t p_free[kPBufs];    // score: the PV that used this P buffer is done
  uint64_t p_ready[kPBufs];   // score: the eight softmax warps staged P
  uint64_t p_full[kPBufs];    // output: P buffer arrived
  uint64_t corr[kPBufs];      // output, even rank: both CTAs hold P and have rescaled O
  uint64_t o_ready[kPBufs];   // output: PV with this P buffer done
  uint64_t o_free;            // output, even rank: both epilogues read O
  uint64_t q_land;            // score: the item's Q rows landed in the (free) KV stages
  uint64_t q_copied;          // score: the row warps moved them into TMEM
  uint64_t mrg_b;             // output: warp 0 published the split's verdict (partial / merge)
  uint64_t mrg_c;             // output: the row warps fenced their partial rows
  uint64_t never;             // failure-path test: nothing ever arrives here
  uint32_t tmem_base;
  int abort;
  int merge_last;
};
static_assert(sizeof(Bars) <= kOffRed, "barrier block too large");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 128-byte swizzle: byte offset of 16-byte unit u of row r inside a chunk.
__device__ __forceinline__ uint32_t swz(int r, int u) { return (uint32_t)(r * 128 + ((u ^ (r & 7)) << 4)); }
// Epilogue staging, 64-byte rows: unit u of row r (bank-conflict free for 8 rows).
__device__ __forceinline__ uint32_t swz64(int r, int u) { return (uint32_t)(r * 64 + ((u ^ ((r >> 1) & 3)) << 4)); }

constexpr long long kAbortDrainCycles = 200000;   // ~100 µs at GB300 clocks

// On a failed wait: record, raise the abort flag in all four CTAs.
__device__ __noinline__ void fail(Bars* bars, const DecodeParams& p, int site) {
  record_error(p.ws_hdr, MLA_DEV_WAIT_TIMEOUT, site);
  bars->abort = 1;
  for (uint32_t r = 0; r < 4; ++r) {
    const uint32_t a = mapa(smem_u32(&bars->abort), r);
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(1) : "memory");
  }
}

// Warp-collective bounded waits: every lane polls, and the warp leaves together
// (to the teardown) if any lane gave up.  WAITC: barrier signalled from another CTA.
#define WAIT(bar, par, site)                                                          \
  if (!__all_sync(0xffffffffu, mbar_wait(bar, par, &bars->abort, p.wait_limit))) {   \
    fail(bars, p, site);                                                              \
    goto done;                                                                        \
  }
#define WAITC(bar, par, site)                                                         \
  if (!__all_sync(0xffffffffu, mbar_wait<true>(bar, par, &bars->abort, p.wait_limit))) { \
    fail(bars, p, site);                                                              \
    goto done;                                                                        \
  }

// Arrive on `bar` in CTA `to` (this CTA or another of the cluster).  Every
// cross-CTA signal here orders only tcgen05 work the caller fenced with
// tcgen05.fence::before_thread_sync (TMEM reads and writes) or data whose landing
// the caller observed on its own barrier, so the remote arrive is relaxed.
__device__ __forceinline__ void arrive_at(uint64_t* bar, uint32_t to, uint32_t self) {
  if (to == self) mbar_arrive(bar);
  else mbar_arrive_remote_relaxed(bar, to);
}

// Static work assignment, identical in every role of all four CTAs: round r
// gives cluster c item r*C + c on even rounds and r*C + (C-1-c) on odd rounds,
// so a cost-sorted item list is dealt out boustrophedon-fashion.
__device__ __forceinline__ int item_of(int r, int c, int C) { return r * C + ((r & 1) ? C - 1 - c : c); }
#define FOR_ITEMS(idx)                                                      \
  for (int r_ = 0, idx = item_of(0, cluster, n_clusters); idx < n_items; \
       ++r_, idx = item_of(r_, cluster, n_clusters))

// Number of 128-entry tiles of an item (the same in all four CTAs).
__device__ __forceinline__ int item_tiles(const Item& it) {
  return it.ok && it.e1 > it.e0 ? (it.e1 - it.e0 + kTileN - 1) / kTileN : 0;
}

// Pull one half's query rows of item `idx` into L2 ahead of their TMEM load.
__device__ __forceinline__ void prefetch_q_rows(const DecodeParams& p, int idx, int n_items, int half) {
  if (idx >= n_items) return;
  const Item it = load_item(p, idx);
  if (!it.ok) return;
  const int hrows = min(max(it.nrows - kHalfRows * half, 0), kHalfRows);
  if (hrows <= 0) return;
  const uint8_t* src = reinterpret_cast<const uint8_t*>(static_cast<const uint16_t*>(p.q) +
                                                        (it.q_row_base + it.row0 + kHalfRows * half) * kDqk);
  const uint32_t bytes = (uint32_t)hrows * kDqk * 2;
  for (uint32_t o = 0; o < bytes; o += 16384) prefetch_l2_bulk(src + o, bytes - o < 16384 ? bytes - o : 16384);
}

// 16 e4m3 values -> two 16-byte bf16 units at dst0 / dst1.  Exact: the f16 bits
// from the hardware e4m3 conversion are placed in a bf16 word with the same
// exponent field, which scales every value by 2^-112 (folded into the scales).
__device__ __forceinline__ void fp8_unit_to_bf16(uint8_t* dst0, uint8_t* dst1, const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h0, h1;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h0) : "h"((uint16_t)(w[q] & 0xFFFF)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h1) : "h"((uint16_t)(w[q] >> 16)));
    o[2 * q] = ((h0 & 0x7FFF7FFFu) >> 3) | (h0 & 0x80008000u);
    o[2 * q + 1] = ((h1 & 0x7FFF7FFFu) >> 3) | (h1 & 0x80008000u);
  }
  *reinterpret_cast<uint4*>(dst0) = make_uint4(o[0], o[1], o[2], o[3]);
  *reinterpret_cast<uint4*>(dst1) = make_uint4(o[4], o[5], o[6], o[7]);
}

// Epilogue write-back of a 64-byte column segment (32 bf16 or 16 fp32 columns
// starting at byte `col_byte` of each row) of a warp's 32 rows, staged at stg as
// [32][64 B]: each store instruction writes eight whole 64-byte row segments.
// Row ri of this CTA's half lives at base + (128*half + ri) * pitch.
__device__ __forceinline__ void epi_rows_out(const uint8_t* stg, int lane, int q4, int col_byte, uint8_t* base,
                                             int64_t pitch, int half, int hrows) {
  uint4 val[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rl = 8 * i + (lane >> 2), u = lane & 3;
    val[i] = *reinterpret_cast<const uint4*>(stg + swz64(rl, u));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rl = 8 * i + (lane >> 2), u = lane & 3;
    const int ri = 32 * q4 + rl;                 // row within this half
    if (ri < hrows)
      *reinterpret_cast<uint4*>(base + (int64_t)(kHalfRows * half + ri) * pitch + col_byte + 16 * u) = val[i];
  }
}

// One thread's 32 values -> its row of the warp's staging block, then the warp
// writes the block out (fp32: two 64-byte halves; bf16: one).
__device__ __forceinline__ void stage_and_write(const float (&v)[32], bool f32, uint8_t* epi, int lane, int q4,
                                                int col, uint8_t* base, int64_t pitch, int half, int hrows) {
  if (f32) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        *reinterpret_cast<float4*>(epi + swz64(lane, k)) =
            make_float4(v[16 * hh + 4 * k], v[16 * hh + 4 * k + 1], v[16 * hh + 4 * k + 2], v[16 * hh + 4 * k + 3]);
      __syncwarp();
      epi_rows_out(epi, lane, q4, 4 * (col + 16 * hh), base, pitch, half, hrows);
      __syncwarp();
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      *reinterpret_cast<uint4*>(epi + swz64(lane, k)) =
          make_uint4(pack_bf16x2(v[8 * k], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                     pack_bf16x2(v[8 * k + 4], v[8 * k + 5]), pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
    __syncwarp();
    epi_rows_out(epi, lane, q4, 2 * col, base, pitch, half, hrows);
    __syncwarp();
  }
}

// Score side, at the start of an item: once the previous item's QK^T is done with
// both KV stages (their `empty` phases for tiles kseq-1 and kseq-2), gather the
// item's live Q rows of this CTA's half into them: 9 chunks of 64 columns, groups of
// 4 rows, one gather4 per lane over `nissue` warps (this one is number `wi`).  The
// last group repeats the half's last live row.  Rows that are not live are not
// loaded: their Q only feeds their own, masked, S rows.  (The caller waits for the
// stages to be free.)
__device__ __forceinline__ uint32_t q_groups(const Item& it, int half) {
  const int hrows = min(max(it.nrows - kHalfRows * half, 0), kHalfRows);
  return (uint32_t)((hrows + 3) / 4);
}
__device__ __forceinline__ void stage_q(const Item& it, int half, uint32_t tiles_u32, const CUtensorMap* tmap_q,
                                        uint64_t* q_land, int wi, int nissue, int lane) {
  const int ng = (int)q_groups(it, half);
  const int64_t row0 = it.q_row_base + it.row0 + kHalfRows * half;
  const int last = min(it.nrows - kHalfRows * half, kHalfRows) - 1;
  for (int o = wi * 32 + lane; o < 9 * ng; o += nissue * 32) {
    const int c = o / ng, g = o - c * ng;
    const int r0 = 4 * g;
    tma_gather4(tiles_u32 + (uint32_t)(c * kQChunk + g * 512), tmap_q, 64 * c, (int32_t)(row0 + min(r0, last)),
                (int32_t)(row0 + min(r0 + 1, last)), (int32_t)(row0 + min(r0 + 2, last)),
                (int32_t)(row0 + min(r0 + 3, last)), q_land);
  }
}

template <bool kFp8>
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kThreads, 1)
mla_decode_tensor_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                         const __grid_constant__ CUtensorMap tmap_q, const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((kSmemAlign - (smem_u32(smem_raw) & (kSmemAlign - 1))) & (kSmemAlign - 1));
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBars);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int half = (int)(rank & 1u);              // row half of the item / B half of the pair
  const bool score_cta = rank < 2;
  const bool even = half == 0;                    // issues the pair's MMAs
  const uint32_t lead = rank & ~1u;               // even rank of this CTA's pair
  const uint32_t out_peer = rank ^ 2u;            // same half on the other side

  const int cluster = (int)cluster_id_x(), n_clusters = (int)num_clusters_x();

  // Set-up first: it reads nothing an earlier kernel writes, so it overlaps the
  // end of that kernel (the device planner, in the re-planning mode).
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], kFp8 ? kConvWarps : 1);
      mbar_init(&bars->peer[s], 1);
      mbar_init(&bars->empty[s], 1);
      mbar_init(&bars->full8[s], 1);
    }
    mbar_init(&bars->cv_sync, kConvWarps);
    mbar_init(&bars->q_full, 2 * kRowWarps);
    mbar_init(&bars->q_free, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 2 * kRowWarps);
    for (int b = 0; b < kPBufs; ++b) {
      mbar_init(&bars->p_free[b], 1);
      mbar_init(&bars->p_ready[b], kRowWarps);
      mbar_init(&bars->p_full[b], 1);
      mbar_init(&bars->corr[b], 2 * kRowWarps);
      mbar_init(&bars->o_ready[b], 1);
    }
    mbar_init(&bars->o_free, 2 * kRowWarps);
    mbar_init(&bars->q_land, 1);
    mbar_init(&bars->q_copied, kRowWarps);
    mbar_init(&bars->mrg_b, 1);
    mbar_init(&bars->mrg_c, kRowWarps);
    mbar_init(&bars->never, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc2(&bars->tmem_base, 512);
    tmem_relinquish2();
  }
  if (warp == kWarpAux0 && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    prefetch_tmap(&tmap_q);
  }
  fence_before_sync();
  __syncthreads();
  cluster_sync();        // barriers of all four CTAs initialised before any remote arrival
  fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  uint8_t* tiles = smem + kOffTiles;
  uint8_t* pbufs = smem + kOffPBuf;
  grid_dependency_wait();
  allow_dependent_launch();
  // A plan that does not match the call runs no item: every CTA goes straight to
  // the teardown.
  const bool plan_ok = plan_header_ok(p.plan, p);
  if (!plan_ok && blockIdx.x == 0 && tid == 0) record_error(p.ws_hdr, MLA_DEV_PLAN_MISMATCH, 0);
  const int n_items = plan_ok ? p.plan[kHNItems] : 0;
  if (blockIdx.x == 0 && tid == 0) p.ws_hdr[kWsCounterWords] = p.counters_words;
  if (score_cta && tid == 0) prefetch_q_rows(p, item_of(0, cluster, n_clusters), n_items, half);
  // Failure-path test: every warp waits on a barrier nothing signals, before any
  // copy or MMA is issued, so the bounded wait runs out with nothing in flight
  // and the kernel records the timeout and tears down.
  if (p.test_stall) {
    WAIT(&bars->never, 0, 99);
  }

  // ======================================================================= producers
  // KV gathers with TMA.  One gather op moves 4 rows (entries 4g..4g+3) x one
  // column box; each lane of an issuing warp owns at most one op of the tile.
  //   score CTA h: entries [64h, 64h+64) of the tile, 9 column chunks (bf16: 144
  //     ops; fp8: three 192-byte boxes per row, 48 ops, into the stage's upper half);
  //   output CTA h: all 128 entries, latent columns [128h, 128h+128) and
  //     [256+128h, 256+128h+128) (bf16: 4 chunks, 128 ops; fp8: two 128-byte
  //     boxes per row, 64 ops, into the upper half of its 64 KB).
  if (warp >= kWarpAux0 && (!kFp8 || warp < kWarpConv0 || warp >= kWarpConv0 + kConvWarps)) {
    constexpr int npw = kFp8 ? 3 : 7;                        // issuing warps
    const int pw = (!kFp8 || warp == kWarpAux0) ? warp - kWarpAux0 : warp - (kWarpConv0 + kConvWarps) + 1;
    const int ngroups = score_cta ? kHalfN / 4 : kTileN / 4;  // 16 | 32 groups of 4 entries
    const int nblk = kFp8 ? (score_cta ? 3 : 2) : (score_cta ? 9 : 4);
    const int nops = ngroups * nblk;
    const int per = (nops + npw - 1) / npw;                   // ops of this warp: [o_begin, o_end), <= 32
    const int o_begin = pw * per, o_end = o_begin + per < nops ? o_begin + per : nops;
    const uint32_t tx = (uint32_t)(score_cta ? (kFp8 ? kHalfN * 576 : kStageBytes)
                                              : (kFp8 ? kTileN * 256 : kOStageUsed));
    const int e_sub = score_cta ? kHalfN * half : 0;          // first tile entry this CTA gathers
    const int nidx = ngroups / 8;                             // index registers in use (2 | 4)
    const void* tmap = score_cta ? (const void*)&tmap_k : (const void*)&tmap_v;
    uint32_t kseq = 0, qseq = 0;
    const bool report = pw == 0;
    // Raw slot indices of tile j: lane holds entries lane + 32k (k < nidx), -1 past
    // the end; checked only when used, one iteration later, so the load is not waited on.
    auto tile_idx = [&](const Item& it, int j, int32_t (&x)[4]) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = it.e0 + j * kTileN + e_sub + lane + 32 * k;
        x[k] = (k < nidx && i < it.e1) ? __ldg(p.kv_indices + it.kv_off + i) : -1;
      }
    };
    // Invalid entries read row -1 (zero fill) and are reported once.
    auto checked = [&](const Item& it, int j, int k, int32_t v) -> int32_t {
      if (v >= 0 && v < p.num_slots) return v;
      const int i = it.e0 + j * kTileN + e_sub + lane + 32 * k;
      if (report && k < nidx && i < it.e1) record_error(p.ws_hdr, MLA_DEV_BAD_INDEX, (int)(it.kv_off + i));
      return -1;
    };
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      const int nt = item_tiles(it);
      int32_t nx[4] = {-1, -1, -1, -1};
      if (nt > 0) tile_idx(it, 0, nx);
      if (score_cta && nt > 0) {
        // The item's Q rows pass through the KV stages (the fp8 conversion warps issue
        // their share too), then the stages go back to the KV tiles.
        for (int k = 1; k <= kStages; ++k)
          if ((int)kseq - k >= 0) {
            const uint32_t s = kseq - k;
            WAITC(&bars->empty[s % kStages], (s / kStages) & 1, 8);
          }
        if (pw == 0 && lane == 0) mbar_arrive_expect_tx(&bars->q_land, 9 * 512 * q_groups(it, half));
        __syncwarp();
        stage_q(it, half, smem_u32(tiles), &tmap_q, &bars->q_land, pw, kQIssuers, lane);
        __syncwarp();
        WAITC(&bars->q_copied, qseq & 1, 9);
        ++qseq;
      }
      for (int j = 0; j < nt; ++j, ++kseq) {
        const int st = kseq % kStages;
        const uint32_t ph = (kseq / kStages) & 1;
        int32_t cx[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) cx[k] = checked(it, j, k, nx[k]);
        if (j + 1 < nt) tile_idx(it, j + 1, nx);
        // slot indices of this lane's op: group g's entries 4g..4g+3 sit in lanes
        // (4g..4g+3) % 32 of index register g / 8
        const int o = o_begin + lane;
        const int g = (o < o_end ? o : o_begin) / nblk;
        int32_t a[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int src = ((4 * g) & 31) + e;
          const int32_t v0 = __shfl_sync(0xffffffffu, cx[0], src);
          const int32_t v1 = __shfl_sync(0xffffffffu, cx[1], src);
          const int32_t v2 = __shfl_sync(0xffffffffu, cx[2], src);
          const int32_t v3 = __shfl_sync(0xffffffffu, cx[3], src);
          const int k = g >> 3;
          a[e] = k == 0 ? v0 : k == 1 ? v1 : k == 2 ? v2 : v3;
        }
        WAITC(&bars->empty[st], ph ^ 1, 1);
        uint64_t* bar = kFp8 ? &bars->full8[st] : &bars->full[st];
        if (pw == 0 && lane == 0) mbar_arrive_expect_tx(bar, tx);
        __syncwarp();
        const uint32_t base = smem_u32(tiles + st * kStageBytes);
        if (o < o_end) {
          const int c = o - g * nblk;
          uint32_t dst;
          int32_t col;
          if (kFp8) {
            if (score_cta) {
              dst = base + (uint32_t)(kF8SOff + c * kF8SBlock + g * 4 * 192);
              col = 192 * c;
            } else {
              dst = base + (uint32_t)(kF8OOff + c * kF8OBlock + g * 4 * 128);
              col = 256 * c + 128 * half;
            }
          } else if (score_cta) {
            dst = base + (uint32_t)(c * kSChunk + g * 512);
            col = 64 * c;
          } else {
            dst = base + (uint32_t)(c * kOChunk + g * 512);
            col = 64 * (c < 2 ? 2 * half + c : 4 + 2 * half + (c - 2));
          }
          tma_gather4(dst, tmap, col, a[0], a[1], a[2], a[3], bar);
        }
        __syncwarp();
      }
    }
    // Drain: the pair's last MMA commits on `empty` must land before this CTA exits.
    if (pw == 0)
      for (int k = 0; k < kStages && (int)kseq - 1 - k >= 0; ++k) {
        const uint32_t s = kseq - 1 - k;
        WAITC(&bars->empty[s % kStages], (s / kStages) & 1, 2);
      }
  }
  // ======================================================================= fp8: convert in place
  // The conversion warps turn the stage's raw e4m3 rows into the swizzled bf16
  // tile.  Rows are split between the warps.  The chunks that land below the raw
  // area are written first; the raw bytes of the rest go to registers, and once
  // every conversion warp holds its share the remaining chunks overwrite the raw area.
  else if (kFp8 && warp >= kWarpConv0 && warp < kWarpConv0 + kConvWarps) {
    const int cw = warp - kWarpConv0;
    uint32_t kseq = 0, cv_ph = 0;
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      const int nt = item_tiles(it);
      if (score_cta && nt > 0) {
        // this warp's share of the item's Q gathers, once both stages are free
        for (int k = 1; k <= kStages; ++k)
          if ((int)kseq - k >= 0) {
            const uint32_t s = kseq - k;
            WAITC(&bars->empty[s % kStages], (s / kStages) & 1, 7);
          }
        stage_q(it, half, smem_u32(tiles), &tmap_q, &bars->q_land, 3 + cw, kQIssuers, lane);
        __syncwarp();
      }
      for (int j = 0; j < nt; ++j, ++kseq) {
        const int st = kseq % kStages;
        WAIT(&bars->full8[st], (kseq / kStages) & 1, 4);
        uint8_t* stage = tiles + st * kStageBytes;
        if (score_cta) {
          // 64 rows x 36 units of 16 e4m3 values; warp cw owns rows kR*cw ...
          // Chunk c, unit u (of 4 per 64 columns) is raw unit 4c+u of the row, in
          // column block (4c+u)/12 at offset ((4c+u)%12)*16.
          constexpr int kR = kHalfN / kConvWarps;     // 16 rows per warp
          const uint8_t* raw = stage + kF8SOff;
#pragma unroll
          for (int k = 0; k < kR * 16 / 32; ++k) {    // chunks 0-3: kR rows x 16 units
            const int f = k * 32 + lane, row = kR * cw + (f >> 4), c = (f >> 2) & 3, u = f & 3;
            const int ru = 4 * c + u;
            const uint4 v = *reinterpret_cast<const uint4*>(raw + (ru / 12) * kF8SBlock + row * 192 + (ru % 12) * 16);
            uint8_t* ch = stage + c * kSChunk;
            fp8_unit_to_bf16(ch + swz(row, 2 * u), ch + swz(row, 2 * u + 1), v);
          }
          uint4 rb[kR * 20 / 32];                     // chunks 4-8: kR rows x 20 units
#pragma unroll
          for (int k = 0; k < kR * 20 / 32; ++k) {
            const int f = k * 32 + lane, row = kR * cw + f / 20, c = 4 + (f % 20) / 4, u = f & 3;
            const int ru = 4 * c + u;
            rb[k] = *reinterpret_cast<const uint4*>(raw + (ru / 12) * kF8SBlock + row * 192 + (ru % 12) * 16);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->cv_sync);
          WAIT(&bars->cv_sync, cv_ph, 5);
          cv_ph ^= 1;
#pragma unroll
          for (int k = 0; k < kR * 20 / 32; ++k) {
            const int f = k * 32 + lane, row = kR * cw + f / 20, c = 4 + (f % 20) / 4, u = f & 3;
            uint8_t* ch = stage + c * kSChunk;
            fp8_unit_to_bf16(ch + swz(row, 2 * u), ch + swz(row, 2 * u + 1), rb[k]);
          }
        } else {
          // 128 rows x 16 units; warp cw owns rows kR*cw ...  Raw unit ru of a row
          // sits in column block ru/8 at offset (ru%8)*16 and becomes units
          // 2(ru%4), 2(ru%4)+1 of chunk slot ru/4.
          constexpr int kR = kTileN / kConvWarps;     // 32 rows per warp
          const uint8_t* raw = stage + kF8OOff;
#pragma unroll
          for (int k = 0; k < kR * 8 / 32; ++k) {     // slots 0-1 (raw block 0): kR rows x 8 units
            const int f = k * 32 + lane, row = kR * cw + (f >> 3), ru = f & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(raw + row * 128 + ru * 16);
            uint8_t* ch = stage + (ru >> 2) * kOChunk;
            fp8_unit_to_bf16(ch + swz(row, 2 * (ru & 3)), ch + swz(row, 2 * (ru & 3) + 1), v);
          }
          uint4 rb[kR * 8 / 32];                      // slots 2-3 (raw block 1)
#pragma unroll
          for (int k = 0; k < kR * 8 / 32; ++k) {
            const int f = k * 32 + lane, row = kR * cw + (f >> 3), ru = f & 7;
            rb[k] = *reinterpret_cast<const uint4*>(raw + kF8OBlock + row * 128 + ru * 16);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->cv_sync);
          WAIT(&bars->cv_sync, cv_ph, 5);
          cv_ph ^= 1;
#pragma unroll
          for (int k = 0; k < kR * 8 / 32; ++k) {
            const int f = k * 32 + lane, row = kR * cw + (f >> 3), ru = f & 7;
            uint8_t* ch = stage + (2 + (ru >> 2)) * kOChunk;
            fp8_unit_to_bf16(ch + swz(row, 2 * (ru & 3)), ch + swz(row, 2 * (ru & 3) + 1), rb[k]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->full[st]);
      }
    }
  }
  // ======================================================================= odd ranks: relay
  // Tell the even rank of the pair that this CTA's share of the tile is in place.
  else if (!even && warp == kWarpMma) {
    uint32_t kseq = 0;
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      const int nt = item_tiles(it);
      for (int j = 0; j < nt; ++j, ++kseq) {
        const int st = kseq % kStages;
        WAIT(&bars->full[st], (kseq / kStages) & 1, 6);
        if (lane == 0) mbar_arrive_remote_relaxed(&bars->peer[st], lead);
        __syncwarp();
      }
    }
  }
  // ======================================================================= score pair: MMA (rank 0)
  else if (score_cta && warp == kWarpMma) {
    uint32_t kseq = 0, qitem = 0;
    const uint32_t idesc = idesc_bf16_f32(256, kTileN, false, false);
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      const int nt = item_tiles(it);
      if (nt == 0) continue;
      WAITC(&bars->q_full, qitem & 1, 10);
      for (int j = 0; j < nt; ++j, ++kseq) {
        const int st = kseq % kStages;
        const uint32_t kph = (kseq / kStages) & 1;
        WAITC(&bars->s_free, (kseq & 1) ^ 1, 11);
        WAIT(&bars->full[st], kph, 12);
        WAITC(&bars->peer[st], kph, 13);
        fence_after_sync();
        if (lane == 0) {
          // B descriptor of K step k: chunk k/4, 32-byte column offset k%4
          const uint64_t bdesc0 = smem_desc_sw128(smem_u32(tiles + st * kStageBytes), 16, 1024);
#pragma unroll
          for (int k = 0; k < kDqk / 16; ++k)
            mma2_ts(tmem + kTmemS, tmem + kTmemQ + 8 * k,
                    bdesc0 + (uint64_t)(((k >> 2) * kSChunk + (k & 3) * 32) >> 4), idesc, k > 0);
          mma2_commit_mc(&bars->empty[st], 0x3);
          mma2_commit_mc(&bars->s_full, 0x3);
        }
        __syncwarp();
      }
      if (lane == 0) mma2_commit_mc(&bars->q_free, 0x3);
      __syncwarp();
      ++qitem;
    }
  }
  // ======================================================================= output pair: MMA (rank 2)
  else if (warp == kWarpMma) {
    uint32_t kseq = 0, oitem = 0;
    const uint32_t idesc = idesc_bf16_f32(256, 256, false, true);
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      const int nt = item_tiles(it);
      if (nt == 0) continue;
      WAITC(&bars->o_free, (oitem & 1) ^ 1, 20);
      for (int j = 0; j < nt; ++j, ++kseq) {
        const int st = kseq % kStages, pb = kseq % kPBufs;
        const uint32_t kph = (kseq / kStages) & 1, pph = (kseq / kPBufs) & 1;
        WAIT(&bars->full[st], kph, 21);
        WAITC(&bars->peer[st], kph, 22);
        WAITC(&bars->corr[pb], pph, 23);
        fence_after_sync();
        if (lane == 0) {
          const uint64_t adesc0 = smem_desc_sw128(smem_u32(pbufs + pb * kPBufBytes), 16, 1024);
          const uint64_t bdesc0 = smem_desc_sw128(smem_u32(tiles + st * kStageBytes), kOChunk, 1024);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int k = 0; k < kTileN / 16; ++k)
              mma2_ss(tmem + kTmemO + 256 * h, adesc0 + (uint64_t)(((k >> 2) * kPChunk + (k & 3) * 32) >> 4),
                      bdesc0 + (uint64_t)(((2 * h) * kOChunk + k * 2048) >> 4), idesc,
                      (j > 0 || k > 0) ? 1u : 0u);
          }
          mma2_commit_mc(&bars->empty[st], 0xC);
          mma2_commit_mc(&bars->p_free[pb], 0x3);
          mma2_commit_mc(&bars->o_ready[pb], 0xC);
        }
        __syncwarp();
      }
      ++oitem;
    }
  }
  // ======================================================================= score pair: softmax
  // Thread (row r, column half ch) owns entries [64ch, 64ch+64) of every tile.
  else if (score_cta && warp < kRowWarps) {
    const int q4 = warp & 3, ch = warp >> 2;
    const int r = 32 * q4 + lane;            // query row within this CTA's half
    const uint32_t lane_addr = (uint32_t)(32 * q4) << 16;
    float* red = reinterpret_cast<float*>(smem + kOffRed);   // [slot][ch][128]
    uint32_t sseq = 0, qitem = 0;
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      const int nt = item_tiles(it);
      if (nt == 0) continue;
      const int hrow0 = it.row0 + kHalfRows * half;
      const int hrows = it.nrows - kHalfRows * half;
      const bool live = r < hrows;
      // Q rows of this half -> TMEM (A operand layout: lane = row, two bf16 per
      // column); column half 0 loads units [0, 40), half 1 units [40, 72).
      WAITC(&bars->q_free, (qitem & 1) ^ 1, 30);
      if (warp == 0 && lane == 0) prefetch_q_rows(p, item_of(r_ + 1, cluster, n_clusters), n_items, half);
      // Q rows of this half -> TMEM (A operand layout: lane = row, two bf16 per
      // column), from the staging the gather warps filled: column half 0 moves chunks
      // [0, 5), half 1 chunks [5, 9).
      WAIT(&bars->q_land, qitem & 1, 35);
      {
        const int rr = 32 * q4 + lane;
        const int c_beg = ch ? 5 : 0, c_end = ch ? 9 : 5;   // 64-column chunks = 32 TMEM columns
        for (int c0 = c_beg; c0 < c_end; ++c0) {
          const uint8_t* chunk = tiles + c0 * kQChunk;
          uint32_t v[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint4 u = *reinterpret_cast<const uint4*>(chunk + swz(rr, k));
            v[4 * k] = u.x;
            v[4 * k + 1] = u.y;
            v[4 * k + 2] = u.z;
            v[4 * k + 3] = u.w;
          }
          tmem_st32(tmem + lane_addr + kTmemQ + 32 * c0, v);
        }
        tmem_wait_st();
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->q_copied);                    // the stages go back to the KV gathers
        arrive_at(&bars->q_full, lead, rank);
      }
      ++qitem;

      // Visibility: local entry i is visible to this row iff ibeg <= i < iend, its
      // index is valid and, with per-entry positions, its position passes the
      // row's causal limit (and window).
      const int t_row = (hrow0 + r) / p.num_heads;
      int ibeg = 0, iend = it.e1;
      if (p.causal && live && !p.kv_pos) {
        const int64_t lim = it.Lg - it.T + t_row - it.base;
        const int64_t cnt = lim < 0 ? 0 : lim / it.stride + 1;
        if (cnt < iend) iend = (int)cnt;
        if (p.window > 0) {              // positions base + i*stride > limit - W
          const int64_t lo = lim - p.window;
          const int64_t first = lo < 0 ? 0 : lo / it.stride + 1;
          ibeg = first < (int64_t)iend ? (int)first : iend;
        }
      }
      if (!live) iend = -1;
      // tokens of this warp's 32 rows (per-entry positions need one mask per token)
      const int t_first = (hrow0 + 32 * q4) / p.num_heads, t_last = (hrow0 + 32 * q4 + 31) / p.num_heads;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j, ++sseq) {
        const int pb = sseq % kPBufs;
        const int i0 = it.e0 + j * kTileN + 64 * ch;   // first entry of this thread's 64
        // validity of the 64 slot indices: word w covers entries i0 + 32w ..
        uint32_t vm[2];
        {
          bool ok[2];
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            const int a = i0 + 32 * w + lane;
            ok[w] = false;
            if (a < it.e1) {
              const int32_t s = __ldg(p.kv_indices + it.kv_off + a);
              ok[w] = s >= 0 && s < p.num_slots;
            }
          }
          if (p.kv_pos && p.causal) {
            int64_t gp[2];
#pragma unroll
            for (int w = 0; w < 2; ++w) {
              const int a = i0 + 32 * w + lane;
              gp[w] = a < it.e1 ? (int64_t)__ldg(p.kv_pos + it.kv_off + a) : INT64_MAX;
              vm[w] = 0;
            }
            for (int t = t_first; t <= t_last; ++t) {
              const int64_t lim = it.Lg - it.T + t;
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                const bool in = gp[w] <= lim && (p.window <= 0 || gp[w] > lim - p.window);
                const uint32_t mk = __ballot_sync(0xffffffffu, ok[w] && in);
                if (t == t_row) vm[w] = mk;
              }
            }
          } else {
#pragma unroll
            for (int w = 0; w < 2; ++w) vm[w] = __ballot_sync(0xffffffffu, ok[w]);
          }
          // entries [ibeg, iend) may be visible: fold the range into the masks
          const int nvis = iend - i0, nbeg = ibeg - i0;
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            const int hi = min(max(nvis - 32 * w, 0), 32), lo = min(max(nbeg - 32 * w, 0), 32);
            const uint32_t range = (hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u)) & (lo >= 32 ? 0u : (0xffffffffu << lo));
            vm[w] &= range;
          }
        }
        WAIT(&bars->s_full, sseq & 1, 31);
        fence_after_sync();
        uint32_t sv[2][32];
        tmem_ld32(tmem + lane_addr + kTmemS + 64 * ch, sv[0]);
        tmem_ld32(tmem + lane_addr + kTmemS + 64 * ch + 32, sv[1]);
        tmem_wait_ld();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_at(&bars->s_free, lead, rank);

        float pmax = -INFINITY;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const bool vis = (vm[w] >> e) & 1u;
            const float x = vis ? __uint_as_float(sv[w][e]) * p.scale_log2 : -INFINITY;
            sv[w][e] = __float_as_uint(x);
            pmax = fmaxf(pmax, x);
          }
        }
        // the row's max over both halves
        const int slot = sseq & 1;
        red[(slot * 2 + ch) * kHalfRows + r] = pmax;
        named_bar_sync(1 + q4, 64);
        const float tmax = fmaxf(pmax, red[(slot * 2 + (ch ^ 1)) * kHalfRows + r]);
        float alpha = 1.f;
        int need = 0;
        if (tmax > m_ref + 8.f) {          // raise the reference max only when it grew a lot
          alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - tmax);
          m_ref = tmax;
          need = 1;
        }
        const int any_need = __any_sync(0xffffffffu, need);
        // Hand P to the output CTA of this half.
        WAITC(&bars->p_free[pb], ((sseq / kPBufs) & 1) ^ 1, 32);
        uint8_t* stg = pbufs + pb * kPBufBytes;
        float psum = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {      // 8 entries per 16-byte unit of chunk ch
          uint32_t pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int e = 8 * u + 2 * q;
            const float x0 = __uint_as_float(sv[e >> 5][e & 31]), x1 = __uint_as_float(sv[e >> 5][(e & 31) + 1]);
            const float a = m_ref == -INFINITY ? 0.f : ex2(x0 - m_ref);
            const float b = m_ref == -INFINITY ? 0.f : ex2(x1 - m_ref);
            psum += a + b;
            pk[q] = pack_bf16x2(a, b);
          }
          *reinterpret_cast<uint4*>(stg + ch * kPChunk + swz(r, u)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        l = l * alpha + psum;              // this half's share of the row sum
        float* stats = reinterpret_cast<float*>(stg + kPStatsOff);
        if (ch == 0) {
          stats[r] = alpha;
          stats[128 + r] = m_ref;
          if (lane == 0) reinterpret_cast<int*>(stats + 512)[q4] = any_need;
        }
        stats[256 + 128 * ch + r] = l;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_ready[pb]);
        if (warp == 0) {
          WAIT(&bars->p_ready[pb], (sseq / kPBufs) & 1, 34);
          if (lane == 0) {
            const uint32_t src = smem_u32(stg);
            bulk_copy_to_peer(mapa(src, out_peer), src, kPCopyBytes, mapa(smem_u32(&bars->p_full[pb]), out_peer));
          }
          __syncwarp();
        }
      }
    }
    // Drain: the output pair's last PV commits on p_free must land before this CTA exits.
    for (int k = 0; k < kPBufs && (int)sseq - 1 - k >= 0; ++k) {
      const uint32_t s = sseq - 1 - k;
      WAITC(&bars->p_free[s % kPBufs], (s / kPBufs) & 1, 33);
    }
  }
  // ======================================================================= output pair: correction + epilogue
  // Thread (row r, column half ch) owns O columns [256ch, 256ch+256).
  else if (!score_cta && warp < kRowWarps) {
    const int q4 = warp & 3, ch = warp >> 2;
    const int r = 32 * q4 + lane;
    const uint32_t lane_addr = (uint32_t)(32 * q4) << 16;
    uint8_t* epi = smem + (warp < 4 ? kOffEpi0 : kOffEpi1) + (warp & 3) * 2048;
    uint32_t pseq = 0, mrg_b_ph = 0, mrg_c_ph = 0;
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      if (!it.ok) continue;
      const int nt = item_tiles(it);
      const int hrows = min(max(it.nrows - kHalfRows * half, 0), kHalfRows);
      const bool live = r < hrows;
      float m_last = -INFINITY, l_last = 0.f;
      for (int j = 0; j < nt; ++j, ++pseq) {
        const int pb = pseq % kPBufs;
        const uint32_t pph = (pseq / kPBufs) & 1;
        if (warp == 0 && lane == 0) mbar_arrive_expect_tx(&bars->p_full[pb], kPCopyBytes);
        WAITC(&bars->p_full[pb], pph, 40);
        const float* stats = reinterpret_cast<const float*>(pbufs + pb * kPBufBytes + kPStatsOff);
        const float alpha = stats[r];
        m_last = stats[128 + r];
        l_last = stats[256 + r] + stats[384 + r];
        if (reinterpret_cast<const int*>(stats + 512)[q4] && j > 0) {
          // O of the previous tile must be complete before rescaling it.
          const uint32_t prev = pseq - 1;
          WAITC(&bars->o_ready[prev % kPBufs], (prev / kPBufs) & 1, 41);
          fence_after_sync();
          for (int c = 0; c < 8; ++c) {
            uint32_t v[32];
            const uint32_t col = kTmemO + 256 * ch + 32 * c;
            tmem_ld32(tmem + lane_addr + col, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tmem_st32(tmem + lane_addr + col, v);
          }
          tmem_wait_st();
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_at(&bars->corr[pb], lead, rank);
      }
      // Epilogue.
      const bool any = l_last > 0.f;
      const float inv = any ? p.out_scale / l_last : 0.f;
      const float lse = any ? (m_last + __log2f(l_last)) * 0.69314718055994531f : -INFINITY;
      const int64_t irow = kHalfRows * half + r;             // row within the item
      const int64_t row = it.q_row_base + it.row0 + irow;
      // Split partials are bf16 unless the call wants fp32 output: O of a split is
      // normalised by its own sum, so its bf16 rounding moves the merged O by at
      // most 2^-9 of the largest partial.
      const bool part_f32 = p.out_fp32 != 0;
      if (nt > 0) {
        const uint32_t last = pseq - 1;
        WAITC(&bars->o_ready[last % kPBufs], (last / kPBufs) & 1, 42);
        fence_after_sync();
      }
      // Split items write their partial (O / l and the LSE of their share of the
      // KV); the last split of a (request, row group, half) to finish then merges
      // every split's partial, in split order, into the output.
      const bool split = it.slot >= 0;
      {
        // O / l of this thread's row and 256 columns, 32 at a time, to the output
        // or to this split's partial
        const bool f32 = split ? part_f32 : p.out_fp32 != 0;
        const int esz = f32 ? 4 : 2;
        uint8_t* base = split ? reinterpret_cast<uint8_t*>(p.part_o) + (int64_t)it.slot * kRows * kDv * esz
                              : static_cast<uint8_t*>(p.o) + (it.q_row_base + it.row0) * kDv * esz;
        for (int c = 0; c < 8; ++c) {
          const int col = 256 * ch + 32 * c;
          float v[32];
          if (nt > 0) {
            uint32_t u[32];
            tmem_ld32(tmem + lane_addr + kTmemO + col, u);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(u[k]) * inv;
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = 0.f;
          }
          stage_and_write(v, f32, epi, lane, q4, col, base, (int64_t)kDv * esz, half, hrows);
        }
        if (live && ch == 0) {
          if (split) p.part_lse[(int64_t)it.slot * kRows + irow] = lse;
          else p.lse[row] = lse;
        }
      }
      if (nt > 0) {
        fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_at(&bars->o_free, lead, rank);
      }
      if (split && hrows > 0) {
        // The row warps meet on a CTA barrier; warp 0 then counts this split in
        // with an acquire-release add at GPU scope: the partial stores ordered
        // before the barrier are published with it, and the last split sees every
        // other split's.
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->mrg_c);
        if (warp == 0) {
          WAIT(&bars->mrg_c, mrg_c_ph, 45);
          if (lane == 0) {
            bars->merge_last = atom_add_acq_rel_gpu(&p.counters[2 * it.group + half], 1) == it.S - 1;
            mbar_arrive(&bars->mrg_b);
          }
          __syncwarp();
        }
        mrg_c_ph ^= 1;
        WAIT(&bars->mrg_b, mrg_b_ph, 44);
        mrg_b_ph ^= 1;
        if (bars->merge_last) {
          const int B = p.batch;
          const int G = p.plan[kPlanHeaderInts + B + it.b + 1] - p.plan[kPlanHeaderInts + B + it.b];
          const int pbase = p.plan[kPlanHeaderInts + 2 * B + 1 + it.b];
          // pass 1 (column half 0, thread = row): every split's weight for the row
          float* wts = reinterpret_cast<float*>(smem + kOffEpi0);   // [S][128], 8 KB
          if (ch == 0) {
            float M = -INFINITY;
            if (live)
              for (int s = 0; s < it.S; ++s)
                M = fmaxf(M, __ldcg(p.part_lse + (int64_t)(pbase + s * G + it.g) * kRows + irow));
            float tot = 0.f;
            for (int s = 0; s < it.S; ++s) {
              const float ls = M == -INFINITY ? -INFINITY
                                              : __ldcg(p.part_lse + (int64_t)(pbase + s * G + it.g) * kRows + irow);
              const float e = ls == -INFINITY ? 0.f : ex2((ls - M) * 1.4426950408889634f);
              wts[s * kHalfRows + r] = e;
              tot += e;
            }
            const float winv = M == -INFINITY ? 0.f : 1.f / tot;
            for (int s = 0; s < it.S; ++s) wts[s * kHalfRows + r] *= winv;
            if (live) p.lse[row] = M == -INFINITY ? -INFINITY : M + logf(tot);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->mrg_c);
          WAIT(&bars->mrg_c, mrg_c_ph, 46);
          mrg_c_ph ^= 1;
          // pass 2: thread t owns 16-byte column unit t % U of rows t / U + kRpp*k
          // (U units per row: 64 bf16, 128 fp32), four rows in flight per split
          const int U = part_f32 ? 128 : 64, kRpp = 256 / U;
          const int cu = tid % U, rp = tid / U;
          const int ocpu = part_f32 ? 4 : 8;                  // columns per unit
          for (int rb = rp; rb < hrows; rb += 4 * kRpp) {
            float acc[4][8];
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[k][e] = 0.f;
            for (int s = 0; s < it.S; ++s) {
              const int64_t slot = pbase + s * G + it.g;
              uint4 q[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int rl = min(rb + kRpp * k, hrows - 1);
                const int64_t off = (slot * kRows + kHalfRows * half + rl) * kDv * (part_f32 ? 4 : 2) + 16 * cu;
                q[k] = __ldcg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.part_o) + off));
              }
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float w = wts[s * kHalfRows + min(rb + kRpp * k, hrows - 1)];
                const uint32_t wd[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
                if (part_f32) {
#pragma unroll
                  for (int e = 0; e < 4; ++e) acc[k][e] += w * __uint_as_float(wd[e]);
                } else {
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    acc[k][2 * e] += w * bf16_bits_to_float(wd[e] & 0xFFFFu);
                    acc[k][2 * e + 1] += w * bf16_bits_to_float(wd[e] >> 16);
                  }
                }
              }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int rl = rb + kRpp * k;
              if (rl >= hrows) break;
              const int64_t orow = it.q_row_base + it.row0 + kHalfRows * half + rl;
              const int c0 = ocpu * cu;
              if (p.out_fp32) {
                float* dst = static_cast<float*>(p.o) + orow * kDv + c0;
                *reinterpret_cast<float4*>(dst) = make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
                if (ocpu == 8) *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[k][4], acc[k][5], acc[k][6], acc[k][7]);
              } else {
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.o) + orow * kDv + c0;
                if (ocpu == 8)
                  *reinterpret_cast<uint4*>(dst) =
                      make_uint4(pack_bf16x2(acc[k][0], acc[k][1]), pack_bf16x2(acc[k][2], acc[k][3]),
                                 pack_bf16x2(acc[k][4], acc[k][5]), pack_bf16x2(acc[k][6], acc[k][7]));
                else
                  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[k][0], acc[k][1]),
                                                              pack_bf16x2(acc[k][2], acc[k][3]));
              }
            }
          }
          if (tid == 0) p.counters[2 * it.group + half] = 0;   // ready for the next call
          // the weights live where the next epilogue stages its rows
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->mrg_c);
          WAIT(&bars->mrg_c, mrg_c_ph, 48);
          mrg_c_ph ^= 1;
        }
      }
    }
  }

done:
  // A CTA that gave up on a wait lets what was issued before the abort (its own
  // gathers and MMAs, the P copies it sent into a peer) land before the cluster
  // releases its memory: a fixed ~100 µs, far longer than any copy or MMA takes.
  // A completed call never takes this branch.
  if (*reinterpret_cast<volatile int*>(&bars->abort)) {
    const long long t0 = clock64();
    while (clock64() - t0 < kAbortDrainCycles) {
    }
  }
  fence_before_sync();
  __syncthreads();
  cluster_sync();        // the pairs' MMAs and every remote arrival are finished
  fence_after_sync();
  if (warp == kWarpMma) tmem_dealloc2(tmem, 512);
}

// ----------------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// Row-gather tensor map over the pool: one row high, `box` elements wide.
bool encode_pool_map(EncodeTiledFn enc, CUtensorMap* tm, const DecodeParams& dp, bool fp8, uint32_t box) {
  const cuuint64_t gdim[2] = {(cuuint64_t)kDqk, (cuuint64_t)dp.num_slots};
  const cuuint64_t gstride[1] = {(cuuint64_t)kDqk * (fp8 ? 1 : 2)};
  const cuuint32_t boxd[2] = {box, 1u};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(dp.kv), gdim, gstride, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-gather tensor map over q [rows, 576] bf16, one row high and 64 columns wide
// (128-byte swizzled).  The row extent is an upper bound of the call's query rows
// (batch x max_q_len x heads): the kernel asks only for rows of its own items.
bool encode_q_map(EncodeTiledFn enc, CUtensorMap* tm, const DecodeParams& dp) {
  const int64_t rows = (int64_t)dp.batch * dp.max_q_len * dp.num_heads;
  const cuuint64_t gdim[2] = {(cuuint64_t)kDqk, (cuuint64_t)(rows > 0 ? rows : 1)};
  const cuuint64_t gstride[1] = {(cuuint64_t)kDqk * 2};
  const cuuint32_t boxd[2] = {64u, 1u};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(dp.q), gdim, gstride, boxd, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of this kernel that fit on the device at once (cached per device).
template <bool kFp8>
int max_active_clusters(int dev) {
  static int cache[kMaxDevices] = {0};
  if (dev < 0) return 0;
  if (cache[dev] == 0) {
    const int smem = kSmemBytes + kSmemAlign;
    auto kern = mla_decode_tensor_kernel<kFp8>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 4;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

template <bool kFp8>
mla_status launch_impl(const DecodeParams& dp, void* stream) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MLA_ERR_CUDA;
  CUtensorMap tk, tv, tq;
  if (!encode_pool_map(enc, &tk, dp, kFp8, kFp8 ? 192u : 64u)) return MLA_ERR_INVALID_ARG;
  if (!encode_pool_map(enc, &tv, dp, kFp8, kFp8 ? 128u : 64u)) return MLA_ERR_INVALID_ARG;
  if (!encode_q_map(enc, &tq, dp)) return MLA_ERR_INVALID_ARG;
  int clusters = max_active_clusters<kFp8>(current_device_slot());
  if (clusters < 1) return MLA_ERR_CUDA;
  if (clusters > dp.items_cap) clusters = dp.items_cap > 0 ? dp.items_cap : 1;
  DecodeParams kp = dp;
  if (kFp8) {
    // The in-register fp8 -> bf16 conversion scales every value by 2^-112.
    kp.scale_log2 = dp.scale_log2 * 5.192296858534828e33f;
    kp.out_scale = dp.out_scale * 5.192296858534828e33f;
  }
  return launch_overlapped(mla_decode_tensor_kernel<kFp8>, dim3(4 * clusters), dim3(kThreads),
                           kSmemBytes + kSmemAlign, (cudaStream_t)stream, tk, tv, tq, kp) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // namespace

int tensor_kernel_available() { return 1; }

int tensor_kernel_workers() {
  const int dev = current_device_slot();
  const int a = max_active_clusters<false>(dev), b = max_active_clusters<true>(dev);
  return a < b ? a : b;
}

mla_status launch_decode_tensor(const DecodeParams& dp, void* stream) {
  return dp.kv_fp8 ? launch_impl<true>(dp, stream) : launch_impl<false>(dp, stream);
}

}  // namespace mla
