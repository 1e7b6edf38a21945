// Tensor-core MLA decode kernel for sm_103a (tcgen05 + TMEM + TMA gathers).
//
// All H*T query rows of a request share one stream of latent KV rows, so QK^T
// over 576 columns and PV over 512 are dense contractions with M = 128 query
// rows.  The fp32 accumulator of O[128, 512] alone fills the 512 TMEM columns of
// an SM, so each work item runs on a cluster of two CTAs with different jobs:
//
//   rank 0, the score CTA: holds the item's Q[128, 576] in TMEM as the MMA's A
//     operand, gathers K tiles [64 entries, 576] with TMA, computes
//     S = Q K^T into a double-buffered TMEM tile, runs the masked online
//     softmax (one thread per query row) and ships P (bf16) plus the per-row
//     rescale factors and running max/sum into the peer's shared memory with a
//     bulk copy.
//   rank 1, the output CTA: gathers V tiles [64 entries, 512], accumulates
//     O += P V in TMEM, rescales O when the score CTA raised its reference max,
//     and writes O / l and the log-sum-exp (or the split partial and the fused
//     split merge).
//
// The KV tile in shared memory is stored as 64-column chunks in the 128-byte
// swizzled layout, so the same bytes serve as the K-major B operand of QK^T and
// as the MN-major B operand of PV.  fp8 e4m3 pools are gathered as bytes and
// converted to bf16 in registers by dedicated warps (exact: e4m3 -> f16 by the
// hardware conversion, then the f16 bits are placed in a bf16 word, which
// scales every value by 2^-112; the factor is folded into the logit and output
// scales).
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

// 12 warps for bf16 pools (seven of them gather), 10 for fp8 (warps 10-11 would
// only slow the conversion warps down).
constexpr int threads_for(bool fp8) { return fp8 ? 320 : 384; }
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpRow0 = 2;           // 4 row warps: softmax (rank 0) / correction+epilogue (rank 1)
constexpr int kWarpConv0 = 6;          // 4 fp8 conversion warps (bf16: KV gathers)
constexpr int kStages = 2;             // KV tile ring
constexpr int kPBufs = 2;              // P hand-off ring

constexpr int kChunkBytes = kBlockN * 128;          // 64 entries x 64 bf16 columns = 8 KB
constexpr int kKTileBytes = 9 * kChunkBytes;        // 576 columns (score CTA)
// fp8: the tile's raw e4m3 rows are gathered into the upper half of the stage
// (three 192-byte column blocks of [64 rows][192 B]) and converted in place.
constexpr int kF8Off = kKTileBytes / 2;             // 36 KB
constexpr int kF8BlockBytes = kBlockN * 192;        // 12 KB
constexpr int kPBytes = kRows * 128;                // P: 128 rows x 64 bf16
constexpr int kPStatsOff = kPBytes;                 // alpha[128], m[128], l[128], flags[4]
constexpr int kPBufBytes = kPBytes + 3 * 512 + 512; // 18 KB, multiple of 16

// Shared-memory map (identical offsets in both CTAs; barriers first).
constexpr int kOffBars = 0;
constexpr int kOffData = 2048;
constexpr int kOffTiles = kOffData;                                   // kStages x 72 KB
constexpr int kOffPBuf = kOffTiles + kStages * kKTileBytes;           // kPBufs x 18 KB
constexpr int kOffEpi = kOffPBuf + kPBufs * kPBufBytes;              // output CTA: 4 x 4 KB epilogue staging
constexpr int kSmemBytes = kOffEpi + 4 * 4096;
constexpr int kSmemAlign = 1024;

// TMEM columns.
constexpr uint32_t kTmemQ = 0;       // score CTA: Q as A operand, 288 columns
constexpr uint32_t kTmemS = 288;     // score CTA: two 64-column S buffers
constexpr uint32_t kTmemO = 0;       // output CTA: O, 512 columns

struct Bars {
  uint64_t full[kStages];     // KV tile landed (TMA or fp8 conversion)
  uint64_t empty[kStages];    // KV tile consumed by this CTA's MMA
  uint64_t full8[kStages];    // fp8: raw e4m3 rows of the tile landed (TMA)
  uint64_t cv_sync;           // fp8: the conversion warps finished reading the raw rows
  uint64_t s_full[2];         // score CTA: S tile computed
  uint64_t s_free[2];         // score CTA: S tile read out
  uint64_t q_full;            // score CTA: Q written to TMEM
  uint64_t q_free;            // score CTA: all QK of the item done
  uint64_t p_empty[kPBufs];   // score CTA: peer finished PV with P buffer
  uint64_t p_ready[kPBufs];   // score CTA: the four softmax warps staged P
  uint64_t p_full[kPBufs];    // output CTA: P buffer arrived
  uint64_t corr_done[kPBufs]; // output CTA: O ready for PV on this P buffer
  uint64_t o_ready[kPBufs];   // output CTA: PV with this P buffer complete
  uint64_t o_free;            // output CTA: epilogue read O
  uint64_t mrg_a;             // output CTA: the 4 row warps fenced their partial rows
  uint64_t mrg_b;             // output CTA: leader published the last-arriver verdict
  uint64_t mrg_c;             // output CTA: per-row merge weights ready
  uint64_t mrg_d;             // output CTA: the 4 row warps are done with the weights
  uint32_t tmem_base;
  int abort;
  int merge_last;
};
static_assert(sizeof(Bars) <= kOffData, "barrier block too large");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 128-byte swizzle: byte offset of 16-byte unit u of row r inside a chunk.
__device__ __forceinline__ uint32_t swz(int r, int u) { return (uint32_t)(r * 128 + ((u ^ (r & 7)) << 4)); }

// On a failed wait: record, raise the abort flag here and in the peer.
__device__ __noinline__ void fail(Bars* bars, const DecodeParams& p, int site) {
  record_error(p.ws_hdr, MLA_DEV_WAIT_TIMEOUT, site);
  bars->abort = 1;
  const uint32_t peer = cluster_rank() ^ 1u;
  const uint32_t a = mapa(smem_u32(&bars->abort), peer);
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(1) : "memory");
}

// Warp-collective bounded waits: every lane polls, and the warp leaves together
// (to the teardown) if any lane gave up.
#define WAIT(bar, par, site)                                                         \
  if (!__all_sync(0xffffffffu, mbar_wait(bar, par, &bars->abort))) {               \
    fail(bars, p, site);                                                             \
    goto done;                                                                       \
  }
#define WAITC(bar, par, site)                                                        \
  if (!__all_sync(0xffffffffu, mbar_wait<true>(bar, par, &bars->abort))) {         \
    fail(bars, p, site);                                                             \
    goto done;                                                                       \
  }

// Static work assignment, identical in every role of both CTAs of a cluster:
// round r gives cluster c item r*C + c on even rounds and r*C + (C-1-c) on odd
// rounds, so a cost-sorted item list is dealt out boustrophedon-fashion.
__device__ __forceinline__ int item_of(int r, int c, int C) { return r * C + ((r & 1) ? C - 1 - c : c); }
#define FOR_ITEMS(idx)                                                      \
  for (int r_ = 0, idx = item_of(0, cluster, n_clusters); idx < n_items; \
       ++r_, idx = item_of(r_, cluster, n_clusters))

// Number of 64-entry tiles of an item.
__device__ __forceinline__ int item_tiles(const Item& it) {
  return it.ok && it.e1 > it.e0 ? (it.e1 - it.e0 + kBlockN - 1) / kBlockN : 0;
}

// 16 e4m3 values (unit u of 64-column chunk c of tile row `row`) -> two 16-byte
// bf16 units of the swizzled tile.  Exact: the f16 bits from the hardware e4m3
// conversion are placed in a bf16 word with the same exponent field, which
// scales every value by 2^-112 (folded into the logit and output scales).
__device__ __forceinline__ void fp8_unit_to_tile(uint8_t* stage, int row, int c, int u, const uint4& v) {
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
  uint8_t* base = stage + c * kChunkBytes;
  *reinterpret_cast<uint4*>(base + swz(row, 2 * u)) = make_uint4(o[0], o[1], o[2], o[3]);
  *reinterpret_cast<uint4*>(base + swz(row, 2 * u + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
}

// Epilogue write-back of one 32-column block of a warp's 32 rows, staged at stg
// (128-byte row pitch, 16-byte unit k of row r at unit k ^ (r & 7)): each store
// instruction writes whole row segments, 128 bytes (fp32) or 64 bytes (bf16).
template <bool kF32>
__device__ __forceinline__ void epi_rows_out(const uint8_t* stg, int lane, int q4, int c, const Item& it,
                                             const DecodeParams& p) {
  constexpr int kUsh = kF32 ? 3 : 2;          // log2 of 16-byte units per row segment
  constexpr int kN = 1 << kUsh;
  uint4 val[kN];
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    const int rl = (i << (5 - kUsh)) + (lane >> kUsh), u = lane & (kN - 1);
    val[i] = *reinterpret_cast<const uint4*>(stg + rl * 128 + ((u ^ (rl & 7)) << 4));
  }
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    const int rl = (i << (5 - kUsh)) + (lane >> kUsh), u = lane & (kN - 1);
    const int ri = 32 * q4 + rl;               // row within the item
    if (ri < it.nrows) {
      void* dst;
      if (!kF32) dst = static_cast<__nv_bfloat16*>(p.o) + (it.q_row_base + it.row0 + ri) * kDv + 32 * c + 8 * u;
      else if (it.slot >= 0) dst = p.part_o + ((int64_t)it.slot * kRows + ri) * kDv + 32 * c + 4 * u;
      else dst = static_cast<float*>(p.o) + (it.q_row_base + it.row0 + ri) * kDv + 32 * c + 4 * u;
      *reinterpret_cast<uint4*>(dst) = val[i];
    }
  }
}

template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(threads_for(kFp8), 1)
mla_decode_tensor_kernel(const __grid_constant__ CUtensorMap tmap_kv, const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((kSmemAlign - (smem_u32(smem_raw) & (kSmemAlign - 1))) & (kSmemAlign - 1));
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBars);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const bool score_cta = rank == 0;

  if (!plan_header_ok(p.plan, p)) {
    if (blockIdx.x == 0 && tid == 0) record_error(p.ws_hdr, MLA_DEV_PLAN_MISMATCH, 0);
    return;   // both CTAs of every cluster leave before touching each other
  }
  const int n_items = p.plan[kHNItems];
  const int cluster = (int)cluster_id_x(), n_clusters = (int)num_clusters_x();

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], kFp8 ? 4 : 1);
      mbar_init(&bars->empty[s], 1);
      mbar_init(&bars->full8[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], 4);
    }
    mbar_init(&bars->q_full, 4);
    mbar_init(&bars->q_free, 1);
    for (int b = 0; b < kPBufs; ++b) {
      mbar_init(&bars->p_empty[b], 1);
      mbar_init(&bars->p_ready[b], 4);
      mbar_init(&bars->p_full[b], 1);
      mbar_init(&bars->corr_done[b], 4);
      mbar_init(&bars->o_ready[b], 1);
    }
    mbar_init(&bars->o_free, 4);
    mbar_init(&bars->cv_sync, 4);
    mbar_init(&bars->mrg_a, 4);
    mbar_init(&bars->mrg_b, 1);
    mbar_init(&bars->mrg_c, 4);
    mbar_init(&bars->mrg_d, 4);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == kWarpProducer && lane == 0) prefetch_tmap(&tmap_kv);
  fence_before_sync();
  __syncthreads();
  cluster_sync();        // barriers of both CTAs initialised before any remote arrival
  fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  uint8_t* tiles = smem + kOffTiles;
  uint8_t* pbufs = smem + kOffPBuf;

  // ======================================================================= producer
  // KV gathers with TMA.  One gather op moves 4 rows (entries 4g..4g+3, row
  // group g) x one column block; a tile needs 16 groups x nblk blocks.  Issue
  // cost is mostly per warp instruction, so each lane owns one op and a warp
  // issues its share of the tile in one instruction (two for fp8).
  //   bf16: each CTA gathers the 64-column chunks it reads into its own ring
  //   (score CTA: all 9, output CTA: the 8 latent chunks), so the score CTA
  //   refills a stage as soon as its QK^T is done with it; warps 0 and 6-11 share
  //   the 144 (128) ops.
  //   fp8: the raw e4m3 rows, three 192-byte column blocks per row, land in the
  //   stage's upper half for the conversion warps; warp 0 issues the 48 ops
  //   alone (more issuing warps slowed the conversion warps beside them).
  if (warp == kWarpProducer || (!kFp8 && warp >= kWarpConv0)) {
    constexpr int npw = kFp8 ? 1 : 7;
    constexpr int kOpsPerLane = kFp8 ? 2 : 1;
    const int pw = warp == kWarpProducer ? 0 : warp - kWarpConv0 + 1;
    const int nblk = kFp8 ? 3 : (score_cta ? 9 : 8);
    const int nops = 16 * nblk;
    const int per = (nops + npw - 1) / npw;             // ops of this warp: [o_begin, o_end)
    const int o_begin = pw * per, o_end = o_begin + per < nops ? o_begin + per : nops;
    const uint32_t tx = (uint32_t)(16 * nblk * (kFp8 ? 4 * 192 : 512));
    uint32_t kseq = 0;
    const bool report = score_cta && pw == 0;
    // Raw slot indices of tile j (lane holds entries lane and lane+32), -1 past the
    // end; checked only when used, one iteration later, so the load is not waited on.
    auto tile_idx = [&](const Item& it, int j, int32_t& x0, int32_t& x1) {
      const int i0 = it.e0 + j * kBlockN + lane, i1 = i0 + 32;
      x0 = i0 < it.e1 ? __ldg(p.kv_indices + it.kv_off + i0) : -1;
      x1 = i1 < it.e1 ? __ldg(p.kv_indices + it.kv_off + i1) : -1;
    };
    // Invalid entries read row -1 (zero fill) and are reported once.
    auto checked = [&](const Item& it, int j, int half, int32_t v) -> int32_t {
      if (v >= 0 && v < p.num_slots) return v;
      const int i = it.e0 + j * kBlockN + lane + 32 * half;
      if (report && i < it.e1) record_error(p.ws_hdr, MLA_DEV_BAD_INDEX, (int)(it.kv_off + i));
      return -1;
    };
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      const int nt = item_tiles(it);
      int32_t n0 = -1, n1 = -1;
      if (nt > 0) tile_idx(it, 0, n0, n1);
      for (int j = 0; j < nt; ++j, ++kseq) {
        const int st = kseq % kStages;
        const uint32_t ph = (kseq / kStages) & 1;
        // this tile's indices were loaded one iteration ago; start the next tile's now
        const int32_t r0 = checked(it, j, 0, n0), r1 = checked(it, j, 1, n1);
        if (j + 1 < nt) tile_idx(it, j + 1, n0, n1);
        // slot indices of the group of each of this lane's ops, from lanes
        // (4g..4g+3) % 32 of r0 (g < 8) or r1 (g >= 8), before the wait
        int32_t a[kOpsPerLane][4];
#pragma unroll
        for (int q = 0; q < kOpsPerLane; ++q) {
          const int g = ((o_begin + 32 * q + lane) / nblk) & 15;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int32_t x0 = __shfl_sync(0xffffffffu, r0, ((4 * g) & 31) + e);
            const int32_t x1 = __shfl_sync(0xffffffffu, r1, ((4 * g) & 31) + e);
            a[q][e] = g < 8 ? x0 : x1;
          }
        }
        WAIT(&bars->empty[st], ph ^ 1, 1);
        uint64_t* bar = kFp8 ? &bars->full8[st] : &bars->full[st];
        if (pw == 0 && lane == 0) mbar_arrive_expect_tx(bar, tx);
        __syncwarp();
        const uint32_t base = smem_u32(tiles + st * kKTileBytes);
#pragma unroll
        for (int q = 0; q < kOpsPerLane; ++q) {
          const int o = o_begin + 32 * q + lane;
          if (o < o_end) {
            const int g = o / nblk, c = o - g * nblk;
            if (kFp8)
              tma_gather4(base + (uint32_t)(kF8Off + c * kF8BlockBytes + g * 4 * 192), &tmap_kv, 192 * c, a[q][0],
                          a[q][1], a[q][2], a[q][3], bar);
            else
              tma_gather4(base + (uint32_t)(c * kChunkBytes + g * 512), &tmap_kv, c * 64, a[q][0], a[q][1], a[q][2],
                          a[q][3], bar);
          }
        }
        __syncwarp();
      }
    }
  }
  // ======================================================================= fp8: convert in place
  // The four conversion warps turn the tile's raw e4m3 rows (gathered by warp 0
  // into the stage's upper half) into the swizzled bf16 tile.  Warp cw owns rows
  // 16cw .. 16cw+15.  Chunks 0-3 are written first (below the raw rows); the raw
  // bytes of chunks 4.. are read into registers, and once all four warps hold
  // theirs the remaining chunks overwrite the raw area.
  else if (kFp8 && warp >= kWarpConv0) {
    const int cw = warp - kWarpConv0;
    uint32_t kseq = 0, cv_ph = 0;
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      const int nt = item_tiles(it);
      for (int j = 0; j < nt; ++j, ++kseq) {
        const int st = kseq % kStages;
        WAIT(&bars->full8[st], (kseq / kStages) & 1, 4);
        uint8_t* stage = tiles + st * kKTileBytes;
        const uint8_t* raw = stage + kF8Off;
        // chunks 0-3: 16 rows x 4 chunks x 4 units of 16 fp8 values, 8 per lane
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int f = k * 32 + lane, row = 16 * cw + (f >> 4), c = (f >> 2) & 3, u = f & 3;
          const uint4 v = *reinterpret_cast<const uint4*>(raw + (c / 3) * kF8BlockBytes + row * 192 + (c % 3) * 64 + u * 16);
          fp8_unit_to_tile(stage, row, c, u, v);
        }
        // chunks 4.. (score: 4-8, output: 4-7) into registers
        uint4 rb[10];
        const int nb = score_cta ? 5 : 4;
#pragma unroll
        for (int k = 0; k < 10; ++k) {
          if (k < 2 * nb) {
            const int f = k * 32 + lane, row = 16 * cw + f / (4 * nb), c = 4 + (f % (4 * nb)) / 4, u = f & 3;
            rb[k] = *reinterpret_cast<const uint4*>(raw + (c / 3) * kF8BlockBytes + row * 192 + (c % 3) * 64 + u * 16);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->cv_sync);
        WAIT(&bars->cv_sync, cv_ph, 5);
        cv_ph ^= 1;
#pragma unroll
        for (int k = 0; k < 10; ++k) {
          if (k < 2 * nb) {
            const int f = k * 32 + lane, row = 16 * cw + f / (4 * nb), c = 4 + (f % (4 * nb)) / 4, u = f & 3;
            fp8_unit_to_tile(stage, row, c, u, rb[k]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->full[st]);
      }
    }
  }
  // ======================================================================= score CTA: MMA
  else if (score_cta && warp == kWarpMma) {
    uint32_t kseq = 0, sseq = 0, qitem = 0;
    const uint32_t idesc = idesc_bf16_f32(128, kBlockN, false, false);
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      const int nt = item_tiles(it);
      if (nt == 0) continue;
      WAIT(&bars->q_full, qitem & 1, 10);
      fence_after_sync();
      for (int j = 0; j < nt; ++j, ++kseq, ++sseq) {
        const int st = kseq % kStages, sb = sseq & 1;
        WAIT(&bars->s_free[sb], ((sseq >> 1) & 1) ^ 1, 11);
        const uint32_t kph = (kseq / kStages) & 1;
        // B descriptor of K step k: chunk k/4, 32-byte column offset k%4 (start address field is addr>>4)
        const uint64_t bdesc0 = smem_desc_sw128(smem_u32(tiles + st * kKTileBytes), 16, 1024);
        const uint32_t dS = tmem + kTmemS + sb * kBlockN;
        WAITC(&bars->full[st], kph, 12);
        fence_after_sync();
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < kDqk / 16; ++k)
            mma_ts(dS, tmem + kTmemQ + 8 * k, bdesc0 + (uint64_t)(((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4),
                   idesc, k > 0);
          mma_commit(&bars->empty[st]);
          mma_commit(&bars->s_full[sb]);
        }
        __syncwarp();
      }
      if (lane == 0) mma_commit(&bars->q_free);
      __syncwarp();
      ++qitem;
    }
  }
  // ======================================================================= output CTA: MMA
  else if (!score_cta && warp == kWarpMma) {
    uint32_t kseq = 0, pseq = 0, oitem = 0;
    const uint32_t idesc = idesc_bf16_f32(128, 256, false, true);
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      const int nt = item_tiles(it);
      if (nt == 0) continue;
      WAIT(&bars->o_free, (oitem & 1) ^ 1, 20);
      for (int j = 0; j < nt; ++j, ++kseq, ++pseq) {
        const int st = kseq % kStages, pb = pseq % kPBufs;
        const uint32_t pph = (pseq / kPBufs) & 1;
        WAITC(&bars->full[st], (kseq / kStages) & 1, 21);
        if (lane == 0) mbar_arrive_expect_tx(&bars->p_full[pb], kPBufBytes);
        __syncwarp();
        WAITC(&bars->p_full[pb], pph, 22);
        WAIT(&bars->corr_done[pb], pph, 23);
        fence_after_sync();
        if (lane == 0) {
          const uint64_t adesc0 = smem_desc_sw128(smem_u32(pbufs + pb * kPBufBytes), 16, 1024);
          const uint64_t bdesc0 = smem_desc_sw128(smem_u32(tiles + st * kKTileBytes), kChunkBytes, 1024);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int k = 0; k < kBlockN / 16; ++k)
              mma_ss(tmem + kTmemO + 256 * h, adesc0 + (uint64_t)((k * 32) >> 4),
                     bdesc0 + (uint64_t)(((4 * h) * kChunkBytes + k * 2048) >> 4), idesc,
                     (j > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&bars->empty[st]);
          mma_commit_mc(&bars->p_empty[pb], 0x1);
          mma_commit(&bars->o_ready[pb]);
        }
        __syncwarp();
      }
      ++oitem;
    }
  }
  // ======================================================================= score CTA: softmax
  else if (score_cta) {
    const int q4 = warp & 3;                 // TMEM lane quadrant of this warp
    const int r = 32 * q4 + lane;            // query row within the group
    const uint32_t lane_addr = (uint32_t)(32 * q4) << 16;
    uint32_t sseq = 0, pseq = 0, qitem = 0;
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      const int nt = item_tiles(it);
      if (nt == 0) continue;
      const bool live = r < it.nrows;
      // Q rows of the item -> TMEM (A operand layout: lane = row, two bf16 per column).
      WAIT(&bars->q_free, (qitem & 1) ^ 1, 30);
      fence_after_sync();
      {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                          (it.q_row_base + it.row0 + (live ? r : 0)) * kDqk);
        // 72 loads of 16 bytes per row: issue 24 at a time (three TMEM chunks) to
        // overlap the global-memory latency.
        for (int c0 = 0; c0 < 9; c0 += 3) {
          uint4 u[24];
#pragma unroll
          for (int k = 0; k < 24; ++k) u[k] = live ? __ldg(src + c0 * 8 + k) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int cc = 0; cc < 3; ++cc) {
            uint32_t v[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              v[4 * k] = u[8 * cc + k].x;
              v[4 * k + 1] = u[8 * cc + k].y;
              v[4 * k + 2] = u[8 * cc + k].z;
              v[4 * k + 3] = u[8 * cc + k].w;
            }
            tmem_st32(tmem + lane_addr + kTmemQ + 32 * (c0 + cc), v);
          }
        }
        tmem_wait_st();
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->q_full);
      ++qitem;

      // Visibility: local entry i is visible to this row iff ibeg <= i < iend, its
      // index is valid and, with per-entry positions, its position passes the
      // row's causal limit (and window).
      const int t_row = (it.row0 + r) / p.num_heads;
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
      const int t_first = (it.row0 + 32 * q4) / p.num_heads, t_last = (it.row0 + 32 * q4 + 31) / p.num_heads;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j, ++sseq, ++pseq) {
        const int sb = sseq & 1, pb = pseq % kPBufs;
        const int i0 = it.e0 + j * kBlockN;
        // validity of the tile's 64 slot indices
        uint32_t vlo, vhi;
        {
          const int a = i0 + lane, b = a + 32;
          bool ok0 = false, ok1 = false;
          if (a < it.e1) {
            const int32_t s = __ldg(p.kv_indices + it.kv_off + a);
            ok0 = s >= 0 && s < p.num_slots;
          }
          if (b < it.e1) {
            const int32_t s = __ldg(p.kv_indices + it.kv_off + b);
            ok1 = s >= 0 && s < p.num_slots;
          }
          if (p.kv_pos && p.causal) {
            const int64_t g0 = a < it.e1 ? (int64_t)__ldg(p.kv_pos + it.kv_off + a) : INT64_MAX;
            const int64_t g1 = b < it.e1 ? (int64_t)__ldg(p.kv_pos + it.kv_off + b) : INT64_MAX;
            vlo = vhi = 0;
            for (int t = t_first; t <= t_last; ++t) {
              const int64_t lim = it.Lg - it.T + t;
              const bool in0 = g0 <= lim && (p.window <= 0 || g0 > lim - p.window);
              const bool in1 = g1 <= lim && (p.window <= 0 || g1 > lim - p.window);
              const uint32_t m0 = __ballot_sync(0xffffffffu, ok0 && in0);
              const uint32_t m1 = __ballot_sync(0xffffffffu, ok1 && in1);
              if (t == t_row) {
                vlo = m0;
                vhi = m1;
              }
            }
          } else {
            vlo = __ballot_sync(0xffffffffu, ok0);
            vhi = __ballot_sync(0xffffffffu, ok1);
          }
        }
        WAIT(&bars->s_full[sb], (sseq >> 1) & 1, 31);
        fence_after_sync();
        uint32_t s0[32], s1[32];
        tmem_ld32(tmem + lane_addr + kTmemS + sb * kBlockN, s0);
        tmem_ld32(tmem + lane_addr + kTmemS + sb * kBlockN + 32, s1);
        tmem_wait_ld();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[sb]);

        // entries [nbeg, nvis) of the tile may be visible: fold the range into the masks
        {
          const int nvis = iend - i0, nbeg = ibeg - i0;
          const int hi = nvis < 0 ? 0 : (nvis > 64 ? 64 : nvis), lo = nbeg < 0 ? 0 : (nbeg > 64 ? 64 : nbeg);
          const uint64_t range = (hi >= 64 ? ~0ull : ((1ull << hi) - 1)) & (lo >= 64 ? 0ull : (~0ull << lo));
          vlo &= (uint32_t)range;
          vhi &= (uint32_t)(range >> 32);
        }
        float x[64];
        float tmax = -INFINITY;
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const uint32_t bits = e < 32 ? s0[e] : s1[e - 32];
          const bool vis = ((e < 32 ? vlo : vhi) >> (e & 31)) & 1u;
          x[e] = vis ? __uint_as_float(bits) * p.scale_log2 : -INFINITY;
          tmax = fmaxf(tmax, x[e]);
        }
        float alpha = 1.f;
        int need = 0;
        if (tmax > m_ref + 8.f) {          // raise the reference max only when it grew a lot
          alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - tmax);
          m_ref = tmax;
          need = 1;
        }
        float psum = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const float a = m_ref == -INFINITY ? 0.f : ex2(x[e] - m_ref);
          const float b = m_ref == -INFINITY ? 0.f : ex2(x[e + 1] - m_ref);
          psum += a + b;
          pk[e / 2] = pack_bf16x2(a, b);
        }
        l = l * alpha + psum;
        const int any_need = __any_sync(0xffffffffu, need);

        // Hand P to the output CTA.
        WAITC(&bars->p_empty[pb], ((pseq / kPBufs) & 1) ^ 1, 32);
        uint8_t* stg = pbufs + pb * kPBufBytes;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(stg + swz(r, u)) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        float* stats = reinterpret_cast<float*>(stg + kPStatsOff);
        stats[r] = alpha;
        stats[128 + r] = m_ref;
        stats[256 + r] = l;
        if (lane == 0) reinterpret_cast<int*>(stats + 384)[q4] = any_need;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_ready[pb]);
        if (warp == kWarpRow0) {
          WAIT(&bars->p_ready[pb], (pseq / kPBufs) & 1, 34);
          if (lane == 0) {
            const uint32_t src = smem_u32(stg);
            bulk_copy_to_peer(mapa(src, 1), src, kPBufBytes, mapa(smem_u32(&bars->p_full[pb]), 1));
          }
          __syncwarp();
        }
      }
    }
    // Drain: the peer's last PV arrivals on p_empty must land before this CTA exits.
    for (int k = 0; k < kPBufs && (int)pseq - 1 - k >= 0; ++k) {
      const uint32_t s = pseq - 1 - k;
      WAITC(&bars->p_empty[s % kPBufs], (s / kPBufs) & 1, 33);
    }
  }
  // ======================================================================= output CTA: correction + epilogue
  else {
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_addr = (uint32_t)(32 * q4) << 16;
    uint32_t pseq = 0, mrg_a_ph = 0, mrg_b_ph = 0, mrg_c_ph = 0, mrg_d_ph = 0;
    FOR_ITEMS(idx) {
      const Item it = load_item(p, idx);
      if (!it.ok) continue;
      const int nt = item_tiles(it);
      const bool live = r < it.nrows;
      float m_last = -INFINITY, l_last = 0.f;
      for (int j = 0; j < nt; ++j, ++pseq) {
        const int pb = pseq % kPBufs;
        const uint32_t pph = (pseq / kPBufs) & 1;
        WAITC(&bars->p_full[pb], pph, 40);
        const uint8_t* pbuf = pbufs + pb * kPBufBytes;
        const float* stats = reinterpret_cast<const float*>(pbuf + kPStatsOff);
        const int* flags = reinterpret_cast<const int*>(stats + 384);
        const float alpha = stats[r];
        m_last = stats[128 + r];
        l_last = stats[256 + r];
        if (flags[q4] && j > 0) {
          // O of the previous tile must be complete before rescaling it.
          const uint32_t prev = pseq - 1;
          WAIT(&bars->o_ready[prev % kPBufs], (prev / kPBufs) & 1, 41);
          fence_after_sync();
          for (int c = 0; c < kDv / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_addr + kTmemO + 32 * c, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tmem_st32(tmem + lane_addr + kTmemO + 32 * c, v);
          }
          tmem_wait_st();
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->corr_done[pb]);
      }
      // Epilogue.
      const bool any = l_last > 0.f;
      const float inv = any ? p.out_scale / l_last : 0.f;
      const float lse = any ? (m_last + __log2f(l_last)) * 0.69314718055994531f : -INFINITY;
      float* dst_f32 = nullptr;
      const int64_t row = it.q_row_base + it.row0 + r;
      if (it.slot >= 0) dst_f32 = p.part_o + ((int64_t)it.slot * kRows + r) * kDv;
      else if (p.out_fp32) dst_f32 = static_cast<float*>(p.o) + row * kDv;
      if (nt > 0) {
        const uint32_t last = pseq - 1;
        WAIT(&bars->o_ready[last % kPBufs], (last / kPBufs) & 1, 42);
        fence_after_sync();
      }
      // O[row = lane][32 columns] per step: staged in this warp's 4 KB (128-byte
      // row pitch, 16-byte units XOR-swizzled by row) and written back as whole
      // row segments, 128 (fp32) or 64 (bf16) contiguous bytes per row.
      uint8_t* stg = smem + kOffEpi + (warp - kWarpRow0) * 4096;
      const bool f32 = dst_f32 != nullptr;
      for (int c = 0; c < kDv / 32; ++c) {
        float v[32];
        if (nt > 0) {
          uint32_t u[32];
          tmem_ld32(tmem + lane_addr + kTmemO + 32 * c, u);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(u[k]) * inv;
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = 0.f;
        }
        if (f32) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                make_uint4(pack_bf16x2(v[8 * k], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                           pack_bf16x2(v[8 * k + 4], v[8 * k + 5]), pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
        }
        __syncwarp();
        if (f32) epi_rows_out<true>(stg, lane, q4, c, it, p);
        else epi_rows_out<false>(stg, lane, q4, c, it, p);
        __syncwarp();
      }
      if (live) {
        if (it.slot >= 0) p.part_lse[(int64_t)it.slot * kRows + r] = lse;
        else p.lse[row] = lse;
      }
      if (nt > 0) {
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->o_free);
      }
      if (it.slot >= 0) {
        // Fused split merge: the last split of this (request, row group) to finish
        // combines every split's partial in split order.  The 4 row warps first
        // agree (leader counts one arrival per split), then merge together.
        __threadfence();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->mrg_a);
        if (warp == kWarpRow0) {
          WAIT(&bars->mrg_a, mrg_a_ph, 43);
          if (lane == 0) {
            bars->merge_last = atomicAdd(&p.counters[it.group], 1) == it.S - 1;
            mbar_arrive(&bars->mrg_b);
          }
          __syncwarp();
        }
        mrg_a_ph ^= 1;
        WAIT(&bars->mrg_b, mrg_b_ph, 44);
        mrg_b_ph ^= 1;
        if (bars->merge_last) {
          __threadfence();
          const int B = p.batch;
          const int G = p.plan[kPlanHeaderInts + B + it.b + 1] - p.plan[kPlanHeaderInts + B + it.b];
          const int pbase = p.plan[kPlanHeaderInts + 2 * B + 1 + it.b];
          // pass 1 (thread = row): max, normaliser and the weight of every split,
          // kept in the epilogue staging area as w[s][row]
          float* wts = reinterpret_cast<float*>(smem + kOffEpi);
          {
            float M = -INFINITY;
            if (live)
              for (int s = 0; s < it.S; ++s)
                M = fmaxf(M, __ldcg(p.part_lse + (int64_t)(pbase + s * G + it.g) * kRows + r));
            float tot = 0.f;
            if (M != -INFINITY)
              for (int s = 0; s < it.S; ++s) {
                const float ls = __ldcg(p.part_lse + (int64_t)(pbase + s * G + it.g) * kRows + r);
                const float e = ls == -INFINITY ? 0.f : ex2((ls - M) * 1.4426950408889634f);
                wts[s * kRows + r] = e;
                tot += e;
              }
            const float inv = M == -INFINITY ? 0.f : 1.f / tot;
            for (int s = 0; s < it.S; ++s) wts[s * kRows + r] = M == -INFINITY ? 0.f : wts[s * kRows + r] * inv;
            if (live) p.lse[row] = M == -INFINITY ? -INFINITY : M + logf(tot);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->mrg_c);
          WAIT(&bars->mrg_c, mrg_c_ph, 45);
          mrg_c_ph ^= 1;
          // pass 2: thread t owns float4 column t of every row; 16 rows in flight
          const int c4 = tid - kWarpRow0 * 32;
          for (int rb = 0; rb < it.nrows; rb += 16) {
            float4 acc[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s = 0; s < it.S; ++s) {
              const int slot = pbase + s * G + it.g;
              float4 ov[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                const int rr = min(rb + k, it.nrows - 1);
                ov[k] = __ldcg(reinterpret_cast<const float4*>(p.part_o + ((int64_t)slot * kRows + rr) * kDv) + c4);
              }
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                const float w = wts[s * kRows + min(rb + k, it.nrows - 1)];
                acc[k].x += w * ov[k].x;
                acc[k].y += w * ov[k].y;
                acc[k].z += w * ov[k].z;
                acc[k].w += w * ov[k].w;
              }
            }
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              if (rb + k >= it.nrows) break;
              const int64_t orow = it.q_row_base + it.row0 + rb + k;
              if (p.out_fp32) {
                reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow * kDv)[c4] = acc[k];
              } else {
                uint2 u;
                u.x = pack_bf16x2(acc[k].x, acc[k].y);
                u.y = pack_bf16x2(acc[k].z, acc[k].w);
                reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.o) + orow * kDv)[c4] = u;
              }
            }
          }
          if (tid == kWarpRow0 * 32) p.counters[it.group] = 0;
          // the weights live where the next epilogue stages its rows
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->mrg_d);
          WAIT(&bars->mrg_d, mrg_d_ph, 46);
          mrg_d_ph ^= 1;
        }
      }
    }
  }

done:
  fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) tmem_dealloc(tmem, 512);
  cluster_sync();
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

template <bool kFp8>
mla_status launch_impl(const DecodeParams& dp, void* stream) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MLA_ERR_CUDA;
  CUtensorMap tmap;
  const cuuint64_t gdim[2] = {(cuuint64_t)kDqk, (cuuint64_t)dp.num_slots};
  const cuuint64_t gstride[1] = {(cuuint64_t)kDqk * (kFp8 ? 1 : 2)};
  const cuuint32_t box[2] = {kFp8 ? 192u : 64u, 1u};
  const cuuint32_t estr[2] = {1, 1};
  CUresult cr = enc(&tmap, kFp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(dp.kv), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    kFp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return MLA_ERR_INVALID_ARG;
  const int smem = kSmemBytes + kSmemAlign;
  auto kern = mla_decode_tensor_kernel<kFp8>;
  static int max_clusters[kMaxDevices][2] = {};
  const int dev = current_device_slot();
  if (dev < 0) return MLA_ERR_CUDA;
  if (max_clusters[dev][kFp8] == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return MLA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(threads_for(kFp8), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) return MLA_ERR_CUDA;
    max_clusters[dev][kFp8] = n;
  }
  int clusters = max_clusters[dev][kFp8];
  if (clusters > dp.items_cap) clusters = dp.items_cap > 0 ? dp.items_cap : 1;
  DecodeParams kp = dp;
  if (kFp8) {
    // The in-register fp8 -> bf16 conversion scales every value by 2^-112.
    kp.scale_log2 = dp.scale_log2 * 5.192296858534828e33f;
    kp.out_scale = dp.out_scale * 5.192296858534828e33f;
  }
  kern<<<2 * clusters, threads_for(kFp8), smem, (cudaStream_t)stream>>>(tmap, kp);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

int tensor_kernel_available() { return 1; }

mla_status launch_decode_tensor(const DecodeParams& dp, void* stream) {
  return dp.kv_fp8 ? launch_impl<true>(dp, stream) : launch_impl<false>(dp, stream);
}

}  // namespace mla
