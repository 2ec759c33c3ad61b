// a2av.cu -- GB300 (sm_103a) variable-size all-to-all with device-resident
// splits: the kernels and the C ABI declared in include/a2av.h.
//
// What is computed ("[a2av] Improve tuning for 4 GPUs", pytorch PR 154580,
// section "Problem"): W ranks; rank r sends S[r][p] rows to peer p; peer p
// receives the chunks back to back in source-rank order; out_splits_offsets
// holds the transposed splits and their exclusive scan.
//
// How (one launch, no host round trip):
//   1. Every CTA loads the W x W split matrix (<= 8 KiB, L2-resident after the
//      first CTA), validates it and builds, in shared memory, the offset
//      tables with warp-shuffle exclusive scans: out_off[p][r] (column scans)
//      and in_off[r][p] (row scans).  All CTAs reach the same verdict, so an
//      invalid matrix stops every CTA before any byte is written, without any
//      inter-CTA synchronisation.
//   2. The received streams of all peers, each contiguous in its output
//      buffer, are cut into equal tiles of at most `max_tile` bytes; the tile
//      size shrinks with the payload so that small exchanges still occupy the
//      whole GPU.  CTAs take tiles round-robin (the bulk engine: blocked runs
//      once every CTA has over a thousand tiles).  A tile maps to one peer p and
//      a contiguous byte range of out[p]; the source chunks it overlaps are
//      found from out_off[p][*].  This is the pages' "shift CTAs onto the
//      data-parallel dimension" (same page, section "Change") taken to its
//      limit: CTAs follow bytes, so one huge chunk gets most CTAs, empty
//      chunks get none and many tiny chunks share a CTA.
//   3. Copy engines:
//      - bulk (every row and buffer 16-byte aligned): one warp per CTA streams
//        tiles global -> shared -> global with cp.async.bulk; lane r loads
//        source r's part of a tile, lane 0 stores the tile; mbarriers track
//        the loads through a ring of shared-memory stages.
//      - staged (any alignment): a producer warp loads, with cp.async.bulk,
//        the 16-byte granules that hold each source segment of a tile into a
//        shared-memory stage; consumer warps rebuild destination-aligned
//        16-byte vectors from shared memory (funnel shifts when source and
//        destination differ mod 16) and store them with st.global.v4; head
//        and tail bytes go one by one.  Full/empty mbarriers pair the warps.
//      - vector (any alignment, no shared-memory staging): 16-byte loads and
//        stores from registers; a misaligned source is realigned with a warp
//        shuffle of neighbouring granules and a funnel shift.
//      No cluster multicast anywhere.  Every mbarrier wait is bounded (~1 s),
//      after which the kernel records A2AV_ERR_TIMEOUT and leaves.
//   CTA 0 writes out_splits_offsets.  Every kernel is launched with
//   programmatic dependent launch and waits for its predecessor on the stream
//   before it reads anything; a2av_run_multi runs up to four exchanges in one
//   launch, each on its own share of the grid.
#include "a2av_device.cuh"
#include "a2av_handle.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

// Engine shapes.  Each can be overridden at compile time (-DA2AV_...) for
// tuning sweeps; the defaults are the measured choices.
#ifndef A2AV_VEC_THREADS
#define A2AV_VEC_THREADS 512
#endif
#ifndef A2AV_VEC_UNROLL
#define A2AV_VEC_UNROLL 4
#endif
#ifndef A2AV_VEC_SHIFT_UNROLL
#define A2AV_VEC_SHIFT_UNROLL 2
#endif
#ifndef A2AV_VEC_MAX_TILE
#define A2AV_VEC_MAX_TILE (64 * 1024)
#endif
#ifndef A2AV_VEC_CTAS_PER_SM
#define A2AV_VEC_CTAS_PER_SM 2
#endif
// Bulk engine ring: 4 x 32 KiB stages, loads one tile ahead of the stores.
// Measured at cfg2 64 MiB / 256 MiB / 4 GiB per rank, each against a torch
// device copy of the same bytes interleaved in the same process: loads one
// tile ahead 0.990 / 1.001 / 0.999 of the copy, two ahead 0.975 / 0.961 /
// 0.972, four ahead of six stages 0.975 (4 GiB), 64 KiB stages 0.959, two
// CTAs an SM 0.950: more bytes in flight per SM is slower here.
#ifndef A2AV_BULK_STAGES
#define A2AV_BULK_STAGES 4
#endif
#ifndef A2AV_BULK_LEAD
#define A2AV_BULK_LEAD 1
#endif
#ifndef A2AV_BULK_STAGE_BYTES
#define A2AV_BULK_STAGE_BYTES (32 * 1024)
#endif
#ifndef A2AV_BULK_CTAS_PER_SM
#define A2AV_BULK_CTAS_PER_SM 1
#endif
#ifndef A2AV_STAGED_STAGES
#define A2AV_STAGED_STAGES 4
#endif
#ifndef A2AV_STAGED_STAGE_BYTES
#define A2AV_STAGED_STAGE_BYTES (32 * 1024)
#endif
#ifndef A2AV_STAGED_CONSUMER_WARPS
// Measured: 8 consumer warps beat 4 by 1-4 % on 13-byte rows at 2^20 rows per
// rank, but cost the latency-bound cases more (the one-launch keyed-jagged
// pair +1.2 us = +9 %, small exchanges +0.2 us), whether or not all of them
// consume: the larger CTA itself is slower to get going.
#define A2AV_STAGED_CONSUMER_WARPS 4
#endif
#ifndef A2AV_STAGED_CTAS_PER_SM
#define A2AV_STAGED_CTAS_PER_SM 1
#endif
// Tile order: round-robin (CTA b takes tiles b, b + G, ...) or blocked (CTA
// b takes a contiguous run of tiles).  Measured (interleaved A/B on one GPU):
// blocked is ~1 % faster for the bulk engine when every CTA has thousands of
// tiles (4 GiB per rank), round-robin equal or up to ~1 % faster below that
// and for the staged engine.  The bulk engine switches to blocked order from
// A2AV_BULK_BLOCKED_TILES tiles per CTA (0 = never).
#ifndef A2AV_BULK_BLOCKED_TILES
#define A2AV_BULK_BLOCKED_TILES 1024
#endif
#ifndef A2AV_STAGED_BLOCKED_TILES
#define A2AV_STAGED_BLOCKED_TILES 0
#endif

namespace {

// Vector engine: 512 threads (64 registers each, two CTAs per SM), 4
// independent 16-byte loads in flight per thread on the aligned path (32 KiB
// per CTA pass) and 2 on the realigning path, tiles of at most 64 KiB.
constexpr int kVecThreads = A2AV_VEC_THREADS;
constexpr int kVecUnroll = A2AV_VEC_UNROLL;
constexpr int kVecShiftUnroll = A2AV_VEC_SHIFT_UNROLL;
constexpr long long kVecMaxTile = A2AV_VEC_MAX_TILE;
constexpr int kVecCtasPerSm = A2AV_VEC_CTAS_PER_SM;

// Bulk engine: a ring of stages, each holding one tile (tiles are powers of
// two, at most the stage size); loads run LEAD tiles ahead of the stores that
// drain them (the stores of the other stages still in flight).
constexpr int kBulkThreads = 128;
constexpr int kBulkStages = A2AV_BULK_STAGES;
constexpr int kBulkLead = A2AV_BULK_LEAD;
constexpr int kBulkStageBytes = A2AV_BULK_STAGE_BYTES;
constexpr int kBulkCtasPerSm = A2AV_BULK_CTAS_PER_SM;

// Staged engine: one producer warp, consumer warps, a ring of stages.  A stage
// holds a tile plus the granule overhang of up to W segments (at most 15 bytes
// before and after each, rounded) so that every segment lands whole.
constexpr int kStagedStages = A2AV_STAGED_STAGES;
constexpr int kStagedStageBytes = A2AV_STAGED_STAGE_BYTES;
constexpr int kStagedConsumerWarps = A2AV_STAGED_CONSUMER_WARPS;
constexpr int kStagedThreads = 32 * (1 + kStagedConsumerWarps);
constexpr int kStagedCtasPerSm = A2AV_STAGED_CTAS_PER_SM;
constexpr int kStagedPad = 32 * kMaxW + 128;
constexpr int kStagedAlloc = kStagedStageBytes + kStagedPad;
static_assert(kStagedPad % 128 == 0 && kStagedStageBytes % 128 == 0, "128-byte aligned stages");

// The k-th of this CTA's tiles, in blocked or round-robin order.
struct TileSeq {
  long long first, step, count;
  __device__ TileSeq(long long ntiles, bool blocked, long long b, long long G) {
    if (blocked) {
      const long long per = (ntiles + G - 1) / G, lo = b * per;
      first = lo;
      step = 1;
      count = ntiles > lo ? (ntiles - lo < per ? ntiles - lo : per) : 0;
    } else {
      first = b;
      step = G;
      count = ntiles > b ? (ntiles - b + G - 1) / G : 0;
    }
  }
  __device__ long long operator[](long long k) const { return first + k * step; }
};

// Each engine is a device function run by CTA `cta` of the `ctas` CTAs that
// work on exchange P; its kernel runs it with the whole grid.
template <int NT, int U, int US>
__device__ __forceinline__ void vector_engine(const Params& P, long long max_tile, int cta,
                                              int ctas) {
  __shared__ Plan pl;
  if (!build_plan(P, pl, max_tile, cta, ctas)) return;
  const int W = P.W, tid = threadIdx.x;
  const long long ntiles = pl.tile_first[W];
  const long long rb = P.rb;
  for (long long t = cta; t < ntiles; t += ctas) {
    long long lo, hi;
    const int p = tile_peer(pl, W, t, rb, &lo, &hi);
    unsigned char* out = P.out[p];
    for (int r = 0; r < W; ++r) {
      const long long c_lo = pl.out_off[p][r] * rb, c_hi = pl.out_off[p][r + 1] * rb;
      const long long a = lo > c_lo ? lo : c_lo, b = hi < c_hi ? hi : c_hi;
      if (a >= b) continue;
      const unsigned char* src = P.in[r] + pl.in_off[r][p] * rb + (a - c_lo);
      copy_span<NT, U, US>(out + a, src, b - a, tid);
    }
  }
}

template <int NT, int U, int US>
__global__ void __launch_bounds__(NT, kVecCtasPerSm)
    a2av_vector_kernel(const __grid_constant__ Params P, long long max_tile) {
  vector_engine<NT, U, US>(P, max_tile, blockIdx.x, gridDim.x);
}

// ------------------------------------------------------------------ bulk --
// Every tile's source segments, destination and size are 16-byte aligned.
// Warp 0 does all the work: each tile is loaded by the lanes of the sources
// it overlaps (lane r, source r) into one stage, and stored by lane 0 in one
// piece, which tracks its own bulk stores.
template <int NS, int LEAD>
__device__ __forceinline__ void bulk_engine(const Params& P, int stage_bytes, int cta, int ctas) {
  static_assert(LEAD >= 1 && LEAD < NS, "loads run 1..NS-1 tiles ahead of stores");
  __shared__ Plan pl;
  __shared__ alignas(8) unsigned long long bars[NS];
  __shared__ unsigned char* stage_dst[NS];
  __shared__ unsigned stage_len[NS];
  extern __shared__ __align__(128) unsigned char stages[];
  if (!build_plan(P, pl, stage_bytes, cta, ctas)) return;
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) != 0) return;

  const int W = P.W;
  const long long ntiles = pl.tile_first[W];
  const TileSeq tiles(ntiles,
                      A2AV_BULK_BLOCKED_TILES > 0 &&
                          ntiles >= (long long)A2AV_BULK_BLOCKED_TILES * ctas,
                      cta, ctas);
  const long long nk = tiles.count;
  if (nk == 0) return;
  const uint32_t bar0 = smem_u32(bars), stage0 = smem_u32(stages);
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_fence_init();
  }
  __syncwarp();

  long long issued = 0;  // tiles whose loads are issued
  long long stored = 0;  // tiles whose stores are issued
  bool ok = true;
  for (long long k = 0; k < nk + LEAD; ++k) {
    if (k < nk) {
      const int s = (int)(k % NS);
      // The store that last read stage s was issued NS - LEAD - 1 stores ago.
      if (k >= NS && lane == 0) bulk_wait_read<NS - LEAD - 1>();
      __syncwarp();
      long long lo, hi, a;
      const unsigned char* src;
      const int p = tile_peer_warp(pl, W, tiles[k], P.rb, lane, &lo, &hi);
      const long long n = lane_segment(P, pl, W, p, lane, lo, hi, &a, &src);
      const uint32_t bar = bar0 + 8 * s, stage = stage0 + (uint32_t)s * stage_bytes;
      if (lane == 0) {
        stage_dst[s] = P.out[p] + lo;
        stage_len[s] = (unsigned)(hi - lo);
        const unsigned starve = (P.starve == 1 && cta == 0 && k == 0) ? 16u : 0u;
        mbar_expect_tx(bar, (unsigned)(hi - lo) + starve);
      }
      __syncwarp();
      if (n > 0) bulk_load(stage + (uint32_t)(a - lo), src, (unsigned)n, bar);
      issued = k + 1;
    }
    const long long j = k - LEAD;
    if (j >= 0 && j < nk) {
      const int s = (int)(j % NS);
      const uint32_t stage = stage0 + (uint32_t)s * stage_bytes;
      if (lane == 0) {
        ok = mbar_wait(bar0 + 8 * s, (unsigned)((j / NS) & 1));
        if (ok) bulk_store(stage_dst[s], stage, stage_len[s]);
      }
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      stored = j + 1;
    }
  }
  if (lane == 0) {
    if (!ok) {
      // A load never completed: report it, give the loads still in flight a
      // bounded chance to land, then leave.
      record_error(P.status, A2AV_ERR_TIMEOUT);
      for (long long j = stored; j < issued; ++j)
        mbar_wait(bar0 + 8 * (int)(j % NS), (unsigned)((j / NS) & 1));
    }
    bulk_wait_all();
  }
}

template <int NS, int LEAD>
__global__ void __launch_bounds__(kBulkThreads)
    a2av_bulk_kernel(const __grid_constant__ Params P, int stage_bytes) {
  bulk_engine<NS, LEAD>(P, stage_bytes, blockIdx.x, gridDim.x);
}

// ---------------------------------------------------------------- staged --
// Where each source segment of a staged tile sits: written by the producer
// warp before it arms the stage's full barrier, read by the consumers after
// they see that barrier complete.
struct StageDesc {
  unsigned char* dst;   // out[p] + lo
  int count;            // segments in the tile
  int seg_dst[kMaxW];   // first byte of the segment, relative to lo
  int seg_len[kMaxW];   // bytes
  int seg_src[kMaxW];   // stage offset of the segment's first byte
};

// n bytes from stage address m to global d, any alignment of either, by the
// NTC consumer threads.
template <int NTC>
__device__ __forceinline__ void copy_span_smem(unsigned char* d, uint32_t m, int n, int ct) {
  int head = (16 - (int)((uintptr_t)d & 15)) & 15;
  if (head > n) head = n;
  if (ct < head) d[ct] = lds8(m + ct);
  d += head;
  m += head;
  n -= head;
  const int nv = n >> 4, tail = n & 15;
  if (ct < tail) d[nv * 16 + ct] = lds8(m + nv * 16 + ct);
  if (nv == 0) return;
  uint4* dv = reinterpret_cast<uint4*>(d);
  const unsigned shift = m & 15;
  if (shift == 0) {
#pragma unroll 4
    for (int i = ct; i < nv; i += NTC) st_stream(dv + i, lds128(m + 16 * i));
    return;
  }
  const uint32_t mb = m - shift;
  const unsigned r8 = (shift & 3) * 8;
#define A2AV_SHIFTED_FROM_SMEM(Q)                                                     \
  _Pragma("unroll 4") for (int i = ct; i < nv; i += NTC)                              \
      st_stream(dv + i, extract16<Q>(lds128(mb + 16 * i), lds128(mb + 16 * i + 16), r8))
  switch (shift >> 2) {
    case 0: A2AV_SHIFTED_FROM_SMEM(0); break;
    case 1: A2AV_SHIFTED_FROM_SMEM(1); break;
    case 2: A2AV_SHIFTED_FROM_SMEM(2); break;
    default: A2AV_SHIFTED_FROM_SMEM(3); break;
  }
#undef A2AV_SHIFTED_FROM_SMEM
}

template <int NS, int NC>
__device__ __forceinline__ void staged_engine(const Params& P, int stage_bytes, int cta,
                                              int ctas) {
  __shared__ Plan pl;
  __shared__ StageDesc desc[NS];
  __shared__ alignas(8) unsigned long long full[NS];
  __shared__ alignas(8) unsigned long long empty[NS];
  __shared__ long long produced;     // tiles whose loads the producer issued
  __shared__ long long consumed[NC];  // tiles each consumer warp finished
  extern __shared__ __align__(128) unsigned char stages[];
  if (!build_plan(P, pl, stage_bytes, cta, ctas)) return;

  const int W = P.W, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TileSeq tiles(pl.tile_first[W], A2AV_STAGED_BLOCKED_TILES != 0, cta, ctas);
  const long long nk = tiles.count;
  if (nk == 0) return;
  const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty), stage0 = smem_u32(stages);
  const uint32_t alloc = (uint32_t)stage_bytes + kStagedPad;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, NC);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == 0) {
    // Producer: one tile per iteration, lane r loading source r's granules.
    long long k = 0;
    for (; k < nk; ++k) {
      const int s = (int)(k % NS);
      if (k >= NS && !mbar_wait_warp(empty0 + 8 * s, (unsigned)((k / NS - 1) & 1))) {
        if (lane == 0) record_error(P.status, A2AV_ERR_TIMEOUT);
        break;
      }
      long long lo, hi, a;
      const unsigned char* src;
      const int p = tile_peer_warp(pl, W, tiles[k], P.rb, lane, &lo, &hi);
      const long long n = lane_segment(P, pl, W, p, lane, lo, hi, &a, &src);
      const uintptr_t g_lo = (uintptr_t)src & ~(uintptr_t)15;
      const unsigned gb =
          n > 0 ? (unsigned)((((uintptr_t)src + (uintptr_t)n + 15) & ~(uintptr_t)15) - g_lo) : 0;
      unsigned inc = gb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += y;
      }
      const unsigned off = inc - gb, total = __shfl_sync(kFull, inc, 31);
      const unsigned has = __ballot_sync(kFull, n > 0);
      StageDesc& d = desc[s];
      if (n > 0) {
        const int idx = __popc(has & ((1u << lane) - 1u));
        d.seg_dst[idx] = (int)(a - lo);
        d.seg_len[idx] = (int)n;
        d.seg_src[idx] = (int)(off + (unsigned)((uintptr_t)src - g_lo));
      }
      if (lane == 0) {
        d.count = __popc(has);
        d.dst = P.out[p] + lo;
      }
      __syncwarp();
      const uint32_t bar = full0 + 8 * s;
      const unsigned starve = (P.starve == 1 && cta == 0 && k == 0) ? 16u : 0u;
      if (lane == 0) mbar_expect_tx(bar, total + starve);
      __syncwarp();
      if (n > 0) bulk_load(stage0 + (uint32_t)s * alloc + off, (const void*)g_lo, gb, bar);
    }
    if (lane == 0) produced = k;
  } else {
    // Consumers: rebuild each tile from its stage with destination-aligned stores.
    const int ct = threadIdx.x - 32;
    long long k = 0;
    for (; k < nk; ++k) {
      const int s = (int)(k % NS);
      if (!mbar_wait_warp(full0 + 8 * s, (unsigned)((k / NS) & 1))) {
        if (lane == 0) record_error(P.status, A2AV_ERR_TIMEOUT);
        break;
      }
      const StageDesc& d = desc[s];
      const int count = d.count;
      unsigned char* dst = d.dst;
      const uint32_t stage = stage0 + (uint32_t)s * alloc;
      for (int i = 0; i < count; ++i)
        copy_span_smem<32 * NC>(dst + d.seg_dst[i], stage + (uint32_t)d.seg_src[i], d.seg_len[i],
                                ct);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
    if (lane == 0) consumed[warp - 1] = k;
  }
  // After a timeout some issued loads may not have been waited for: before
  // the CTA leaves (and its shared memory is reused), wait -- bounded -- for
  // every tile the producer issued that some consumer did not finish.  The
  // producer never runs more than NS tiles ahead, so these tiles sit in
  // distinct stages and their phases are the ones the consumers waited on.
  __syncthreads();
  if (threadIdx.x == 0) {
    long long lo = produced;
    for (int c = 0; c < NC; ++c) lo = consumed[c] < lo ? consumed[c] : lo;
    for (long long k = lo; k < produced; ++k)
      mbar_wait(full0 + 8 * (int)(k % NS), (unsigned)((k / NS) & 1));
  }
}

template <int NS, int NC>
__global__ void __launch_bounds__(32 * (NC + 1))
    a2av_staged_kernel(const __grid_constant__ Params P, int stage_bytes) {
  staged_engine<NS, NC>(P, stage_bytes, blockIdx.x, gridDim.x);
}

// ------------------------------------------------------ several at once --
// Up to A2AV_MAX_EXCHANGES independent exchanges over the same ranks in one
// launch (a2av_run_multi).  The grid is divided among them in proportion to
// their bytes, each getting at least one CTA; every CTA computes the same
// division from the split matrices, then runs its exchange's engine as if
// that exchange had the launch to itself.
constexpr int kMaxExchanges = A2AV_MAX_EXCHANGES;
static_assert(kBulkThreads >= 32 * kMaxExchanges && kStagedThreads >= 32 * kMaxExchanges &&
                  kVecThreads >= 32 * kMaxExchanges,
              "multi_slot gives each exchange a warp");

struct MultiParams {
  Params ex[kMaxExchanges];
  int count;
};

// This CTA's exchange, its index among that exchange's CTAs and their
// number; false for a CTA left over by the rounding.  An exchange whose
// splits are out of range weighs nothing (its one CTA finds them invalid).
__device__ __forceinline__ bool multi_slot(const MultiParams& M, int* which, int* cta, int* ctas) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ double weight[kMaxExchanges];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, n = M.count;
  if (warp < n) {  // warp x sums exchange x's bytes (every engine has >= 4 warps)
    const Params& P = M.ex[warp];
    const int W = P.W;
    double rows = 0.0;
    int bad = 0;
    for (int e = lane; e < W * W; e += 32) {
      const long long v = P.splits[(long long)(e / W) * P.split_stride + e % W];
      if (v < 0 || v > P.limit)
        bad = 1;
      else
        rows += (double)v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rows += __shfl_xor_sync(kFull, rows, o);
    bad = __any_sync(kFull, bad);
    if (lane == 0) weight[warp] = bad ? 0.0 : rows * (double)P.rb;
  }
  __syncthreads();
  double total = 0.0;
  for (int x = 0; x < n; ++x) total += weight[x];
  const int G = gridDim.x, spare = G - n;
  int start = 0;
  for (int x = 0; x < n; ++x) {
    int g = 1 + (total > 0.0 ? (int)floor((double)spare * (weight[x] / total)) : 0);
    const int room = G - (n - 1 - x) - start;  // keep one CTA for each later exchange
    if (g > room) g = room;
    if ((int)blockIdx.x >= start && (int)blockIdx.x < start + g) {
      *which = x;
      *cta = (int)blockIdx.x - start;
      *ctas = g;
      return true;
    }
    start += g;
  }
  return false;
}

template <int NT, int U, int US>
__global__ void __launch_bounds__(NT, kVecCtasPerSm)
    a2av_vector_multi_kernel(const __grid_constant__ MultiParams M, long long max_tile) {
  int x, cta, ctas;
  if (multi_slot(M, &x, &cta, &ctas)) vector_engine<NT, U, US>(M.ex[x], max_tile, cta, ctas);
}

template <int NS, int LEAD>
__global__ void __launch_bounds__(kBulkThreads)
    a2av_bulk_multi_kernel(const __grid_constant__ MultiParams M, int stage_bytes) {
  int x, cta, ctas;
  if (multi_slot(M, &x, &cta, &ctas)) bulk_engine<NS, LEAD>(M.ex[x], stage_bytes, cta, ctas);
}

template <int NS, int NC>
__global__ void __launch_bounds__(32 * (NC + 1))
    a2av_staged_multi_kernel(const __grid_constant__ MultiParams M, int stage_bytes) {
  int x, cta, ctas;
  if (multi_slot(M, &x, &cta, &ctas)) staged_engine<NS, NC>(M.ex[x], stage_bytes, cta, ctas);
}

}  // namespace

// ================================================================ host ABI ==

namespace {

using BulkKernel = void (*)(Params, int);
const BulkKernel kBulk = a2av_bulk_kernel<kBulkStages, kBulkLead>;
const BulkKernel kStaged = a2av_staged_kernel<kStagedStages, kStagedConsumerWarps>;
using VecKernel = void (*)(Params, long long);
const VecKernel kVec = a2av_vector_kernel<kVecThreads, kVecUnroll, kVecShiftUnroll>;
using BulkMultiKernel = void (*)(MultiParams, int);
const BulkMultiKernel kBulkMulti = a2av_bulk_multi_kernel<kBulkStages, kBulkLead>;
const BulkMultiKernel kStagedMulti = a2av_staged_multi_kernel<kStagedStages, kStagedConsumerWarps>;
using VecMultiKernel = void (*)(MultiParams, long long);
const VecMultiKernel kVecMulti =
    a2av_vector_multi_kernel<kVecThreads, kVecUnroll, kVecShiftUnroll>;

int env_int(const char* name, int fallback) {
  const char* v = std::getenv(name);
  if (v == nullptr || *v == '\0') return fallback;
  return std::atoi(v);
}

// Shared-memory opt-in of the staging engines (once per device).
int configure_kernels() {
  if (cudaFuncSetAttribute(kBulk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kBulkStages * kBulkStageBytes) != cudaSuccess)
    return A2AV_ERR_CUDA;
  if (cudaFuncSetAttribute(kStaged, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kStagedStages * kStagedAlloc) != cudaSuccess)
    return A2AV_ERR_CUDA;
  if (cudaFuncSetAttribute(kBulkMulti, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kBulkStages * kBulkStageBytes) != cudaSuccess)
    return A2AV_ERR_CUDA;
  if (cudaFuncSetAttribute(kStagedMulti, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kStagedStages * kStagedAlloc) != cudaSuccess)
    return A2AV_ERR_CUDA;
  return A2AV_OK;
}

// Fill the kernel parameters; returns whether every row and buffer is
// 16-byte aligned (the bulk engine's precondition).
bool fill_params(Params* P, int W, const void* const* in_ptrs, const int64_t* in_splits_dev,
                 void* const* out_ptrs, int64_t* out_splits_offsets_dev, int64_t row_bytes,
                 long long in_cap, long long out_cap, int* status, long long split_stride,
                 int starve = 0) {
  std::memset(P, 0, sizeof(*P));
  bool aligned = (row_bytes % 16) == 0;
  for (int r = 0; r < W; ++r) {
    P->in[r] = static_cast<const unsigned char*>(in_ptrs[r]);
    P->out[r] = static_cast<unsigned char*>(out_ptrs[r]);
    aligned = aligned && ((uintptr_t)P->in[r] & 15) == 0 && ((uintptr_t)P->out[r] & 15) == 0;
  }
  P->splits = reinterpret_cast<const long long*>(in_splits_dev);
  P->split_stride = split_stride;
  P->out_so = reinterpret_cast<long long*>(out_splits_offsets_dev);
  P->status = status;
  P->rb = row_bytes;
  P->limit = split_limit(W, row_bytes);
  P->in_cap = in_cap;
  P->out_cap = out_cap;
  P->W = W;
  P->starve = starve;
  return aligned;
}

// Engine actually used for a request: buffers that are not all device memory
// take the vector engine (plain loads and stores reach host memory; the
// cp.async.bulk engines are kept to device memory); BULK needs full
// alignment (else STAGED); AUTO is BULK when aligned, STAGED otherwise.
int resolve_path(int requested, bool aligned, bool device_memory) {
  if (!device_memory || requested == A2AV_PATH_VECTOR) return A2AV_PATH_VECTOR;
  if (requested == A2AV_PATH_STAGED) return requested;
  return aligned ? A2AV_PATH_BULK : A2AV_PATH_STAGED;
}

bool classify(const void* const* a, int na, const void* const* b, int nb) {
  for (int k = 0; k < na + nb; ++k) {
    const void* p = k < na ? a[k] : b[k - na];
    if (p == nullptr) continue;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      cudaGetLastError();  // (not sticky) -- an unknown pointer is not device memory
      return false;
    }
    if (at.type != cudaMemoryTypeDevice) return false;
  }
  return true;
}

// One launch of the chosen engine.  With `pdl` the launch may overlap the
// tail of the previous kernel on the stream (build_plan waits for it).
int launch(const Params& P, int path, int ctas_per_sm, int sms, cudaStream_t s, bool pdl,
           int* grid, int* block) {
  cudaError_t e;
  if (path == A2AV_PATH_BULK) {
    *grid = sms * (ctas_per_sm ? ctas_per_sm : kBulkCtasPerSm);
    *block = kBulkThreads;
    e = launch_kernel(kBulk, dim3(*grid), *block, kBulkStages * kBulkStageBytes, s, pdl, P,
                      (int)kBulkStageBytes);
  } else if (path == A2AV_PATH_STAGED) {
    *grid = sms * (ctas_per_sm ? ctas_per_sm : kStagedCtasPerSm);
    *block = kStagedThreads;
    e = launch_kernel(kStaged, dim3(*grid), *block, kStagedStages * kStagedAlloc, s, pdl, P,
                      (int)kStagedStageBytes);
  } else {
    *grid = sms * (ctas_per_sm ? ctas_per_sm : kVecCtasPerSm);
    *block = kVecThreads;
    e = launch_kernel(kVec, dim3(*grid), *block, 0, s, pdl, P, (long long)kVecMaxTile);
  }
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? A2AV_OK : A2AV_ERR_CUDA;
}

}  // namespace

bool a2av_device_buffers(a2av_handle* h, const void* const* a, int na, const void* const* b,
                         int nb) {
  const int n = na + nb;
  if (h == nullptr || n > 2 * kMaxExchanges * kMaxW) return classify(a, na, b, nb);
  ++h->cache_clock;
  for (a2av_ptr_cache& c : h->cache) {
    if (c.n != n) continue;
    bool same = true;
    for (int k = 0; k < n && same; ++k) same = c.ptrs[k] == (k < na ? a[k] : b[k - na]);
    if (same) {
      c.stamp = h->cache_clock;
      return c.device;
    }
  }
  a2av_ptr_cache& c = h->cache[0].stamp <= h->cache[1].stamp ? h->cache[0] : h->cache[1];
  c.device = classify(a, na, b, nb);
  for (int k = 0; k < n; ++k) c.ptrs[k] = k < na ? a[k] : b[k - na];
  c.n = n;
  c.stamp = h->cache_clock;
  return c.device;
}

extern "C" {

int a2av_version(void) { return 10200; }

const char* a2av_error_string(int code) {
  switch (code) {
    case A2AV_OK: return "ok";
    case A2AV_ERR_INVALID_ARG: return "invalid argument";
    case A2AV_ERR_UNSUPPORTED: return "unsupported (world size above A2AV_MAX_RANKS)";
    case A2AV_ERR_CUDA: return "CUDA runtime error";
    case A2AV_ERR_BAD_SPLITS: return "invalid split matrix (detected on the device)";
    case A2AV_ERR_TIMEOUT: return "a bounded device wait timed out";
    case A2AV_ERR_BAD_INDEX:
      return "a dispatch key, source row or combine position is out of range (detected on the device)";
    default: return "unknown status";
  }
}

int a2av_create(int world_size, int64_t in_capacity_rows, int64_t out_capacity_rows,
                a2av_handle** out) {
  if (out == nullptr) return A2AV_ERR_INVALID_ARG;
  *out = nullptr;
  if (world_size < 1 || in_capacity_rows < 0 || out_capacity_rows < 0) return A2AV_ERR_INVALID_ARG;
  if (world_size > kMaxW) return A2AV_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return A2AV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return A2AV_ERR_CUDA;
  if (configure_kernels() != A2AV_OK) return A2AV_ERR_CUDA;
  int* status = nullptr;
  if (cudaMalloc(&status, 256) != cudaSuccess) return A2AV_ERR_CUDA;
  if (cudaMemset(status, 0, 256) != cudaSuccess) {
    cudaFree(status);
    return A2AV_ERR_CUDA;
  }
  a2av_handle* h = new (std::nothrow) a2av_handle();
  if (h == nullptr) {
    cudaFree(status);
    return A2AV_ERR_CUDA;
  }
  h->W = world_size;
  h->in_cap = in_capacity_rows;
  h->out_cap = out_capacity_rows;
  h->device = dev;
  h->sms = sms;
  h->d_status = status;
  h->path = env_int("A2AV_PATH", A2AV_PATH_AUTO);
  if (h->path < A2AV_PATH_AUTO || h->path > A2AV_PATH_STAGED) h->path = A2AV_PATH_AUTO;
  h->ctas_per_sm = env_int("A2AV_CTAS_PER_SM", 0);
  if (h->ctas_per_sm < 0 || h->ctas_per_sm > 32) h->ctas_per_sm = 0;
  h->starve = env_int("A2AV_DEBUG_STARVE", 0);
  if (h->starve < 0 || h->starve > 2) h->starve = 0;
  h->pdl = env_int("A2AV_PDL", 1) != 0;
  h->gather_ready = false;
  h->order_grid = 0;
  h->order_level = env_int("A2AV_DISPATCH_ORDER", A2AV_DISPATCH_ORDER);
  if (h->order_level < 0 || h->order_level > 3) h->order_level = A2AV_DISPATCH_ORDER;
  h->last_path = h->last_grid = h->last_block = 0;
  h->last_kernels = h->last_memsets = 0;
  h->last_copy = "";
  h->cache[0].n = h->cache[1].n = 0;
  h->cache[0].stamp = h->cache[1].stamp = 0;
  h->cache_clock = 0;
  *out = h;
  return A2AV_OK;
}

int a2av_set_path(a2av_handle* h, int path) {
  if (h == nullptr || path < A2AV_PATH_AUTO || path > A2AV_PATH_STAGED) return A2AV_ERR_INVALID_ARG;
  h->path = path;
  h->cache[0].n = h->cache[1].n = 0;  // the pointers are looked at afresh
  return A2AV_OK;
}

int a2av_set_grid(a2av_handle* h, int ctas_per_sm) {
  if (h == nullptr || ctas_per_sm < 0 || ctas_per_sm > 32) return A2AV_ERR_INVALID_ARG;
  h->ctas_per_sm = ctas_per_sm;
  h->cache[0].n = h->cache[1].n = 0;
  return A2AV_OK;
}

int a2av_last_launch(const a2av_handle* h, int* path, int* grid, int* block) {
  if (h == nullptr) return A2AV_ERR_INVALID_ARG;
  if (path) *path = h->last_path;
  if (grid) *grid = h->last_grid;
  if (block) *block = h->last_block;
  return A2AV_OK;
}

}  // extern "C"

namespace {

// a2av_run and a2av_combine: the split matrix's rows are split_stride apart.
int run_exchange(a2av_handle* h, const void* const* in_ptrs, const int64_t* in_splits_dev,
                 void* const* out_ptrs, int64_t* out_splits_offsets_dev, int64_t row_bytes,
                 void* stream, long long split_stride) {
  if (h == nullptr || in_ptrs == nullptr || out_ptrs == nullptr || in_splits_dev == nullptr ||
      out_splits_offsets_dev == nullptr || row_bytes < 1)
    return A2AV_ERR_INVALID_ARG;
  if (((uintptr_t)in_splits_dev & 7) != 0 || ((uintptr_t)out_splits_offsets_dev & 7) != 0)
    return A2AV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return A2AV_ERR_CUDA;
  if (dev != h->device) return A2AV_ERR_INVALID_ARG;

  Params P;
  const bool aligned = fill_params(&P, h->W, in_ptrs, in_splits_dev, out_ptrs,
                                   out_splits_offsets_dev, row_bytes, h->in_cap, h->out_cap,
                                   h->d_status, split_stride, h->starve);
  const bool device_memory = a2av_device_buffers(h, in_ptrs, h->W, out_ptrs, h->W);
  const int path = resolve_path(h->path, aligned, device_memory);
  int grid = 0, block = 0;
  const int rc = launch(P, path, h->ctas_per_sm, h->sms, static_cast<cudaStream_t>(stream),
                        h->pdl, &grid, &block);
  if (rc != A2AV_OK) return rc;
  h->last_path = path;
  h->last_grid = grid;
  h->last_block = block;
  return A2AV_OK;
}

}  // namespace

extern "C" {

int a2av_run(a2av_handle* h, const void* const* in_ptrs, const int64_t* in_splits_dev,
             void* const* out_ptrs, int64_t* out_splits_offsets_dev, int64_t row_bytes,
             void* stream) {
  if (h == nullptr) return A2AV_ERR_INVALID_ARG;
  return run_exchange(h, in_ptrs, in_splits_dev, out_ptrs, out_splits_offsets_dev, row_bytes,
                      stream, h->W);
}

int a2av_combine(a2av_handle* h, const void* const* in_ptrs,
                 const int64_t* dispatch_splits_offsets_dev, void* const* out_ptrs,
                 int64_t* out_splits_offsets_dev, int64_t row_bytes, void* stream) {
  if (h == nullptr) return A2AV_ERR_INVALID_ARG;
  // Rank p sends back to rank r the S[r][p] rows it received from it:
  // the reverse splits S'[p][r] = S[r][p] are row 0 of the dispatch's
  // out_splits_offsets block of peer p, i.e. rows 2W apart.
  return run_exchange(h, in_ptrs, dispatch_splits_offsets_dev, out_ptrs,
                      out_splits_offsets_dev, row_bytes, stream, 2LL * h->W);
}

int a2av_run_multi(a2av_handle* h, int count, const a2av_exchange_t* exchanges, void* stream) {
  if (h == nullptr || exchanges == nullptr || count < 1) return A2AV_ERR_INVALID_ARG;
  if (count > kMaxExchanges) return A2AV_ERR_UNSUPPORTED;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return A2AV_ERR_CUDA;
  if (dev != h->device) return A2AV_ERR_INVALID_ARG;
  MultiParams M;
  std::memset(&M, 0, sizeof(M));
  M.count = count;
  bool aligned = true;
  const void* bufs[2 * kMaxExchanges * kMaxW];  // every buffer of the call, classified at once
  int nbufs = 0;
  for (int x = 0; x < count; ++x) {
    const a2av_exchange_t& e = exchanges[x];
    if (e.in_ptrs == nullptr || e.out_ptrs == nullptr || e.in_splits_dev == nullptr ||
        e.out_splits_offsets_dev == nullptr || e.row_bytes < 1)
      return A2AV_ERR_INVALID_ARG;
    if (((uintptr_t)e.in_splits_dev & 7) != 0 || ((uintptr_t)e.out_splits_offsets_dev & 7) != 0)
      return A2AV_ERR_INVALID_ARG;
    aligned = fill_params(&M.ex[x], h->W, e.in_ptrs, e.in_splits_dev, e.out_ptrs,
                          e.out_splits_offsets_dev, e.row_bytes, h->in_cap, h->out_cap,
                          h->d_status, h->W, h->starve) &&
              aligned;
    for (int r = 0; r < h->W; ++r) {
      bufs[nbufs++] = e.in_ptrs[r];
      bufs[nbufs++] = e.out_ptrs[r];
    }
  }
  const bool device_memory = a2av_device_buffers(h, bufs, nbufs, nullptr, 0);
  // One engine for the launch: bulk only when every exchange allows it.
  const int path = resolve_path(h->path, aligned, device_memory);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int grid, block;
  cudaError_t err;
  if (path == A2AV_PATH_BULK) {
    grid = h->sms * (h->ctas_per_sm ? h->ctas_per_sm : kBulkCtasPerSm);
    block = kBulkThreads;
    err = launch_kernel(kBulkMulti, dim3(grid), block, kBulkStages * kBulkStageBytes, s, h->pdl,
                        M, (int)kBulkStageBytes);
  } else if (path == A2AV_PATH_STAGED) {
    grid = h->sms * (h->ctas_per_sm ? h->ctas_per_sm : kStagedCtasPerSm);
    block = kStagedThreads;
    err = launch_kernel(kStagedMulti, dim3(grid), block, kStagedStages * kStagedAlloc, s, h->pdl,
                        M, (int)kStagedStageBytes);
  } else {
    grid = h->sms * (h->ctas_per_sm ? h->ctas_per_sm : kVecCtasPerSm);
    block = kVecThreads;
    err = launch_kernel(kVecMulti, dim3(grid), block, 0, s, h->pdl, M, (long long)kVecMaxTile);
  }
  if (err != cudaSuccess || cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
  h->last_path = path;
  h->last_grid = grid;
  h->last_block = block;
  return A2AV_OK;
}

int a2av_status(a2av_handle* h, void* stream, int* device_status) {
  if (h == nullptr || device_status == nullptr) return A2AV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int value = 0;
  if (cudaMemcpyAsync(&value, h->d_status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return A2AV_ERR_CUDA;
  if (cudaMemsetAsync(h->d_status, 0, sizeof(int), s) != cudaSuccess) return A2AV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return A2AV_ERR_CUDA;
  *device_status = value;
  return A2AV_OK;
}

int a2av_destroy(a2av_handle* h) {
  if (h == nullptr) return A2AV_OK;
  const cudaError_t err = cudaFree(h->d_status);
  delete h;
  return err == cudaSuccess ? A2AV_OK : A2AV_ERR_CUDA;
}

}  // extern "C"

// ===================================================== allocation-free call ==
// The status word of a2av_run_noalloc.  Host code never touches this name:
// on the host it is only a stand-in, so its device address is looked up once
// per device (with that device current) and passed to the kernels.
static __device__ __align__(256) int g_noalloc_scratch[A2AV_NOALLOC_SCRATCH_BYTES / sizeof(int)];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
int* g_noalloc_status[kNoAllocMaxDevices];  // device address of g_noalloc_scratch
int g_noalloc_sms[kNoAllocMaxDevices];

int noalloc_setup(int dev, int** status, int* sms) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_status[dev] == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess) return A2AV_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return A2AV_ERR_CUDA;
    if (configure_kernels() != A2AV_OK) return A2AV_ERR_CUDA;
    g_noalloc_sms[dev] = n;
    g_noalloc_status[dev] = static_cast<int*>(addr);
  }
  *status = g_noalloc_status[dev];
  *sms = g_noalloc_sms[dev];
  return A2AV_OK;
}

}  // namespace

extern "C" int a2av_run_noalloc(int world_size, int64_t in_capacity_rows,
                                int64_t out_capacity_rows, const void* const* in_ptrs,
                                const int64_t* in_splits_dev, void* const* out_ptrs,
                                int64_t* out_splits_offsets_dev, int64_t row_bytes, void* stream,
                                int* device_status) {
  static_assert(sizeof(int) <= A2AV_NOALLOC_SCRATCH_BYTES, "the status word fits the scratch");
  if (world_size < 1 || in_capacity_rows < 0 || out_capacity_rows < 0 || in_ptrs == nullptr ||
      out_ptrs == nullptr || in_splits_dev == nullptr || out_splits_offsets_dev == nullptr ||
      row_bytes < 1)
    return A2AV_ERR_INVALID_ARG;
  if (world_size > kMaxW) return A2AV_ERR_UNSUPPORTED;
  if (((uintptr_t)in_splits_dev & 7) != 0 || ((uintptr_t)out_splits_offsets_dev & 7) != 0)
    return A2AV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return A2AV_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return A2AV_ERR_UNSUPPORTED;
  int* status = nullptr;
  int sms = 0;
  int rc = noalloc_setup(dev, &status, &sms);
  if (rc != A2AV_OK) return rc;

  Params P;
  const bool aligned = fill_params(&P, world_size, in_ptrs, in_splits_dev, out_ptrs,
                                   out_splits_offsets_dev, row_bytes, in_capacity_rows,
                                   out_capacity_rows, status, world_size);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The kernels only ever set the status word, so it must start at zero.
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return A2AV_ERR_CUDA;
  int grid = 0, block = 0;
  const bool device_memory = a2av_device_buffers(nullptr, in_ptrs, world_size, out_ptrs,
                                                 world_size);
  rc = launch(P, resolve_path(A2AV_PATH_AUTO, aligned, device_memory), 0, sms, s, true, &grid,
              &block);
  if (rc != A2AV_OK) return rc;
  if (device_status != nullptr) {
    int value = 0;
    if (cudaMemcpyAsync(&value, status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return A2AV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return A2AV_ERR_CUDA;
    *device_status = value;
  }
  return A2AV_OK;
}
