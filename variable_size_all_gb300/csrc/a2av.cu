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
//      whole GPU.  CTAs take tiles round-robin.  A tile maps to one peer p and
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
//   CTA 0 writes out_splits_offsets.
#include "a2av.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

namespace {

constexpr int kMaxW = A2AV_MAX_RANKS;
constexpr long long kMaxBytes = 1LL << 62;  // byte offsets stay below 2^62
constexpr unsigned kFull = 0xffffffffu;
constexpr long long kTileGranule = 4096;         // tile sizes are multiples of this
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at GB300 clocks

}  // namespace

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
#ifndef A2AV_BULK_STAGES
#define A2AV_BULK_STAGES 4
#endif
#ifndef A2AV_BULK_LEAD
#define A2AV_BULK_LEAD 2
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
#define A2AV_STAGED_CONSUMER_WARPS 4
#endif
#ifndef A2AV_STAGED_CTAS_PER_SM
#define A2AV_STAGED_CTAS_PER_SM 1
#endif
#ifndef A2AV_TILES_PER_CTA
#define A2AV_TILES_PER_CTA 1
#endif
// L2 eviction hints of the bulk engine: bit 0 marks loaded lines
// evict-first, bit 1 stored lines (each byte is used exactly once; marking
// the stored lines measured best).
#ifndef A2AV_L2_HINT
#define A2AV_L2_HINT 2
#endif

namespace {

// Tiles each CTA gets at least, when the payload allows (smaller tiles for
// small payloads keep more of them in flight per CTA).
constexpr long long kTilesPerCta = A2AV_TILES_PER_CTA;

// Vector engine: 512 threads (64 registers each, two CTAs per SM), 4
// independent 16-byte loads in flight per thread on the aligned path (32 KiB
// per CTA pass) and 2 on the realigning path, tiles of at most 64 KiB.
constexpr int kVecThreads = A2AV_VEC_THREADS;
constexpr int kVecUnroll = A2AV_VEC_UNROLL;
constexpr int kVecShiftUnroll = A2AV_VEC_SHIFT_UNROLL;
constexpr long long kVecMaxTile = A2AV_VEC_MAX_TILE;
constexpr int kVecCtasPerSm = A2AV_VEC_CTAS_PER_SM;

// Bulk engine: a ring of stages (tile = stage size); loads run LEAD tiles
// ahead of the stores that drain them.
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

struct Params {
  const unsigned char* in[kMaxW];
  unsigned char* out[kMaxW];
  const long long* splits;  // S[r][p] at splits[r * split_stride + p]
  long long split_stride;   // W for a2av_run; 2W when the splits are a previous
                            // exchange's out_splits_offsets (a2av_combine)
  long long* out_so;        // [W][2][W]
  int* status;
  long long rb;             // row bytes
  long long in_cap;         // rows, 0 = unchecked
  long long out_cap;        // rows, 0 = unchecked
  int W;
};

// Per-CTA plan in shared memory.  Once build_plan returns, offsets are BYTES.
struct Plan {
  long long out_off[kMaxW][kMaxW + 1];  // [p][r] = rb * sum_{q<r} S[q][p]; [p][W] = bytes p receives
  long long in_off[kMaxW][kMaxW];       // [r][p] = rb * sum_{q<p} S[r][q]
  long long tile_first[kMaxW + 1];      // first tile of peer p; [W] = number of tiles
  long long tile;                       // tile size in bytes
};

__device__ __forceinline__ long long warp_inclusive_scan(long long x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

__device__ __forceinline__ void record_error(int* status, int code) {
  atomicCAS(status, 0, code);
}

// Step 1 of the header comment.  Returns false (in every thread of the CTA)
// when the splits are invalid; CTA 0 then records A2AV_ERR_BAD_SPLITS.
__device__ bool build_plan(const Params& P, Plan& pl, long long max_tile) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
  const int W = P.W;
  const long long rb = P.rb;
  const long long limit = kMaxBytes / ((long long)W * rb);

  int bad = 0;
  for (int e = tid; e < W * W; e += nt) {
    const long long s = P.splits[(long long)(e / W) * P.split_stride + e % W];
    if (s < 0 || s > limit) bad = 1;
    pl.in_off[e / W][e % W] = s;  // raw S[r][p] until the row scans below
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) record_error(P.status, A2AV_ERR_BAD_SPLITS);
    return false;
  }

  // Column scans: lane r holds S[r][p]; out_off[p][r] is its exclusive prefix.
  for (int p = warp; p < W; p += nwarps) {
    const long long x = lane < W ? pl.in_off[lane][p] : 0;
    const long long inc = warp_inclusive_scan(x, lane);
    if (lane < W) pl.out_off[p][lane] = inc - x;
    if (lane == 31) {
      pl.out_off[p][W] = inc;
      if ((P.out_cap > 0 && inc > P.out_cap) || (P.out[p] == nullptr && inc > 0)) bad = 1;
    }
  }
  __syncthreads();
  // Row scans, in place: lane p holds S[r][p]; in_off[r][p] is its exclusive prefix.
  for (int r = warp; r < W; r += nwarps) {
    const long long x = lane < W ? pl.in_off[r][lane] : 0;
    const long long inc = warp_inclusive_scan(x, lane);
    if (lane < W) pl.in_off[r][lane] = inc - x;
    if (lane == 31) {
      if ((P.in_cap > 0 && inc > P.in_cap) || (P.in[r] == nullptr && inc > 0)) bad = 1;
    }
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) record_error(P.status, A2AV_ERR_BAD_SPLITS);
    return false;
  }

  // Tiles: peer p's received stream (out_off[p][W] * rb bytes) is cut into
  // ceil(bytes / tile) tiles; tile_first is their exclusive prefix.
  if (warp == 0) {
    const long long bytes = lane < W ? pl.out_off[lane][W] * rb : 0;
    const long long total = __shfl_sync(kFull, warp_inclusive_scan(bytes, lane), 31);
    const long long per_cta =
        (total + kTilesPerCta * gridDim.x - 1) / (kTilesPerCta * gridDim.x);
    long long tile = (per_cta + kTileGranule - 1) / kTileGranule * kTileGranule;
    tile = tile < kTileGranule ? kTileGranule : (tile > max_tile ? max_tile : tile);
    const long long n = (bytes + tile - 1) / tile;
    const long long inc = warp_inclusive_scan(n, lane);
    if (lane < W) pl.tile_first[lane] = inc - n;
    if (lane == 31) {
      pl.tile_first[W] = inc;
      pl.tile = tile;
    }
  }
  __syncthreads();

  if (blockIdx.x == 0) {
    for (int e = tid; e < W * W; e += nt) {
      const int p = e / W, r = e % W;
      long long* so = P.out_so + (long long)p * 2 * W;
      so[r] = pl.out_off[p][r + 1] - pl.out_off[p][r];
      so[W + r] = pl.out_off[p][r];
    }
  }
  __syncthreads();
  // From here on the tables hold bytes.
  for (int e = tid; e < W * (W + 1); e += nt) pl.out_off[e / (W + 1)][e % (W + 1)] *= rb;
  for (int e = tid; e < W * W; e += nt) pl.in_off[e / W][e % W] *= rb;
  __syncthreads();
  return true;
}

// Tile t -> peer p and the byte range [lo, hi) of out[p] it covers (all
// threads of the caller compute the same).
__device__ __forceinline__ int tile_peer(const Plan& pl, int W, long long t, long long* lo,
                                         long long* hi) {
  int p = 0;
  while (p + 1 < W && pl.tile_first[p + 1] <= t) ++p;
  *lo = (t - pl.tile_first[p]) * pl.tile;
  const long long end = *lo + pl.tile;
  *hi = end < pl.out_off[p][W] ? end : pl.out_off[p][W];
  return p;
}

// The same for a whole warp at once: the largest p with tile_first[p] <= t
// (peers without tiles share their successor's tile_first, so the largest
// such p is the one that owns tile t).
__device__ __forceinline__ int tile_peer_warp(const Plan& pl, int W, long long t, int lane,
                                              long long* lo, long long* hi) {
  const unsigned m = __ballot_sync(kFull, lane < W && pl.tile_first[lane] <= t);
  const int p = 31 - __clz(m);
  *lo = (t - pl.tile_first[p]) * pl.tile;
  const long long end = *lo + pl.tile;
  *hi = end < pl.out_off[p][W] ? end : pl.out_off[p][W];
  return p;
}

// Lane r's part of the tile [lo, hi) of peer p: the destination offset a, the
// byte count n (0 when source r contributes nothing) and the source address.
__device__ __forceinline__ long long lane_segment(const Params& P, const Plan& pl, int W, int p,
                                                  int r, long long lo, long long hi, long long* a,
                                                  const unsigned char** src) {
  *a = 0;
  *src = nullptr;
  if (r >= W) return 0;
  const long long c_lo = pl.out_off[p][r], c_hi = pl.out_off[p][r + 1];
  const long long x = lo > c_lo ? lo : c_lo, y = hi < c_hi ? hi : c_hi;
  if (x >= y) return 0;
  *a = x;
  *src = P.in[r] + pl.in_off[r][p] + (x - c_lo);
  return y - x;
}

// ------------------------------------------------------- memory helpers --
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ unsigned char lds8(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
  return (unsigned char)v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Bytes [s, s + 16) of the 32-byte little-endian concatenation a:b, where
// s = 4*Q + r8/8.
template <int Q>
__device__ __forceinline__ uint4 extract16(const uint4& a, const uint4& b, unsigned r8) {
  const unsigned w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint4 o;
  o.x = __funnelshift_r(w[Q + 0], w[Q + 1], r8);
  o.y = __funnelshift_r(w[Q + 1], w[Q + 2], r8);
  o.z = __funnelshift_r(w[Q + 2], w[Q + 3], r8);
  o.w = __funnelshift_r(w[Q + 3], w[Q + 4], r8);
  return o;
}

// ------------------------------------------------------------ mbarriers --
__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait for phase `parity` of the mbarrier; false after ~1 s.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, unsigned parity) {
  const long long start = clock64();
  for (;;) {
    unsigned done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if (clock64() - start > kWaitCycles) return false;
  }
}

// Every lane of the warp waits (so each one observes the phase, and the data
// it guards); the warp agrees on the outcome, so a timeout is warp-uniform.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, unsigned parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(kFull, ok) != 0;
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

__device__ __forceinline__ void bulk_load(uint32_t dst_smem, const void* src, unsigned bytes,
                                          uint32_t bar) {
  if (A2AV_L2_HINT & 1) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst_smem),
        "l"(src), "r"(bytes), "r"(bar), "l"(evict_first_policy())
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst_smem),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
  }
}

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src_smem, unsigned bytes) {
  if (A2AV_L2_HINT & 2) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::
                     "l"(dst),
                 "r"(src_smem), "r"(bytes), "l"(evict_first_policy())
                 : "memory");
  } else {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(src_smem), "r"(bytes)
                 : "memory");
  }
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------- vector --
// nv 16-byte vectors, source and destination both 16-byte aligned.
template <int NT, int U>
__device__ __forceinline__ void copy_aligned(uint4* dst, const uint4* src, long long nv, int tid) {
  for (long long base = 0; base < nv; base += (long long)NT * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = base + (long long)u * NT + tid;
      if (i < nv) v[u] = ld_stream(src + i);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = base + (long long)u * NT + tid;
      if (i < nv) st_stream(dst + i, v[u]);
    }
  }
}

// nv destination-aligned vectors whose source starts 4*Q + r8/8 bytes
// (1..15) past the aligned granule `src`: vector i is built from source
// granules i and i + 1.  A warp owns 32*U consecutive vectors per pass, lane
// l of step u holding vector 32*u + l, so granule i + 1 is the next lane's
// granule i, or for lane 31 lane 0's granule of step u + 1: one rotated
// shuffle per step delivers both.  Only lane 31 of the last step and the
// last vector of the span load their second granule themselves.
template <int NT, int U, int Q>
__device__ __forceinline__ void copy_shifted(uint4* dst, const uint4* src, long long nv,
                                             unsigned r8, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  for (long long base = 0; base < nv; base += (long long)NT * U) {
    const long long wbase = base + (long long)warp * 32 * U + lane;
    uint4 a[U];
    uint4 extra = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = wbase + 32 * u;
      a[u] = make_uint4(0, 0, 0, 0);
      if (i < nv) {
        a[u] = ld_stream(src + i);
        if (i == nv - 1 || (lane == 31 && u == U - 1)) extra = ld_stream(src + i + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = wbase + 32 * u;
      const uint4 give = (u + 1 < U && lane == 0) ? a[u + 1 < U ? u + 1 : u] : a[u];
      uint4 n;
      n.x = __shfl_sync(kFull, give.x, lane + 1);
      n.y = __shfl_sync(kFull, give.y, lane + 1);
      n.z = __shfl_sync(kFull, give.z, lane + 1);
      n.w = __shfl_sync(kFull, give.w, lane + 1);
      if (i < nv) {
        const bool own = i == nv - 1 || (lane == 31 && u == U - 1);
        st_stream(dst + i, extract16<Q>(a[u], own ? extra : n, r8));
      }
    }
  }
}

// n bytes from s to d, any alignment, by all NT threads of the CTA.
template <int NT, int U, int US>
__device__ __forceinline__ void copy_span(unsigned char* d, const unsigned char* s, long long n,
                                          int tid) {
  long long head = (16 - (long long)((uintptr_t)d & 15)) & 15;
  if (head > n) head = n;
  if (tid < head) d[tid] = __ldg(s + tid);
  d += head;
  s += head;
  n -= head;
  const long long nv = n >> 4;
  const int tail = (int)(n & 15);
  if (tid < tail) d[nv * 16 + tid] = __ldg(s + nv * 16 + tid);
  if (nv == 0) return;
  uint4* dv = reinterpret_cast<uint4*>(d);
  const unsigned shift = (unsigned)((uintptr_t)s & 15);
  if (shift == 0) {
    copy_aligned<NT, U>(dv, reinterpret_cast<const uint4*>(s), nv, tid);
    return;
  }
  const uint4* sa = reinterpret_cast<const uint4*>(s - shift);
  const unsigned r8 = (shift & 3) * 8;
  switch (shift >> 2) {
    case 0: copy_shifted<NT, US, 0>(dv, sa, nv, r8, tid); break;
    case 1: copy_shifted<NT, US, 1>(dv, sa, nv, r8, tid); break;
    case 2: copy_shifted<NT, US, 2>(dv, sa, nv, r8, tid); break;
    default: copy_shifted<NT, US, 3>(dv, sa, nv, r8, tid); break;
  }
}

template <int NT, int U, int US>
__global__ void __launch_bounds__(NT, kVecCtasPerSm)
    a2av_vector_kernel(const __grid_constant__ Params P, long long max_tile) {
  __shared__ Plan pl;
  if (!build_plan(P, pl, max_tile)) return;
  const int W = P.W, tid = threadIdx.x;
  const long long ntiles = pl.tile_first[W];
  for (long long t = blockIdx.x; t < ntiles; t += gridDim.x) {
    long long lo, hi;
    const int p = tile_peer(pl, W, t, &lo, &hi);
    unsigned char* out = P.out[p];
    for (int r = 0; r < W; ++r) {
      const long long c_lo = pl.out_off[p][r], c_hi = pl.out_off[p][r + 1];
      const long long a = lo > c_lo ? lo : c_lo, b = hi < c_hi ? hi : c_hi;
      if (a >= b) continue;
      const unsigned char* src = P.in[r] + pl.in_off[r][p] + (a - c_lo);
      copy_span<NT, U, US>(out + a, src, b - a, tid);
    }
  }
}

// ------------------------------------------------------------------ bulk --
// Every tile's source segments, destination and size are 16-byte aligned.
// Warp 0 does all the work: each tile is loaded by the lanes of the sources
// it overlaps (lane r, source r) into one stage, and stored by lane 0 in one
// piece, which tracks its own bulk stores.
template <int NS, int LEAD>
__global__ void __launch_bounds__(kBulkThreads)
    a2av_bulk_kernel(const __grid_constant__ Params P, int stage_bytes) {
  static_assert(LEAD >= 1 && LEAD < NS, "loads run 1..NS-1 tiles ahead of stores");
  __shared__ Plan pl;
  __shared__ alignas(8) unsigned long long bars[NS];
  __shared__ unsigned char* stage_dst[NS];
  __shared__ unsigned stage_len[NS];
  extern __shared__ __align__(128) unsigned char stages[];
  if (!build_plan(P, pl, stage_bytes)) return;
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) != 0) return;

  const int W = P.W;
  const long long ntiles = pl.tile_first[W], G = gridDim.x, b0 = blockIdx.x;
  const long long nk = ntiles > b0 ? (ntiles - b0 + G - 1) / G : 0;
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
      const int p = tile_peer_warp(pl, W, b0 + k * G, lane, &lo, &hi);
      const long long n = lane_segment(P, pl, W, p, lane, lo, hi, &a, &src);
      const uint32_t bar = bar0 + 8 * s, stage = stage0 + (uint32_t)s * stage_bytes;
      if (lane == 0) {
        stage_dst[s] = P.out[p] + lo;
        stage_len[s] = (unsigned)(hi - lo);
        mbar_expect_tx(bar, (unsigned)(hi - lo));
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
__global__ void __launch_bounds__(32 * (NC + 1))
    a2av_staged_kernel(const __grid_constant__ Params P, int stage_bytes) {
  __shared__ Plan pl;
  __shared__ StageDesc desc[NS];
  __shared__ alignas(8) unsigned long long full[NS];
  __shared__ alignas(8) unsigned long long empty[NS];
  extern __shared__ __align__(128) unsigned char stages[];
  if (!build_plan(P, pl, stage_bytes)) return;

  const int W = P.W, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long ntiles = pl.tile_first[W], G = gridDim.x, b0 = blockIdx.x;
  const long long nk = ntiles > b0 ? (ntiles - b0 + G - 1) / G : 0;
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
    for (long long k = 0; k < nk; ++k) {
      const int s = (int)(k % NS);
      if (k >= NS && !mbar_wait_warp(empty0 + 8 * s, (unsigned)((k / NS - 1) & 1))) {
        if (lane == 0) record_error(P.status, A2AV_ERR_TIMEOUT);
        break;
      }
      long long lo, hi, a;
      const unsigned char* src;
      const int p = tile_peer_warp(pl, W, b0 + k * G, lane, &lo, &hi);
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
      if (lane == 0) mbar_expect_tx(bar, total);
      __syncwarp();
      if (n > 0) bulk_load(stage0 + (uint32_t)s * alloc + off, (const void*)g_lo, gb, bar);
    }
    return;
  }

  // Consumers: rebuild each tile from its stage with destination-aligned stores.
  const int ct = threadIdx.x - 32;
  for (long long k = 0; k < nk; ++k) {
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
      copy_span_smem<32 * NC>(dst + d.seg_dst[i], stage + (uint32_t)d.seg_src[i], d.seg_len[i], ct);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
}

}  // namespace

// ================================================================ host ABI ==
struct a2av_handle {
  int W;
  long long in_cap, out_cap;
  int device;
  int sms;
  int* d_status;
  int path;         // a2av_path_t
  int ctas_per_sm;  // 0 = engine default
  int last_path, last_grid, last_block;
};

namespace {

using BulkKernel = void (*)(Params, int);
const BulkKernel kBulk = a2av_bulk_kernel<kBulkStages, kBulkLead>;
const BulkKernel kStaged = a2av_staged_kernel<kStagedStages, kStagedConsumerWarps>;
using VecKernel = void (*)(Params, long long);
const VecKernel kVec = a2av_vector_kernel<kVecThreads, kVecUnroll, kVecShiftUnroll>;

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
  return A2AV_OK;
}

// Fill the kernel parameters; returns whether every row and buffer is
// 16-byte aligned (the bulk engine's precondition).
bool fill_params(Params* P, int W, const void* const* in_ptrs, const int64_t* in_splits_dev,
                 void* const* out_ptrs, int64_t* out_splits_offsets_dev, int64_t row_bytes,
                 long long in_cap, long long out_cap, int* status, long long split_stride) {
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
  P->in_cap = in_cap;
  P->out_cap = out_cap;
  P->W = W;
  return aligned;
}

// Engine actually used for a request: BULK needs full alignment (else STAGED);
// AUTO is BULK when aligned, STAGED otherwise.
int resolve_path(int requested, bool aligned) {
  if (requested == A2AV_PATH_VECTOR || requested == A2AV_PATH_STAGED) return requested;
  return aligned ? A2AV_PATH_BULK : A2AV_PATH_STAGED;
}

int launch(const Params& P, int path, int ctas_per_sm, int sms, cudaStream_t s, int* grid,
           int* block) {
  if (path == A2AV_PATH_BULK) {
    *grid = sms * (ctas_per_sm ? ctas_per_sm : kBulkCtasPerSm);
    *block = kBulkThreads;
    kBulk<<<*grid, *block, kBulkStages * kBulkStageBytes, s>>>(P, kBulkStageBytes);
  } else if (path == A2AV_PATH_STAGED) {
    *grid = sms * (ctas_per_sm ? ctas_per_sm : kStagedCtasPerSm);
    *block = kStagedThreads;
    kStaged<<<*grid, *block, kStagedStages * kStagedAlloc, s>>>(P, kStagedStageBytes);
  } else {
    *grid = sms * (ctas_per_sm ? ctas_per_sm : kVecCtasPerSm);
    *block = kVecThreads;
    kVec<<<*grid, *block, 0, s>>>(P, kVecMaxTile);
  }
  return cudaGetLastError() == cudaSuccess ? A2AV_OK : A2AV_ERR_CUDA;
}

}  // namespace

extern "C" {

int a2av_version(void) { return 10100; }

const char* a2av_error_string(int code) {
  switch (code) {
    case A2AV_OK: return "ok";
    case A2AV_ERR_INVALID_ARG: return "invalid argument";
    case A2AV_ERR_UNSUPPORTED: return "unsupported (world size above A2AV_MAX_RANKS)";
    case A2AV_ERR_CUDA: return "CUDA runtime error";
    case A2AV_ERR_BAD_SPLITS: return "invalid split matrix (detected on the device)";
    case A2AV_ERR_TIMEOUT: return "a bounded device wait timed out";
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
  h->last_path = h->last_grid = h->last_block = 0;
  *out = h;
  return A2AV_OK;
}

int a2av_set_path(a2av_handle* h, int path) {
  if (h == nullptr || path < A2AV_PATH_AUTO || path > A2AV_PATH_STAGED) return A2AV_ERR_INVALID_ARG;
  h->path = path;
  return A2AV_OK;
}

int a2av_set_grid(a2av_handle* h, int ctas_per_sm) {
  if (h == nullptr || ctas_per_sm < 0 || ctas_per_sm > 32) return A2AV_ERR_INVALID_ARG;
  h->ctas_per_sm = ctas_per_sm;
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
                                   h->d_status, split_stride);
  const int path = resolve_path(h->path, aligned);
  int grid = 0, block = 0;
  const int rc = launch(P, path, h->ctas_per_sm, h->sms, static_cast<cudaStream_t>(stream),
                        &grid, &block);
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
  rc = launch(P, resolve_path(A2AV_PATH_AUTO, aligned), 0, sms, s, &grid, &block);
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
