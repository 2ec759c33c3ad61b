// a2av_device.cuh -- device code shared by the exchange (a2av.cu) and the
// fused dispatch (dispatch.cu): the per-CTA plan built from the split matrix
// (warp-shuffle scans, validation, tiling), memory and mbarrier helpers, and
// the register-path span copy.  Everything has internal linkage; each
// translation unit gets its own copy.
#pragma once

#include "a2av.h"

#include <cuda_runtime.h>

#include <cstdint>

#ifndef A2AV_TILES_PER_CTA
#define A2AV_TILES_PER_CTA 2
#endif
// L2 eviction hints of the bulk engine: bit 0 marks loaded lines
// evict-first, bit 1 stored lines (each byte is used exactly once; marking
// the stored lines measured best).
#ifndef A2AV_L2_HINT
#define A2AV_L2_HINT 2
#endif

namespace {

constexpr int kMaxW = A2AV_MAX_RANKS;
constexpr long long kMaxBytes = 1LL << 62;  // byte offsets stay below 2^62
constexpr unsigned kFull = 0xffffffffu;
constexpr long long kTileGranule = 4096;         // tile sizes are multiples of this
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at GB300 clocks

}  // namespace

namespace {

// Tiles each CTA gets at least, when the payload allows (smaller tiles for
// small payloads keep more of them in flight per CTA).
constexpr long long kTilesPerCta = A2AV_TILES_PER_CTA;

struct Params {
  const unsigned char* in[kMaxW];
  unsigned char* out[kMaxW];
  const long long* splits;  // S[r][p] at splits[r * split_stride + p]
  long long split_stride;   // W for a2av_run; 2W when the splits are a previous
                            // exchange's out_splits_offsets (a2av_combine)
  long long* out_so;        // [W][2][W]
  int* status;
  long long rb;             // row bytes
  long long limit;          // largest valid split: 2^62 / (W * rb), computed on the host
  long long in_cap;         // rows, 0 = unchecked
  long long out_cap;        // rows, 0 = unchecked
  int W;
  int starve;               // test hook: 1 -- CTA 0 arms its first stage for 16 bytes too
                            // many; 2 -- grid barriers wait for one CTA more than the grid
};

// Host side of Params::limit: every byte offset then stays below 2^62.
inline long long split_limit(int W, long long rb) { return kMaxBytes / ((long long)W * rb); }

// Host: launch with programmatic stream serialization when `pdl` is set, so
// that the kernel's CTAs may be scheduled while the previous kernel on the
// stream is still running (its griddepcontrol.wait keeps the data order).
template <typename... Args, typename... Vals>
cudaError_t launch_kernel(void (*kernel)(Args...), dim3 grid, int block, size_t smem,
                          cudaStream_t s, bool pdl, Vals... vals) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, vals...);
}

// Per-CTA plan in shared memory.  Offsets are in ROWS; callers multiply by the
// row size where they need bytes.  Tiles are a power of two bytes long.
// Rows are padded to kMaxW + 1 entries so that lanes reading a column (lane
// r at [r][k]) hit 32 different shared-memory banks.
struct Plan {
  long long s[kMaxW][kMaxW + 1];        // S[r][p] as loaded
  long long out_off[kMaxW][kMaxW + 1];  // [p][r] = sum_{q<r} S[q][p]; [p][W] = rows p receives
  long long in_off[kMaxW][kMaxW + 1];   // [r][p] = sum_{q<p} S[r][q]
  long long tile_first[kMaxW + 1];      // first tile of peer p; [W] = number of tiles
  int tile_shift;                       // tile size = 1 << tile_shift bytes
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

// Ranks for which one warp builds the whole plan (below).
constexpr int kWarpPlanRanks = 8;

// Steps 2 and 3 of the plan for W <= kWarpPlanRanks, by warp 0 alone once it
// sees a range-checked pl.s: lane j scans column j (out_off[j][*]) and row j
// (in_off[j][*]) in shared memory and checks peer j's and rank j's
// capacities; then the tiles and CTA 0's out_splits_offsets.  Returns true
// (warp-uniform) when a capacity or NULL-buffer rule is broken.  No block
// barrier: the caller publishes the plan with one.
__device__ __forceinline__ bool plan_one_warp(const Params& P, Plan& pl, long long max_tile, int cta,
                                              int ctas, int lane) {
  const int W = P.W;
  int bad = 0;
  long long col = 0, row = 0;
  if (lane < W) {
    for (int r = 0; r < W; ++r) {
      pl.out_off[lane][r] = col;
      col += pl.s[r][lane];
    }
    pl.out_off[lane][W] = col;
    for (int p = 0; p < W; ++p) {
      pl.in_off[lane][p] = row;
      row += pl.s[lane][p];
    }
    if ((P.out_cap > 0 && col > P.out_cap) || (P.out[lane] == nullptr && col > 0)) bad = 1;
    if ((P.in_cap > 0 && row > P.in_cap) || (P.in[lane] == nullptr && row > 0)) bad = 1;
  }
  if (__any_sync(kFull, bad)) return true;
  // tiles, as in plan_from_splits
  const long long bytes = lane < W ? col * P.rb : 0;
  const long long total = __shfl_sync(kFull, warp_inclusive_scan(bytes, lane), 31);
  const long long slots = kTilesPerCta * (long long)ctas;
  const long long per_cta = (total + slots - 1) / slots;
  int shift = per_cta > 1 ? 64 - __clzll(per_cta - 1) : 0;
  const int lo_shift = 63 - __clzll(kTileGranule), hi_shift = 63 - __clzll(max_tile);
  shift = shift < lo_shift ? lo_shift : (shift > hi_shift ? hi_shift : shift);
  const long long n = (bytes + (1LL << shift) - 1) >> shift;
  const long long inc = warp_inclusive_scan(n, lane);
  if (lane < W) pl.tile_first[lane] = inc - n;
  if (lane == 31) {
    pl.tile_first[W] = inc;
    pl.tile_shift = shift;
  }
  __syncwarp();
  if (cta == 0) {
    for (int e = lane; e < W * W; e += 32) {
      const int p = e / W, r = e - p * W;
      long long* so = P.out_so + (long long)p * 2 * W;
      so[r] = pl.s[r][p];
      so[W + r] = pl.out_off[p][r];
    }
  }
  return false;
}

// Steps 2 and 3 of the plan, once pl.s holds a range-checked split matrix:
// column scans (out_off) and row scans (in_off) side by side + capacity
// checks; tiles and out_splits_offsets.  Two barriers.  Returns false (in
// every thread of the CTA) when a capacity or NULL-buffer rule is broken;
// CTA 0 then records A2AV_ERR_BAD_SPLITS.
__device__ bool plan_from_splits(const Params& P, Plan& pl, long long max_tile, int cta, int ctas) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
  const int W = P.W;
  if (W <= kWarpPlanRanks) {  // one warp, one barrier
    __shared__ int plan_bad;
    if (warp == 0) {
      const bool b = plan_one_warp(P, pl, max_tile, cta, ctas, lane);
      if (lane == 0) {
        plan_bad = b;
        if (b && cta == 0) record_error(P.status, A2AV_ERR_BAD_SPLITS);
      }
    }
    __syncthreads();
    return !plan_bad;
  }
  int bad = 0;

  // Task k < W: column scan of peer k (lane r holds S[r][k]); task W + k: row
  // scan of rank k (lane p holds S[k][p]).  Exclusive prefix = inclusive - own.
  for (int task = warp; task < 2 * W; task += nwarps) {
    const bool column = task < W;
    const int k = column ? task : task - W;
    const long long x = lane < W ? (column ? pl.s[lane][k] : pl.s[k][lane]) : 0;
    const long long inc = warp_inclusive_scan(x, lane);
    if (column) {
      if (lane < W) pl.out_off[k][lane] = inc - x;
      if (lane == 31) {
        pl.out_off[k][W] = inc;
        if ((P.out_cap > 0 && inc > P.out_cap) || (P.out[k] == nullptr && inc > 0)) bad = 1;
      }
    } else {
      if (lane < W) pl.in_off[k][lane] = inc - x;
      if (lane == 31 && ((P.in_cap > 0 && inc > P.in_cap) || (P.in[k] == nullptr && inc > 0)))
        bad = 1;
    }
  }
  if (__syncthreads_or(bad)) {
    if (cta == 0 && tid == 0) record_error(P.status, A2AV_ERR_BAD_SPLITS);
    return false;
  }

  // Tiles: the smallest power of two (>= 4 KiB, <= max_tile, itself a power
  // of two) that gives every CTA about kTilesPerCta tiles; peer p's received
  // stream is cut into ceil(bytes / tile) of them.
  if (warp == 0) {
    const long long bytes = lane < W ? pl.out_off[lane][W] * P.rb : 0;
    const long long total = __shfl_sync(kFull, warp_inclusive_scan(bytes, lane), 31);
    const long long slots = kTilesPerCta * (long long)ctas;
    const long long per_cta = (total + slots - 1) / slots;
    int shift = per_cta > 1 ? 64 - __clzll(per_cta - 1) : 0;  // ceil(log2(per_cta))
    const int lo_shift = 63 - __clzll(kTileGranule), hi_shift = 63 - __clzll(max_tile);
    shift = shift < lo_shift ? lo_shift : (shift > hi_shift ? hi_shift : shift);
    const long long n = (bytes + (1LL << shift) - 1) >> shift;
    const long long inc = warp_inclusive_scan(n, lane);
    if (lane < W) pl.tile_first[lane] = inc - n;
    if (lane == 31) {
      pl.tile_first[W] = inc;
      pl.tile_shift = shift;
    }
  }
  if (cta == 0) {
    for (int e = tid; e < W * W; e += nt) {
      const int p = e / W, r = e - p * W;
      long long* so = P.out_so + (long long)p * 2 * W;
      so[r] = pl.s[r][p];
      so[W + r] = pl.out_off[p][r];
    }
  }
  __syncthreads();
  return true;
}

// Step 1 of the exchange, then the rest of the plan: load the split matrix
// into shared memory and check its range (one barrier), then
// plan_from_splits; for at most kWarpPlanRanks ranks warp 0 does all of it
// and one barrier publishes the plan (measured on a cold 0.5 MiB exchange:
// the three-barrier plan took ~1.3 us of CTA 0's time).  `ctas` CTAs work on this exchange and this one is
// number `cta` among them (the whole grid, unless several exchanges share a
// launch).  Returns false (in every thread of the CTA) when the splits are
// invalid; CTA 0 then records A2AV_ERR_BAD_SPLITS.
__device__ bool build_plan(const Params& P, Plan& pl, long long max_tile, int cta, int ctas) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int W = P.W;

  // Programmatic dependent launch (both no-ops for a plain launch): let the
  // next kernel of the stream start launching, then wait until the previous
  // one has finished and its writes are visible -- it may have produced the
  // splits or the inputs, and it may still be reading our outputs.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (W <= kWarpPlanRanks) {
    // Few ranks: warp 0 loads the split matrix (at most two entries a lane),
    // checks it and builds the whole plan; one block barrier publishes it.
    __shared__ int plan_bad;
    if ((tid >> 5) == 0) {
      const int lane = tid & 31;
      int bad = 0;
      long long v[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int e = lane + 32 * q;
        v[q] = e < W * W ? __ldcg(P.splits + (long long)(e / W) * P.split_stride + e % W) : 0;
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int e = lane + 32 * q;
        if (e < W * W) {
          if (v[q] < 0 || v[q] > P.limit) bad = 1;
          pl.s[e / W][e % W] = v[q];
        }
      }
      bool b = __any_sync(kFull, bad) != 0;
      __syncwarp();
      if (!b) b = plan_one_warp(P, pl, max_tile, cta, ctas, lane);
      if (lane == 0) {
        plan_bad = b;
        if (b && cta == 0) record_error(P.status, A2AV_ERR_BAD_SPLITS);
      }
    }
    __syncthreads();
    return !plan_bad;
  }
  int bad = 0;
  for (int e = tid; e < W * W; e += nt) {
    const int r = e / W, p = e - r * W;
    // (L2 loads: the splits may have been written during this very launch
    // by other CTAs, as in the fused dispatch's scan kernel)
    const long long s = __ldcg(P.splits + (long long)r * P.split_stride + p);
    if (s < 0 || s > P.limit) bad = 1;
    pl.s[r][p] = s;
  }
  if (__syncthreads_or(bad)) {
    if (cta == 0 && tid == 0) record_error(P.status, A2AV_ERR_BAD_SPLITS);
    return false;
  }
  return plan_from_splits(P, pl, max_tile, cta, ctas);
}

// The whole grid on one exchange.
__device__ __forceinline__ bool build_plan(const Params& P, Plan& pl, long long max_tile) {
  return build_plan(P, pl, max_tile, blockIdx.x, gridDim.x);
}

// Tile t -> peer p and the byte range [lo, hi) of out[p] it covers (all
// threads of the caller compute the same).
__device__ __forceinline__ int tile_peer(const Plan& pl, int W, long long t, long long rb,
                                         long long* lo, long long* hi) {
  int p = 0;
  while (p + 1 < W && pl.tile_first[p + 1] <= t) ++p;
  const long long bytes = pl.out_off[p][W] * rb;
  *lo = (t - pl.tile_first[p]) << pl.tile_shift;
  const long long end = *lo + (1LL << pl.tile_shift);
  *hi = end < bytes ? end : bytes;
  return p;
}

// The same for a whole warp at once: the largest p with tile_first[p] <= t
// (peers without tiles share their successor's tile_first, so the largest
// such p is the one that owns tile t).
__device__ __forceinline__ int tile_peer_warp(const Plan& pl, int W, long long t, long long rb,
                                              int lane, long long* lo, long long* hi) {
  const unsigned m = __ballot_sync(kFull, lane < W && pl.tile_first[lane] <= t);
  const int p = 31 - __clz(m);
  const long long bytes = pl.out_off[p][W] * rb;
  *lo = (t - pl.tile_first[p]) << pl.tile_shift;
  const long long end = *lo + (1LL << pl.tile_shift);
  *hi = end < bytes ? end : bytes;
  return p;
}

// Source r's part of the byte range [lo, hi) of peer p's output: the
// destination offset a, the byte count (0 when source r contributes nothing)
// and the source address.
__device__ __forceinline__ long long lane_segment(const Params& P, const Plan& pl, int W, int p,
                                                  int r, long long lo, long long hi, long long* a,
                                                  const unsigned char** src) {
  *a = 0;
  *src = nullptr;
  if (r >= W) return 0;
  const long long rb = P.rb;
  const long long c_lo = pl.out_off[p][r] * rb, c_hi = pl.out_off[p][r + 1] * rb;
  const long long x = lo > c_lo ? lo : c_lo, y = hi < c_hi ? hi : c_hi;
  if (x >= y) return 0;
  *a = x;
  *src = P.in[r] + pl.in_off[r][p] * rb + (x - c_lo);
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

}  // namespace
