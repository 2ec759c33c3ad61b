// dispatch.cu -- fused dispatch preparation for the variable-size all-to-all:
// the exchange of rows that are not yet grouped by destination (declared in
// include/a2av.h, a2av_dispatch).
//
// Each rank's items carry a key (destination = key / K) and a source row.
// The exchange runs on the rank's items ordered stably by key -- the input
// a2av_run would expect -- without ever materialising that order:
//   1. count  (a warp per range of 256 items, eight per CTA): per range, the
//      key histogram in shared memory; keys and source rows are validated here.
//   2. scan   (grid keys x W, 256 threads): per (key, rank), the exclusive
//      prefix of the key's count over the ranges (in place); the last CTA of
//      each rank to finish turns the key totals into key start offsets and
//      the split matrix row S[r][*].
//   3. rank   (grid ranges x W, one warp): items of a range in order, 32 at a
//      time; __match_any_sync groups equal keys, a lane's rank among them
//      plus the running count of its key gives its stable position (kept in
//      the workspace).
//   When every rank has at most 2048 items and there are at most 256 keys,
//   one kernel (one CTA per rank, a warp per 256 items) does 1-3 instead.
//   Rows shorter than 64 bytes (not that small): the rank kernel also does
//   the exchange's prologue for its own rank (every CTA validates the whole
//   split matrix, as the a2av prologue does, and derives its rank's row
//   displacement per peer) and copies every item's row as soon as it knows
//   its position: rank + copy in one kernel, step 4 below not launched.
//   4. copy   (grid SMs x 4): build the exchange plan from S (the a2av
//      prologue, which also checks capacities and NULL buffers), publish the
//      positions and the split matrix, then gather every item's row straight
//      into its place in the output of its destination: with cp.async.bulk
//      through shared memory for 16-byte aligned rows of 2..32 KiB, else 32
//      rows per warp (flat 16-byte vector runs when aligned) for rows of 64
//      bytes or more and a thread per row below.
// Invalid keys or source rows set a workspace flag (cleared first) that stops
// every later kernel; invalid splits stop the copy kernel in its prologue.
// Either way nothing the caller owns is written.
#include "a2av_device.cuh"
#include "a2av_handle.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

namespace {

constexpr int kRange = 256;                       // items per histogram range
constexpr int kMaxBins = A2AV_MAX_DISPATCH_KEYS;  // W * K at most
constexpr int kScanThreads = 256;
constexpr int kScanBatch = 16;  // counts a scan thread loads at once
static_assert(kMaxBins <= 4 * kScanThreads, "the finishing scan CTA holds 4 keys per thread");
constexpr int kCopyThreads = 256;
constexpr int kCopyCtasPerSm = 4;
#ifndef A2AV_COPY_WARP_ROWS_CTAS_PER_SM
#define A2AV_COPY_WARP_ROWS_CTAS_PER_SM 3  // the vector runs want up to 85 registers
#endif
constexpr int kCopyCtasPerSmWarpRows = A2AV_COPY_WARP_ROWS_CTAS_PER_SM;
constexpr long long kWarpRowBytes = 64;  // rows this long get a warp each
constexpr int kItemsPerThread = 4;      // items a thread copies at once (short rows)
#ifndef A2AV_COPY_VEC_ROWS
#define A2AV_COPY_VEC_ROWS 4
#endif
constexpr int kVecRows = A2AV_COPY_VEC_ROWS;  // 16-byte vectors a lane keeps in flight (warp rows)
// The combine's aligned warp rows: twice the vectors in flight at two CTAs an
// SM (123 registers, no spill).  Measured on MoE rows of 512 B and 1 KiB: the
// combine 5-9 % faster than at 4 vectors and three CTAs; the dispatch, which
// reads each token's row once for its two experts, no faster; rows that need
// realigning 7-20 % slower at two CTAs.
constexpr int kVecRowsWide = 8;
constexpr int kCopyCtasPerSmWide = 2;
constexpr long long kVecMaxRow = 64 * 1024;  // flat vector runs up to this row size

struct DispatchParams {
  const int* key[kMaxW];
  const int* src[kMaxW];
  long long* sorted_pos[kMaxW];
  long long items[kMaxW];           // m_r
  long long rows[kMaxW];            // source rows per rank
  long long item_first[kMaxW + 1];  // exclusive prefix of m_r
  int* flag;                        // workspace: set once input is found invalid
  int* done;                        // workspace: [W] CTAs finished per rank (the one that scans)
  long long* S;                     // workspace: [W][W]
  long long* key_start;             // workspace: [W][NB]
  long long* key_total;             // workspace: [W][NB]
  int* hist;                        // workspace: [W][ranges_max][NB]
  int* grp;                         // workspace: [W][groups_max][NB]
  int* pos;                         // workspace: [W][pos_stride] item positions in key order
  int* status;
  long long* in_splits_out;         // optional [W][W]
  int vec16;                        // every row and buffer 16-byte aligned
  int combine;                      // the fused combine: rows move the other way (below)
  long long ranges_max;
  long long groups_max;             // ranges_max / kCountWarps, rounded up
  int fuse_scan;                    // the count kernel's last CTA per rank scans the groups
  long long pos_stride;
  int W, K;
};

// Programmatic dependent launch: a kernel of the chain launched with the
// programmatic-serialization attribute may start while its predecessor runs;
// it waits here before reading anything the predecessor wrote (a no-op when
// the launch had no such dependency).  A predecessor lets its successor's
// CTAs start launching once its own CTAs have begun.
__device__ __forceinline__ void chain_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void chain_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ bool flagged(const DispatchParams& D) {
  return *reinterpret_cast<volatile int*>(D.flag) != 0;
}

__device__ __forceinline__ void fail(const DispatchParams& D, int code) {
  atomicExch(D.flag, 1);
  record_error(D.status, code);
}

// Block-wide exclusive scan of one value per thread (kScanThreads threads);
// returns the exclusive prefix, *total gets the sum.  `warp_sums` holds
// kScanThreads / 32 entries.
__device__ __forceinline__ long long block_exclusive_scan(long long x, long long* warp_sums,
                                                          long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long inc = warp_inclusive_scan(x, lane);
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  long long base = 0, all = 0;
  for (int w = 0; w < kScanThreads / 32; ++w) {
    if (w < warp) base += warp_sums[w];
    all += warp_sums[w];
  }
  *total = all;
  __syncthreads();
  return base + inc - x;
}

// Rank r's key totals (tot[b], in shared memory, NB <= kScanThreads) become
// key_total[r][*], key_start[r][*] (items with a smaller key) and S[r][p]
// (items with key / K = p).  Every thread of the CTA calls it.
__device__ __forceinline__ void finish_rank(const DispatchParams& D, int r, const long long* tot,
                                            long long* warp_sums) {
  const int t = threadIdx.x, NB = D.W * D.K;
  const long long x = t < NB ? tot[t] : 0;
  long long all;
  const long long start = block_exclusive_scan(x, warp_sums, &all);
  if (t < NB) {
    D.key_total[(long long)r * NB + t] = x;
    D.key_start[(long long)r * NB + t] = start;
  }
  if (t < D.W) {
    long long sum = 0;
    for (int k = 0; k < D.K; ++k) sum += tot[t * D.K + k];
    D.S[(long long)r * D.W + t] = sum;
  }
}

// Items are counted in ranges of kRange, ranges in groups of kCountWarps (a
// count CTA).  After the count kernel, hist[r][j][b] holds the items with key
// b in the earlier ranges of range j's group, and grp[r][c][b] the group's
// count; the scan (below) turns grp[r][*][b] into exclusive prefixes over the
// groups, so that an item's place among the equal keys of its rank is
// key_start[b] + grp[c][b] + hist[j][b] + its rank within the range.
//
// A warp per range of 256 items (8 per lane, all loads issued together),
// eight ranges per CTA, registers capped for six CTAs an SM so that 7296
// ranges (1.8 M items) are resident in one wave; each warp counts its keys in
// its own slice of shared memory (dynamic: 8 x W*K ints).  With D.fuse_scan
// (at most kFuseScanPer groups per thread and key) the last count CTA of each
// rank to finish does the scan itself and the scan kernel is not launched:
// one launch and one kernel boundary fewer (MoE dispatch of 8192 tokens).
constexpr int kCountWarps = 8;
constexpr int kGroupItems = kCountWarps * kRange;  // 2048
constexpr int kFuseScanPer = 4;                    // groups a thread scans in the fused scan
static_assert(32 * kCountWarps == kScanThreads, "a count CTA can run the block scan");

// The fused scan: one CTA (kScanThreads threads) over rank r's C groups.
// Thread t takes key b = t % NB and the slice g = t / NB of at most
// kFuseScanPer consecutive groups (G = kScanThreads / NB slices per key).
__device__ __forceinline__ void scan_groups_in_cta(const DispatchParams& D, int r, long long C) {
  const int t = threadIdx.x, NB = D.W * D.K, G = kScanThreads / NB;
  const int b = t % NB, g = t / NB;
  const long long per = (C + G - 1) / G;
  const long long c0 = g < G ? g * per : C, c1 = c0 + per < C ? c0 + per : C;
  int* A = D.grp + (long long)r * D.groups_max * NB + b;  // group c at A[c * NB]
  __shared__ long long part[kScanThreads];
  __shared__ long long tot[kScanThreads];
  __shared__ long long warp_sums[kScanThreads / 32];
  int v[kFuseScanPer];
  long long local = 0;
#pragma unroll
  for (int q = 0; q < kFuseScanPer; ++q) {
    v[q] = c0 + q < c1 ? __ldcg(A + (c0 + q) * NB) : 0;
    local += v[q];
  }
  part[t] = local;
  __syncthreads();
  long long base = 0, total = 0;
  if (g < G)
    for (int h = 0; h < G; ++h) {
      const long long x = part[h * NB + b];
      if (h < g) base += x;
      total += x;
    }
#pragma unroll
  for (int q = 0; q < kFuseScanPer; ++q) {
    if (c0 + q < c1) A[(c0 + q) * NB] = (int)base;
    base += v[q];
  }
  if (g == 0) tot[b] = total;
  __syncthreads();
  finish_rank(D, r, tot, warp_sums);
}

__global__ void __launch_bounds__(32 * kCountWarps, 6) dispatch_count_kernel(const __grid_constant__ DispatchParams D) {
  chain_release();
  chain_wait();
  const int r = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
  const long long c = blockIdx.x;
  const long long range = c * kCountWarps + warp;
  const long long i0 = range * kRange, m = D.items[r];
  const int NB = D.W * D.K;
  if (c * kGroupItems >= m) {  // no items in this CTA's ranges (uniform over the CTA)
    if (c == 0 && D.fuse_scan) {  // a rank without items: zero counts and splits
      __shared__ long long zero[kScanThreads];
      __shared__ long long zero_sums[kScanThreads / 32];
      zero[t] = 0;
      __syncthreads();
      finish_rank(D, r, zero, zero_sums);
    }
    return;
  }
  extern __shared__ int count_hist[];
  int* hist = count_hist + warp * NB;
  for (int b = lane; b < NB; b += 32) hist[b] = 0;
  if (i0 < m) {
    int keys[kRange / 32], srcs[kRange / 32];
#pragma unroll
    for (int q = 0; q < kRange / 32; ++q) {
      const long long i = i0 + q * 32 + lane;
      keys[q] = i < m ? D.key[r][i] : 0;
      srcs[q] = i < m ? D.src[r][i] : 0;
    }
    __syncwarp();
    int bad = 0;
#pragma unroll
    for (int q = 0; q < kRange / 32; ++q) {
      if (i0 + q * 32 + lane >= m) continue;
      if (keys[q] < 0 || keys[q] >= NB || srcs[q] < 0 || srcs[q] >= D.rows[r])
        bad = 1;
      else
        atomicAdd(&hist[keys[q]], 1);
    }
    if (__any_sync(kFull, bad) && lane == 0) fail(D, A2AV_ERR_BAD_INDEX);
  }
  __syncthreads();
  // in-group prefixes of the ranges that hold items, and the group's count
  const long long R = (m + kRange - 1) / kRange;
  for (int b = t; b < NB; b += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kCountWarps; ++w) {
      const long long j = c * kCountWarps + w;
      if (j < R) D.hist[((long long)r * D.ranges_max + j) * NB + b] = run;
      run += count_hist[w * NB + b];
    }
    D.grp[((long long)r * D.groups_max + c) * NB + b] = run;
  }
  if (!D.fuse_scan) return;
  // The rank's last CTA to finish (an atomic count, after a fence) scans.
  __shared__ int last;
  __threadfence();
  __syncthreads();
  const long long C = (m + kGroupItems - 1) / kGroupItems;
  if (t == 0) last = atomicAdd(&D.done[r], 1) == (int)(C - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  scan_groups_in_cta(D, r, C);
}

// CTA (b, r): key b of rank r.  grp[c][b] becomes the number of items with
// key b in groups < c (thread t scans a run of consecutive groups), and
// key_total[r][b] the key's count.  The last CTA of rank r to finish (an
// atomic count, after a fence) turns the totals into key_start[r][*] (items
// with a smaller key) and S[r][p] (items with key / K = p).
__global__ void __launch_bounds__(kScanThreads) dispatch_scan_kernel(const __grid_constant__ DispatchParams D) {
  chain_wait();
  chain_release();
  if (flagged(D)) return;
  const int b = blockIdx.x, r = blockIdx.y, NB = D.W * D.K, t = threadIdx.x;
  __shared__ long long warp_sums[kScanThreads / 32];
  __shared__ long long tot[kMaxBins];
  __shared__ int last;
  const long long C = (D.items[r] + kGroupItems - 1) / kGroupItems;
  int* H = D.grp + (long long)r * D.groups_max * NB + b;  // group j at H[j * NB]
  const long long per = (C + kScanThreads - 1) / kScanThreads;
  const long long j0 = t * per, j1 = j0 + per < C ? j0 + per : C;
  // A thread's first kScanBatch counts are loaded together and kept in
  // registers for the rewrite (runs longer than that are walked in batches).
  int first[kScanBatch];
  long long local = 0;
#pragma unroll
  for (int q = 0; q < kScanBatch; ++q) {
    first[q] = j0 + q < j1 ? H[(j0 + q) * NB] : 0;
    local += first[q];
  }
  for (long long base = j0 + kScanBatch; base < j1; base += kScanBatch) {
    int v[kScanBatch];
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q) v[q] = base + q < j1 ? H[(base + q) * NB] : 0;
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q) local += v[q];
  }
  long long total;
  long long run = block_exclusive_scan(local, warp_sums, &total);
#pragma unroll
  for (int q = 0; q < kScanBatch; ++q) {
    if (j0 + q < j1) H[(j0 + q) * NB] = (int)run;
    run += first[q];
  }
  for (long long base = j0 + kScanBatch; base < j1; base += kScanBatch) {
    int v[kScanBatch];
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q) v[q] = base + q < j1 ? H[(base + q) * NB] : 0;
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q) {
      if (base + q < j1) H[(base + q) * NB] = (int)run;
      run += v[q];
    }
  }
  if (t == 0) D.key_total[(long long)r * NB + b] = total;
  __threadfence();
  __syncthreads();
  if (t == 0) last = atomicAdd(&D.done[r], 1) == NB - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // key starts: thread t owns keys [4t, 4t + 4) (NB <= 4 * kScanThreads)
  long long v[4], sum = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int k = 4 * t + q;
    v[q] = k < NB ? __ldcg(D.key_total + (long long)r * NB + k) : 0;
    sum += v[q];
  }
  long long start = block_exclusive_scan(sum, warp_sums, &total);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int k = 4 * t + q;
    if (k < NB) {
      D.key_start[(long long)r * NB + k] = start;
      tot[k] = v[q];
    }
    start += v[q];
  }
  __syncthreads();
  if (t < D.W) {
    long long s = 0;
    for (int k = 0; k < D.K; ++k) s += tot[t * D.K + k];
    D.S[(long long)r * D.W + t] = s;
  }
}

__global__ void __launch_bounds__(32) dispatch_rank_kernel(const __grid_constant__ DispatchParams D) {
  chain_wait();
  chain_release();
  if (flagged(D)) return;
  const int r = blockIdx.y, lane = threadIdx.x, NB = D.W * D.K;
  const long long i0 = (long long)blockIdx.x * kRange, m = D.items[r];
  if (i0 >= m) return;
  __shared__ long long next[kMaxBins];  // next position of each key in this range
  const int* H = D.hist + ((long long)r * D.ranges_max + blockIdx.x) * NB;
  const int* A = D.grp + ((long long)r * D.groups_max + blockIdx.x / kCountWarps) * NB;
  for (int k = lane; k < NB; k += 32) next[k] = D.key_start[(long long)r * NB + k] + A[k] + H[k];
  __syncwarp();
  // All keys of the range are loaded at once (8 per lane), then ranked in order.
  int keys[kRange / 32];
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {
    const long long i = i0 + c * 32 + lane;
    keys[c] = i < m ? D.key[r][i] : -1 - lane;  // invalid lanes match nobody
  }
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {
    const long long i = i0 + c * 32 + lane;
    const bool valid = i < m;
    const int key = keys[c];
    const unsigned same = __match_any_sync(kFull, key);
    long long pos = 0;
    if (valid) pos = next[key] + __popc(same & ((1u << lane) - 1u));
    __syncwarp();
    if (valid && lane == 31 - __clz(same)) next[key] += __popc(same);
    __syncwarp();
    if (valid) D.pos[(long long)r * D.pos_stride + i] = (int)pos;
  }
}

// A row of n bytes, any alignment, copied by one thread.
__device__ __forceinline__ void copy_row_thread(unsigned char* d, const unsigned char* s,
                                                long long n) {
  const uintptr_t a = (uintptr_t)d | (uintptr_t)s | (uintptr_t)n;
  if ((a & 7) == 0) {
    for (long long k = 0; k < n; k += 8)
      *reinterpret_cast<unsigned long long*>(d + k) =
          __ldg(reinterpret_cast<const unsigned long long*>(s + k));
  } else if ((a & 3) == 0) {
    for (long long k = 0; k < n; k += 4)
      *reinterpret_cast<unsigned*>(d + k) = __ldg(reinterpret_cast<const unsigned*>(s + k));
  } else {
    for (long long k = 0; k < n; ++k) d[k] = __ldg(s + k);
  }
}

// Rank and copy (rows shorter than 64 bytes): the rank kernel's ranking,
// then each lane copies its items' rows straight to their place in the
// output of their destination and publishes their positions.  The plan was
// validated by the scan kernel, whose flag stops this kernel otherwise.  Two
// warps per CTA, a range each, registers capped so that a whole GPU of them
// is resident at once (the ranking is a serial chain per warp: more warps
// in flight, not more work per warp).
#ifndef A2AV_RANK_COPY_WARPS
#define A2AV_RANK_COPY_WARPS 2
#endif
#ifndef A2AV_RANK_COPY_MIN_CTAS
#define A2AV_RANK_COPY_MIN_CTAS 18
#endif
constexpr int kRankCopyWarps = A2AV_RANK_COPY_WARPS;

__global__ void __launch_bounds__(32 * kRankCopyWarps, A2AV_RANK_COPY_MIN_CTAS)
    dispatch_rank_copy_kernel(const __grid_constant__ Params P,
                              const __grid_constant__ DispatchParams D) {
  chain_wait();
  chain_release();
  if (flagged(D)) return;
  const int r = blockIdx.y, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int W = D.W, K = D.K, NB = W * K;
  const long long range = (long long)blockIdx.x * kRankCopyWarps + warp;
  const long long i0 = range * kRange, m = D.items[r];
  __shared__ int next_all[kRankCopyWarps][kMaxBins];  // next position of each key in the range
  __shared__ long long disp[kMaxW];  // out_off[p][r] - in_off[r][p], rows
  __shared__ int bad_splits;
  if (warp == 0) {
    // The a2av prologue's checks on the whole split matrix (identical in
    // every CTA, so all reach the same verdict): lane p owns column p and
    // row p.  S was completed by the scan kernel.
    const int p = lane;
    long long col = 0, above = 0, row = 0, own = 0;
    int bad = 0;
    if (p < W) {
      for (int q = 0; q < W; ++q) {
        const long long v = __ldcg(D.S + (long long)q * W + p);  // S[q][p]
        const long long h = __ldcg(D.S + (long long)p * W + q);  // S[p][q]
        if (v < 0 || v > P.limit || h < 0 || h > P.limit) bad = 1;
        if (q < r) above += v;
        if (q == r) own = v;
        col += v;
        row += h;
      }
      if ((P.out_cap > 0 && col > P.out_cap) || (P.out[p] == nullptr && col > 0)) bad = 1;
      if ((P.in_cap > 0 && row > P.in_cap) || (P.in[p] == nullptr && row > 0)) bad = 1;
    }
    const long long in_off = warp_inclusive_scan(own, lane) - own;  // in_off[r][p]
    if (p < W) disp[p] = above - in_off;
    bad = __any_sync(kFull, bad);
    if (lane == 0) bad_splits = bad;
    if (blockIdx.x == 0 && r == 0) {  // one CTA records the verdict and the offsets
      if (bad) {
        if (lane == 0) record_error(D.status, A2AV_ERR_BAD_SPLITS);
      } else if (p < W) {
        long long* so = P.out_so + (long long)p * 2 * W;
        long long run = 0;
        for (int q = 0; q < W; ++q) {
          const long long v = __ldcg(D.S + (long long)q * W + p);
          so[q] = v;
          so[W + q] = run;
          run += v;
          if (D.in_splits_out != nullptr) D.in_splits_out[(long long)q * W + p] = v;
        }
      }
    }
  }
  __syncthreads();
  if (bad_splits || i0 >= m) return;
  int* next = next_all[warp];
  const int* H = D.hist + ((long long)r * D.ranges_max + range) * NB;
  const int* A = D.grp + ((long long)r * D.groups_max + range / kCountWarps) * NB;
  for (int k = lane; k < NB; k += 32) next[k] = (int)D.key_start[(long long)r * NB + k] + A[k] + H[k];
  int keys[kRange / 32];
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {
    const long long i = i0 + c * 32 + lane;
    keys[c] = i < m ? D.key[r][i] : -1 - lane;  // invalid lanes match nobody
  }
  __syncwarp();
  int pos[kRange / 32];  // positions within the rank: below 2^31 items
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {
    const bool valid = i0 + c * 32 + lane < m;
    const int key = keys[c];
    const unsigned same = __match_any_sync(kFull, key);
    pos[c] = valid ? next[key] + __popc(same & ((1u << lane) - 1u)) : 0;
    __syncwarp();
    if (valid && lane == 31 - __clz(same)) next[key] += __popc(same);
    __syncwarp();
  }
  const long long rb = P.rb;
  int srcs[kRange / 32];  // loaded together, after the ranking (fewer live registers)
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {
    const long long i = i0 + c * 32 + lane;
    srcs[c] = i < m ? D.src[r][i] : 0;
  }
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {
    const long long i = i0 + c * 32 + lane;
    if (i >= m) continue;
    const int p = keys[c] / K;
    D.sorted_pos[r][i] = pos[c];
    copy_row_thread(P.out[p] + (disp[p] + (long long)pos[c]) * rb,
                    P.in[r] + (long long)srcs[c] * rb, rb);
  }
}

// Small dispatches (every rank at most kSmallItems items, at most
// kSmallKeys keys): count, scan and rank in one kernel, one CTA per rank.
// Warp w owns items [256 w, 256 w + 256) with their keys in registers: it
// counts them per key (warp match, its own row of `cnt`), the rows are
// turned into per-key prefixes over the warps, a block scan of the key
// totals gives the key starts, and each warp ranks its items in order.
constexpr int kSmallWarps = 8;
constexpr int kSmallItems = kSmallWarps * kRange;  // 2048
constexpr int kSmallKeys = kScanThreads;           // one key per thread in the key scan

__global__ void __launch_bounds__(kScanThreads) dispatch_small_kernel(const __grid_constant__ DispatchParams D) {
  chain_release();
  chain_wait();
  const int r = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NB = D.W * D.K;
  const long long m = D.items[r];
  __shared__ int cnt[kSmallWarps][kSmallKeys];
  __shared__ long long key_start[kSmallKeys];
  __shared__ long long warp_sums[kScanThreads / 32];
  for (int e = tid; e < kSmallWarps * NB; e += kScanThreads) cnt[e / NB][e % NB] = 0;
  __syncthreads();
  int keys[kRange / 32];
  int bad = 0;
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {
    const long long i = (long long)warp * kRange + c * 32 + lane;
    int key = -1 - lane;  // absent items match nobody
    if (i < m) {
      key = D.key[r][i];
      const int src = D.src[r][i];
      if (key < 0 || key >= NB || src < 0 || src >= D.rows[r]) {
        bad = 1;
        key = -1 - lane;
      }
    }
    keys[c] = key;
    const unsigned same = __match_any_sync(kFull, key);
    if (key >= 0 && lane == 31 - __clz(same)) cnt[warp][key] += __popc(same);
    __syncwarp();
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) fail(D, A2AV_ERR_BAD_INDEX);
    return;
  }
  long long total_k = 0;
  if (tid < NB) {
    int run = 0;
    for (int w = 0; w < kSmallWarps; ++w) {
      const int x = cnt[w][tid];
      cnt[w][tid] = run;
      run += x;
    }
    total_k = run;
  }
  long long all;
  const long long start = block_exclusive_scan(total_k, warp_sums, &all);
  if (tid < NB) {
    key_start[tid] = start;
    D.key_total[(long long)r * NB + tid] = total_k;
  }
  __syncthreads();
  if (tid < D.W) {
    long long sum = 0;
    for (int k = 0; k < D.K; ++k) sum += __ldcg(D.key_total + (long long)r * NB + tid * D.K + k);
    D.S[(long long)r * D.W + tid] = sum;
  }
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {
    const long long i = (long long)warp * kRange + c * 32 + lane;
    const int key = keys[c];
    const unsigned same = __match_any_sync(kFull, key);
    int pos = 0;
    if (key >= 0) pos = (int)key_start[key] + cnt[warp][key] + __popc(same & ((1u << lane) - 1u));
    __syncwarp();
    if (key >= 0 && lane == 31 - __clz(same)) cnt[warp][key] += __popc(same);
    __syncwarp();
    if (i < m) D.pos[(long long)r * D.pos_stride + i] = pos;
  }
}

// Once build_plan has accepted the split matrix: CTA 0 writes it out.
__device__ __forceinline__ void publish_splits(const DispatchParams& D) {
  if (blockIdx.x == 0 && D.in_splits_out != nullptr)
    for (int e = threadIdx.x; e < D.W * D.W; e += blockDim.x) D.in_splits_out[e] = D.S[e];
}

// The warp's n rows one at a time with the realigning span copy (rows not
// 16-byte aligned, or very long); kept out of line so that its registers do
// not weigh on the vector path of the kernel that calls it.
__device__ __noinline__ void copy_rows_unaligned(long long mdst, long long msrc, int n,
                                                 long long rb, int lane) {
  for (int j = 0; j < n; ++j) {
    unsigned char* dst = reinterpret_cast<unsigned char*>(__shfl_sync(kFull, mdst, j));
    const unsigned char* src = reinterpret_cast<const unsigned char*>(__shfl_sync(kFull, msrc, j));
    copy_span<32, 4, 2>(dst, src, rb, lane);
  }
}

// kWarpRows: rows of kWarpRowBytes or more, a warp per row (each kernel
// instantiation holds one of the two loops, so neither pays the other's
// registers); kVec: the 16-byte vectors a lane keeps in flight on aligned
// warp rows.
template <bool kWarpRows, int kVec = kVecRows>
__global__ void __launch_bounds__(kCopyThreads, !kWarpRows          ? kCopyCtasPerSm
                                                : kVec > kVecRows ? kCopyCtasPerSmWide
                                                                  : kCopyCtasPerSmWarpRows)
    dispatch_copy_kernel(const __grid_constant__ Params P, const __grid_constant__ DispatchParams D) {
  chain_wait();
  if (flagged(D)) return;
  __shared__ Plan pl;
  if (!build_plan(P, pl, kTileGranule)) return;
  publish_splits(D);
  const int W = D.W, K = D.K;
  const long long rb = P.rb, total = D.item_first[W];
  constexpr bool warp_rows = kWarpRows;
  const long long team = warp_rows ? (long long)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5)
                                   : (long long)blockIdx.x * kCopyThreads + threadIdx.x;
  const long long teams = warp_rows ? (long long)gridDim.x * (kCopyThreads / 32)
                                    : (long long)gridDim.x * kCopyThreads;
  if constexpr (warp_rows) {
    // A warp takes a batch of up to 32 consecutive items: lane l reads item
    // l's key, position and source row (one round trip for the batch), then
    // the warp copies the batch's rows.  16-byte aligned rows are copied as
    // one flat run of vectors over the batch, kVec x 16 bytes per lane in
    // flight; other rows one at a time with the realigning span copy.  The
    // batch size gives every warp the same number of batches: with 32 items
    // a batch, 131072 items over 3648 warps would leave a second round to one
    // warp in eight, and the kernel would take twice the time of the rest.
    const int lane = threadIdx.x & 31;
    const long long rounds = (total + teams * 32 - 1) / (teams * 32);
    const long long batch = rounds > 0 ? (total + teams * rounds - 1) / (teams * rounds) : 32;
    for (long long g0 = team * batch; g0 < total; g0 += teams * batch) {
      const long long g = g0 + lane;
      const int n = total - g0 < batch ? (int)(total - g0) : (int)batch;
      long long mdst = 0, msrc = 0;
      if (lane < n) {
        int r = 0;
        while (r + 1 < W && D.item_first[r + 1] <= g) ++r;
        const long long i = g - D.item_first[r];
        const int p = D.key[r][i] / K;
        const long long grouped = pl.out_off[p][r] - pl.in_off[r][p];  // + pos: the row in p's buffer
        if (D.combine) {  // from the peer's buffer back to the item's row
          msrc = (long long)(P.out[p] + (grouped + D.sorted_pos[r][i]) * rb);
          mdst = (long long)(P.in[r] + i * rb);
        } else {
          const long long pos = D.pos[(long long)r * D.pos_stride + i];
          D.sorted_pos[r][i] = pos;
          mdst = (long long)(P.out[p] + (grouped + pos) * rb);
          msrc = (long long)(P.in[r] + (long long)D.src[r][i] * rb);
        }
      }
      if (D.vec16 && rb <= kVecMaxRow) {
        const unsigned V = (unsigned)(rb >> 4), nv = (unsigned)n * V;  // < 2^17
        for (unsigned b0 = 0; b0 < nv; b0 += 32 * kVec) {  // warp-uniform trip count
          uint4 v[kVec];
          long long d[kVec];
#pragma unroll
          for (int q = 0; q < kVec; ++q) {
            const unsigned idx = b0 + q * 32 + lane;
            const bool ok = idx < nv;
            const unsigned j = ok ? idx / V : 0, c = ok ? idx - j * V : 0;
            const long long s = __shfl_sync(kFull, msrc, (int)j);
            d[q] = __shfl_sync(kFull, mdst, (int)j) + 16LL * c;
            if (ok) v[q] = ld_stream(reinterpret_cast<const uint4*>(s) + c);
          }
#pragma unroll
          for (int q = 0; q < kVec; ++q)
            if (b0 + q * 32 + lane < nv) st_stream(reinterpret_cast<uint4*>(d[q]), v[q]);
        }
      } else {
        copy_rows_unaligned(mdst, msrc, n, rb, lane);
      }
    }
  } else {
  // Short rows: a thread takes kItemsPerThread items, their key, source row
  // and position loads issued together, then copies the rows.
  for (long long g0 = team; g0 < total; g0 += teams * kItemsPerThread) {
    int rank[kItemsPerThread], key[kItemsPerThread], src_row[kItemsPerThread];
    long long pos[kItemsPerThread];
#pragma unroll
    for (int q = 0; q < kItemsPerThread; ++q) {
      const long long g = g0 + q * teams;
      rank[q] = -1;
      if (g < total) {
        int r = 0;
        while (r + 1 < W && D.item_first[r + 1] <= g) ++r;
        const long long i = g - D.item_first[r];
        rank[q] = r;
        key[q] = D.key[r][i];
        if (D.combine) {
          src_row[q] = (int)i;  // the item's own row of the rank's buffer
          pos[q] = D.sorted_pos[r][i];
        } else {
          src_row[q] = D.src[r][i];
          pos[q] = D.pos[(long long)r * D.pos_stride + i];
          D.sorted_pos[r][i] = pos[q];
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kItemsPerThread; ++q) {
      const int r = rank[q];
      if (r < 0) continue;
      const int p = key[q] / K;
      unsigned char* grouped = P.out[p] + (pl.out_off[p][r] + pos[q] - pl.in_off[r][p]) * rb;
      unsigned char* own = const_cast<unsigned char*>(P.in[r]) + (long long)src_row[q] * rb;
      if (D.combine)
        copy_row_thread(own, grouped, rb);
      else
        copy_row_thread(grouped, own, rb);
    }
  }
  }
}

// The fused combine's checks, before any row moves: the split matrix (the
// a2av prologue, which records A2AV_ERR_BAD_SPLITS), then every item's key
// and position -- the position must lie in its destination's group of the
// rank's key order, [in_off[r][p], in_off[r][p] + S[r][p]) -- else the flag
// that stops the copy kernel, and A2AV_ERR_BAD_INDEX.
__global__ void __launch_bounds__(kCopyThreads)
    combine_check_kernel(const __grid_constant__ Params P, const __grid_constant__ DispatchParams D) {
  chain_wait();
  chain_release();
  __shared__ Plan pl;
  if (!build_plan(P, pl, kTileGranule)) return;
  const int W = D.W, K = D.K, NB = W * K;
  const long long total = D.item_first[W];
  int bad = 0;
  for (long long g = (long long)blockIdx.x * kCopyThreads + threadIdx.x; g < total;
       g += (long long)gridDim.x * kCopyThreads) {
    int r = 0;
    while (r + 1 < W && D.item_first[r + 1] <= g) ++r;
    const long long i = g - D.item_first[r];
    const int key = D.key[r][i];
    if (key < 0 || key >= NB) {
      bad = 1;
      continue;
    }
    const int p = key / K;
    const long long pos = D.sorted_pos[r][i], lo = pl.in_off[r][p];
    if (pos < lo || pos >= lo + pl.s[r][p]) bad = 1;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) fail(D, A2AV_ERR_BAD_INDEX);
}

// Workspace: [0, 256) the flag (int) and the per-rank done counters (W ints),
// cleared before every dispatch; then S, key starts, key totals, histograms.
// Rows of 2..32 KiB, every row and buffer 16-byte aligned: NWK warps per CTA
// each stream their share of the CTA's items, row by row, global -> shared ->
// global with cp.async.bulk through a ring of NS stages of their own (loads
// LEAD rows ahead of the stores).  A warp reads the metadata of 32 items at
// a time, lane i item i; its lane 0 issues the copies and tracks its own
// bulk stores.
template <int NS, int LEAD, int NWK>
__global__ void __launch_bounds__(128)
    dispatch_copy_bulk_kernel(const __grid_constant__ Params P,
                              const __grid_constant__ DispatchParams D, int stage_bytes) {
  static_assert(LEAD >= 1 && LEAD < NS, "loads run 1..NS-1 rows ahead of stores");
  static_assert(NWK >= 1 && NWK <= 4, "one to four issuing warps");
  chain_wait();
  if (flagged(D)) return;
  __shared__ Plan pl;
  __shared__ alignas(8) unsigned long long bars[NWK * NS];
  __shared__ unsigned char* stage_dst[NWK * NS];
  extern __shared__ __align__(128) unsigned char stages[];
  if (!build_plan(P, pl, kTileGranule)) return;
  publish_splits(D);
  const int lane = threadIdx.x & 31;
  if ((int)(threadIdx.x >> 5) >= NWK) return;
  const int warp = NWK == 1 ? 0 : (int)(threadIdx.x >> 5);  // a constant for one warp
  // Warp w owns every NWK-th of the CTA's items, its own NS stages and
  // barriers: NWK independent pipelines, so NWK lanes issue copies at once.
  const int W = D.W, K = D.K;
  const long long rb = P.rb, total = D.item_first[W], G = gridDim.x, b0 = blockIdx.x;
  const long long nc = total > b0 ? (total - b0 + G - 1) / G : 0;  // the CTA's items
  const long long nk = nc > warp ? (nc - warp + NWK - 1) / NWK : 0;  // this warp's
  if (nk == 0) return;
  const uint32_t bar0 = smem_u32(bars) + 8u * NS * warp,
                 stage0 = smem_u32(stages) + (uint32_t)(NS * warp) * (uint32_t)stage_bytes;
  unsigned char** const sdst = stage_dst + NS * warp;
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_fence_init();
  }
  __syncwarp();
  long long msrc = 0, mdst = 0;  // this lane's item of the current batch of 32
  long long issued = 0, stored = 0;
  bool ok = true;
  for (long long k = 0; k < nk + LEAD; ++k) {
    if (k < nk) {
      if ((k & 31) == 0) {
        const long long kk = k + lane;
        if (kk < nk) {
          const long long g = b0 + (warp + kk * NWK) * G;
          int r = 0;
          while (r + 1 < W && D.item_first[r + 1] <= g) ++r;
          const long long i = g - D.item_first[r];
          const int p = D.key[r][i] / K;
          const long long grouped = pl.out_off[p][r] - pl.in_off[r][p];
          if (D.combine) {  // from the peer's buffer back to the item's row
            msrc = (long long)(P.out[p] + (grouped + D.sorted_pos[r][i]) * rb);
            mdst = (long long)(P.in[r] + i * rb);
          } else {
            const long long pos = D.pos[(long long)r * D.pos_stride + i];
            D.sorted_pos[r][i] = pos;
            msrc = (long long)(P.in[r] + (long long)D.src[r][i] * rb);
            mdst = (long long)(P.out[p] + (grouped + pos) * rb);
          }
        }
      }
      const int t = (int)(k & 31);
      const long long src = __shfl_sync(kFull, msrc, t), dst = __shfl_sync(kFull, mdst, t);
      if (lane == 0) {
        const int s = (int)(k % NS);
        if (k >= NS) bulk_wait_read<NS - LEAD - 1>();
        sdst[s] = reinterpret_cast<unsigned char*>(dst);
        mbar_expect_tx(bar0 + 8 * s, (unsigned)rb);
        bulk_load(stage0 + (uint32_t)s * stage_bytes, reinterpret_cast<const void*>(src),
                  (unsigned)rb, bar0 + 8 * s);
      }
      issued = k + 1;
    }
    const long long j = k - LEAD;
    if (j >= 0 && j < nk) {
      const int s = (int)(j % NS);
      if (lane == 0) {
        ok = mbar_wait(bar0 + 8 * s, (unsigned)((j / NS) & 1));
        if (ok) bulk_store(sdst[s], stage0 + (uint32_t)s * stage_bytes, (unsigned)rb);
      }
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      stored = j + 1;
    }
  }
  if (lane == 0) {
    if (!ok) {
      record_error(P.status, A2AV_ERR_TIMEOUT);
      for (long long j = stored; j < issued; ++j)
        mbar_wait(bar0 + 8 * (int)(j % NS), (unsigned)((j / NS) & 1));
    }
    bulk_wait_all();
  }
}

// The two ring shapes: rows up to 16 KiB (16 KiB stages) and up to 32 KiB
// (half as many 32 KiB stages).
// The gather's ring: measured on the cfg3 dispatch (14 KiB rows), 12 x 16
// KiB stages with loads 10 rows ahead beat 8 stages / 6 ahead by 3 % and two
// CTAs per SM with smaller rings by 4-6 %: bytes in flight per SM decide.
#ifndef A2AV_GATHER_STAGES
#define A2AV_GATHER_STAGES 12  // 16 KiB stages of the small ring
#endif
#ifndef A2AV_GATHER_LEAD
#define A2AV_GATHER_LEAD 10
#endif
#ifndef A2AV_GATHER_CTAS_PER_SM
#define A2AV_GATHER_CTAS_PER_SM 1
#endif
// Rows of at most 8 KiB go through 8 KiB stages, several warps issuing at
// once, each with its own ring (one lane issuing every row was the limit:
// ~480 ns a row whatever its size).  Measured on the MoE dispatch (8192
// tokens, top-2, W=8, us): 2 / 4 KiB rows 113 / 154 with four warps x 6
// stages (two warps x 12: 193 / 197; the warp copy: 141 / 263); 8 KiB rows 279
// with two warps x 12 stages (four x 6: 300; one warp, 16 KiB stages: 411).
constexpr int kGatherTinyStage = 8 * 1024;
constexpr int kGatherSmallStage = 16 * 1024, kGatherLargeStage = 32 * 1024;
using GatherKernel = void (*)(Params, DispatchParams, int);
const GatherKernel kGatherTiny4 = dispatch_copy_bulk_kernel<6, 4, 4>;    // rows <= 4 KiB
const GatherKernel kGatherTiny2 = dispatch_copy_bulk_kernel<12, 10, 2>;  // rows <= 8 KiB
// 8..16 KiB rows: one issuing warp, 12 x 16 KiB (two warps x 6: 2-4 % slower).
const GatherKernel kGatherSmall = dispatch_copy_bulk_kernel<A2AV_GATHER_STAGES, A2AV_GATHER_LEAD, 1>;
// Few items per CTA (decode-size dispatches) of 8..16 KiB rows: four warps x
// 3 x 16 KiB, so that a CTA's handful of rows are issued four at a time
// (14 KiB rows, 128 / 512 tokens a rank: 26.3 / 44.0 -> 25.2 / 41.8 us; no
// gain for 8 KiB rows, which keep the two-warp ring).
#ifndef A2AV_GATHER_FEW_ITEMS
#define A2AV_GATHER_FEW_ITEMS 64  // items per CTA at or below which the four-warp ring is used
#endif
const GatherKernel kGatherSmallFew = dispatch_copy_bulk_kernel<3, 1, 4>;
const GatherKernel kGatherLarge =
    dispatch_copy_bulk_kernel<A2AV_GATHER_STAGES / 2, (A2AV_GATHER_LEAD + 1) / 2 - 1 >= 1
                                                          ? (A2AV_GATHER_LEAD + 1) / 2 - 1
                                                          : 1, 1>;
constexpr int kGatherSmem = A2AV_GATHER_STAGES * kGatherSmallStage;
static_assert(4 * 6 * kGatherTinyStage <= kGatherSmem && 2 * 12 * kGatherTinyStage <= kGatherSmem,
              "the 8 KiB rings fit the same shared memory");
static_assert(kGatherSmem <= 192 * 1024, "shared memory per CTA");
static_assert(A2AV_GATHER_STAGES % 2 == 0 && A2AV_GATHER_LEAD < A2AV_GATHER_STAGES,
              "the large ring halves the small one");
// Aligned rows this long or longer take the bulk gather; shorter ones the
// warp copy's flat vector runs.  Measured on the MoE dispatch (8192 tokens,
// top-2, W=8): 1 KiB rows 78 us by warp copy against 117 by the gather; from
// 2 KiB the gather wins (above); 14 KiB rows 459 us against 868 by warp copy.
#ifndef A2AV_GATHER_MIN_ROW
#define A2AV_GATHER_MIN_ROW 2048
#endif
constexpr long long kGatherMinRow = A2AV_GATHER_MIN_ROW;


struct Layout {
  long long flag, done, S, key_start, key_total, pos, hist, grp, total;
};

Layout layout(int W, int K, long long max_items) {
  auto up = [](long long x) { return (x + 255) / 256 * 256; };
  const long long NB = (long long)W * K;
  const long long ranges = (max_items + kRange - 1) / kRange;
  Layout L;
  L.flag = 0;
  L.done = 4;
  L.S = 256;
  L.key_start = L.S + up(8LL * W * W);
  L.key_total = L.key_start + up(8LL * W * NB);
  L.pos = L.key_total + up(8LL * W * NB);
  const long long groups = (ranges + kCountWarps - 1) / kCountWarps;
  L.hist = L.pos + up(4LL * W * (max_items < 1 ? 1 : max_items));
  L.grp = L.hist + up(4LL * W * (ranges < 1 ? 1 : ranges) * NB);
  L.total = L.grp + up(4LL * W * (groups < 1 ? 1 : groups) * NB);
  return L;
}

}  // namespace

extern "C" int64_t a2av_dispatch_workspace_bytes(int world_size, int keys_per_peer,
                                                 int64_t max_items_per_rank) {
  if (world_size < 1 || world_size > kMaxW || keys_per_peer < 1 || max_items_per_rank < 0 ||
      (long long)world_size * keys_per_peer > kMaxBins || max_items_per_rank > 0x7fffffffLL)
    return -1;
  return layout(world_size, keys_per_peer, max_items_per_rank).total;
}

namespace {

// The row copy of a dispatch or a combine: the cp.async.bulk gather for
// 16-byte aligned rows of 2..32 KiB (its ring chosen by row size and by the
// items per CTA), else the warp copy (rows of 64 bytes or more) or the
// thread copy.
cudaError_t launch_copy(a2av_handle* h, const Params& P, const DispatchParams& D,
                        long long row_bytes, cudaStream_t s) {
  const bool aligned = D.vec16 && row_bytes >= kGatherMinRow && row_bytes <= kGatherLargeStage;
  if (!aligned) {
    if (row_bytes < kWarpRowBytes)
      return launch_kernel(dispatch_copy_kernel<false>, dim3(h->sms * kCopyCtasPerSm),
                           kCopyThreads, 0, s, true, P, D);
    if (D.combine && D.vec16 && row_bytes <= kVecMaxRow)
      return launch_kernel(dispatch_copy_kernel<true, kVecRowsWide>,
                           dim3(h->sms * kCopyCtasPerSmWide), kCopyThreads, 0, s, true, P, D);
    return launch_kernel(dispatch_copy_kernel<true>, dim3(h->sms * kCopyCtasPerSmWarpRows),
                         kCopyThreads, 0, s, true, P, D);
  }
  const bool tiny = row_bytes <= kGatherTinyStage, small = row_bytes <= kGatherSmallStage;
  const bool few = D.item_first[D.W] <= (long long)A2AV_GATHER_FEW_ITEMS *
                                             (h->sms * A2AV_GATHER_CTAS_PER_SM);
  const GatherKernel k = row_bytes <= 4096 ? kGatherTiny4
                         : tiny            ? kGatherTiny2
                         : small           ? (few ? kGatherSmallFew : kGatherSmall)
                                           : kGatherLarge;
  if (!h->gather_ready) {  // shared-memory opt-in, once per handle (a host call per launch otherwise)
    for (GatherKernel g : {kGatherTiny4, kGatherTiny2, kGatherSmall, kGatherSmallFew, kGatherLarge})
      if (cudaFuncSetAttribute(g, cudaFuncAttributeMaxDynamicSharedMemorySize, kGatherSmem) !=
          cudaSuccess)
        return cudaErrorInvalidValue;
    h->gather_ready = true;
  }
  return launch_kernel(k, dim3(h->sms * A2AV_GATHER_CTAS_PER_SM), 128, kGatherSmem, s, true, P, D,
                       tiny ? kGatherTinyStage : small ? kGatherSmallStage : kGatherLargeStage);
}

}  // namespace

extern "C" int a2av_dispatch(a2av_handle* h, int keys_per_peer, const void* const* rows_ptrs,
                             const int64_t* rows_per_rank, const int32_t* const* src_row_ptrs,
                             const int32_t* const* key_ptrs, const int64_t* items_per_rank,
                             void* const* out_ptrs, int64_t* out_splits_offsets_dev,
                             int64_t* const* sorted_pos_ptrs, int64_t* in_splits_dev,
                             int64_t row_bytes, void* workspace, int64_t workspace_bytes,
                             void* stream) {
  if (h == nullptr || rows_ptrs == nullptr || rows_per_rank == nullptr || src_row_ptrs == nullptr ||
      key_ptrs == nullptr || items_per_rank == nullptr || out_ptrs == nullptr ||
      out_splits_offsets_dev == nullptr || sorted_pos_ptrs == nullptr || workspace == nullptr ||
      row_bytes < 1 || keys_per_peer < 1)
    return A2AV_ERR_INVALID_ARG;
  const int W = h->W, K = keys_per_peer;
  if ((long long)W * K > kMaxBins) return A2AV_ERR_UNSUPPORTED;
  if (((uintptr_t)workspace & 255) != 0 || ((uintptr_t)out_splits_offsets_dev & 7) != 0 ||
      ((uintptr_t)in_splits_dev & 7) != 0)
    return A2AV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return A2AV_ERR_CUDA;
  if (dev != h->device) return A2AV_ERR_INVALID_ARG;

  DispatchParams D;
  std::memset(&D, 0, sizeof(D));
  long long ranges_max = 0, max_items = 0;
  D.item_first[0] = 0;
  for (int r = 0; r < W; ++r) {
    const long long m = items_per_rank[r], n = rows_per_rank[r];
    if (m < 0 || n < 0) return A2AV_ERR_INVALID_ARG;
    if (m > 0x7fffffffLL || n > 0x7fffffffLL) return A2AV_ERR_UNSUPPORTED;
    if (m > 0 && (key_ptrs[r] == nullptr || src_row_ptrs[r] == nullptr ||
                  sorted_pos_ptrs[r] == nullptr))
      return A2AV_ERR_INVALID_ARG;
    D.key[r] = key_ptrs[r];
    D.src[r] = src_row_ptrs[r];
    D.sorted_pos[r] = reinterpret_cast<long long*>(sorted_pos_ptrs[r]);
    D.items[r] = m;
    D.rows[r] = n;
    D.item_first[r + 1] = D.item_first[r] + m;
    const long long R = (m + kRange - 1) / kRange;
    ranges_max = R > ranges_max ? R : ranges_max;
    max_items = m > max_items ? m : max_items;
  }
  const Layout L = layout(W, K, max_items);
  if (workspace_bytes < L.total) return A2AV_ERR_INVALID_ARG;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  D.flag = reinterpret_cast<int*>(ws + L.flag);
  D.done = reinterpret_cast<int*>(ws + L.done);
  D.S = reinterpret_cast<long long*>(ws + L.S);
  D.key_start = reinterpret_cast<long long*>(ws + L.key_start);
  D.key_total = reinterpret_cast<long long*>(ws + L.key_total);
  D.pos = reinterpret_cast<int*>(ws + L.pos);
  D.pos_stride = max_items < 1 ? 1 : max_items;
  D.hist = reinterpret_cast<int*>(ws + L.hist);
  D.grp = reinterpret_cast<int*>(ws + L.grp);
  D.status = h->d_status;
  D.in_splits_out = reinterpret_cast<long long*>(in_splits_dev);
  D.ranges_max = ranges_max;
  D.groups_max = (ranges_max + kCountWarps - 1) / kCountWarps;
  D.W = W;
  D.K = K;
  // One count CTA per rank scans its groups when a thread's share of one key
  // fits kFuseScanPer registers; the scan kernel and its launch are skipped.
  const int slices = kScanThreads / (W * K);
  D.fuse_scan = slices > 0 && D.groups_max <= (long long)kFuseScanPer * slices;
  bool vec16 = row_bytes % 16 == 0;
  for (int r = 0; r < W; ++r)
    vec16 = vec16 && ((uintptr_t)rows_ptrs[r] & 15) == 0 && ((uintptr_t)out_ptrs[r] & 15) == 0;
  D.vec16 = vec16 ? 1 : 0;

  Params P;
  std::memset(&P, 0, sizeof(P));
  for (int r = 0; r < W; ++r) {
    P.in[r] = static_cast<const unsigned char*>(rows_ptrs[r]);
    P.out[r] = static_cast<unsigned char*>(out_ptrs[r]);
  }
  P.splits = D.S;
  P.split_stride = W;
  P.out_so = reinterpret_cast<long long*>(out_splits_offsets_dev);
  P.status = h->d_status;
  P.rb = row_bytes;
  P.limit = split_limit(W, row_bytes);
  P.in_cap = 0;  // sources are checked by row index in the count kernel
  P.out_cap = h->out_cap;
  P.W = W;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  static_assert(4 + 4 * kMaxW <= 256, "flag and done counters fit the first 256 bytes");
  if (cudaMemsetAsync(D.flag, 0, 256, s) != cudaSuccess) return A2AV_ERR_CUDA;
  // Every kernel of the chain is launched with programmatic stream
  // serialization: it may be scheduled while its predecessor runs and waits
  // for that predecessor's results in chain_wait.
  cudaError_t e;
  const bool small_path = max_items <= kSmallItems && W * K <= kSmallKeys;
  const bool fuse = !small_path && row_bytes < kWarpRowBytes;  // rank kernel copies the rows
  if (small_path) {
    e = launch_kernel(dispatch_small_kernel, dim3(W), kScanThreads, 0, s, h->pdl, D);
  } else {
    // (at least one CTA per rank: a batch without items still gets its
    // counts, splits and offsets written)
    const long long ranges = ranges_max > 0 ? ranges_max : 1;
    const dim3 grid((unsigned)ranges, (unsigned)W);
    const dim3 grid_count((unsigned)((ranges + kCountWarps - 1) / kCountWarps), (unsigned)W);
    e = launch_kernel(dispatch_count_kernel, grid_count, 32 * kCountWarps,
                      (size_t)kCountWarps * W * K * sizeof(int), s, h->pdl, D);
    if (e == cudaSuccess && !D.fuse_scan)
      e = launch_kernel(dispatch_scan_kernel, dim3((unsigned)(W * K), (unsigned)W), kScanThreads,
                        0, s, true, D);
    if (e == cudaSuccess && fuse) {
      const dim3 grid2((unsigned)((ranges + kRankCopyWarps - 1) / kRankCopyWarps),
                       (unsigned)W);
      e = launch_kernel(dispatch_rank_copy_kernel, grid2, 32 * kRankCopyWarps, 0, s, true, P, D);
      if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
      return A2AV_OK;
    }
    if (e == cudaSuccess) e = launch_kernel(dispatch_rank_kernel, grid, 32, 0, s, true, D);
  }
  if (e != cudaSuccess) return A2AV_ERR_CUDA;
  e = launch_copy(h, P, D, row_bytes, s);
  if (e != cudaSuccess) return A2AV_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
  return A2AV_OK;
}

extern "C" int a2av_combine_items(a2av_handle* h, int keys_per_peer,
                                  const void* const* peer_ptrs, const int64_t* in_splits_dev,
                                  const int32_t* const* key_ptrs,
                                  const int64_t* const* sorted_pos_ptrs,
                                  const int64_t* items_per_rank, void* const* item_out_ptrs,
                                  int64_t row_bytes, void* workspace, int64_t workspace_bytes,
                                  void* stream) {
  if (h == nullptr || peer_ptrs == nullptr || in_splits_dev == nullptr || key_ptrs == nullptr ||
      sorted_pos_ptrs == nullptr || items_per_rank == nullptr || item_out_ptrs == nullptr ||
      workspace == nullptr || row_bytes < 1 || keys_per_peer < 1)
    return A2AV_ERR_INVALID_ARG;
  const int W = h->W, K = keys_per_peer;
  if ((long long)W * K > kMaxBins) return A2AV_ERR_UNSUPPORTED;
  if (((uintptr_t)workspace & 255) != 0 || ((uintptr_t)in_splits_dev & 7) != 0 ||
      workspace_bytes < A2AV_COMBINE_WORKSPACE_BYTES)
    return A2AV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return A2AV_ERR_CUDA;
  if (dev != h->device) return A2AV_ERR_INVALID_ARG;

  DispatchParams D;
  std::memset(&D, 0, sizeof(D));
  D.item_first[0] = 0;
  for (int r = 0; r < W; ++r) {
    const long long m = items_per_rank[r];
    if (m < 0) return A2AV_ERR_INVALID_ARG;
    if (m > 0x7fffffffLL) return A2AV_ERR_UNSUPPORTED;
    if (m > 0 && (key_ptrs[r] == nullptr || sorted_pos_ptrs[r] == nullptr ||
                  item_out_ptrs[r] == nullptr))
      return A2AV_ERR_INVALID_ARG;
    D.key[r] = key_ptrs[r];
    D.sorted_pos[r] = const_cast<long long*>(reinterpret_cast<const long long*>(sorted_pos_ptrs[r]));
    D.items[r] = m;
    D.item_first[r + 1] = D.item_first[r] + m;
  }
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  D.flag = reinterpret_cast<int*>(ws);
  D.status = h->d_status;
  D.W = W;
  D.K = K;
  D.combine = 1;
  bool vec16 = row_bytes % 16 == 0;
  for (int r = 0; r < W; ++r)
    vec16 = vec16 && ((uintptr_t)peer_ptrs[r] & 15) == 0 && ((uintptr_t)item_out_ptrs[r] & 15) == 0;
  D.vec16 = vec16 ? 1 : 0;

  // Rank-side buffers (the items' rows, written) in P.in, peer-side buffers
  // (the dispatch layout, read) in P.out: the prologue's checks and offsets
  // are those of the dispatch; its offsets table goes to the workspace.
  Params P;
  std::memset(&P, 0, sizeof(P));
  for (int r = 0; r < W; ++r) {
    P.in[r] = static_cast<const unsigned char*>(item_out_ptrs[r]);
    P.out[r] = static_cast<unsigned char*>(const_cast<void*>(peer_ptrs[r]));
  }
  P.splits = reinterpret_cast<const long long*>(in_splits_dev);
  P.split_stride = W;
  P.out_so = reinterpret_cast<long long*>(ws + 256);
  P.status = h->d_status;
  P.rb = row_bytes;
  P.limit = split_limit(W, row_bytes);
  P.in_cap = 0;
  P.out_cap = 0;
  P.W = W;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(D.flag, 0, 256, s) != cudaSuccess) return A2AV_ERR_CUDA;
  cudaError_t e = launch_kernel(combine_check_kernel, dim3(h->sms * kCopyCtasPerSm), kCopyThreads,
                                0, s, h->pdl, P, D);
  if (e != cudaSuccess) return A2AV_ERR_CUDA;
  e = launch_copy(h, P, D, row_bytes, s);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
  return A2AV_OK;
}
