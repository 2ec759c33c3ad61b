// dispatch.cu -- fused dispatch preparation for the variable-size all-to-all:
// the exchange of rows that are not yet grouped by destination (declared in
// include/a2av.h, a2av_dispatch), and its return path in item order
// (a2av_combine_items).
//
// Each rank's items carry a key (destination = key / K) and a source row.
// The exchange runs on the rank's items ordered stably by key -- the input
// a2av_run would expect -- without ever materialising that order.  An item's
// place in it is
//     pos = key_start[r][k] + grp[r][c][k] + hist[r][j][k] + inrank[i]
// for item i of rank r with key k in range j (256 items) of group c (8 or 32
// ranges): the items of smaller keys, of key k in earlier groups, in earlier
// ranges of the group, and earlier in the item's own range.
//   1. count  (eight warps per CTA, one to four ranges each): a warp ranks
//      its range's items 32 at a time (equal keys found by ballots), which gives
//      every item its inrank byte and the range's key histogram; keys and
//      source rows are validated here.  The CTA's histograms give each range
//      its in-group prefix (hist) and the group its count (grp).  The last
//      CTA of each rank to finish (an atomic count after a fence) turns the
//      group counts into prefixes over the groups, the key totals into key
//      starts and the split matrix row S[r][*].
//   2. scan   (only when a rank has too many groups for one CTA): the same
//      per-key scan over groups as a kernel of its own.
//   When every rank has at most 2048 items and there are at most 256 keys,
//   one kernel (one CTA per rank) does 1-2 instead.
//   3. copy   (the a2av prologue builds the plan from S, which also checks
//      capacities and NULL buffers; then S is published and every item's row
//      goes straight to its place in the output of its destination):
//      - 16-byte aligned rows above 2 KiB .. 32 KiB (the combine: from 64 B):
//        the cp.async.bulk gather -- up to 2 KiB, every lane of a warp
//        issues the copy of its own item's row into its slot of a 16-row
//        shared-memory stage (one mbarrier per stage), then its own bulk
//        store, with as many warps per CTA as keep ~96 KiB of loads in flight
//        per SM; above 2 KiB one row a stage, issued by one lane per warp;
//        the item metadata is loaded two and one batches ahead;
//      - other rows of 64 bytes or more: a warp per batch of rows (registers);
//      - rows under 64 bytes: the count kernel's successor places and copies
//        the rows of a whole range per warp (thread per row).
// Rows under 64 bytes, when every item fits the grid's registers, take one
// cooperative launch instead of 1-3 (the order kernel): each CTA counts a
// chunk of one rank's items, the CTAs exchange their counts through the
// workspace and one bounded grid barrier, and each CTA then ranks, places
// and copies its chunk.
// Decode-size batches (at most 4096 items over all ranks) take one kernel
// instead: every CTA reads all keys, counts them, derives the split matrix
// and the plan itself (so all CTAs reach the same verdict without any
// inter-CTA communication), then places and copies its own share of the
// items -- no workspace, no memset, one launch.
// The combine moves rows back with the same copy kernels after a check
// kernel; short rows check and copy in one cooperative launch, and the
// gather checks its items itself (grid barrier) for rows up to 2 KiB.
// Invalid keys or source rows set a workspace flag (cleared first) that stops
// every later kernel; invalid splits stop the copy kernel in its prologue.
// Either way nothing the caller owns is written.
#include "a2av_device.cuh"
#include "a2av_handle.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <type_traits>

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
constexpr long long kVecMaxRow = 64 * 1024;  // flat vector runs up to this row size

struct DispatchParams {
  const int* key[kMaxW];
  const int* src[kMaxW];
  long long* sorted_pos[kMaxW];
  long long items[kMaxW];            // m_r
  long long rows[kMaxW];             // source rows per rank
  long long item_first[kMaxW + 1];   // exclusive prefix of m_r
  long long batch_first[kMaxW + 1];  // exclusive prefix of ceil(m_r / bs) (gather)
  int* flag;                         // workspace: set once input is found invalid
  int* done;                         // workspace: [W] CTAs finished per rank (the one that scans)
  long long* S;                      // workspace: [W][W]
  long long* key_start;              // workspace: [W][NB]
  long long* key_total;              // workspace: [W][NB]
  int* hist;                         // workspace: [W][ranges_max][NB]
  int* grp;                          // workspace: [W][groups_max][NB]
  unsigned char* inrank;             // workspace: [W][pos_stride] rank within the item's range
  int* status;
  long long* in_splits_out;          // optional [W][W]
  int vec16;                         // every row and buffer 16-byte aligned
  int combine;                       // the fused combine: rows move the other way (below)
  long long ranges_max;
  long long groups_max;
  int group_log2;                    // a group is 1 << group_log2 ranges (8 or 32)
  int fuse_scan;                     // the count kernel's last CTA per rank scans the groups
  int bs;                            // items per gather batch (8, 16 or 32)

  long long pos_stride;
  int W, K;
  // the one-launch order kernel (below)
  int* cta_cnt;                      // workspace: [grid][NB] key counts of each CTA's chunk
  unsigned* barrier;                 // workspace (cleared): CTAs past the grid barrier
  long long chunk;                   // items per CTA
  int cta_first[kMaxW + 1];          // CTAs of rank r: [cta_first[r], cta_first[r + 1])
  int pos_ready;                     // sorted_pos already holds every item's position
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

// The lanes of the warp holding the same key as this lane (valid lanes only;
// an invalid lane gets 0 and matches nobody): one ballot per key bit, keys in
// [0, 2^bits).  Same result as __match_any_sync on the valid keys, at the
// throughput of plain ballots (the match instruction is far slower per SM,
// measured: ranking 640 K items a rank in 8-warp blocks took 28 us with it).
__device__ __forceinline__ unsigned same_key_lanes(int key, bool valid, int bits) {
  unsigned m = __ballot_sync(kFull, valid);
  for (int b = 0; b < bits; ++b) {
    const bool one = (key >> b) & 1;
    const unsigned v = __ballot_sync(kFull, one);
    m &= one ? v : ~v;
  }
  return valid ? m : 0u;
}

// Bits that hold every key below nb (0 for one key).
__device__ __forceinline__ int key_bits(int nb) { return nb > 1 ? 32 - __clz(nb - 1) : 0; }

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
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

// Items are counted in ranges of kRange, ranges in groups of 8 * RW (a count
// CTA: eight warps of RW ranges each).  After the count kernel, hist[r][j][b]
// holds the items with key b in the earlier ranges of range j's group and
// grp[r][c][b] the group's count; the scan (below) turns grp[r][*][b] into
// exclusive prefixes over the groups.
constexpr int kCountWarps = 8;
constexpr int kFuseScanMax = 32;  // groups a thread may scan in the fused scan
static_assert(32 * kCountWarps == kScanThreads, "a count CTA can run the block scan");

// The fused scan: one CTA (kScanThreads threads) over rank r's C groups.
// Thread t takes key b = t % NB and the slice g = t / NB of consecutive
// groups (G = kScanThreads / NB slices per key): it sums its slice, the
// slices' sums give it its base, and it rewrites its slice with running
// prefixes.  Counts are loaded kFuseScanBatch at a time, from L2 (the other
// count CTAs wrote them during this launch); the first batch is kept in
// registers for the second pass, so a slice of at most kFuseScanBatch groups
// is loaded once.
constexpr int kFuseScanBatch = 8;
__device__ void scan_groups_in_cta(const DispatchParams& D, int r, long long C) {
  const int t = threadIdx.x, NB = D.W * D.K, G = kScanThreads / NB;
  const int b = t % NB, g = t / NB;
  const long long per = (C + G - 1) / G;
  const long long c0 = g < G ? g * per : C;
  const long long c1 = g < G ? (c0 + per < C ? c0 + per : C) : C;
  int* A = D.grp + (long long)r * D.groups_max * NB + b;  // group c at A[c * NB]
  __shared__ long long part[kScanThreads];
  __shared__ long long tot[kScanThreads];
  __shared__ long long warp_sums[kScanThreads / 32];
  long long local = 0;
  int v0[kFuseScanBatch];  // the first batch, kept for the second pass
  for (long long c = c0; c < c1; c += kFuseScanBatch) {
    int v[kFuseScanBatch];
#pragma unroll
    for (int q = 0; q < kFuseScanBatch; ++q) v[q] = c + q < c1 ? __ldcg(A + (c + q) * NB) : 0;
#pragma unroll
    for (int q = 0; q < kFuseScanBatch; ++q) {
      local += v[q];
      if (c == c0) v0[q] = v[q];
    }
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
  for (long long c = c0; c < c1; c += kFuseScanBatch) {
    int v[kFuseScanBatch];
#pragma unroll
    for (int q = 0; q < kFuseScanBatch; ++q)
      v[q] = c == c0 ? v0[q] : (c + q < c1 ? __ldcg(A + (c + q) * NB) : 0);
#pragma unroll
    for (int q = 0; q < kFuseScanBatch; ++q) {
      if (c + q < c1) A[(c + q) * NB] = (int)base;
      base += v[q];
    }
  }
  if (g == 0) tot[b] = total;
  __syncthreads();
  finish_rank(D, r, tot, warp_sums);
}

// Count: CTA (c, r) holds group c of rank r; warp w ranks ranges
// 8RW c + RW w .. + RW - 1 (all their keys and source rows loaded at once),
// 32 items at a time: a ballot per key bit groups equal keys, a lane's rank
// among them plus the range's running count of its key is its inrank, and
// each key's leader advances that count.  RW = 1 (the default) at five CTAs
// an SM (48 registers) keeps a batch of 760 groups of 2048 items (1.5 M items) resident
// in one wave; RW = 4 (fewer, longer CTAs, for sweeps) was measured slower.
template <int RW, bool kRank = true>
__global__ void __launch_bounds__(32 * kCountWarps, RW == 1 ? 5 : 2)
    dispatch_count_kernel(const __grid_constant__ DispatchParams D) {
  chain_release();
  chain_wait();
  constexpr int kGroupRanges = kCountWarps * RW;
  const int r = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
  const long long c = blockIdx.x;
  const long long m = D.items[r];
  const int NB = D.W * D.K;
  if (c * kGroupRanges * kRange >= m) {  // no items in this CTA's ranges (uniform over the CTA)
    if (c == 0 && D.fuse_scan) {  // a rank without items: zero counts and splits
      __shared__ long long zero[kScanThreads];
      __shared__ long long zero_sums[kScanThreads / 32];
      zero[t] = 0;
      __syncthreads();
      finish_rank(D, r, zero, zero_sums);
    }
    return;
  }
  extern __shared__ int count_hist[];  // [kGroupRanges][NB], range by range
  for (int e = t; e < kGroupRanges * NB; e += blockDim.x) count_hist[e] = 0;
  const long long j0 = c * kGroupRanges + (long long)warp * RW;  // this warp's first range
  // Every load unconditional (an index past the rank's last item reads its
  // last item again, then counts for nothing), so all of them issue at once.
  const int* const kp = D.key[r];
  const int* const sp = D.src[r];
  const long long rows_r = D.rows[r];
  int keys[RW][kRange / 32], srcs[RW][kRange / 32];
#pragma unroll
  for (int u = 0; u < RW; ++u)
#pragma unroll
    for (int q = 0; q < kRange / 32; ++q) {
      const long long i = (j0 + u) * kRange + q * 32 + lane;
      const long long ii = i < m ? i : m - 1;
      keys[u][q] = __ldg(kp + ii);
      srcs[u][q] = __ldg(sp + ii);
    }
  int bad = 0;
#pragma unroll
  for (int u = 0; u < RW; ++u)
#pragma unroll
    for (int q = 0; q < kRange / 32; ++q) {
      const long long i = (j0 + u) * kRange + q * 32 + lane;
      const int k = keys[u][q], s = srcs[u][q];
      const bool ok = i < m && k >= 0 && k < NB && s >= 0 && s < rows_r;
      if (i < m && !ok) bad = 1;
      keys[u][q] = ok ? k : -1 - lane;  // absent or invalid items match nobody
    }
  __syncthreads();
  if constexpr (kRank) {
    const unsigned lt = (1u << lane) - 1u;
    const int bits = key_bits(NB);
#pragma unroll
    for (int u = 0; u < RW; ++u) {
      int* hist = count_hist + (warp * RW + u) * NB;
#pragma unroll
      for (int q = 0; q < kRange / 32; ++q) {
        const int k = keys[u][q];
        const unsigned same = same_key_lanes(k, k >= 0, bits);
        const int inr = k >= 0 ? hist[k] + __popc(same & lt) : 0;
        __syncwarp();
        if (k >= 0 && lane == 31 - __clz(same)) hist[k] += __popc(same);
        __syncwarp();
        if (k >= 0)
          D.inrank[(long long)r * D.pos_stride + (j0 + u) * kRange + q * 32 + lane] =
              (unsigned char)inr;
      }
    }
  } else {  // counts only: the place-and-copy kernel ranks the items itself
#pragma unroll
    for (int u = 0; u < RW; ++u)
#pragma unroll
      for (int q = 0; q < kRange / 32; ++q)
        if (keys[u][q] >= 0) atomicAdd(&count_hist[(warp * RW + u) * NB + keys[u][q]], 1);
  }
  if (__any_sync(kFull, bad) && lane == 0) fail(D, A2AV_ERR_BAD_INDEX);
  __syncthreads();
  // in-group prefixes of the ranges that hold items, and the group's count
  const long long R = (m + kRange - 1) / kRange;
  for (int b = t; b < NB; b += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kGroupRanges; ++w) {
      const long long j = c * kGroupRanges + w;
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
  const long long C = (m + kGroupRanges * kRange - 1) / (kGroupRanges * kRange);
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
  const long long GI = (long long)kRange << D.group_log2;
  const long long C = (D.items[r] + GI - 1) / GI;
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

// Small dispatches (every rank at most kSmallItems items, at most
// kSmallKeys keys): count and scan in one kernel, one CTA per rank.  Warp w
// ranks range w of the rank (items [256 w, 256 w + 256)) like the count
// kernel; the per-warp counts become the ranges' prefixes (one group), a
// block scan of the key totals gives the key starts.
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
  __shared__ long long warp_sums[kScanThreads / 32];
  for (int e = tid; e < kSmallWarps * NB; e += kScanThreads) cnt[e / NB][e % NB] = 0;
  int keys[kRange / 32], srcs[kRange / 32];
  const int* const kp = D.key[r];
  const int* const sp = D.src[r];
  const long long rows_r = D.rows[r];
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {  // (unconditional loads, as in the count kernel)
    const long long i = (long long)warp * kRange + c * 32 + lane;
    const long long ii = i < m ? i : (m > 0 ? m - 1 : 0);
    keys[c] = m > 0 ? __ldg(kp + ii) : 0;
    srcs[c] = m > 0 ? __ldg(sp + ii) : 0;
  }
  int bad = 0;
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {
    const long long i = (long long)warp * kRange + c * 32 + lane;
    const bool ok = i < m && keys[c] >= 0 && keys[c] < NB && srcs[c] >= 0 && srcs[c] < rows_r;
    if (i < m && !ok) bad = 1;
    keys[c] = ok ? keys[c] : -1 - lane;  // absent or invalid items match nobody
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  const int bits = key_bits(NB);
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {
    const int key = keys[c];
    const unsigned same = same_key_lanes(key, key >= 0, bits);
    const int inr = key >= 0 ? cnt[warp][key] + __popc(same & lt) : 0;
    __syncwarp();
    if (key >= 0 && lane == 31 - __clz(same)) cnt[warp][key] += __popc(same);
    __syncwarp();
    if (key >= 0)
      D.inrank[(long long)r * D.pos_stride + (long long)warp * kRange + c * 32 + lane] =
          (unsigned char)inr;
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) fail(D, A2AV_ERR_BAD_INDEX);
    return;
  }
  const long long R = (m + kRange - 1) / kRange;
  long long total_k = 0;
  if (tid < NB) {
    int run = 0;
    for (int w = 0; w < kSmallWarps; ++w) {
      if (w < R) D.hist[((long long)r * D.ranges_max + w) * NB + tid] = run;
      run += cnt[w][tid];
    }
    total_k = run;
    D.grp[(long long)r * D.groups_max * NB + tid] = 0;  // one group
  }
  long long all;
  const long long start = block_exclusive_scan(total_k, warp_sums, &all);
  if (tid < NB) {
    D.key_start[(long long)r * NB + tid] = start;
    D.key_total[(long long)r * NB + tid] = total_k;
  }
  __syncthreads();
  if (tid < D.W) {
    long long sum = 0;
    for (int k = 0; k < D.K; ++k) sum += __ldcg(D.key_total + (long long)r * NB + tid * D.K + k);
    D.S[(long long)r * D.W + tid] = sum;
  }
}

// Position of item i (key k) of rank r in the rank's key order, less its
// inrank byte: items of smaller keys, of key k in earlier groups and in
// earlier ranges of its group.
__device__ __forceinline__ long long key_base(const DispatchParams& D, int r, long long i, int k) {
  const int NB = D.W * D.K;
  const long long j = i >> 8, c = j >> D.group_log2;
  return D.key_start[(long long)r * NB + k] + D.grp[((long long)r * D.groups_max + c) * NB + k] +
         D.hist[((long long)r * D.ranges_max + j) * NB + k];
}

// Defensive check of a computed position: it must lie in its destination's
// group of the rank's key order, [in_off[r][p], in_off[r][p] + S[r][p]).
// Positions are derived from validated keys, so this never fails unless the
// position arithmetic itself is wrong; if it did, the row is not copied (no
// write outside the outputs) and A2AV_ERR_BAD_INDEX is recorded.
__device__ __forceinline__ bool in_group(const Plan& pl, int r, int p, long long pos, int* status) {
  const long long lo = pl.in_off[r][p];
  if (pos >= lo && pos < lo + pl.s[r][p]) return true;
  record_error(status, A2AV_ERR_BAD_INDEX);
  return false;
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

// Place and copy (rows shorter than 64 bytes): warp w takes one range of 256
// items; its keys and source rows and the range's key bases (key_base for
// every key, into shared memory) are loaded at once; the warp ranks the
// items 32 at a time (ballots on the key; the count kernel only counted
// them on this path), then each lane puts its items' rows straight at their
// place in the output of their destination and publishes their positions.  Every CTA first repeats
// the a2av prologue's checks on the whole split matrix (so all reach the
// same verdict) and derives its rank's row displacement per peer.  Two warps
// per CTA, registers capped so that a whole GPU of them is resident at once.
#ifndef A2AV_PLACE_WARPS
#define A2AV_PLACE_WARPS 2
#endif
#ifndef A2AV_PLACE_MIN_CTAS
#define A2AV_PLACE_MIN_CTAS 18
#endif
constexpr int kPlaceWarps = A2AV_PLACE_WARPS;

__global__ void __launch_bounds__(32 * kPlaceWarps, A2AV_PLACE_MIN_CTAS)
    dispatch_place_copy_kernel(const __grid_constant__ Params P,
                               const __grid_constant__ DispatchParams D) {
  chain_wait();
  chain_release();
  if (flagged(D)) return;
  const int r = blockIdx.y, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int W = D.W, K = D.K, NB = W * K;
  const long long range = (long long)blockIdx.x * kPlaceWarps + warp;
  const long long i0 = range * kRange, m = D.items[r];
  const bool live = i0 < m;
  extern __shared__ int place_base[];  // [kPlaceWarps][NB]
  __shared__ long long disp[kMaxW];    // out_off[p][r] - in_off[r][p], rows
  __shared__ long long glo[kMaxW], gcnt[kMaxW];  // in_off[r][p], S[r][p]: p's group
  __shared__ int bad_splits;
  int keys[kRange / 32], srcs[kRange / 32];
  int* base = place_base + warp * NB;  // the next position of each key in this range
  if (live) {
    const int* const kp = D.key[r];
    const int* const sp = D.src[r];
#pragma unroll
    for (int c = 0; c < kRange / 32; ++c) {  // (unconditional loads, as in the count kernel)
      const long long i = i0 + c * 32 + lane;
      const long long ii = i < m ? i : m - 1;
      keys[c] = __ldg(kp + ii);
      srcs[c] = __ldg(sp + ii);
    }
    for (int k = lane; k < NB; k += 32) base[k] = (int)key_base(D, r, i0, k);
  }
  if (warp == 0) {
    // The a2av prologue's checks on the whole split matrix (identical in
    // every CTA, so all reach the same verdict): lane p owns column p and
    // row p.  S was completed by the count (or scan) kernel.
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
    if (p < W) {
      disp[p] = above - in_off;
      glo[p] = in_off;
      gcnt[p] = own;
    }
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
  if (bad_splits || !live) return;
  // the range's items ranked 32 at a time (ballots on the key), in order
  int pos32[kRange / 32];
  {
    const unsigned lt = (1u << lane) - 1u;
    const int bits = key_bits(NB);
#pragma unroll
    for (int c = 0; c < kRange / 32; ++c) {
      const bool v = i0 + c * 32 + lane < m;
      const int k = keys[c];
      const unsigned same = same_key_lanes(k, v, bits);
      pos32[c] = v ? base[k] + __popc(same & lt) : 0;
      __syncwarp();
      if (v && lane == 31 - __clz(same)) base[k] += __popc(same);
      __syncwarp();
    }
  }
  const long long rb = P.rb;
#pragma unroll
  for (int c = 0; c < kRange / 32; ++c) {
    const long long i = i0 + c * 32 + lane;
    if (i >= m) continue;
    const int p = keys[c] / K;
    const long long pos = pos32[c];
    D.sorted_pos[r][i] = pos;
    if (pos < glo[p] || pos >= glo[p] + gcnt[p]) {  // never: see in_group
      record_error(D.status, A2AV_ERR_BAD_INDEX);
      continue;
    }
    copy_row_thread(P.out[p] + (disp[p] + pos) * rb, P.in[r] + (long long)srcs[c] * rb, rb);
  }
}

// ------------------------------------------------------------ one launch --
// The whole ordering in one cooperative launch (every CTA resident at once)
// when every item fits the grid's registers: CTA b takes a chunk of
// consecutive items of one rank, warp w of it a run of at most kOrderRunMax
// consecutive items of the chunk.
//   1. Each warp loads its run's keys and source rows (validated, kept in
//      registers); the CTA counts its keys with shared atomics, publishes
//      them to cta_cnt[b][*] and adds its counts per destination to S[r][*]
//      (cleared with the flag), then arrives at a grid barrier (bounded:
//      A2AV_ERR_TIMEOUT after ~1 s).
//   2. While the other CTAs arrive, each warp ranks its run's items 32 at a
//      time (ballots on the key), keeping every item's rank among the run's
//      equal keys beside its key, and the runs' counts become their offsets
//      in the chunk; then the CTA waits at the barrier.
//   3. Every CTA loads the counts of its rank's CTAs, builds the plan from
//      the completed S (the a2av prologue's checks) while they are in
//      flight, sums them -- over all of the rank's CTAs (the key totals,
//      whose exclusive scan gives the key starts) and over the earlier ones
//      (its chunk's base per key) -- and adds those bases to the runs'
//      offsets; an item's position is its run's offset for its key plus its
//      rank.  Positions go to sorted_pos; rows under 64 bytes are copied
//      here (kRow != 0), longer ones by the copy kernel that follows.
constexpr int kOrderWarps = 16, kOrderThreads = 32 * kOrderWarps;
constexpr int kOrderIpt = 10;                          // items a lane holds
constexpr long long kOrderRunMax = 32LL * kOrderIpt;   // items of a warp's run
constexpr long long kOrderCtaItems = kOrderWarps * kOrderRunMax;
constexpr int kOrderPrefixLoads = 16;  // most 16-byte count loads a thread makes in step 3
#ifndef A2AV_ORDER_PREFIX_BATCH
#define A2AV_ORDER_PREFIX_BATCH 4
#endif
constexpr int kOrderPrefixBatch = A2AV_ORDER_PREFIX_BATCH;  // of them in flight at once
constexpr int kOrderBarrierOffset = 192;  // workspace byte of the grid barrier's counter
constexpr int kOrderKeyBits = 10;          // a key and its rank in the run share an int
static_assert(kMaxBins <= (1 << kOrderKeyBits) && kOrderRunMax < (1 << (31 - kOrderKeyBits)),
              "key and rank fit one int");
static_assert(kMaxBins <= 2 * kOrderThreads, "the key scan holds two keys a thread");

// Exclusive scan over the CTA of one value per thread (NT threads); *total
// gets the sum.  `warp_sums` holds NT / 32 entries.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan_int(int x, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  int base = 0, all = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    if (w < warp) base += warp_sums[w];
    all += warp_sums[w];
  }
  *total = all;
  __syncthreads();
  return base + inc - x;
}

#ifndef A2AV_BARRIER_SLEEP_NS
#define A2AV_BARRIER_SLEEP_NS 32
#endif
// A grid barrier in two halves, so that a CTA can work between its arrival
// and its wait.  The counter starts at zero (the workspace memset) and serves
// one barrier.  Arrival: after a block barrier, thread 0 publishes the CTA's
// writes (fence) and counts itself in.
__device__ __forceinline__ void grid_arrive(unsigned* ctr) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
  }
}

// One thread polls (bounded) until all `ctas` CTAs have arrived; false when
// the wait ran out.  The fence after the relaxed polls orders the thread's
// later reads after the other CTAs' published writes.
__device__ __forceinline__ bool grid_poll(unsigned* ctr, unsigned ctas) {
  const long long start = clock64();
  bool ok = false;
  for (;;) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= ctas) {
      ok = true;
      break;
    }
    if (clock64() - start > kWaitCycles) break;
    if (A2AV_BARRIER_SLEEP_NS > 0) __nanosleep(A2AV_BARRIER_SLEEP_NS);
  }
  __threadfence();
  return ok;
}

// The whole CTA waits (thread 0 polls); false (in every thread) when the wait
// ran out.
__device__ __forceinline__ bool grid_wait(unsigned* ctr, unsigned ctas) {
  __shared__ int passed;
  if (threadIdx.x == 0) passed = grid_poll(ctr, ctas) ? 1 : 0;
  __syncthreads();
  return passed != 0;
}

__device__ __forceinline__ bool grid_barrier(unsigned* ctr, unsigned ctas) {
  grid_arrive(ctr);
  return grid_wait(ctr, ctas);
}

// Step 3's last part for a lane's items: position (its run's base for its
// key plus its rank), published; with T a row type (rows of exactly sizeof(T)
// bytes at that alignment) every row is loaded first, then stored, so that a
// lane's loads are in flight together; T = void: rows of any other size one
// at a time (kCopy), or positions only.
template <typename T, bool kCopy>
__device__ __forceinline__ void order_place(const Params& P, const DispatchParams& D,
                                            const Plan& pl, int r, long long w0, int lane, int nc,
                                            const int* wb, const int* keys, const int* srcs) {
  constexpr int kMask = (1 << kOrderKeyBits) - 1;
  long long* const out_pos = D.sorted_pos[r];
  if constexpr (std::is_void<T>::value) {
    const long long rb = P.rb;
#pragma unroll
    for (int c = 0; c < kOrderIpt; ++c) {
      if (c >= nc || keys[c] < 0) continue;
      const int k = keys[c] & kMask, p = k / D.K;
      const long long pos = wb[k] + (keys[c] >> kOrderKeyBits);
      out_pos[w0 + c * 32 + lane] = pos;
      if (kCopy && in_group(pl, r, p, pos, D.status))
        copy_row_thread(P.out[p] + (pl.out_off[p][r] - pl.in_off[r][p] + pos) * rb,
                        P.in[r] + (long long)srcs[c] * rb, rb);
    }
  } else {
    T v[kOrderIpt];
    const T* const in = reinterpret_cast<const T*>(P.in[r]);
#pragma unroll
    for (int c = 0; c < kOrderIpt; ++c)
      if (c < nc && keys[c] >= 0) v[c] = __ldg(in + srcs[c]);
#pragma unroll
    for (int c = 0; c < kOrderIpt; ++c) {
      if (c >= nc || keys[c] < 0) continue;
      const int k = keys[c] & kMask, p = k / D.K;
      const long long pos = wb[k] + (keys[c] >> kOrderKeyBits);
      out_pos[w0 + c * 32 + lane] = pos;
      if (in_group(pl, r, p, pos, D.status))
        reinterpret_cast<T*>(P.out[p])[pl.out_off[p][r] - pl.in_off[r][p] + pos] = v[c];
    }
  }
}

// kRow: 0 -- positions only (rows of 64 bytes or more, copied next); 4, 8,
// 16 -- rows of that many bytes at that alignment, copied here; -1 -- other
// rows under 64 bytes, copied here one at a time.
template <int kRow>
__global__ void __launch_bounds__(kOrderThreads, 2)
    dispatch_order_kernel(const __grid_constant__ Params P, const __grid_constant__ DispatchParams D) {
  chain_release();
  chain_wait();
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int W = D.W, K = D.K, NB = W * K;
  const int b = blockIdx.x;
  int r = 0;
  while (r + 1 < W && D.cta_first[r + 1] <= b) ++r;
  extern __shared__ int order_cnt[];  // [kOrderWarps][NB]: runs' key counts, then bases
  __shared__ int cta_k[kMaxBins];     // the CTA's key counts
  __shared__ int tot_k[kMaxBins], pre_k[kMaxBins];
  __shared__ int dest_cnt[kMaxW];
  __shared__ int warp_sums[kOrderWarps];
  __shared__ Plan pl;
  const int NBP = (NB + 3) & ~3;  // count row stride (int4 loads)
  const long long m = D.items[r];
  const long long lo = (long long)(b - D.cta_first[r]) * D.chunk;
  const long long hi = lo + D.chunk < m ? lo + D.chunk : m;
  const long long run = (D.chunk + 32 * kOrderWarps - 1) / (32 * kOrderWarps) * 32;
  const long long w0 = lo + warp * run, w1 = w0 + run < hi ? w0 + run : hi;
  const int nc = w1 > w0 ? (int)((w1 - w0 + 31) / 32) : 0;  // warp-uniform
  for (int e = t; e < kOrderWarps * NB; e += kOrderThreads) order_cnt[e] = 0;
  for (int e = t; e < NBP; e += kOrderThreads) cta_k[e] = tot_k[e] = pre_k[e] = 0;
  if (t < W) dest_cnt[t] = 0;

  // 1. load and validate; count the CTA's keys (shared atomics) and publish
  const int* const kp = D.key[r];
  const int* const sp = D.src[r];
  const long long rows_r = D.rows[r];
  // keys[c]: the item's key, then key | rank << kOrderKeyBits (-1: no item)
  int keys[kOrderIpt], srcs[kOrderIpt];
#pragma unroll
  for (int c = 0; c < kOrderIpt; ++c) {  // (unconditional loads, clamped index)
    keys[c] = -1;
    srcs[c] = 0;
    if (c < nc) {
      const long long i = w0 + c * 32 + lane;
      const long long ii = i < w1 ? i : w1 - 1;
      keys[c] = __ldg(kp + ii);
      srcs[c] = __ldg(sp + ii);
    }
  }
  int bad = 0;
#pragma unroll
  for (int c = 0; c < kOrderIpt; ++c) {
    const long long i = w0 + c * 32 + lane;
    const bool in = c < nc && i < w1;
    const bool ok = in && keys[c] >= 0 && keys[c] < NB && srcs[c] >= 0 && srcs[c] < rows_r;
    if (in && !ok) bad = 1;
    keys[c] = ok ? keys[c] : -1;
  }
  __syncthreads();  // (counters zeroed)
#pragma unroll
  for (int c = 0; c < kOrderIpt; ++c)
    if (keys[c] >= 0) atomicAdd(&cta_k[keys[c]], 1);
  if (__syncthreads_or(bad)) {
    if (t == 0) fail(D, A2AV_ERR_BAD_INDEX);
  } else {
    for (int k = t; k < NBP; k += kOrderThreads) {
      const int sum = cta_k[k];  // (0 in the padding)
      D.cta_cnt[(long long)b * NBP + k] = sum;
      if (sum != 0) atomicAdd(&dest_cnt[k / K], sum);
    }
    __syncthreads();
    if (t < W && dest_cnt[t] != 0)
      atomicAdd(reinterpret_cast<unsigned long long*>(D.S + (long long)r * W + t),
                (unsigned long long)dest_cnt[t]);
  }
  grid_arrive(D.barrier);

  // 2. while the other CTAs arrive: rank each run's items 32 at a time
  // (ballots on the key) and turn the runs' counts into their offsets in
  // the chunk, key by key (ranking after the wait, beside the loads of
  // step 3, measured slower: 25.6 against 23.6 us on the embedding keys)
  {
    int* cnt = order_cnt + warp * NB;
    const unsigned lt = (1u << lane) - 1u;
    const int bits = key_bits(NB);
#pragma unroll
    for (int c = 0; c < kOrderIpt; ++c) {
      if (c < nc) {
        const int k = keys[c];
        const unsigned same = same_key_lanes(k, k >= 0, bits);
        if (k >= 0) keys[c] = k | (cnt[k] + __popc(same & lt)) << kOrderKeyBits;
        __syncwarp();
        if (k >= 0 && lane == 31 - __clz(same)) cnt[k] += __popc(same);
        __syncwarp();
      }
    }
  }
  __syncthreads();
  for (int k = t; k < NB; k += kOrderThreads) {
    int base = 0;
#pragma unroll 4
    for (int w = 0; w < kOrderWarps; ++w) {
      const int c = order_cnt[w * NB + k];
      order_cnt[w * NB + k] = base;
      base += c;
    }
  }
  if (!grid_wait(D.barrier, gridDim.x + (P.starve == 2))) {  // (also publishes order_cnt)
    if (t == 0) fail(D, A2AV_ERR_TIMEOUT);
    return;
  }
  if (flagged(D)) return;

  // 3. the counts of the rank's CTAs (int4 loads: thread t takes keys
  // 4q .. 4q + 3, q = t % Q, of every S-th CTA from t / Q), issued before
  // the plan is built; sums over all of them (key totals) and over the
  // earlier ones (the chunk's base per key)
  const int c0 = D.cta_first[r], gr = D.cta_first[r + 1] - c0;
  const int Q = NBP / 4, S = kOrderThreads / Q, q = t % Q, s0 = t / Q;
  int tot4[4] = {0, 0, 0, 0}, pre4[4] = {0, 0, 0, 0};
  {
    const int4* const cnt4 = reinterpret_cast<const int4*>(D.cta_cnt);
    int4 v[kOrderPrefixBatch];
    auto load = [&](int j0) {
#pragma unroll
      for (int u = 0; u < kOrderPrefixBatch; ++u) {
        const int j = j0 + u * S;
        v[u] = make_int4(0, 0, 0, 0);
        if (s0 < S && j < gr) v[u] = __ldcg(cnt4 + (long long)(c0 + j) * Q + q);
      }
    };
    load(s0);
    if (!build_plan(P, pl, kTileGranule)) return;  // (while the first loads are in flight)
    for (int j0 = s0; j0 < gr; j0 += kOrderPrefixBatch * S) {
      if (j0 != s0) load(j0);
#pragma unroll
      for (int u = 0; u < kOrderPrefixBatch; ++u) {
        const int e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        const bool earlier = c0 + j0 + u * S < b;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          tot4[i] += e[i];
          if (earlier) pre4[i] += e[i];
        }
      }
    }
  }
  if (b == 0 && D.in_splits_out != nullptr)
    for (int e = t; e < W * W; e += kOrderThreads) D.in_splits_out[e] = pl.s[e / W][e % W];
  if (s0 < S)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (tot4[i] != 0) atomicAdd(&tot_k[4 * q + i], tot4[i]);
      if (pre4[i] != 0) atomicAdd(&pre_k[4 * q + i], pre4[i]);
    }
  __syncthreads();
  {  // key starts (two keys a thread) plus the chunk's base
    const int k0 = 2 * t;
    const int x0 = k0 < NB ? tot_k[k0] : 0, x1 = k0 + 1 < NB ? tot_k[k0 + 1] : 0;
    int all;
    const int start = block_exclusive_scan_int<kOrderThreads>(x0 + x1, warp_sums, &all);
    if (k0 < NB) pre_k[k0] += start;
    if (k0 + 1 < NB) pre_k[k0 + 1] += start + x0;
  }
  __syncthreads();
  for (int e = t; e < kOrderWarps * NB; e += kOrderThreads) order_cnt[e] += pre_k[e % NB];
  __syncthreads();
  const int* const wb = order_cnt + warp * NB;
  if constexpr (kRow == 4)
    order_place<unsigned, true>(P, D, pl, r, w0, lane, nc, wb, keys, srcs);
  else if constexpr (kRow == 8)
    order_place<unsigned long long, true>(P, D, pl, r, w0, lane, nc, wb, keys, srcs);
  else if constexpr (kRow == 16)
    order_place<uint4, true>(P, D, pl, r, w0, lane, nc, wb, keys, srcs);
  else
    order_place<void, kRow != 0>(P, D, pl, r, w0, lane, nc, wb, keys, srcs);
}

// The fused combine of rows under 64 bytes in one cooperative launch, items
// partitioned as in the order kernel: every CTA loads its items' keys and
// positions, builds the plan from the split matrix while they are in flight
// (the a2av prologue's checks), and checks them (a position must lie in its destination's group
// of the rank's key order), then a grid barrier; if no CTA found an invalid
// item, each moves its items' rows back -- rows of exactly kRow = 4, 8 or 16
// bytes at that alignment all loaded first, then stored; kRow = -1 one row
// at a time.
template <int kRow>
__global__ void __launch_bounds__(kOrderThreads, 2)
    combine_order_kernel(const __grid_constant__ Params P, const __grid_constant__ DispatchParams D) {
  __shared__ Plan pl;
  // the positions come from the previous kernel: wait for it, then load the
  // items' keys and positions and build the plan while they are in flight
  chain_release();
  chain_wait();
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int W = D.W, K = D.K, NB = W * K;
  const int b = blockIdx.x;
  int r = 0;
  while (r + 1 < W && D.cta_first[r + 1] <= b) ++r;
  const long long m = D.items[r];
  const long long lo = (long long)(b - D.cta_first[r]) * D.chunk;
  const long long hi = lo + D.chunk < m ? lo + D.chunk : m;
  const long long run = (D.chunk + 32 * kOrderWarps - 1) / (32 * kOrderWarps) * 32;
  const long long w0 = lo + warp * run, w1 = w0 + run < hi ? w0 + run : hi;
  const int nc = w1 > w0 ? (int)((w1 - w0 + 31) / 32) : 0;  // warp-uniform
  const int* const kp = D.key[r];
  const long long* const pp = D.sorted_pos[r];
  int kraw[kOrderIpt];
  long long praw[kOrderIpt];
#pragma unroll
  for (int c = 0; c < kOrderIpt; ++c) {  // (unconditional loads, clamped index)
    kraw[c] = 0;
    praw[c] = 0;
    if (c < nc) {
      const long long i = w0 + c * 32 + lane;
      const long long ii = i < w1 ? i : w1 - 1;
      kraw[c] = __ldg(kp + ii);
      praw[c] = __ldg(pp + ii);
    }
  }
  if (!build_plan(P, pl, kTileGranule)) return;  // (same verdict in every CTA)
  int keys[kOrderIpt], pos[kOrderIpt];  // -1: no item; positions are below 2^31
#pragma unroll
  for (int c = 0; c < kOrderIpt; ++c) {
    keys[c] = -1;
    pos[c] = 0;
    if (c < nc) {
      const long long i = w0 + c * 32 + lane;
      const int k = kraw[c];
      const long long q = praw[c];
      bool ok = false;
      if (i < w1 && k >= 0 && k < NB) {
        const int p = k / K;
        const long long g0 = pl.in_off[r][p];
        ok = q >= g0 && q < g0 + pl.s[r][p];
      }
      keys[c] = ok ? k : (i < w1 ? -2 : -1);
      pos[c] = ok ? (int)q : 0;
    }
  }
  int bad = 0;
#pragma unroll
  for (int c = 0; c < kOrderIpt; ++c) bad |= keys[c] == -2;
  if (__syncthreads_or(bad) && t == 0) fail(D, A2AV_ERR_BAD_INDEX);
  if (!grid_barrier(D.barrier, gridDim.x + (P.starve == 2))) {
    if (t == 0) fail(D, A2AV_ERR_TIMEOUT);
    return;
  }
  if (flagged(D)) return;
  const long long rb = P.rb;
  unsigned char* const own = const_cast<unsigned char*>(P.in[r]);
  if constexpr (kRow > 0) {
    using T = typename std::conditional<
        kRow == 4, unsigned, typename std::conditional<kRow == 8, unsigned long long, uint4>::type>::type;
    T v[kOrderIpt];
#pragma unroll
    for (int c = 0; c < kOrderIpt; ++c)
      if (keys[c] >= 0) {
        const int p = keys[c] / K;
        v[c] = __ldg(reinterpret_cast<const T*>(P.out[p]) + (pl.out_off[p][r] - pl.in_off[r][p] + pos[c]));
      }
#pragma unroll
    for (int c = 0; c < kOrderIpt; ++c)
      if (keys[c] >= 0) reinterpret_cast<T*>(own)[w0 + c * 32 + lane] = v[c];
  } else {
#pragma unroll
    for (int c = 0; c < kOrderIpt; ++c)
      if (keys[c] >= 0) {
        const int p = keys[c] / K;
        copy_row_thread(own + (w0 + c * 32 + lane) * rb,
                        P.out[p] + (pl.out_off[p][r] - pl.in_off[r][p] + pos[c]) * rb, rb);
      }
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

// Register copies (rows the gather does not take):
// kWarpRows -- rows of kWarpRowBytes or more, a warp per batch of rows; else
// a thread per row.  kRows512: every row and buffer 16-byte aligned and rows
// a multiple of 512 bytes (the host checks).  Each instantiation holds one
// loop, so none pays another's registers.
#ifndef A2AV_ROWS512_CTAS_PER_SM
#define A2AV_ROWS512_CTAS_PER_SM 4  // 64 registers: four CTAs an SM, 2 KiB a warp in flight
#endif
constexpr int kRows512CtasPerSm = A2AV_ROWS512_CTAS_PER_SM;
#ifndef A2AV_COPY_PRELOAD
#define A2AV_COPY_PRELOAD 1
#endif
template <bool kWarpRows, bool kRows512 = false>
__global__ void __launch_bounds__(kCopyThreads, kRows512    ? kRows512CtasPerSm
                                                : kWarpRows ? kCopyCtasPerSmWarpRows
                                                            : kCopyCtasPerSm)
    dispatch_copy_kernel(const __grid_constant__ Params P, const __grid_constant__ DispatchParams D) {
  chain_wait();
  if (flagged(D)) return;
  const int W = D.W, K = D.K;
  const long long rb = P.rb, total = D.item_first[W];
  constexpr bool warp_rows = kWarpRows;
  const long long team = warp_rows ? (long long)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5)
                                   : (long long)blockIdx.x * kCopyThreads + threadIdx.x;
  const long long teams = warp_rows ? (long long)gridDim.x * (kCopyThreads / 32)
                                    : (long long)gridDim.x * kCopyThreads;
  const long long rounds = (total + teams * 32 - 1) / (teams * 32);
  const long long batch = rounds > 0 ? (total + teams * rounds - 1) / (teams * rounds) : 32;
  // (512-byte pieces, the dispatch) the first batch's keys, source rows and
  // in-range ranks are loaded before the plan is built
  const bool pre = kRows512 && !D.combine && !D.pos_ready && A2AV_COPY_PRELOAD;
  int pre_k = 0, pre_s = 0, pre_in = 0;
  if (pre) {
    const long long g = team * batch + (threadIdx.x & 31);
    if (team * batch < total && g < total && (threadIdx.x & 31) < batch) {
      int r = 0;
      while (r + 1 < W && D.item_first[r + 1] <= g) ++r;
      const long long i = g - D.item_first[r];
      pre_k = D.key[r][i];
      pre_s = D.src[r][i];
      pre_in = D.inrank[(long long)r * D.pos_stride + i];
    }
  }
  __shared__ Plan pl;
  if (!build_plan(P, pl, kTileGranule)) return;
  publish_splits(D);
  if constexpr (warp_rows) {
    // A warp takes a batch of up to 32 consecutive items: lane l reads item
    // l's metadata (one round trip for the batch, a second for the key
    // bases), then the warp copies the batch's rows.  16-byte aligned rows
    // are copied as one flat run of vectors over the batch, kVecRows x 16
    // bytes per lane in flight; other rows one at a time with the
    // realigning span copy.  The batch size gives every warp the same
    // number of batches.
    const int lane = threadIdx.x & 31;
    for (long long g0 = team * batch; g0 < total; g0 += teams * batch) {
      const long long g = g0 + lane;
      const int n = total - g0 < batch ? (int)(total - g0) : (int)batch;
      const bool first = pre && g0 == team * batch;  // this batch's metadata loaded already
      long long mdst = 0, msrc = 0;
      if (lane < n) {
        int r = 0;
        while (r + 1 < W && D.item_first[r + 1] <= g) ++r;
        const long long i = g - D.item_first[r];
        const int k = first ? pre_k : D.key[r][i];
        const int p = k / K;
        const long long grouped = pl.out_off[p][r] - pl.in_off[r][p];  // + pos: the row in p's buffer
        if (D.combine) {  // from the peer's buffer back to the item's row
          msrc = (long long)(P.out[p] + (grouped + D.sorted_pos[r][i]) * rb);
          mdst = (long long)(P.in[r] + i * rb);
        } else {
          const int s = first ? pre_s : D.src[r][i];
          long long pos;
          if (D.pos_ready) {
            pos = D.sorted_pos[r][i];
          } else {
            pos = key_base(D, r, i, k) +
                  (first ? pre_in : (int)D.inrank[(long long)r * D.pos_stride + i]);
            D.sorted_pos[r][i] = pos;
          }
          mdst = (long long)(P.out[p] + (grouped + pos) * rb);
          msrc = (long long)(P.in[r] + (long long)s * rb);
          if (!in_group(pl, r, p, pos, D.status)) mdst = msrc = 0;
        }
      }
      if (!D.combine && __any_sync(kFull, lane < n && mdst == 0)) continue;  // (never: in_group)
      if constexpr (kRows512) {
        // rows of a multiple of 512 bytes: lane l takes pieces l, l + 32, ...
        // of every row; (row, piece) advance by a counter, no division.
        // Consecutive items with the same source row (a token routed to
        // several experts) form a run: the row is loaded once and stored to
        // every destination of the run.  `heads` marks the first item of
        // each run; the loop walks the runs in order with the current run
        // [h, hn) warp-uniform.
        const long long prev = __shfl_up_sync(kFull, msrc, 1);
        unsigned hm = __ballot_sync(kFull, lane < n && (lane == 0 || prev != msrc));
        const int nu = __popc(hm);
        auto next_head = [&](unsigned m) { return m != 0u ? __ffs(m) - 1 : n; };
        int h = next_head(hm), hn = next_head(hm & (hm - 1u));
        const unsigned vpl = (unsigned)(rb >> 9), np = (unsigned)nu * vpl;  // a lane's pieces
        unsigned c = 0;
        for (unsigned b0 = 0; b0 < np; b0 += kVecRows) {  // warp-uniform trip count
          uint4 v[kVecRows];
          int first[kVecRows], end[kVecRows];
          long long off[kVecRows];
#pragma unroll
          for (int q = 0; q < kVecRows; ++q) {
            const bool ok = b0 + q < np;
            first[q] = h;
            end[q] = hn;
            const long long s = __shfl_sync(kFull, msrc, h & 31);
            off[q] = 16LL * (lane + 32 * c);
            if (ok) v[q] = ld_stream(reinterpret_cast<const uint4*>(s + off[q]));
            if (++c == vpl) {  // the next run
              c = 0;
              hm &= hm - 1u;
              h = hn;
              hn = next_head(hm & (hm - 1u));
            }
          }
#pragma unroll
          for (int q = 0; q < kVecRows; ++q) {
            if (b0 + q >= np) continue;  // (warp-uniform)
            for (int e = first[q]; e < end[q]; ++e)
              st_stream(reinterpret_cast<uint4*>(__shfl_sync(kFull, mdst, e) + off[q]), v[q]);
          }
        }
      } else if (D.vec16 && rb <= kVecMaxRow) {
        const unsigned V = (unsigned)(rb >> 4), nv = (unsigned)n * V;  // < 2^17
        for (unsigned b0 = 0; b0 < nv; b0 += 32 * kVecRows) {  // warp-uniform trip count
          uint4 v[kVecRows];
          long long d[kVecRows];
#pragma unroll
          for (int q = 0; q < kVecRows; ++q) {
            const unsigned idx = b0 + q * 32 + lane;
            const bool ok = idx < nv;
            const unsigned j = ok ? idx / V : 0, c = ok ? idx - j * V : 0;
            const long long s = __shfl_sync(kFull, msrc, (int)j);
            d[q] = __shfl_sync(kFull, mdst, (int)j) + 16LL * c;
            if (ok) v[q] = ld_stream(reinterpret_cast<const uint4*>(s) + c);
          }
#pragma unroll
          for (int q = 0; q < kVecRows; ++q)
            if (b0 + q * 32 + lane < nv) st_stream(reinterpret_cast<uint4*>(d[q]), v[q]);
        }
      } else {
        copy_rows_unaligned(mdst, msrc, n, rb, lane);
      }
    }
  } else {
  // Short rows: a thread takes kItemsPerThread items, their metadata loads
  // issued together, then copies the rows.
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
          pos[q] = D.pos_ready ? D.sorted_pos[r][i] : D.inrank[(long long)r * D.pos_stride + i];
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kItemsPerThread; ++q) {
      const int r = rank[q];
      if (r < 0 || D.combine) continue;
      const long long i = g0 + q * teams - D.item_first[r];
      if (!D.pos_ready) {
        pos[q] += key_base(D, r, i, key[q]);
        D.sorted_pos[r][i] = pos[q];
      }
      if (!in_group(pl, r, key[q] / K, pos[q], D.status)) rank[q] = -1;
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
// Whether the items [g0 + u * stride] (u < B, below total) all have a valid
// key and a position in their destination's group; their keys and positions
// are loaded together.
template <int B>
__device__ __forceinline__ bool combine_items_ok(const DispatchParams& D, const Plan& pl,
                                                 long long g0, long long stride, long long total) {
  const int W = D.W, K = D.K, NB = W * K;
  int key[B], rank[B];
  long long pos[B];
#pragma unroll
  for (int u = 0; u < B; ++u) {
    const long long g = g0 + u * stride;
    rank[u] = -1;
    if (g < total) {
      int r = 0;
      while (r + 1 < W && D.item_first[r + 1] <= g) ++r;
      const long long i = g - D.item_first[r];
      rank[u] = r;
      key[u] = D.key[r][i];
      pos[u] = D.sorted_pos[r][i];
    }
  }
  bool ok = true;
#pragma unroll
  for (int u = 0; u < B; ++u) {
    const int r = rank[u];
    if (r < 0) continue;
    if (key[u] < 0 || key[u] >= NB) {
      ok = false;
      continue;
    }
    const int p = key[u] / K;
    const long long lo = pl.in_off[r][p];
    if (pos[u] < lo || pos[u] >= lo + pl.s[r][p]) ok = false;
  }
  return ok;
}

// Every item of the combine checked by the whole grid (thread x of the grid
// takes items x, x + G, ... in batches of B); true (in every thread of the
// CTA) when the CTA found no invalid item -- else it has raised the flag and
// recorded A2AV_ERR_BAD_INDEX.
template <int B>
__device__ __forceinline__ bool combine_check_all(const DispatchParams& D, const Plan& pl) {
  const long long total = D.item_first[D.W];
  const long long G = (long long)gridDim.x * blockDim.x;
  int bad = 0;
  for (long long g0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; g0 < total; g0 += B * G)
    if (!combine_items_ok<B>(D, pl, g0, G, total)) bad = 1;
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) fail(D, A2AV_ERR_BAD_INDEX);
    return false;
  }
  return true;
}

__global__ void __launch_bounds__(kCopyThreads)
    combine_check_kernel(const __grid_constant__ Params P, const __grid_constant__ DispatchParams D) {
  chain_wait();
  chain_release();
  __shared__ Plan pl;
  if (!build_plan(P, pl, kTileGranule)) return;
  combine_check_all<4>(D, pl);
}

// ------------------------------------------------------------- gather --
// One lane's item of a gather batch: where it is and its raw metadata.
struct GatherItem {
  long long i;     // index within its rank
  long long spos;  // combine: the item's position in its rank's key order
  int r, key, src, inr;
  bool v;          // the lane holds an item
};

// Item g of the global order (rank-major) when `ok`, else none.
__device__ __forceinline__ GatherItem gather_item_at(const DispatchParams& D, long long g, bool ok) {
  GatherItem x;
  x.i = 0;
  x.spos = 0;
  x.r = 0;
  x.key = 0;
  x.src = 0;
  x.inr = 0;
  x.v = false;
  if (!ok) return x;
  int r = 0;
  while (r + 1 < D.W && D.item_first[r + 1] <= g) ++r;
  const long long i = g - D.item_first[r];
  x.r = r;
  x.i = i;
  x.v = true;
  x.key = D.key[r][i];
  if (D.combine || D.pos_ready) x.spos = D.sorted_pos[r][i];
  if (!D.combine) {
    x.src = D.src[r][i];
    if (!D.pos_ready) x.inr = D.inrank[(long long)r * D.pos_stride + i];
  }
  return x;
}

// Batch b (global over the ranks, bs items each) -> lane's item; b < 0: none.
__device__ __forceinline__ GatherItem gather_item(const DispatchParams& D, long long b, int lane) {
  GatherItem x;
  x.i = 0;
  x.spos = 0;
  x.r = 0;
  x.key = 0;
  x.src = 0;
  x.inr = 0;
  x.v = false;
  if (b < 0) return x;
  int r = 0;
  while (r + 1 < D.W && D.batch_first[r + 1] <= b) ++r;
  const long long i = (b - D.batch_first[r]) * D.bs + lane;
  x.r = r;
  x.i = i;
  if (lane < D.bs && i < D.items[r]) {
    x.v = true;
    x.key = D.key[r][i];
    if (D.combine || D.pos_ready) x.spos = D.sorted_pos[r][i];
    if (!D.combine) {
      x.src = D.src[r][i];
      if (!D.pos_ready) x.inr = D.inrank[(long long)r * D.pos_stride + i];
    }
  }
  return x;
}

// The cp.async.bulk gather for 16-byte aligned rows of 64 B .. 32 KiB.  NWK
// warps per CTA, each an independent pipeline with a ring of NS stages of
// IPS row slots (its own mbarriers, its own bulk groups).  Rings of one row
// a stage (IPS == 1) run the one-row loop below: the warp's k-th row is item
// wg + k WG of the global order, lane 0 loads row k and stores row k - LEAD.
// Rings of several rows a stage: a warp takes every
// (grid x NWK)-th batch of bs consecutive items of one rank; a batch is
// copied as bs / min(bs, IPS) stages.  In a stage every lane that holds an
// item issues the bulk load of its row into its slot (one mbarrier per
// stage, armed by lane 0 with the stage's byte count); LEAD stages later the
// lanes wait for the stage and issue one bulk store each (the combine: one
// store of the whole stage, whose rows are consecutive items of one rank),
// and every lane commits one bulk group per stage, so that
// cp.async.bulk.wait_group.read NS - LEAD - 1 frees the stage reused next.
// A batch's addresses need two dependent round trips (its keys, then their
// key bases), so they are loaded two and one batches ahead.  Waits are
// bounded: on a timeout the warp records A2AV_ERR_TIMEOUT, waits (bounded)
// for every load it issued and leaves.
#ifndef A2AV_GATHER_ROW_LANE0
#define A2AV_GATHER_ROW_LANE0 0
#endif
#ifndef A2AV_GATHER_SIMPLE_COMBINE
#define A2AV_GATHER_SIMPLE_COMBINE 1
#endif
#ifndef A2AV_GATHER_SIMPLE_DISPATCH
#define A2AV_GATHER_SIMPLE_DISPATCH 1
#endif
#ifndef A2AV_GATHER_EARLY
#define A2AV_GATHER_EARLY 1
#endif
constexpr int kGatherSmemBound = 192 * 1024;  // the stages' dynamic shared memory (kGatherSmem)
template <int NS, int LEAD, int NWK, int IPS>
__global__ void __launch_bounds__(32 * NWK, 1)
    dispatch_gather_kernel(const __grid_constant__ Params P, const __grid_constant__ DispatchParams D) {
  static_assert(LEAD >= 1 && LEAD < NS, "loads run 1..NS-1 stages ahead of stores");
  static_assert(NWK >= 1 && NWK <= 16 && IPS >= 1 && IPS <= 32 && (IPS & (IPS - 1)) == 0,
                "one to sixteen warps, a power-of-two number of slots per stage");
  static_assert(sizeof(Plan) + NWK * NS * (8 + 8 * IPS + 4) + 256 + kGatherSmemBound <= 227 * 1024,
                "the ring's static shared memory and the stages fit a CTA's 227 KiB");
  chain_wait();
  // (the combine's checking launch follows the workspace clear directly:
  // nothing before it can have raised the flag)
  if (!(D.combine && D.barrier != nullptr) && flagged(D)) return;
  __shared__ Plan pl;
  __shared__ alignas(8) unsigned long long bars[NWK][NS];
  __shared__ unsigned long long sdst[NWK][NS][IPS];  // each slot's destination
  __shared__ unsigned smask[NWK][NS];               // slots holding a row, per stage
  extern __shared__ __align__(128) unsigned char stages[];
  if (!build_plan(P, pl, kTileGranule)) return;
  publish_splits(D);
  // The combine's checks in this launch (cooperative: every CTA resident):
  // the whole grid checks every item (few threads: 16 items a thread in
  // flight), then a grid barrier; no row is stored unless every CTA found its
  // items valid.  With several rows a stage each warp waits at the barrier
  // only before its first store (`gate`): its first LEAD stages load, from
  // items it checked itself, while the last CTAs finish their checks.
  const unsigned ctas = gridDim.x + (P.starve == 2);
  bool gate = false;
  if (D.combine && D.barrier != nullptr) {
    combine_check_all<16>(D, pl);
    grid_arrive(D.barrier);
    if (IPS == 1 || !A2AV_GATHER_EARLY) {
      if (!grid_wait(D.barrier, ctas)) {
        if (threadIdx.x == 0) fail(D, A2AV_ERR_TIMEOUT);
        return;
      }
      if (flagged(D)) return;
    } else {
      gate = true;
    }
  }
  const int lane = threadIdx.x & 31;
  const int warp = NWK == 1 ? 0 : (int)(threadIdx.x >> 5);  // a constant for one warp
  // One-row stages (IPS == 1) take the items in a strided order: the warp's
  // k-th row is item wg + k WG of the global order, so that the warps of the
  // grid work on neighbouring items at any time.  Otherwise batches of bs
  // consecutive items of one rank.  With one row a stage, only lane 0 waits,
  // stores and tracks bulk groups (the row's lane issues its load).
  constexpr bool kStrided = IPS == 1;
  const int W = D.W, K = D.K, bs = kStrided ? 32 : D.bs;
  const int unit = bs < IPS ? bs : IPS, spb = bs / unit;  // slots used per stage, stages per batch
  const long long rb = P.rb;
  const long long WG = (long long)gridDim.x * NWK, wg = (long long)blockIdx.x * NWK + warp;
  const long long total = D.item_first[W], nbatch = D.batch_first[W];
  const long long mine = total > wg ? (total - wg + WG - 1) / WG : 0;  // strided: this warp's items
  const long long nt = kStrided ? (mine + 31) / 32
                                : (nbatch > wg ? (nbatch - wg + WG - 1) / WG : 0);  // its batches
  if (nt == 0) return;
  auto fetch = [&](long long t) -> GatherItem {  // the lane's item of the warp's batch t
    if (kStrided) {
      const long long k = t * 32 + lane;
      return gather_item_at(D, wg + k * WG, t < nt && k < mine);
    }
    return gather_item(D, t < nt ? wg + t * WG : -1, lane);
  };
  const uint32_t stage_bytes = (uint32_t)(IPS * rb);
  const uint32_t bar0 = smem_u32(&bars[warp][0]);
  const uint32_t st0 = smem_u32(stages) + (uint32_t)(NS * warp) * stage_bytes;
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_fence_init();
  }
  __syncwarp();

#if A2AV_GATHER_SIMPLE_COMBINE
  if constexpr (IPS == 1) {
    if (D.combine || A2AV_GATHER_SIMPLE_DISPATCH) {
      // One row a stage: lane 0 issues row k's load and stores row k - LEAD,
      // the rows' addresses fetched 32 at a time (lane l: the warp's row
      // k0 + l).  (Measured against the batched issue below on the MoE
      // combine: 603.4 against 617.6 us at 14 KiB rows, 174.5 against 179.3
      // at 4 KiB, 343.0 against 353.7 at 8 KiB; on the MoE dispatch, with
      // the 14 KiB ring on two warps: 457.6 against 471.4 us at 14 KiB,
      // 147.2 against 148.7 at 4 KiB, 278.9 against 279.5 at 8 KiB.)
      long long msrc = 0, mdst = 0, stored = 0, loaded = 0;
      bool fine = true;
      for (long long k = 0; k < mine + LEAD; ++k) {
        if (k < mine) {
          if ((k & 31) == 0) {
            GatherItem x = gather_item_at(D, wg + (k + lane) * WG, k + lane < mine);
            msrc = mdst = 0;
            if (x.v) {
              const int p = x.key / K;
              const long long grouped = pl.out_off[p][x.r] - pl.in_off[x.r][p];
              if (D.combine) {
                msrc = (long long)(P.out[p] + (grouped + x.spos) * rb);
                mdst = (long long)(P.in[x.r] + x.i * rb);
              } else {
                const long long pos = D.pos_ready ? x.spos : key_base(D, x.r, x.i, x.key) + x.inr;
                if (!D.pos_ready) D.sorted_pos[x.r][x.i] = pos;
                if (in_group(pl, x.r, p, pos, D.status)) {
                  msrc = (long long)(P.in[x.r] + (long long)x.src * rb);
                  mdst = (long long)(P.out[p] + (grouped + pos) * rb);
                }
              }
            }
          }
          const long long src = __shfl_sync(kFull, msrc, (int)(k & 31));
          const long long dst = __shfl_sync(kFull, mdst, (int)(k & 31));
          if (lane == 0) {
            const int s = (int)(k % NS);
            if (k >= NS) bulk_wait_read<NS - LEAD - 1>();
            sdst[warp][s][0] = (unsigned long long)dst;
            if (dst != 0) {
              const unsigned starve =
                  (P.starve == 1 && blockIdx.x == 0 && warp == 0 && k == 0) ? 16u : 0u;
              mbar_expect_tx(bar0 + 8 * s, (unsigned)rb + starve);
              bulk_load(st0 + (uint32_t)s * stage_bytes, reinterpret_cast<const void*>(src),
                        (unsigned)rb, bar0 + 8 * s);
            } else {  // a row whose position failed its check (never): the stage only completes
              mbar_expect_tx(bar0 + 8 * s, 0u);
            }
          }
          loaded = k + 1;
        }
        const long long j = k - LEAD;
        if (j >= 0 && j < mine) {
          const int s = (int)(j % NS);
          bool done = true;
          if (lane == 0) {
            done = mbar_wait(bar0 + 8 * s, (unsigned)((j / NS) & 1));
            if (done && sdst[warp][s][0] != 0)
              bulk_store(reinterpret_cast<void*>(sdst[warp][s][0]), st0 + (uint32_t)s * stage_bytes,
                         (unsigned)rb);
          }
          fine = __shfl_sync(kFull, done ? 1 : 0, 0) != 0;
          if (!fine) break;
          stored = j + 1;
        }
      }
      if (lane == 0) {
        if (!fine) {  // a row never landed: report, let the loads in flight land (bounded)
          record_error(P.status, A2AV_ERR_TIMEOUT);
          for (long long j = stored; j < loaded; ++j)
            mbar_wait(bar0 + 8 * (int)(j % NS), (unsigned)((j / NS) & 1));
        }
        bulk_wait_all();
      }
      return;
    }
  }
#endif

  long long issued = 0, drained = 0;  // stages
  bool ok = true, stop = false;  // stop: the gate found an invalid item somewhere
  // Wait for stage j's loads and store its rows; false on a timeout, or when
  // the gate (before the first store) finds the grid's verdict negative.
  auto drain = [&](long long j) -> bool {
    if (gate) {
      gate = false;
      int g = 0;  // 0: every CTA passed its checks, 1: one failed, 2: the wait ran out
      if (lane == 0) g = !grid_poll(D.barrier, ctas) ? 2 : flagged(D) ? 1 : 0;
      g = __shfl_sync(kFull, g, 0);
      if (g == 2 && lane == 0) fail(D, A2AV_ERR_TIMEOUT);
      if (g != 0) {
        stop = true;
        return false;
      }
    }
    const int s = (int)(j % NS);
    if (IPS == 1) {
      bool done = true;
      if (lane == 0) {
        done = mbar_wait(bar0 + 8 * s, (unsigned)((j / NS) & 1));
        if (done && smask[warp][s] != 0)
          bulk_store(reinterpret_cast<void*>(sdst[warp][s][0]), st0 + (uint32_t)s * stage_bytes,
                     (unsigned)rb);
        else if (done)
          bulk_commit();
      }
      return __shfl_sync(kFull, done ? 1 : 0, 0) != 0;
    }
    if (!mbar_wait_warp(bar0 + 8 * s, (unsigned)((j / NS) & 1))) return false;
    const unsigned mask = smask[warp][s];
    const uint32_t st = st0 + (uint32_t)s * stage_bytes;
    if (D.combine) {  // the slots in use are a prefix, consecutive items of one rank
      if (lane == 0 && mask != 0)
        bulk_store(reinterpret_cast<void*>(sdst[warp][s][0]), st, (unsigned)(__popc(mask) * rb));
      else
        bulk_commit();
    } else if ((mask >> lane) & 1u) {
      bulk_store(reinterpret_cast<void*>(sdst[warp][s][lane]), st + (uint32_t)(lane * rb),
                 (unsigned)rb);
    } else {
      bulk_commit();
    }
    return true;
  };

  GatherItem a0 = fetch(0);
  GatherItem a1 = fetch(1);
  const bool bases = !D.combine && !D.pos_ready;  // positions from key bases + inrank
  long long b0 = a0.v && bases ? key_base(D, a0.r, a0.i, a0.key) : 0;
  for (long long t = 0; t < nt && ok; ++t) {
    const GatherItem a2 = fetch(t + 2);
    const long long b1 = a1.v && bases ? key_base(D, a1.r, a1.i, a1.key) : 0;
    // batch t's row addresses
    long long src = 0, dst = 0;
    // loads ahead of the grid's verdict (the combine's gate): only from items
    // whose key and position are valid
    if (gate && (a0.key < 0 || a0.key >= W * K)) a0.v = false;
    if (a0.v) {
      const int p = a0.key / K;
      const long long grouped = pl.out_off[p][a0.r] - pl.in_off[a0.r][p];
      if (D.combine) {
        const long long lo = pl.in_off[a0.r][p];
        if (gate && (a0.spos < lo || a0.spos >= lo + pl.s[a0.r][p])) a0.v = false;
        src = (long long)(P.out[p] + (grouped + a0.spos) * rb);
        dst = (long long)(P.in[a0.r] + a0.i * rb);
      } else {
        const long long pos = bases ? b0 + a0.inr : a0.spos;
        if (bases) D.sorted_pos[a0.r][a0.i] = pos;
        src = (long long)(P.in[a0.r] + (long long)a0.src * rb);
        dst = (long long)(P.out[p] + (grouped + pos) * rb);
        if (!in_group(pl, a0.r, p, pos, D.status)) a0.v = false;
      }
    }
#if A2AV_GATHER_ROW_LANE0
    if constexpr (IPS == 1) {
      // one row a stage: lane 0 issues the batch's loads one by one
      const unsigned held = __ballot_sync(kFull, a0.v);
      for (int u = 0; u < 32 && ok; ++u) {
        const long long su = __shfl_sync(kFull, src, u), du = __shfl_sync(kFull, dst, u);
        if (!((held >> u) & 1u)) continue;
        if (lane == 0) {
          const int s = (int)(issued % NS);
          if (issued >= NS) bulk_wait_read<NS - LEAD - 1>();
          const uint32_t bar = bar0 + 8 * s;
          sdst[warp][s][0] = (unsigned long long)du;
          smask[warp][s] = 1u;
          const unsigned starve = (P.starve == 1 && blockIdx.x == 0 && warp == 0 && issued == 0) ? 16u : 0u;
          mbar_expect_tx(bar, (unsigned)rb + starve);
          bulk_load(st0 + (uint32_t)s * stage_bytes, reinterpret_cast<const void*>(su),
                    (unsigned)rb, bar);
        }
        ++issued;
        while (issued - drained > LEAD) {
          if (!drain(drained)) {
            ok = false;
            break;
          }
          ++drained;
        }
      }
      a0 = a1;
      a1 = a2;
      b0 = b1;
      continue;
    }
#endif
    for (int u = 0; u < spb; ++u) {
      const int s = (int)(issued % NS);
      if (issued >= NS && (IPS > 1 || lane == 0))
        bulk_wait_read<NS - LEAD - 1>();  // the store that last read stage s
      __syncwarp();
      const int slot = lane - u * unit;
      const bool mine = a0.v && slot >= 0 && slot < unit;
      const unsigned held = __ballot_sync(kFull, mine);
      const unsigned n = __popc(held);
      const uint32_t bar = bar0 + 8 * s;
      if (mine) sdst[warp][s][slot] = (unsigned long long)dst;
      if (lane == 0) {
        smask[warp][s] = unit == 32 ? held : (held >> (u * unit)) & ((1u << unit) - 1u);
        const unsigned starve = (P.starve == 1 && blockIdx.x == 0 && warp == 0 && issued == 0) ? 16u : 0u;
        mbar_expect_tx(bar, (unsigned)(n * rb) + starve);
      }
      __syncwarp();
      if (mine)
        bulk_load(st0 + (uint32_t)s * stage_bytes + (uint32_t)(slot * rb),
                  reinterpret_cast<const void*>(src), (unsigned)rb, bar);
      ++issued;
      while (issued - drained > LEAD) {
        if (!drain(drained)) {
          ok = false;
          break;
        }
        ++drained;
      }
      if (!ok) break;
    }
    a0 = a1;
    a1 = a2;
    b0 = b1;
  }
  while (ok && drained < issued) {
    if (!drain(drained)) {
      ok = false;
      break;
    }
    ++drained;
  }
  if (!ok) {
    // A stage never completed (reported here), or the gate said stop: give
    // every load still in flight a bounded chance to land, then leave.
    if (lane == 0) {
      if (!stop) record_error(P.status, A2AV_ERR_TIMEOUT);
      for (long long j = drained; j < issued; ++j)
        mbar_wait(bar0 + 8 * (int)(j % NS), (unsigned)((j / NS) & 1));
    }
    __syncwarp();
  }
  if (IPS > 1 || lane == 0) bulk_wait_all();
}

// The gather's ring shapes by row size: NWK x NS stages of IPS slots, at most
// 192 KiB of shared memory (1 CTA per SM, 4 x 32 KiB .. 12 x 16 KiB of loads
// in flight per SM).
#ifndef A2AV_GATHER_NS
#define A2AV_GATHER_NS 6
#endif
#ifndef A2AV_GATHER_LEAD
#define A2AV_GATHER_LEAD 4
#endif
// Aligned rows this long or longer take the gather (the combine from
// A2AV_GATHER_MIN_ROW, the dispatch from A2AV_DISPATCH_GATHER_MIN_ROW).
// Measured on the MoE workload (8192 tokens, W=8, us, gather / register warp
// copy): combine 24.3 / 27.6 at 128 B rows, 50.1 / 51.7 at 1 KiB; dispatch
// 34.9 / 31.8 at 128 B, 57.2 / 52.5 at 1 KiB (the dispatch's batch metadata
// -- key bases -- costs the gather's few issuing warps more), and, with the
// register copy loading a token's row once for all its experts, 88.1 / 84.5
// at 2 KiB, 152.5 / 150.9 at 4 KiB (but 150.7 / 155.5 in bench lines taken on
// other boxes), 286.0 / 285.8 at 8 KiB, 476.7 / 485.6 at 14 KiB: the
// dispatch's gather starts above 2 KiB.
#ifndef A2AV_GATHER_MIN_ROW
#define A2AV_GATHER_MIN_ROW 64
#endif
#ifndef A2AV_DISPATCH_GATHER_MIN_ROW
#define A2AV_DISPATCH_GATHER_MIN_ROW 2049
#endif
constexpr int kGatherNs = A2AV_GATHER_NS, kGatherLead = A2AV_GATHER_LEAD;
constexpr long long kGatherMinRow = A2AV_GATHER_MIN_ROW;
constexpr long long kDispatchGatherMinRow = A2AV_DISPATCH_GATHER_MIN_ROW;
constexpr long long kGatherMaxRow = 32 * 1024;
constexpr long long kGatherCheckMaxRow = 2048;  // the combine's gather checks its items up to here
constexpr int kGatherSmem = kGatherSmemBound;

using GatherKernel = void (*)(Params, DispatchParams);
struct GatherShape {
  long long max_row;
  GatherKernel kernel;
  int nwk, ns, ips;
};
// Rows of 64 B .. 2 KiB: every lane of a warp issues its own row's copy,
// 16-row stages, loads two stages ahead, and as many warps as keep ~96 KiB
// of loads in flight per SM (3 warps at 1 KiB rows .. 16 at 128 B).  A
// standalone probe (256 MiB of rows to scattered destinations) measured this
// shape at 3134 / 3060 / 2990 GB/s moved for 1 KiB / 512 B / 256 B rows,
// against 1877 / 994 / 511 with one warp of 32-row stages and 2580 / 2155 /
// 1283 by register copies: with enough warps issuing, the per-copy cost of
// small cp.async.bulk operations is hidden.  (The combine takes its own
// one-row rings for 1 and 2 KiB rows, below; the dispatch takes the
// register copy up to 2 KiB.)
const GatherShape kGatherShapes[] = {
    {128, dispatch_gather_kernel<4, 2, 16, 16>, 16, 4, 16},
    {256, dispatch_gather_kernel<4, 2, 12, 16>, 12, 4, 16},
    {512, dispatch_gather_kernel<4, 2, 6, 16>, 6, 4, 16},
    {1024, dispatch_gather_kernel<4, 2, 3, 16>, 3, 4, 16},
    {2048, dispatch_gather_kernel<4, 2, 3, 8>, 3, 4, 8},
    // one row a stage, one issuing lane per warp, several warps with rings of
    // their own (MoE dispatch / combine, 8192 tokens, W=8, the one-row loop:
    // 4 KiB rows 142.1 / 173.3 us on eight warps x 6 stages, loads 3 ahead,
    // against 145.5 / 174.6 on four x 6 and 145.4 / 174.2 on four x 12; 8
    // KiB rows 268.4 / 337.3 on three x 8, loads 6 ahead, against 277.6 /
    // 341.8 on two x 12 and 268.3 / 337.9 on four x 6)
    {4096, dispatch_gather_kernel<6, 3, 8, 1>, 8, 6, 1},
    {8192, dispatch_gather_kernel<8, 6, 3, 1>, 3, 8, 1},
    // 14 KiB MoE rows: two warps x 6 x 16 KiB stages, loads 4 ahead (with
    // the one-row loop: 462.8 us against 468.0 with three warps x 4 and
    // 470.8 with one warp x 12, the ring that was best for the batched
    // issue)
    {16384, dispatch_gather_kernel<6, 4, 2, 1>, 2, 6, 1},
    {32768, dispatch_gather_kernel<kGatherNs, kGatherLead, 1, 1>, 1, kGatherNs, 1},
};
// The combine's own rings where they differ from the dispatch's, measured
// with the one-row loop (MoE combine, 8192 tokens, W=8): 1 and 2 KiB rows
// on sixteen warps of one-row stages (12 and 6 stages, loads 6 and 3 ahead:
// 48.5 against 49.7 us and 89.0 against 90.8 for the lane-per-row stages
// above, which keep 64 B .. 512 B rows -- at 512 B one-row rings took 44.0
// against 29.7); rows above 8 KiB up to 16 KiB on three warps x 4 stages,
// loads two ahead (14 KiB rows: 584.6 against 597.1 us for one warp x 12;
// the dispatch's own ring there is two warps x 6).
#ifndef A2AV_C16K_NS
#define A2AV_C16K_NS 4
#define A2AV_C16K_LEAD 2
#define A2AV_C16K_NWK 3
#endif
#ifndef A2AV_C1K_NS
#define A2AV_C1K_NS 12
#define A2AV_C1K_LEAD 6
#define A2AV_C1K_NWK 16
#endif
#ifndef A2AV_C2K_NS
#define A2AV_C2K_NS 6
#define A2AV_C2K_LEAD 3
#define A2AV_C2K_NWK 16
#endif
const GatherShape kCombineShapes[] = {
    {1024, dispatch_gather_kernel<A2AV_C1K_NS, A2AV_C1K_LEAD, A2AV_C1K_NWK, 1>, A2AV_C1K_NWK,
     A2AV_C1K_NS, 1},
    {2048, dispatch_gather_kernel<A2AV_C2K_NS, A2AV_C2K_LEAD, A2AV_C2K_NWK, 1>, A2AV_C2K_NWK,
     A2AV_C2K_NS, 1},
    {16384, dispatch_gather_kernel<A2AV_C16K_NS, A2AV_C16K_LEAD, A2AV_C16K_NWK, 1>, A2AV_C16K_NWK,
     A2AV_C16K_NS, 1},
};
static_assert(A2AV_C16K_NWK * A2AV_C16K_NS * 16384 <= kGatherSmem &&
                  A2AV_C1K_NWK * A2AV_C1K_NS * 1024 <= kGatherSmem &&
                  A2AV_C2K_NWK * A2AV_C2K_NS * 2048 <= kGatherSmem,
              "the combine's rings fit the gather's shared memory");
static_assert(16 * 4 * 16 * 128 <= kGatherSmem && 12 * 4 * 16 * 256 <= kGatherSmem &&
                  6 * 4 * 16 * 512 <= kGatherSmem && 3 * 4 * 16 * 1024 <= kGatherSmem &&
                  3 * 4 * 8 * 2048 <= kGatherSmem && 8 * 6 * 4096 <= kGatherSmem &&
                  3 * 8 * 8192 <= kGatherSmem && 2 * 6 * 16384 <= kGatherSmem &&
                  kGatherNs * 32768 <= kGatherSmem,
              "every ring fits the gather's shared memory");

// ------------------------------------------------------------ one kernel --
// Decode-size batches: at most kTinyItems items over all ranks.  Every CTA
// reads every key, so all reach the same verdict and the same plan without
// any exchange between CTAs; CTA b then places and copies the items
// [b n / G, (b + 1) n / G) of the global item order (at most kTinyOwn).
constexpr int kTinyThreads = 256;
constexpr int kTinyItems = 4096;
constexpr int kTinyCounts = 2048;  // W * W * K counters in shared memory
constexpr int kTinyOwn = 64;
// Dynamic shared memory of the one-kernel paths: row slots, then (dispatch)
// the counters; 199 KiB with the ~28 KB of static shared memory (the plan,
// the CTA's share) stays within the 227 KiB a CTA may have (14 slots of
// 14 KiB MoE rows plus counters).  The shared-memory opt-in of both kernels
// fails, and so every decode-size call with it, if the sum goes above.
constexpr int kTinyDynBytes = 199 * 1024;

// The CTA's c rows (addresses listed in shared memory; 0: a row the position
// check dropped), by warp 0 with cp.async.bulk when slots > 0 (rows and
// buffers 16-byte aligned): when every row has a slot, each row has its own
// mbarrier and the lane that loaded it stores it as soon as it lands;
// otherwise rounds of min(32, slots) rows on one mbarrier.  With slots == 0
// every warp copies with registers (a warp per row from 64 bytes, a thread
// per row below).  A bounded wait that gives up records A2AV_ERR_TIMEOUT and
// waits (bounded) once more for its load before the warp leaves.
__device__ void copy_listed_rows(const unsigned long long* src, const unsigned long long* dst,
                                 int c, long long rb, int slots, uint32_t slot0, uint32_t bar0,
                                 int* status) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (slots == 0) {
    if (rb >= kWarpRowBytes) {
      for (int x = warp; x < c; x += kTinyThreads / 32)
        if (dst[x] != 0)
          copy_span<32, 4, 2>(reinterpret_cast<unsigned char*>(dst[x]),
                              reinterpret_cast<const unsigned char*>(src[x]), rb, lane);
    } else {
      for (int x = tid; x < c; x += kTinyThreads)
        if (dst[x] != 0)
          copy_row_thread(reinterpret_cast<unsigned char*>(dst[x]),
                          reinterpret_cast<const unsigned char*>(src[x]), rb);
    }
    return;
  }
  if (warp != 0 || c == 0) return;
  if (c <= slots) {  // one slot and one mbarrier a row; lane l takes rows l, l + 32
    for (int x = lane; x < c; x += 32) {
      mbar_init(bar0 + 8 * x, 1);
      mbar_fence_init();
    }
    for (int x = lane; x < c; x += 32) {
      mbar_expect_tx(bar0 + 8 * x, (unsigned)rb);
      bulk_load(slot0 + (uint32_t)(x * rb), reinterpret_cast<const void*>(src[x]), (unsigned)rb,
                bar0 + 8 * x);
    }
    for (int x = lane; x < c; x += 32) {
      if (!mbar_wait(bar0 + 8 * x, 0)) {
        record_error(status, A2AV_ERR_TIMEOUT);
        mbar_wait(bar0 + 8 * x, 0);
        continue;
      }
      if (dst[x] != 0)
        bulk_store(reinterpret_cast<void*>(dst[x]), slot0 + (uint32_t)(x * rb), (unsigned)rb);
    }
    bulk_wait_all();
    return;
  }
  const uint32_t bar = bar0;
  if (lane == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  __syncwarp();
  const int per = slots < 32 ? slots : 32;
  unsigned phase = 0;
  for (int base = 0; base < c; base += per) {
    const int nr = c - base < per ? c - base : per;
    if (base > 0) bulk_wait_read<0>();  // the previous round's stores have read their slots
    __syncwarp();
    if (lane == 0) mbar_expect_tx(bar, (unsigned)(nr * rb));
    __syncwarp();
    if (lane < nr)
      bulk_load(slot0 + (uint32_t)(lane * rb), reinterpret_cast<const void*>(src[base + lane]),
                (unsigned)rb, bar);
    if (!mbar_wait_warp(bar, phase)) {
      if (lane == 0) {
        record_error(status, A2AV_ERR_TIMEOUT);
        mbar_wait(bar, phase);
      }
      __syncwarp();
      break;
    }
    phase ^= 1;
    if (lane < nr && dst[base + lane] != 0)
      bulk_store(reinterpret_cast<void*>(dst[base + lane]), slot0 + (uint32_t)(lane * rb),
                 (unsigned)rb);
    else
      bulk_commit();
  }
  bulk_wait_all();
}

// This CTA's share [a, e) of the n items (global order, rank-major).
__device__ __forceinline__ void tiny_share(const DispatchParams& D, long long* a, long long* e) {
  const long long n = D.item_first[D.W];
  *a = (long long)blockIdx.x * n / gridDim.x;
  *e = (long long)(blockIdx.x + 1) * n / gridDim.x;
}

__global__ void __launch_bounds__(kTinyThreads, 1)
    dispatch_tiny_kernel(const __grid_constant__ Params P, const __grid_constant__ DispatchParams D,
                         int slots) {
  chain_release();
  chain_wait();
  __shared__ Plan pl;
  __shared__ unsigned long long own_src[kTinyOwn], own_dst[kTinyOwn];
  __shared__ int own_key[kTinyOwn], own_row[kTinyOwn];  // the share's keys and source rows
  __shared__ alignas(8) unsigned long long bars[kTinyOwn];
  extern __shared__ __align__(128) unsigned char slot_mem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int W = D.W, K = D.K, NB = W * K;
  const long long rb = P.rb;
  // The counters follow the row slots in dynamic shared memory.
  int* const cnt = reinterpret_cast<int*>(slot_mem + (((long long)slots * rb + 15) & ~15LL));
  int* const run = cnt + W * NB;  // [r][key]: counts, then key starts; running count of each key
  long long a, e;
  tiny_share(D, &a, &e);
  int ra = 0;  // the rank of item a
  while (ra + 1 < W && D.item_first[ra + 1] <= a) ++ra;
  const long long ia = a - D.item_first[ra];
  // Thread t takes items t, t + 256, ... of the global order (at most
  // kTinyItems / kTinyThreads), all their keys and source rows loaded at
  // once, first: the counts wait for them.
  constexpr int kPer = kTinyItems / kTinyThreads;
  const long long n = D.item_first[W];
  int kk[kPer], ss[kPer], rr[kPer];
  long long ii[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const long long g = (long long)q * kTinyThreads + tid;
    int r = 0;
    while (r + 1 < W && D.item_first[r + 1] <= g) ++r;
    rr[q] = g < n ? r : -1;
    ii[q] = g - D.item_first[r];
    kk[q] = g < n ? __ldg(D.key[r] + ii[q]) : 0;
    ss[q] = g < n ? __ldg(D.src[r] + ii[q]) : 0;
  }
  // When every row of this CTA's share has a slot, thread t loads the share's
  // t-th source row at once (its index range-checked first; an invalid item
  // loads nothing and is never stored): the loads land while the items are
  // counted, the plan built and the rows placed.  Every exit below waits for
  // them first.
  const int c = (int)(e - a);
  const bool early = slots > 0 && c <= slots;
  if (early && tid < c) {
    const long long g = a + tid;
    int r = ra;
    while (r + 1 < W && D.item_first[r + 1] <= g) ++r;
    const int src = __ldg(D.src[r] + (g - D.item_first[r]));
    const uint32_t bar = smem_u32(&bars[tid]);
    mbar_init(bar, 1);
    mbar_fence_init();
    if (src >= 0 && src < D.rows[r]) {
      mbar_expect_tx(bar, (unsigned)rb);
      bulk_load(smem_u32(slot_mem) + (uint32_t)(tid * rb), P.in[r] + (long long)src * rb,
                (unsigned)rb, bar);
    } else {
      mbar_arrive(bar);
    }
  }
  auto settle = [&]() {  // (bounded) every early load has landed
    if (early && tid < c) mbar_wait(smem_u32(&bars[tid]), 0);
  };
  for (int x = tid; x < W * NB; x += kTinyThreads) cnt[x] = 0;
  for (int x = tid; x < NB; x += kTinyThreads) run[x] = 0;
  __syncthreads();
  // every item: validity, its rank's key counts, and for rank ra the counts
  // of the items before this CTA's share.
  int bad = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int r = rr[q];
    if (r < 0) continue;
    if (kk[q] < 0 || kk[q] >= NB || ss[q] < 0 || ss[q] >= D.rows[r]) {
      bad = 1;
      continue;
    }
    atomicAdd(&cnt[r * NB + kk[q]], 1);
    if (r == ra && ii[q] < ia) atomicAdd(&run[kk[q]], 1);
    const long long g = (long long)q * kTinyThreads + tid;
    if (g >= a && g < e) {  // this CTA's share: kept for the placement below
      own_key[g - a] = kk[q];
      own_row[g - a] = ss[q];
    }
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) record_error(D.status, A2AV_ERR_BAD_INDEX);
    settle();
    return;
  }
  // per rank: key starts (exclusive scan in place) and S[r][*]
  for (int r = warp; r < W; r += kTinyThreads / 32) {
    int carry = 0;
    for (int k0 = 0; k0 < NB; k0 += 32) {
      const int k = k0 + lane;
      const int x = k < NB ? cnt[r * NB + k] : 0;
      const int inc = (int)warp_inclusive_scan(x, lane);
      if (k < NB) cnt[r * NB + k] = carry + inc - x;
      carry += __shfl_sync(kFull, inc, 31);
    }
    __syncwarp();
    for (int p = lane; p < W; p += 32) {
      const long long hi = p + 1 < W ? cnt[r * NB + (p + 1) * K] : D.items[r];
      pl.s[r][p] = hi - cnt[r * NB + p * K];
    }
  }
  __syncthreads();
  int over = 0;
  for (int x = tid; x < W * W; x += kTinyThreads)
    if (pl.s[x / W][x % W] > P.limit) over = 1;
  if (__syncthreads_or(over)) {
    if (blockIdx.x == 0 && tid == 0) record_error(D.status, A2AV_ERR_BAD_SPLITS);
    settle();
    return;
  }
  if (!plan_from_splits(P, pl, kTileGranule, blockIdx.x, gridDim.x)) {
    settle();
    return;
  }
  if (blockIdx.x == 0 && D.in_splits_out != nullptr)
    for (int x = tid; x < W * W; x += kTinyThreads) D.in_splits_out[x] = pl.s[x / W][x % W];
  // place the CTA's items, rank by rank, 32 at a time (warp 0)
  if (warp == 0) {
    const unsigned lt = (1u << lane) - 1u;
    int idx = 0, r = ra;
    for (long long g = a; g < e;) {
      while (D.item_first[r + 1] <= g) ++r;
      const long long seg_end = e < D.item_first[r + 1] ? e : D.item_first[r + 1];
      if (r != ra) {  // a later rank starts at its first item
        for (int k = lane; k < NB; k += 32) run[k] = 0;
        __syncwarp();
      }
      for (long long g0 = g; g0 < seg_end; g0 += 32) {
        const long long gi = g0 + lane;
        const bool v = gi < seg_end;
        const long long i = gi - D.item_first[r];
        const int key = v ? own_key[gi - a] : -1 - lane;
        const int s = v ? own_row[gi - a] : 0;
        const unsigned same = same_key_lanes(key, v, key_bits(NB));
        long long pos = 0;
        if (v) pos = (long long)cnt[r * NB + key] + run[key] + __popc(same & lt);
        __syncwarp();
        if (v && lane == 31 - __clz(same)) run[key] += __popc(same);
        __syncwarp();
        if (v) {
          const int p = key / K;
          D.sorted_pos[r][i] = pos;
          const bool ok = in_group(pl, r, p, pos, D.status);
          own_dst[idx + lane] =
              ok ? (unsigned long long)(P.out[p] + (pl.out_off[p][r] - pl.in_off[r][p] + pos) * rb)
                 : 0ull;
          own_src[idx + lane] = (unsigned long long)(P.in[r] + (long long)s * rb);
        }
        idx += (int)(seg_end - g0 < 32 ? seg_end - g0 : 32);
      }
      g = seg_end;
    }
  }
  __syncthreads();
  if (early) {  // each loaded row stored by the thread that loaded it
    if (tid < c) {
      const uint32_t bar = smem_u32(&bars[tid]);
      if (!mbar_wait(bar, 0)) {
        record_error(D.status, A2AV_ERR_TIMEOUT);
        mbar_wait(bar, 0);
      } else if (own_dst[tid] != 0) {
        bulk_store(reinterpret_cast<void*>(own_dst[tid]), smem_u32(slot_mem) + (uint32_t)(tid * rb),
                   (unsigned)rb);
      }
    }
    bulk_wait_all();
    return;
  }
  copy_listed_rows(own_src, own_dst, c, rb, slots, smem_u32(slot_mem), smem_u32(bars), D.status);
}

// The fused combine in one kernel (decode sizes): every CTA checks the split
// matrix (the a2av prologue) and every item's key and position, then copies
// its own share of the items' rows back to their item rows.
__global__ void __launch_bounds__(kTinyThreads, 1)
    combine_tiny_kernel(const __grid_constant__ Params P, const __grid_constant__ DispatchParams D,
                        int slots) {
  __shared__ Plan pl;
  __shared__ unsigned long long own_src[kTinyOwn], own_dst[kTinyOwn];
  __shared__ alignas(8) unsigned long long bars[kTinyOwn];
  __shared__ int own_key[kTinyOwn];
  __shared__ long long own_pos[kTinyOwn];
  extern __shared__ __align__(128) unsigned char slot_mem[];
  // The previous kernel of the stream (a dispatch) writes the positions:
  // wait for it, then load every item's key and position at once (thread
  // t: items t, t + 256, ... of the global order) and build the plan while
  // they are in flight.
  chain_release();
  chain_wait();
  const int tid = threadIdx.x, W = D.W, K = D.K, NB = W * K;
  constexpr int kPer = kTinyItems / kTinyThreads;
  const long long n = D.item_first[W];
  int kk[kPer], rr[kPer];
  long long pp[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const long long g = (long long)q * kTinyThreads + tid;
    int r = 0;
    while (r + 1 < W && D.item_first[r + 1] <= g) ++r;
    rr[q] = g < n ? r : -1;
    const long long i = g - D.item_first[r];
    kk[q] = g < n ? __ldg(D.key[r] + i) : 0;
    pp[q] = g < n ? __ldg(D.sorted_pos[r] + i) : 0;
  }
  if (!build_plan(P, pl, kTileGranule)) return;
  long long a, e;
  tiny_share(D, &a, &e);
  const long long rb = P.rb;
  // When every row of the share has a slot, the thread holding a share item
  // that it found valid loads its row at once (slot and mbarrier of the
  // item), while the other items are checked; the rows are stored only once
  // every item of the batch has passed.
  const int c = (int)(e - a);
  const bool early = slots > 0 && c <= slots;
  const uint32_t slot0 = smem_u32(slot_mem);
  unsigned armed = 0;  // bit q: this thread armed the mbarrier of its q-th item
  int bad = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int r = rr[q];
    if (r < 0) continue;
    bool ok = kk[q] >= 0 && kk[q] < NB;
    const int p = ok ? kk[q] / K : 0;
    if (ok) {
      const long long lo = pl.in_off[r][p];
      ok = pp[q] >= lo && pp[q] < lo + pl.s[r][p];
    }
    if (!ok) bad = 1;
    const long long g = (long long)q * kTinyThreads + tid;
    if (g >= a && g < e) {  // this CTA's share: kept for its copy
      own_key[g - a] = kk[q];
      own_pos[g - a] = pp[q];
      if (early) {
        const uint32_t bar = smem_u32(&bars[g - a]);
        mbar_init(bar, 1);
        mbar_fence_init();
        if (ok) {
          mbar_expect_tx(bar, (unsigned)rb);
          bulk_load(slot0 + (uint32_t)((g - a) * rb),
                    P.out[p] + (pl.out_off[p][r] - pl.in_off[r][p] + pp[q]) * rb, (unsigned)rb, bar);
        } else {
          mbar_arrive(bar);
        }
        armed |= 1u << q;
      }
    }
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) record_error(D.status, A2AV_ERR_BAD_INDEX);
#pragma unroll
    for (int q = 0; q < kPer; ++q)  // (bounded) the loads this thread issued land first
      if ((armed >> q) & 1u) mbar_wait(smem_u32(&bars[(long long)q * kTinyThreads + tid - a]), 0);
    return;
  }
  for (long long g = a + tid; g < e; g += kTinyThreads) {
    int r = 0;
    while (r + 1 < W && D.item_first[r + 1] <= g) ++r;
    const long long i = g - D.item_first[r];
    const int p = own_key[g - a] / K;
    own_src[g - a] = (unsigned long long)(P.out[p] +
                                          (pl.out_off[p][r] - pl.in_off[r][p] + own_pos[g - a]) * rb);
    own_dst[g - a] = (unsigned long long)(P.in[r] + i * rb);
  }
  __syncthreads();
  if (early) {  // row x stored by thread x once it has landed
    if (tid < c) {
      const uint32_t bar = smem_u32(&bars[tid]);
      if (!mbar_wait(bar, 0)) {
        record_error(D.status, A2AV_ERR_TIMEOUT);
        mbar_wait(bar, 0);
      } else {
        bulk_store(reinterpret_cast<void*>(own_dst[tid]), slot0 + (uint32_t)(tid * rb), (unsigned)rb);
      }
    }
    bulk_wait_all();
    return;
  }
  copy_listed_rows(own_src, own_dst, c, rb, slots, slot0, smem_u32(bars), D.status);
}

// Workspace: [0, 256) the flag (int) and the per-rank done counters (W ints),
// cleared before every dispatch that uses them; then S, key starts, key
// totals, inrank bytes, range prefixes, group counts.
struct Layout {
  long long flag, done, S, key_start, key_total, inrank, hist, grp, total;
};

Layout layout(int W, int K, long long max_items) {
  auto up = [](long long x) { return (x + 255) / 256 * 256; };
  const long long NB = (long long)W * K;
  const long long ranges = (max_items + kRange - 1) / kRange;
  const long long groups = (ranges + kCountWarps - 1) / kCountWarps;  // groups of 8 ranges at most
  Layout L;
  L.flag = 0;
  L.done = 4;
  L.S = 256;
  L.key_start = L.S + up(8LL * W * W);
  L.key_total = L.key_start + up(8LL * W * NB);
  L.inrank = L.key_total + up(8LL * W * NB);
  L.hist = L.inrank + up((long long)W * (max_items < 1 ? 1 : max_items));
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

using OrderKernel = void (*)(Params, DispatchParams);
const OrderKernel kOrderKernels[] = {
    dispatch_order_kernel<0>,  dispatch_order_kernel<4>, dispatch_order_kernel<8>,
    dispatch_order_kernel<16>, dispatch_order_kernel<-1>, combine_order_kernel<4>,
    combine_order_kernel<8>,   combine_order_kernel<16>, combine_order_kernel<-1>};

// The row word of rows under 64 bytes: 4, 8 or 16 when rows are exactly that
// long and every buffer is aligned to it, else -1 (rows one at a time).
int row_word(const Params& P, long long rb) {
  uintptr_t a = (uintptr_t)rb;
  for (int r = 0; r < P.W; ++r) a |= (uintptr_t)P.in[r] | (uintptr_t)P.out[r];
  if ((rb == 4 || rb == 8 || rb == 16) && (a & (uintptr_t)(rb - 1)) == 0) return (int)rb;
  return -1;
}

// The order kernel for a batch: positions only for rows of 64 bytes or more;
// else the copying one for the row size and alignment.
OrderKernel order_kernel(const Params& P, long long rb, bool combine) {
  if (rb >= kWarpRowBytes) return dispatch_order_kernel<0>;
  switch (row_word(P, rb)) {
    case 4: return combine ? combine_order_kernel<4> : dispatch_order_kernel<4>;
    case 8: return combine ? combine_order_kernel<8> : dispatch_order_kernel<8>;
    case 16: return combine ? combine_order_kernel<16> : dispatch_order_kernel<16>;
    default: return combine ? combine_order_kernel<-1> : dispatch_order_kernel<-1>;
  }
}

// Shared-memory opt-in of the gather and one-kernel paths, once per handle
// (a host call per launch otherwise).
cudaError_t prepare_kernels(a2av_handle* h) {
  if (h->gather_ready) return cudaSuccess;
  for (const GatherShape& g : kGatherShapes)
    if (cudaFuncSetAttribute(g.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGatherSmem) !=
        cudaSuccess)
      return cudaErrorInvalidValue;
  for (const GatherShape& g : kCombineShapes)
    if (cudaFuncSetAttribute(g.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGatherSmem) !=
        cudaSuccess)
      return cudaErrorInvalidValue;
  // (count histograms: 8 ranges a warp x 4 x W * K ints, up to 128 KiB)
  if (cudaFuncSetAttribute(dispatch_count_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kCountWarps * 4 * kMaxBins * (int)sizeof(int)) != cudaSuccess ||
      cudaFuncSetAttribute(dispatch_tiny_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kTinyDynBytes) != cudaSuccess ||
      cudaFuncSetAttribute(combine_tiny_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kTinyDynBytes) != cudaSuccess)
    return cudaErrorInvalidValue;
  // The order kernel's grid: as many CTAs as are resident at once with the
  // largest run-count table (a cooperative launch needs every CTA resident).
  constexpr int kOrderSmemMax = kOrderWarps * kMaxBins * (int)sizeof(int);
  int per_sm = 1 << 30;
  for (OrderKernel k : kOrderKernels) {
    int n = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kOrderSmemMax) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kOrderThreads, kOrderSmemMax) !=
            cudaSuccess)
      return cudaErrorInvalidValue;
    per_sm = n < per_sm ? n : per_sm;
  }
  h->order_grid = h->sms * per_sm;
  h->gather_ready = true;
  return cudaSuccess;
}

// Host side of the order kernels: the chunk and each rank's CTAs, or 0 when
// the batch does not fit one launch (more items than the grid's registers
// hold; for the dispatch -- L given -- also too many counts for step 3, or a
// workspace too small for the CTA counts: the count / scan chain takes it
// then).
int order_grid(const a2av_handle* h, DispatchParams& D, const Layout* L) {
  const int W = D.W;
  const long long NB = (long long)W * D.K, M = D.item_first[W], G = h->order_grid;
  if (M == 0 || G <= W) return 0;
  long long chunk = (M + (G - W) - 1) / (G - W);
  chunk = chunk < 32 * kOrderWarps ? 32 * kOrderWarps : chunk;  // a 32-item run per warp at least
  if (chunk > kOrderCtaItems) return 0;
  long long ctas = 0, most = 0;
  for (int r = 0; r < W; ++r) {
    const long long g = (D.items[r] + chunk - 1) / chunk;
    D.cta_first[r] = (int)ctas;
    ctas += g;
    most = g > most ? g : most;
  }
  D.cta_first[W] = (int)ctas;
  // (step 3: thread t loads the counts of every S-th CTA of its rank, S =
  // threads / (NBP / 4), NBP = NB rounded up to a multiple of 4)
  const long long NBP = (NB + 3) & ~3LL, S = kOrderThreads / (NBP / 4);
  if (ctas > G ||
      (L != nullptr && ((most + S - 1) / S > kOrderPrefixLoads ||
                        4 * ctas * NBP > L->total - L->hist)))
    return 0;
  D.chunk = chunk;
  return (int)ctas;
}

// A cooperative launch (every CTA resident at once: the order kernel's grid
// barrier relies on it).
template <typename... Args, typename... Vals>
cudaError_t launch_cooperative(void (*kernel)(Args...), dim3 grid, int block, size_t smem,
                               cudaStream_t s, Vals... vals) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, vals...);
}

// Row slots of the one-kernel paths: 0 (register copies) unless every row
// and buffer is 16-byte aligned and a row fits beside `reserved` bytes.
int tiny_slots(const DispatchParams& D, long long rb, long long reserved) {
  if (!D.vec16 || rb < kWarpRowBytes || rb > kTinyDynBytes - reserved) return 0;
  const long long n = (kTinyDynBytes - reserved) / rb;
  return (int)(n < kTinyOwn ? n : kTinyOwn);
}

// The dispatch's counters: [W][W*K] key counts and a W*K running count.
long long tiny_count_bytes(const DispatchParams& D) {
  return ((long long)D.W * D.W * D.K + (long long)D.W * D.K) * (long long)sizeof(int);
}

// One-kernel path: at most kTinyItems items, their counts fit shared memory,
// and no CTA gets more than kTinyOwn of them.
bool tiny_fits(const a2av_handle* h, const DispatchParams& D) {
  const long long n = D.item_first[D.W];
  return n <= kTinyItems && (long long)D.W * D.W * D.K <= kTinyCounts &&
         (long long)h->sms * kTinyOwn >= n;
}

int tiny_grid(const a2av_handle* h, const DispatchParams& D) {
  const long long n = D.item_first[D.W];
  return (int)(n < 1 ? 1 : (n < h->sms ? n : h->sms));
}

// What the last dispatch or combine enqueued (a2av_last_dispatch).
void record_chain(a2av_handle* h, int kernels, int memsets, const char* copy) {
  h->last_kernels = kernels;
  h->last_memsets = memsets;
  h->last_copy = copy;
}

// Whether the cp.async.bulk gather moves rows of this size.
bool takes_gather(const DispatchParams& D, long long row_bytes) {
  return D.vec16 && row_bytes >= (D.combine ? kGatherMinRow : kDispatchGatherMinRow) &&
         row_bytes <= kGatherMaxRow;
}

// The row copy of a dispatch or a combine: the cp.async.bulk gather for
// 16-byte aligned rows of kGatherMinRow (the dispatch: kDispatchGatherMinRow)
// .. 32 KiB (its ring by row size), else the warp copy (rows of 64 bytes or
// more) or the thread copy.
cudaError_t launch_copy(a2av_handle* h, const Params& P, DispatchParams D, long long row_bytes,
                        cudaStream_t s, const char** name) {
  const bool gather = takes_gather(D, row_bytes);
  if (!gather) {
    *name = "dispatch_copy_kernel";
    if (row_bytes < kWarpRowBytes)
      return launch_kernel(dispatch_copy_kernel<false>, dim3(h->sms * kCopyCtasPerSm),
                           kCopyThreads, 0, s, true, P, D);
    if (D.vec16 && row_bytes <= kVecMaxRow && row_bytes % 512 == 0)
      return launch_kernel(dispatch_copy_kernel<true, true>, dim3(h->sms * kRows512CtasPerSm),
                           kCopyThreads, 0, s, true, P, D);
    return launch_kernel(dispatch_copy_kernel<true>, dim3(h->sms * kCopyCtasPerSmWarpRows),
                         kCopyThreads, 0, s, true, P, D);
  }
  *name = "dispatch_gather_kernel";
  const cudaError_t e = prepare_kernels(h);
  if (e != cudaSuccess) return e;
  const GatherShape* g = &kGatherShapes[0];
  while (g->max_row < row_bytes) ++g;
  if (D.combine)
    for (const GatherShape& c : kCombineShapes)
      if (c.max_row == g->max_row) g = &c;
  // Batches of 32 items, or of 16 / 8 when that gives every warp at least
  // four (balance for mid-size batches).
  const long long warps = (long long)h->sms * g->nwk;
  int bs = 32;
  for (;;) {
    long long nb = 0;
    for (int r = 0; r < D.W; ++r) nb += (D.items[r] + bs - 1) / bs;
    if (bs == 8 || nb >= 4 * warps) break;
    bs >>= 1;
  }
  D.bs = bs;
  D.batch_first[0] = 0;
  for (int r = 0; r < D.W; ++r) D.batch_first[r + 1] = D.batch_first[r] + (D.items[r] + bs - 1) / bs;
  const size_t smem = (size_t)g->nwk * g->ns * g->ips * row_bytes;
  if (D.combine && D.barrier != nullptr)  // (the combine's checks in the gather: a grid barrier)
    return launch_cooperative(g->kernel, dim3(h->sms), 32 * g->nwk, smem, s, P, D);
  return launch_kernel(g->kernel, dim3(h->sms), 32 * g->nwk, smem, s, true, P, D);
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
  D.inrank = ws + L.inrank;
  D.pos_stride = max_items < 1 ? 1 : max_items;
  D.hist = reinterpret_cast<int*>(ws + L.hist);
  D.grp = reinterpret_cast<int*>(ws + L.grp);
  D.status = h->d_status;
  D.in_splits_out = reinterpret_cast<long long*>(in_splits_dev);
  D.ranges_max = ranges_max;
  D.W = W;
  D.K = K;
  // (16-byte vectors and cp.async.bulk only on aligned device memory; rows in
  // host memory are copied with plain loads and stores)
  bool vec16 = row_bytes % 16 == 0;
  for (int r = 0; r < W; ++r)
    vec16 = vec16 && ((uintptr_t)rows_ptrs[r] & 15) == 0 && ((uintptr_t)out_ptrs[r] & 15) == 0;
  D.vec16 = vec16 && a2av_device_buffers(h, rows_ptrs, W, out_ptrs, W) ? 1 : 0;


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
  P.starve = h->starve;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (tiny_fits(h, D)) {  // decode sizes: one kernel, no workspace
    if ((e = prepare_kernels(h)) != cudaSuccess) return A2AV_ERR_CUDA;
    const long long counters = tiny_count_bytes(D);
    const int slots = tiny_slots(D, row_bytes, counters + 16);
    const size_t smem = (size_t)((((long long)slots * row_bytes + 15) & ~15LL) + counters);
    e = launch_kernel(dispatch_tiny_kernel, dim3(tiny_grid(h, D)), kTinyThreads, smem, s, h->pdl,
                      P, D, slots);
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
    record_chain(h, 1, 0, "dispatch_tiny_kernel");
    return A2AV_OK;
  }
  const bool small_path = max_items <= kSmallItems && W * K <= kSmallKeys;
  // The one-launch order kernel (the handle's A2AV_DISPATCH_ORDER level: 1
  // for rows under 64 bytes, 2 for every row size, 3 also for batches the
  // small kernel takes)
  if (h->order_level >= (row_bytes < kWarpRowBytes ? 1 : 2) &&
      (h->order_level >= 3 || !small_path)) {
    if ((e = prepare_kernels(h)) != cudaSuccess) return A2AV_ERR_CUDA;
    const int ctas = order_grid(h, D, &L);
    if (ctas > 0) {
      static_assert(4 + 4 * kMaxW <= kOrderBarrierOffset, "done counters below the barrier");
      D.barrier = reinterpret_cast<unsigned*>(ws + kOrderBarrierOffset);
      D.cta_cnt = reinterpret_cast<int*>(ws + L.hist);
      if (cudaMemsetAsync(ws, 0, (size_t)L.key_start, s) != cudaSuccess) return A2AV_ERR_CUDA;
      const bool fused = row_bytes < kWarpRowBytes;  // rows copied by the order kernel
      const size_t smem = (size_t)kOrderWarps * W * K * sizeof(int);
      e = launch_cooperative(order_kernel(P, row_bytes, false), dim3((unsigned)ctas),
                             kOrderThreads, smem, s, P, D);
      if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
      if (fused) {
        record_chain(h, 1, 1, "dispatch_order_kernel");
        return A2AV_OK;
      }
      D.pos_ready = 1;
      const char* copy = nullptr;
      e = launch_copy(h, P, D, row_bytes, s, &copy);
      if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
      record_chain(h, 2, 1, copy);
      return A2AV_OK;
    }
  }
// Four ranges a count warp (fewer, longer count CTAs) measured slower on the
// embedding-key dispatch (640 K items a rank: 56.5 against 35.8 us); kept
// for sweeps.
#ifndef A2AV_COUNT_RW4
#define A2AV_COUNT_RW4 0
#endif
  const int rw = A2AV_COUNT_RW4 && !small_path &&
                         (long long)W * ((ranges_max + 31) / 32) >= h->sms ? 4 : 1;
  D.group_log2 = rw == 4 ? 5 : 3;
  D.groups_max = (ranges_max + (1LL << D.group_log2) - 1) >> D.group_log2;
  // One count CTA per rank scans its groups when a thread's share of one key
  // stays short; the scan kernel and its launch are skipped.
  const int slices = kScanThreads / (W * K);
  D.fuse_scan = small_path || (slices > 0 && D.groups_max <= (long long)kFuseScanMax * slices);

  static_assert(4 + 4 * kMaxW <= 256, "flag and done counters fit the first 256 bytes");
  if (cudaMemsetAsync(D.flag, 0, 256, s) != cudaSuccess) return A2AV_ERR_CUDA;
  // Every kernel of the chain is launched with programmatic stream
  // serialization: it may be scheduled while its predecessor runs and waits
  // for that predecessor's results in chain_wait.
  if (small_path) {
    e = launch_kernel(dispatch_small_kernel, dim3(W), kScanThreads, 0, s, h->pdl, D);
  } else {
    // (at least one CTA per rank: a batch without items still gets its
    // counts, splits and offsets written)
    const long long groups = D.groups_max > 0 ? D.groups_max : 1;
    const size_t hist_smem = (size_t)kCountWarps * rw * W * K * sizeof(int);
    if ((e = prepare_kernels(h)) != cudaSuccess) return A2AV_ERR_CUDA;
    const bool place = row_bytes < kWarpRowBytes;  // the place-and-copy kernel ranks
    if (rw == 4)
      e = launch_kernel(dispatch_count_kernel<4>, dim3((unsigned)groups, (unsigned)W),
                        32 * kCountWarps, hist_smem, s, h->pdl, D);
    else if (place)
      e = launch_kernel(dispatch_count_kernel<1, false>, dim3((unsigned)groups, (unsigned)W),
                        32 * kCountWarps, hist_smem, s, h->pdl, D);
    else
      e = launch_kernel(dispatch_count_kernel<1>, dim3((unsigned)groups, (unsigned)W),
                        32 * kCountWarps, hist_smem, s, h->pdl, D);
    if (e == cudaSuccess && !D.fuse_scan)
      e = launch_kernel(dispatch_scan_kernel, dim3((unsigned)(W * K), (unsigned)W), kScanThreads,
                        0, s, true, D);
    if (e == cudaSuccess && row_bytes < kWarpRowBytes) {  // place and copy in one kernel
      const long long ranges = ranges_max > 0 ? ranges_max : 1;
      const dim3 grid2((unsigned)((ranges + kPlaceWarps - 1) / kPlaceWarps), (unsigned)W);
      e = launch_kernel(dispatch_place_copy_kernel, grid2, 32 * kPlaceWarps,
                        (size_t)kPlaceWarps * W * K * sizeof(int), s, true, P, D);
      if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
      record_chain(h, D.fuse_scan ? 2 : 3, 1, "dispatch_place_copy_kernel");
      return A2AV_OK;
    }
  }
  if (e != cudaSuccess) return A2AV_ERR_CUDA;
  const char* copy = nullptr;
  e = launch_copy(h, P, D, row_bytes, s, &copy);
  if (e != cudaSuccess) return A2AV_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
  record_chain(h, small_path || D.fuse_scan ? 2 : 3, 1, copy);
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
  D.vec16 = vec16 && a2av_device_buffers(h, peer_ptrs, W, item_out_ptrs, W) ? 1 : 0;


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
  P.starve = h->starve;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (tiny_fits(h, D)) {  // decode sizes: one kernel, no flag
    if ((e = prepare_kernels(h)) != cudaSuccess) return A2AV_ERR_CUDA;
    const int slots = tiny_slots(D, row_bytes, 0);
    e = launch_kernel(combine_tiny_kernel, dim3(tiny_grid(h, D)), kTinyThreads,
                      (size_t)slots * row_bytes, s, h->pdl, P, D, slots);
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
    record_chain(h, 1, 0, "combine_tiny_kernel");
    return A2AV_OK;
  }
  if (cudaMemsetAsync(D.flag, 0, 256, s) != cudaSuccess) return A2AV_ERR_CUDA;
  if (row_bytes < kWarpRowBytes && h->order_level >= 1) {  // check and copy in one launch
    if ((e = prepare_kernels(h)) != cudaSuccess) return A2AV_ERR_CUDA;
    const int ctas = order_grid(h, D, nullptr);
    if (ctas > 0) {
      D.barrier = reinterpret_cast<unsigned*>(ws + kOrderBarrierOffset);
      e = launch_cooperative(order_kernel(P, row_bytes, true), dim3((unsigned)ctas),
                             kOrderThreads, 0, s, P, D);
      if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
      record_chain(h, 1, 1, "combine_order_kernel");
      return A2AV_OK;
    }
  }
  // Aligned rows of 64 B .. 2 KiB: the gather checks every item itself
  // (grid barrier) -- 1 KiB rows: the gather with its checks 45.8 us against
  // 40.0 + 6.0 us for the check kernel and the gather, one launch less; the
  // one-row rings above 2 KiB have too few threads to check quickly (14 KiB
  // rows: 625.6 against 619.5 us), so they keep the check kernel.
  if (takes_gather(D, row_bytes) && row_bytes <= kGatherCheckMaxRow && h->order_level >= 1) {
    if ((e = prepare_kernels(h)) != cudaSuccess) return A2AV_ERR_CUDA;
    D.barrier = reinterpret_cast<unsigned*>(ws + kOrderBarrierOffset);
    const char* copy = nullptr;
    e = launch_copy(h, P, D, row_bytes, s, &copy);
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
    record_chain(h, 1, 1, copy);
    return A2AV_OK;
  }
  e = launch_kernel(combine_check_kernel, dim3(h->sms * kCopyCtasPerSm), kCopyThreads, 0, s,
                    h->pdl, P, D);
  if (e != cudaSuccess) return A2AV_ERR_CUDA;
  const char* copy = nullptr;
  e = launch_copy(h, P, D, row_bytes, s, &copy);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
  record_chain(h, 2, 1, copy);
  return A2AV_OK;
}

extern "C" int a2av_last_dispatch(const a2av_handle* h, int* kernels, int* memsets,
                                  const char** copy_kernel) {
  if (h == nullptr) return A2AV_ERR_INVALID_ARG;
  if (kernels) *kernels = h->last_kernels;
  if (memsets) *memsets = h->last_memsets;
  if (copy_kernel) *copy_kernel = h->last_copy;
  return A2AV_OK;
}
