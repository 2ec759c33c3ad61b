// a2av_handle.h -- the opaque handle behind include/a2av.h (host side only).
#pragma once

#include "a2av.h"

// The last pointer sets classified by a2av_device_buffers (two slots, the
// older one replaced), so that repeated calls on the same buffers skip the
// CUDA pointer queries.
struct a2av_ptr_cache {
  const void* ptrs[2 * A2AV_MAX_EXCHANGES * A2AV_MAX_RANKS];
  int n;           // pointers in the set; 0 = empty slot
  bool device;     // every non-NULL pointer is device memory
  unsigned stamp;  // last use
};

// Default of A2AV_DISPATCH_ORDER (see a2av_create in a2av.h).
#ifndef A2AV_DISPATCH_ORDER
#define A2AV_DISPATCH_ORDER 1
#endif

struct a2av_handle {
  int W;
  long long in_cap, out_cap;  // rows, 0 = unchecked
  int device;
  int sms;
  int* d_status;              // device status word (first device-detected error)
  int path;                   // a2av_path_t
  int ctas_per_sm;            // 0 = engine default
  int last_path, last_grid, last_block;
  int starve;                 // test hook (A2AV_DEBUG_STARVE): see a2av_create in a2av.h
  bool pdl;                   // programmatic dependent launch (A2AV_PDL, default on)
  bool gather_ready;          // the dispatch gather kernels' shared-memory opt-in is done
  int order_grid;             // CTAs of the dispatch's one-launch order kernel (all resident)
  int order_level;            // A2AV_DISPATCH_ORDER: batches the order kernel takes
  int last_kernels;           // kernels the last dispatch / combine_items enqueued
  int last_memsets;           // and workspace memsets
  const char* last_copy;      // the kernel of that call that moved the rows (static string)
  a2av_ptr_cache cache[2];
  unsigned cache_clock;
};

// Whether every non-NULL pointer of a[0..na) and b[0..nb) is device memory
// (cudaMemoryTypeDevice).  Host-resident buffers -- pinned, registered, or
// system memory the GPU reaches through the host link -- must not be handed
// to cp.async.bulk; the callers route them to plain loads and stores.  With a
// handle (may be NULL) the answer for the last two pointer sets is cached
// (a2av_set_path and a2av_set_grid clear it).
__attribute__((visibility("hidden"))) bool a2av_device_buffers(a2av_handle* h,
                                                              const void* const* a, int na,
                                                              const void* const* b, int nb);
