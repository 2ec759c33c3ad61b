// a2av_handle.h -- the opaque handle behind include/a2av.h (host side only).
#pragma once

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
};
