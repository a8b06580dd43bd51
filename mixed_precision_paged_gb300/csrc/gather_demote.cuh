// gather_demote.cuh -- parameters of the gather and demotion kernels.
#pragma once

#include "common.cuh"

namespace ekv {

constexpr int kMaxRanges = 128;   // page ranges per gather launch (kernel-parameter sized)

struct GatherRanges {
  int n;
  int seq[kMaxRanges];
  int first[kMaxRanges];
  int off[kMaxRanges + 1];        // exclusive prefix sum of the ranges' page counts
};

struct GatherParams {
  const __half* k_pages;
  const uint8_t* v_pages;
  long long v_page_stride;
  int num_pages;
  const float* v_scales;
  int scale_mode;
  const uint8_t* page_mode;       // null -> uniform_mode
  int uniform_mode;
  const int32_t* block_table;
  int bt_stride;
  __half* ws_k;
  __half* ws_v;
  int32_t* ws_indices;
  int ws_base;                    // first workspace slot of this launch
  int Hkv, D;
  int apply_scale;
  int* err;
  // pair-structured value layout (ElasticKV): value location (half-slot index) of each
  // logical page; null -> the plain layout (location 2 * page id)
  const int32_t* v_block_table;
  int num_v_slots;                // slots of v_pages (elastic layout only)
  const int32_t* boundaries;      // [B][2] T-B-T boundaries or null (elastic layout only)
  int has_base;                   // 0: every page TARGET (elastic layout only)
  // 1: launched with programmatic serialization. Before its griddepcontrol.wait the
  // kernel reads only the block tables, page metadata, scales and pool pages; it writes
  // the workspace, the indices and the error word after it.
  int pdl;
};

// Page-mode transitions run by the same streaming kernel.
enum TransitionOp { kToE4M3 = 0, kToBase = 1, kPromote = 2 };

struct DemoteParams {
  uint8_t* v_pages;
  long long v_page_stride;
  int num_pages;
  const int32_t* page_ids;
  uint8_t* page_mode;
  float* scale_out;       // kToE4M3: fp32 [num_pages][H_kv]
  uint8_t* low;           // kToBase: low bytes out [n][16*H_kv*D] (may be null);
                          // kPromote: low bytes in, same layout
  const int32_t* src_loc; // per item, or null (in place): demotions: the TARGET page's
  const int32_t* dst_loc; // even location; promotion: the BASE half. dst: the half a
                          // demotion writes / the even location a promotion fills.
  int num_slots;          // value slots of v_pages (locations 0 .. 2*num_slots-1)
  int Hkv, D;
  int* err;
};

// K16/V8 cache writer: one new token per sequence.
struct AppendParams {
  const __half* k_new;      // [B][H_kv][D]
  const __half* v_new;      // [B][H_kv][D]
  __half* k_pages;
  uint8_t* v_pages;
  long long v_page_stride;
  int num_pages;
  const float* v_scales;
  int scale_mode;
  const uint8_t* page_mode;
  int uniform_mode;
  const int32_t* block_table;
  int bt_stride;
  const int32_t* positions; // [B], < 0: no token
  int Hkv, D;
  int* err;
};

cudaError_t launch_gather(const GatherParams& p, const GatherRanges& r, int pages, cudaStream_t st);
cudaError_t launch_append(const AppendParams& p, int batch, cudaStream_t st);
cudaError_t launch_transition(const DemoteParams& p, int op, int n, int num_sms, cudaStream_t st);

}  // namespace ekv
