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
};

struct DemoteParams {
  uint8_t* v_pages;
  long long v_page_stride;
  int num_pages;
  const int32_t* page_ids;
  uint8_t* page_mode;
  float* scale_out;
  int Hkv, D;
  int* err;
};

cudaError_t launch_gather(const GatherParams& p, const GatherRanges& r, int pages, cudaStream_t st);
cudaError_t launch_demote(const DemoteParams& p, int n, int num_sms, cudaStream_t st);

}  // namespace ekv
