// decode.cuh -- parameters and shared-memory layout of the split-K paged decode.
#pragma once

#include "common.cuh"

namespace ekv {

// Value-page handling, fixed per launch:
//   kVE4M3  every page compact (page_mode == NULL, uniform COMPACT)
//   kVFP16  every page TARGET  (page_mode == NULL, uniform TARGET): the native path,
//           no mode bytes, no scales
//   kVMixed per-page mode byte, FP16-sized value slots in shared memory
enum VMode { kVE4M3 = 0, kVFP16 = 1, kVMixed = 2 };

// Consumer algorithm: CUDA-core FP32 FMAs or mma.sync tensor-core tiles.
enum Algo { kAlgoSimt = 0, kAlgoMma = 1 };

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;   // + 1 TMA producer warp
constexpr int kSmemBudget = 196608;                    // bytes of pipeline stages
constexpr int kSplitSmemMax = 225280;                  // dynamic smem opt-in of the split kernels

// plan buffer (int32), zeroed at context creation:
//   [kPlanBad + b * 8 + h]    set when sequence b read bad data (page id, mode, scale,
//                             length); the merge of (b, h) zeroes the output and clears it
//   [kPlanTicket + b * 8 + h] partial records written so far for (b, KV head h); the
//                             warp that brings it to its final count merges and resets it
constexpr int kPlanBad = 0;
constexpr int kPlanTicket = kPlanBad + kMaxBatch * kMaxKvHeads;
constexpr int kPlanInts = kPlanTicket + kMaxBatch * kMaxKvHeads;

struct DecodeParams {
  const __half* q;          // [B][Hq][D]
  const int32_t* block_table;
  const int32_t* seq_lens;
  const uint8_t* page_mode; // kVMixed only
  const float* v_scales;
  float* part_acc;          // [records][Hq][D]
  float2* part_ml;          // [records][Hq]   (m in log2 units, l)
  int* plan;
  int* err;
  __half* out;              // [B][Hq][D]
  float* lse;               // [B][Hq] or null
  int bt_stride;
  int batch;
  int num_pages;
  int uniform_mode;
  int scale_mode;
  int Hq, Hkv, G, NG;       // NG = 8 / Hkv page groups per stage
  int D;
  float qscale;             // sm_scale * log2(e)
};

// Metadata of one page slot of a pipeline stage, written by the producer.
struct PageMeta {
  int page;
  int ntok;     // valid tokens of this page (1..16)
  int flags;    // kMetaCompact | kMetaSkip
  int pad;
  float scale[kMaxKvHeads];
};
constexpr int kMetaCompact = 1;
constexpr int kMetaSkip = 2;

template <int D, int VMODE>
struct StageLayout {
  // One stage holds 8 (page, KV head) slices: NG = 8 / Hkv pages of Hkv heads.
  static constexpr int kKStage = 8 * kPage * D * 2;                           // fp16 K
  static constexpr int kVStage = 8 * kPage * D * (VMODE == kVE4M3 ? 1 : 2);   // V slot
  static constexpr int kStageBytes = kKStage + kVStage;
  static constexpr int kStages = kSmemBudget / kStageBytes;
  static constexpr int kMetaOff = kStages * kStageBytes;
  static constexpr int kBarOff = kMetaOff + kStages * 8 * (int)sizeof(PageMeta);
  static constexpr int kCuOff = kBarOff + 2 * kStages * 8;
  static_assert(kStages >= 2, "pipeline needs two stages");
};

cudaError_t set_smem_attr(const void* kern);
size_t split_smem_bytes(int D, int vmode, int algo, int batch);

}  // namespace ekv
