// decode.cuh -- parameters and shared-memory layout of the split-K paged decode.
#pragma once

#include "common.cuh"

namespace ekv {

// Value-page handling, fixed per launch:
//   kVE4M3  every page compact (page_mode == NULL, uniform COMPACT)
//   kVFP16  every page TARGET  (page_mode == NULL, uniform TARGET): the native path,
//           no mode bytes, no scales
//   kVMixed per-page mode byte, FP16-sized value slots in shared memory
// Value pool of a launch: all E4M3, all FP16, or per-page modes (TARGET / E4M3 / BASE;
// also a uniform BASE pool, which has the mixed layout).
enum VMode { kVE4M3 = 0, kVFP16 = 1, kVMixed = 2 };

// Consumer algorithm: CUDA-core FP32 FMAs or mma.sync tensor-core tiles.
enum Algo { kAlgoSimt = 0, kAlgoMma = 1 };

constexpr int kWarps = 8;                              // one warp per (KV head, page group)
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSlots = 32;                          // ring slots per warp
constexpr int kSplitSmemMax = 232448 - 1024;           // dynamic smem opt-in (static smem < 1 KB)

// plan buffer (int32), zeroed at context creation and left zeroed by every launch:
//   [kPlanTicket + b * 8 + h] partial records counted so far for (b, KV head h) of a
//                             sequence split across CTAs; the warp that brings it to
//                             its final count merges and resets it
constexpr int kPlanTicket = 0;
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
  int Hq, Hkv, G, NG;       // NG = 8 / Hkv page groups (warps sharing a KV head)
  int D;
  float qscale;             // sm_scale * log2(e)
  // shared-memory layout of the launch (set by the host for the slot size and batch)
  int nsl;                  // ring slots per warp
  int bar_off, cu_off, pbuf_off;
  // elastic layout (ElasticKV Sec. 3.1-3.2), all null / 0 for the plain call:
  const int32_t* v_block_table;   // [B][bt_stride] value locations (half-slot indices)
  const int32_t* boundaries;      // [B][2] TARGET-BASE-TARGET boundaries, or null
  int num_v_slots;                // value slots (locations 0 .. 2*num_v_slots-1)
  int elastic;                    // 1: values read through v_block_table
  // 1: launched with programmatic serialization (tensor-core consumer only). Before its
  // griddepcontrol.wait the kernel reads only seq_lens, the block tables, page metadata
  // and the K/V pages that are not the last page of their sequence; q is read and every
  // output, record and ticket written after it.
  int pdl;
#ifdef EKV_TEST_WAIT_TIMEOUT
  // test build only: 1 makes the first ring wait of CTA 0, warp 0 run out
  int inject_timeout;
#endif
};

constexpr int kMetaCompact = 1;   // E4M3 value page
constexpr int kMetaSkip = 2;      // no page, or a page that failed its checks
constexpr int kMetaBase = 4;      // BASE value page (FP16 high bytes)

// One ring slot holds one (page, KV head) slice: K [16][D] fp16 as D/64 blocks of 16
// rows x 128 B (one 5-D TMA box), then V [16][D] as E4M3 rows (one box of 16 x D
// bytes) or fp16 (D/64 blocks, one box). Slots are 1024-byte aligned, as the 128B
// swizzle requires.
template <int D, int VMODE>
struct Slot {
  static constexpr int kK = kPage * D * 2;
  static constexpr int kV = kPage * D * (VMODE == kVE4M3 ? 1 : 2);
  static constexpr int kBytes = kK + kV;
};

// Opt a kernel into `bytes` of dynamic shared memory, once per (kernel, device).
cudaError_t set_smem_attr(const void* kern, int bytes = kSplitSmemMax);
size_t split_layout(DecodeParams& p, int D, int vmode, int algo);

}  // namespace ekv
