// pool_maps.h -- host-side TMA tensor maps of the page pools (decode entry points).
//
// A ring slot receives one (page, KV head) slice per tensor, each with a single
// cp.async.bulk.tensor:
//   K and FP16 V: 5-D view (d mod 64, token, d / 64, head, page) of [P][16][H_kv][D]
//                 fp16; the box {64, 16, D/64, 1, 1} lands as [D/64][16][128 B] with
//                 the 128B swizzle, i.e. D/64 blocks of 16 rows x 128 B.
//   byte V:       4-D view (d, head, token, page) of [P][16][H_kv][D] bytes (E4M3 codes
//                 or BASE high bytes); the box {D, 1, 16, 1} lands as [16][D B] (128B
//                 swizzle for D = 128, 64B for D = 64).
// One instruction per tensor matters: issuing a bulk tensor copy costs the issuing
// warp the same time whatever the box size, and the consumer warps issue their own.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "decode.cuh"

namespace ekv {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// fp16 pool [P][16][H_kv][D] with `page_stride` bytes between pages.
inline bool encode_fp16_slice_map(CUtensorMap* tm, const void* base, int D, int Hkv, int num_pages,
                                  long long page_stride) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[5] = {64, (cuuint64_t)kPage, (cuuint64_t)(D / 64), (cuuint64_t)Hkv, (cuuint64_t)num_pages};
  cuuint64_t strides[4] = {(cuuint64_t)Hkv * D * 2, 128, (cuuint64_t)D * 2, (cuuint64_t)page_stride};
  cuuint32_t box[5] = {64, (cuuint32_t)kPage, (cuuint32_t)(D / 64), 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 pool [P][16][H_kv][D] bytes with `page_stride` bytes between pages.
inline bool encode_e4m3_slice_map(CUtensorMap* tm, const void* base, int D, int Hkv, int num_pages,
                                  long long page_stride) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)kPage, (cuuint64_t)num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)D, (cuuint64_t)Hkv * D, (cuuint64_t)page_stride};
  cuuint32_t box[4] = {(cuuint32_t)D, 1, (cuuint32_t)kPage, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Byte values addressed by half-slot location (the elastic layout): 5-D view (d, head,
// token, half, slot) of slots of `slot_stride` bytes, each two halves of 16*H_kv*D bytes;
// the box {D, 1, 16, 1, 1} lands as [16][D B] like the 4-D byte view.
inline bool encode_byte_half_map(CUtensorMap* tm, const void* base, int D, int Hkv, int num_slots,
                                 long long slot_stride) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t half = (cuuint64_t)kPage * Hkv * D;
  cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)kPage, 2, (cuuint64_t)num_slots};
  cuuint64_t strides[4] = {(cuuint64_t)D, (cuuint64_t)Hkv * D, half, (cuuint64_t)slot_stride};
  cuuint32_t box[5] = {(cuuint32_t)D, 1, (cuuint32_t)kPage, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Value-pool kind of a decode call: per-page modes (a mode table, or a uniform BASE
// pool, which has the mixed layout), uniform E4M3, or uniform FP16. -1: bad uniform_mode.
inline int decode_vmode(const uint8_t* page_mode, int uniform_mode) {
  if (uniform_mode < EKV_MODE_TARGET_FP16 || uniform_mode > EKV_MODE_BASE) return -1;
  if (page_mode || uniform_mode == EKV_MODE_BASE) return kVMixed;
  return uniform_mode == EKV_MODE_COMPACT_E4M3 ? kVE4M3 : kVFP16;
}

// The three maps of one decode call; unused ones stay zeroed. False on an encode error.
// num_v_slots > 0: the elastic layout (values located by half-slot index over
// num_v_slots slots); 0: the value page of logical page p is slot p.
inline bool decode_pool_maps(CUtensorMap* tk, CUtensorMap* t8, CUtensorMap* t16, const void* k_pages,
                             const void* v_pages, int D, int Hkv, int num_pages, long long v_page_stride,
                             int vmode, int num_v_slots = 0) {
  memset(tk, 0, sizeof(*tk));
  memset(t8, 0, sizeof(*t8));
  memset(t16, 0, sizeof(*t16));
  if (!encode_fp16_slice_map(tk, k_pages, D, Hkv, num_pages, (long long)kPage * Hkv * D * 2)) return false;
  const int vp = num_v_slots > 0 ? num_v_slots : num_pages;
  if (vmode != kVFP16) {
    const bool ok = num_v_slots > 0 ? encode_byte_half_map(t8, v_pages, D, Hkv, vp, v_page_stride)
                                    : encode_e4m3_slice_map(t8, v_pages, D, Hkv, vp, v_page_stride);
    if (!ok) return false;
  }
  if (vmode != kVE4M3 && !encode_fp16_slice_map(t16, v_pages, D, Hkv, vp, v_page_stride)) return false;
  return true;
}

}  // namespace ekv
