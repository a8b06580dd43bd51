// noalloc.cu -- ekv_paged_decode_noalloc: the paged decode without a context, with
// its split-K scratch in a fixed device array owned by the library.
//
// Who needs it: code that must not call cudaMalloc on the decode path -- for example
// a serving runtime whose memory pool owns all device memory and forbids side
// allocations, a plugin whose enqueue hook runs where the host framework does not
// allow allocation, or a caller with a fixed memory budget decided at start-up. Such
// callers can still pass their own inputs and outputs; the only memory the decode adds
// (split-K partial records, per-(sequence, KV head) tickets, the error word) lives in
// one file-scope array below, which every GPU that loads this library keeps until the
// process exits.
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "decode.cuh"
#include "pool_maps.h"

namespace ekv {
cudaError_t launch_split_mma(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                             const DecodeParams& p, int D, int vmode, int grid, size_t smem, cudaStream_t st);
}  // namespace ekv

using namespace ekv;

namespace {

// Fixed scratch: 16 MiB per device. Layout: [plan ints kPlanInts][error word, 4 ints]
// [(m, l) records][acc records]. The records need (batch + #SMs) * (8 / H_kv) * H_q *
// (D + 2) floats; calls that need more are refused with EKV_ERR_CAPACITY.
constexpr size_t kScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr size_t kPlanBytes = (size_t)kPlanInts * 4;
constexpr size_t kErrBytes = 256;                      // 4 ints, padded for alignment

struct DeviceSetup {
  bool ready;
  unsigned char* scratch;                              // device address of g_decode_scratch
  int num_sms;
};
constexpr int kMaxDevices = 64;
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;

// Once per device, with that device current: the array's device address (host code
// only sees a stand-in for the symbol, never usable as a pointer) and the SM count.
cudaError_t device_setup(int dev, DeviceSetup* out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    s.scratch = static_cast<unsigned char*>(ptr);
    s.num_sms = sms;
    s.ready = true;
  }
  *out = s;
  return cudaSuccess;
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" ekv_status ekv_paged_decode_noalloc(int num_q_heads, int num_kv_heads, int head_dim, const void* q,
                                               const void* k_pages, const void* v_pages,
                                               long long v_page_stride_bytes, int num_pages,
                                               const float* v_scales, int scale_mode, const uint8_t* page_mode,
                                               int uniform_mode, const int32_t* block_table,
                                               int block_table_stride, const int32_t* seq_lens, int batch,
                                               float sm_scale, void* out, float* lse, int* err_out,
                                               void* stream) {
  const int Hq = num_q_heads, Hkv = num_kv_heads, D = head_dim;
  if (D != 64 && D != 128) return EKV_ERR_UNSUPPORTED;
  if (Hkv != 1 && Hkv != 2 && Hkv != 4 && Hkv != 8) return EKV_ERR_UNSUPPORTED;
  if (Hq <= 0 || Hq % Hkv != 0 || Hq / Hkv > 8) return EKV_ERR_UNSUPPORTED;
  if (batch < 0) return EKV_ERR_INVALID_ARG;
  if (batch > kMaxBatch) return EKV_ERR_CAPACITY;
  if (batch == 0) return EKV_OK;
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !out) return EKV_ERR_INVALID_ARG;
  if (num_pages < 1 || block_table_stride < 1) return EKV_ERR_INVALID_ARG;
  if (scale_mode != EKV_SCALE_PER_TENSOR && scale_mode != EKV_SCALE_PER_PAGE_HEAD) return EKV_ERR_INVALID_ARG;
  const int vmode = decode_vmode(page_mode, uniform_mode);
  if (vmode < 0) return EKV_ERR_INVALID_ARG;
  const long long n_elem = (long long)kPage * Hkv * D;
  if (v_page_stride_bytes < (vmode == kVE4M3 ? n_elem : 2 * n_elem) || (v_page_stride_bytes & 15))
    return EKV_ERR_INVALID_ARG;
  if (vmode == kVE4M3 && !v_scales) return EKV_ERR_INVALID_ARG;   // mixed: a compact page without scales is a device error
  if (!is_aligned16(q) || !is_aligned16(k_pages) || !is_aligned16(v_pages) || !is_aligned16(out))
    return EKV_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return EKV_ERR_INVALID_ARG;
  if (err_out && (reinterpret_cast<uintptr_t>(err_out) & 3u)) return EKV_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !isfinite(sm_scale)) sm_scale = 1.0f / sqrtf((float)D);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return EKV_ERR_CUDA;
  DeviceSetup ds;
  if (device_setup(dev, &ds) != cudaSuccess) return EKV_ERR_CUDA;

  // fit the partial records into the fixed array, or refuse the call
  const int NG = kWarps / Hkv;
  const size_t records = (size_t)(batch + ds.num_sms) * NG;
  const size_t ml_bytes = records * Hq * sizeof(float2);
  const size_t acc_bytes = records * Hq * D * sizeof(float);
  const size_t ml_off = kPlanBytes + kErrBytes;
  const size_t acc_off = (ml_off + ml_bytes + 255) & ~(size_t)255;
  if (acc_off + acc_bytes > kScratchBytes) return EKV_ERR_CAPACITY;

  CUtensorMap tk, t8, t16;
  if (!decode_pool_maps(&tk, &t8, &t16, k_pages, v_pages, D, Hkv, num_pages, v_page_stride_bytes, vmode))
    return EKV_ERR_INVALID_ARG;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* plan = reinterpret_cast<int*>(ds.scratch);
  int* err = err_out ? err_out : reinterpret_cast<int*>(ds.scratch + kPlanBytes);
  // The array keeps whatever the previous call left: clear the tickets of this batch
  // and the error word before the launch (records need no clearing).
  if (cudaMemsetAsync(plan + kPlanTicket, 0, (size_t)batch * kMaxKvHeads * 4, st) != cudaSuccess ||
      cudaMemsetAsync(err, 0, 4 * sizeof(int), st) != cudaSuccess)
    return EKV_ERR_CUDA;

  DecodeParams p;
  memset(&p, 0, sizeof(p));
  p.q = static_cast<const __half*>(q);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.page_mode = page_mode;
  p.v_scales = v_scales;
  p.part_ml = reinterpret_cast<float2*>(ds.scratch + ml_off);
  p.part_acc = reinterpret_cast<float*>(ds.scratch + acc_off);
  p.plan = plan;
  p.err = err;
  p.out = static_cast<__half*>(out);
  p.lse = lse;
  p.bt_stride = block_table_stride;
  p.batch = batch;
  p.num_pages = num_pages;
  p.uniform_mode = uniform_mode;
  p.scale_mode = scale_mode;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.NG = NG;
  p.D = D;
  p.qscale = sm_scale * 1.4426950408889634f;
  const size_t smem = split_layout(p, D, vmode, kAlgoMma);
  return launch_split_mma(tk, t8, t16, p, D, vmode, ds.num_sms, smem, st) == cudaSuccess ? EKV_OK : EKV_ERR_CUDA;
}
