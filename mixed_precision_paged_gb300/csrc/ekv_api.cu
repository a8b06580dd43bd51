// ekv_api.cu -- the C ABI (include/ekv.h): argument checks, tensor maps, launches.
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "decode.cuh"
#include "gather_demote.cuh"
#include "pool_maps.h"
#include "prefill.cuh"

namespace ekv {
cudaError_t launch_split_simt(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                              const DecodeParams& p, int D, int vmode, int grid, size_t smem, cudaStream_t st);
cudaError_t launch_split_mma(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                             const DecodeParams& p, int D, int vmode, int grid, size_t smem, cudaStream_t st);

// ------------------------------------------------------------- launch floor
// An empty kernel with the split kernel's block, shared memory and parameter list: what
// a timed launch costs before any work (ekv_profile_launch_floor).
__global__ void __launch_bounds__(kThreads, 1)
launch_floor_kernel(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                    const __grid_constant__ CUtensorMap, const DecodeParams) {}

// One thread that returns `ns` nanoseconds after it starts: keeps the stream busy while
// the host queues the timed launches behind it (bounded by construction).
__global__ void hold_stream_kernel(uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) __nanosleep(1000);
}

static cudaError_t launch_floor(int grid, size_t smem, cudaStream_t st, int reps, cudaEvent_t* ev) {
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(launch_floor_kernel));
  if (e != cudaSuccess) return e;
  hold_stream_kernel<<<1, 1, 0, st>>>(2000000ull + 20000ull * (uint64_t)reps);
  CUtensorMap tm{};
  DecodeParams p{};
  for (int i = 0; i < reps; ++i) {
    cudaEventRecord(ev[2 * i], st);
    launch_floor_kernel<<<grid, kThreads, smem, st>>>(tm, tm, tm, p);
    cudaEventRecord(ev[2 * i + 1], st);
  }
  return cudaGetLastError();
}
}  // namespace ekv

using namespace ekv;

struct ekv_ctx {
  int device = 0;
  int num_sms = 0;
  int split_ctas = 0;
  ekv_config cfg{};
  int NG = 1;
  int variant = 0;            // 0 tensor-core consumer, 1 CUDA-core consumer
  int pdl = 0;                // 1: decode launched with programmatic serialization
  float* part_acc = nullptr;
  float2* part_ml = nullptr;
  int* plan = nullptr;
  int* err = nullptr;
  cudaStream_t last_stream = nullptr;
  bool profiling = false;
  std::vector<cudaEvent_t> ev;   // pairs (start, stop)
  size_t ev_used = 0;            // pairs recorded since the last read
  double prof_ms = 0.0;
  long long prof_launches = 0;
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
    else prev = -1;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

// The kind of the last kernel this library (any context) enqueued on each stream, kept
// for the streams where it writes what a programmatically launched kernel of the
// library reads before its griddepcontrol.wait: the page-mode transitions write value
// pages, mode bytes and scales; the cache writer writes the last page of each sequence.
// CUDA makes a preceding grid's writes visible to a programmatically launched kernel
// only after that kernel's wait, so a decode after a transition, and a gather after a
// transition or the writer, is launched in plain stream order. Other launches (decode,
// gather, prefill) remove their stream from the map.
enum LastKernel { kAfterReader = 0, kAfterAppend = 1, kAfterTransition = 2 };
std::mutex g_last_mu;
std::unordered_map<cudaStream_t, int> g_last_kernel;

void note_launch(cudaStream_t st, int kind) {
  std::lock_guard<std::mutex> lock(g_last_mu);
  if (kind != kAfterReader) g_last_kernel[st] = kind;
  else g_last_kernel.erase(st);
}

int last_kernel(cudaStream_t st) {
  std::lock_guard<std::mutex> lock(g_last_mu);
  auto it = g_last_kernel.find(st);
  return it == g_last_kernel.end() ? kAfterReader : it->second;
}

#ifdef EKV_TEST_WAIT_TIMEOUT
// test build only: decode calls left that run their first ring wait out
int g_inject_timeout_calls = 0;
#endif

bool supported_shape(int Hq, int Hkv, int D) {
  if (D != 64 && D != 128) return false;
  if (Hkv != 1 && Hkv != 2 && Hkv != 4 && Hkv != 8) return false;
  if (Hq <= 0 || Hq % Hkv != 0) return false;
  const int G = Hq / Hkv;
  return G >= 1 && G <= 8;
}

}  // namespace

extern "C" {

const char* ekv_status_string(int s) {
  switch (s) {
    case EKV_OK: return "EKV_OK";
    case EKV_ERR_INVALID_ARG: return "EKV_ERR_INVALID_ARG";
    case EKV_ERR_UNSUPPORTED: return "EKV_ERR_UNSUPPORTED";
    case EKV_ERR_CAPACITY: return "EKV_ERR_CAPACITY";
    case EKV_ERR_CUDA: return "EKV_ERR_CUDA";
    case EKV_ERR_DEVICE_CHECK: return "EKV_ERR_DEVICE_CHECK";
    default: return "EKV_UNKNOWN_STATUS";
  }
}

ekv_status ekv_create(ekv_ctx** out, const ekv_config* cfg) {
  if (!out) return EKV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg) return EKV_ERR_INVALID_ARG;
  if (cfg->max_batch < 1 || cfg->num_q_heads < 1 || cfg->num_kv_heads < 1 || cfg->head_dim < 1)
    return EKV_ERR_INVALID_ARG;
  if (!supported_shape(cfg->num_q_heads, cfg->num_kv_heads, cfg->head_dim) || cfg->max_batch > kMaxBatch)
    return EKV_ERR_UNSUPPORTED;
  ekv_ctx* c = new (std::nothrow) ekv_ctx();
  if (!c) return EKV_ERR_CUDA;
  c->cfg = *cfg;
  c->NG = kWarps / cfg->num_kv_heads;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    delete c;
    return EKV_ERR_CUDA;
  }
  c->split_ctas = c->num_sms;                     // one 256-thread CTA per SM (~220 KB smem)
  const size_t records = (size_t)(cfg->max_batch + c->split_ctas) * c->NG;
  const size_t hq = (size_t)cfg->num_q_heads;
  bool ok = cudaMalloc(&c->part_acc, records * hq * cfg->head_dim * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&c->part_ml, records * hq * sizeof(float2)) == cudaSuccess &&
            cudaMalloc(&c->plan, kPlanInts * sizeof(int)) == cudaSuccess &&
            cudaMalloc(&c->err, 4 * sizeof(int)) == cudaSuccess &&
            cudaMemset(c->plan, 0, kPlanInts * sizeof(int)) == cudaSuccess &&
            cudaMemset(c->err, 0, 4 * sizeof(int)) == cudaSuccess &&
            cudaDeviceSynchronize() == cudaSuccess;
  if (!ok || !encode_fn()) {
    ekv_destroy(c);
    return EKV_ERR_CUDA;
  }
  *out = c;
  return EKV_OK;
}

ekv_status ekv_destroy(ekv_ctx* c) {
  if (!c) return EKV_OK;
  DeviceGuard g(c->device);
  cudaDeviceSynchronize();
  for (cudaEvent_t e : c->ev) cudaEventDestroy(e);
  cudaFree(c->part_acc);
  cudaFree(c->part_ml);
  cudaFree(c->plan);
  cudaFree(c->err);
  delete c;
  return EKV_OK;
}

ekv_status ekv_set_decode_variant(ekv_ctx* c, int variant) {
  if (!c || (variant != 0 && variant != 1)) return EKV_ERR_INVALID_ARG;
  c->variant = variant;
  return EKV_OK;
}

ekv_status ekv_set_pdl(ekv_ctx* c, int enable) {
  if (!c || (enable != 0 && enable != 1)) return EKV_ERR_INVALID_ARG;
  c->pdl = enable;
  return EKV_OK;
}

namespace {

// Shared body of the plain and the elastic decode. Elastic: v_block_table != null
// (num_v_slots value slots), boundaries optional, has_base = 0 forces the native path.
ekv_status decode_impl(ekv_ctx* c, const void* q, const void* k_pages, const void* v_pages,
                       long long v_page_stride_bytes, int num_pages, int num_v_slots, const float* v_scales,
                       int scale_mode, const uint8_t* page_mode, int uniform_mode, const int32_t* block_table,
                       const int32_t* v_block_table, int block_table_stride, const int32_t* boundaries,
                       int has_base, const int32_t* seq_lens, int batch, float sm_scale, void* out, float* lse,
                       void* stream) {
  if (!c) return EKV_ERR_INVALID_ARG;
  if (batch < 0) return EKV_ERR_INVALID_ARG;
  if (batch > c->cfg.max_batch) return EKV_ERR_CAPACITY;
  if (batch == 0) return EKV_OK;
  const int Hq = c->cfg.num_q_heads, Hkv = c->cfg.num_kv_heads, D = c->cfg.head_dim;
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !out) return EKV_ERR_INVALID_ARG;
  if (num_pages < 1 || block_table_stride < 1) return EKV_ERR_INVALID_ARG;
  if (scale_mode != EKV_SCALE_PER_TENSOR && scale_mode != EKV_SCALE_PER_PAGE_HEAD) return EKV_ERR_INVALID_ARG;
  const bool elastic = v_block_table != nullptr;
  if (elastic && num_v_slots < 1) return EKV_ERR_INVALID_ARG;
  int vmode = decode_vmode(page_mode, uniform_mode);
  if (vmode < 0) return EKV_ERR_INVALID_ARG;
  if (elastic) vmode = has_base ? kVMixed : kVFP16;       // ElasticKV's batch-level indicator
  const long long n_elem = (long long)kPage * Hkv * D;
  const long long need = vmode == kVE4M3 ? n_elem : 2 * n_elem;
  if (v_page_stride_bytes < need || (v_page_stride_bytes & 15)) return EKV_ERR_INVALID_ARG;
  if (vmode == kVE4M3 && !v_scales) return EKV_ERR_INVALID_ARG;   // mixed: a compact page without scales is a device error
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out)) return EKV_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return EKV_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !isfinite(sm_scale)) sm_scale = 1.0f / sqrtf((float)D);

  DeviceGuard g(c->device);
  CUtensorMap tk, t8, t16;
  if (!decode_pool_maps(&tk, &t8, &t16, k_pages, v_pages, D, Hkv, num_pages, v_page_stride_bytes, vmode,
                        elastic ? num_v_slots : 0))
    return EKV_ERR_INVALID_ARG;

  DecodeParams p;
  memset(&p, 0, sizeof(p));
  p.q = static_cast<const __half*>(q);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.page_mode = page_mode;
  p.v_scales = v_scales;
  p.part_acc = c->part_acc;
  p.part_ml = c->part_ml;
  p.plan = c->plan;
  p.err = c->err;
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
  p.NG = c->NG;
  p.D = D;
  p.qscale = sm_scale * 1.4426950408889634f;
  p.v_block_table = v_block_table;
  p.boundaries = elastic ? boundaries : nullptr;
  p.num_v_slots = elastic ? num_v_slots : num_pages;
  p.elastic = elastic ? 1 : 0;
  p.pdl = c->pdl && c->variant == 0 ? 1 : 0;
#ifdef EKV_TEST_WAIT_TIMEOUT
  if (g_inject_timeout_calls > 0 && c->variant == 0) {
    p.inject_timeout = 1;
    --g_inject_timeout_calls;
  }
#endif

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  c->last_stream = st;
  if (p.pdl && last_kernel(st) == kAfterTransition) p.pdl = 0;   // plain stream order after a transition
  const bool timed = c->profiling && c->ev_used * 2 + 1 < c->ev.size();
  if (timed) cudaEventRecord(c->ev[2 * c->ev_used], st);
  const int algo = c->variant == 1 ? kAlgoSimt : kAlgoMma;
  const size_t smem = split_layout(p, D, vmode, algo);
  cudaError_t e = algo == kAlgoSimt ? launch_split_simt(tk, t8, t16, p, D, vmode, c->split_ctas, smem, st)
                                    : launch_split_mma(tk, t8, t16, p, D, vmode, c->split_ctas, smem, st);
  if (e != cudaSuccess) return EKV_ERR_CUDA;
  note_launch(st, kAfterReader);
  if (timed) {
    cudaEventRecord(c->ev[2 * c->ev_used + 1], st);
    ++c->ev_used;
  }
  return EKV_OK;
}

}  // namespace

ekv_status ekv_paged_decode(ekv_ctx* c, const void* q, const void* k_pages, const void* v_pages,
                            long long v_page_stride_bytes, int num_pages, const float* v_scales,
                            int scale_mode, const uint8_t* page_mode, int uniform_mode,
                            const int32_t* block_table, int block_table_stride,
                            const int32_t* seq_lens, int batch, float sm_scale, void* out,
                            float* lse, void* stream) {
  return decode_impl(c, q, k_pages, v_pages, v_page_stride_bytes, num_pages, 0, v_scales, scale_mode, page_mode,
                     uniform_mode, block_table, nullptr, block_table_stride, nullptr, 1, seq_lens, batch, sm_scale,
                     out, lse, stream);
}

ekv_status ekv_paged_decode_elastic(ekv_ctx* c, const void* q, const void* k_pages, const void* v_pages,
                                    long long v_page_stride_bytes, int num_pages, int num_v_slots,
                                    const float* v_scales, int scale_mode, const uint8_t* page_mode,
                                    int uniform_mode, const int32_t* block_table, const int32_t* v_block_table,
                                    int block_table_stride, const int32_t* boundaries, int has_base,
                                    const int32_t* seq_lens, int batch, float sm_scale, void* out, float* lse,
                                    void* stream) {
  if (!v_block_table) return EKV_ERR_INVALID_ARG;
  return decode_impl(c, q, k_pages, v_pages, v_page_stride_bytes, num_pages, num_v_slots, v_scales, scale_mode,
                     page_mode, uniform_mode, block_table, v_block_table, block_table_stride, boundaries, has_base,
                     seq_lens, batch, sm_scale, out, lse, stream);
}

namespace {

// The gather of both layouts: v_block_table null -> the plain layout (values at the
// logical page id; num_v_slots, boundaries and has_base unused).
ekv_status gather_impl(ekv_ctx* c, const void* k_pages, const void* v_pages, long long v_page_stride_bytes,
                       int num_pages, int num_v_slots, const float* v_scales, int scale_mode,
                       const uint8_t* page_mode, int uniform_mode, const int32_t* block_table,
                       const int32_t* v_block_table, int block_table_stride, const int32_t* boundaries,
                       int has_base, int block_table_rows, const int32_t* page_range, int n, void* ws_k,
                       void* ws_v, int32_t* ws_indices, int ws_pages, int apply_scale, void* stream) {
  if (!c || n < 0 || ws_pages < 0) return EKV_ERR_INVALID_ARG;
  if (n == 0) return EKV_OK;
  const int Hkv = c->cfg.num_kv_heads, D = c->cfg.head_dim;
  if (!page_range || !k_pages || !v_pages || !block_table || !ws_k || !ws_v || !ws_indices)
    return EKV_ERR_INVALID_ARG;
  if (num_pages < 1 || block_table_stride < 1 || block_table_rows < 1) return EKV_ERR_INVALID_ARG;
  if (scale_mode != EKV_SCALE_PER_TENSOR && scale_mode != EKV_SCALE_PER_PAGE_HEAD) return EKV_ERR_INVALID_ARG;
  if (uniform_mode < EKV_MODE_TARGET_FP16 || uniform_mode > EKV_MODE_BASE) return EKV_ERR_INVALID_ARG;
  const bool any_compact = uniform_mode == EKV_MODE_COMPACT_E4M3;   // a mode table: checked per page
  const bool any_target = page_mode || uniform_mode != EKV_MODE_COMPACT_E4M3;
  const long long n_elem = (long long)kPage * Hkv * D;
  // the pair-structured layout: every slot holds a TARGET page or two halves
  if (v_page_stride_bytes < (v_block_table || any_target ? 2 * n_elem : n_elem) || (v_page_stride_bytes & 15))
    return EKV_ERR_INVALID_ARG;
  if (v_block_table && num_v_slots < 1) return EKV_ERR_INVALID_ARG;
  if (any_compact && apply_scale && !v_scales) return EKV_ERR_INVALID_ARG;
  if (!aligned16(k_pages) || !aligned16(v_pages) || !aligned16(ws_k) || !aligned16(ws_v))
    return EKV_ERR_INVALID_ARG;
  long long total = 0;
  for (int i = 0; i < n; ++i) {
    const int seq = page_range[3 * i], first = page_range[3 * i + 1], num = page_range[3 * i + 2];
    if (seq < 0 || seq >= block_table_rows || first < 0 || num < 0 ||
        (long long)first + num > block_table_stride)
      return EKV_ERR_INVALID_ARG;
    total += num;
  }
  if (total > ws_pages) return EKV_ERR_CAPACITY;

  DeviceGuard g(c->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  c->last_stream = st;
  GatherParams p;
  p.k_pages = static_cast<const __half*>(k_pages);
  p.v_pages = static_cast<const uint8_t*>(v_pages);
  p.v_page_stride = v_page_stride_bytes;
  p.num_pages = num_pages;
  p.v_scales = v_scales;
  p.scale_mode = scale_mode;
  p.page_mode = page_mode;
  p.uniform_mode = uniform_mode;
  p.block_table = block_table;
  p.bt_stride = block_table_stride;
  p.ws_k = static_cast<__half*>(ws_k);
  p.ws_v = static_cast<__half*>(ws_v);
  p.ws_indices = ws_indices;
  p.Hkv = Hkv;
  p.D = D;
  p.apply_scale = apply_scale ? 1 : 0;
  p.err = c->err;
  p.v_block_table = v_block_table;
  p.num_v_slots = num_v_slots;
  p.boundaries = v_block_table ? boundaries : nullptr;
  p.has_base = v_block_table ? has_base : 1;
  p.pdl = c->pdl && last_kernel(st) == kAfterReader ? 1 : 0;   // not right after a writer of the pool
  int base = 0;
  for (int i0 = 0; i0 < n; i0 += kMaxRanges) {
    GatherRanges r;
    memset(&r, 0, sizeof(r));
    r.n = n - i0 < kMaxRanges ? n - i0 : kMaxRanges;
    int off = 0;
    for (int k = 0; k < r.n; ++k) {
      r.seq[k] = page_range[3 * (i0 + k)];
      r.first[k] = page_range[3 * (i0 + k) + 1];
      r.off[k] = off;
      off += page_range[3 * (i0 + k) + 2];
    }
    r.off[r.n] = off;
    p.ws_base = base;
    if (launch_gather(p, r, off, st) != cudaSuccess) return EKV_ERR_CUDA;
    base += off;
  }
  note_launch(st, kAfterReader);
  return EKV_OK;
}

}  // namespace

ekv_status ekv_gather_prefill(ekv_ctx* c, const void* k_pages, const void* v_pages,
                              long long v_page_stride_bytes, int num_pages, const float* v_scales,
                              int scale_mode, const uint8_t* page_mode, int uniform_mode,
                              const int32_t* block_table, int block_table_stride, int block_table_rows,
                              const int32_t* page_range, int n, void* ws_k, void* ws_v,
                              int32_t* ws_indices, int ws_pages, int apply_scale, void* stream) {
  return gather_impl(c, k_pages, v_pages, v_page_stride_bytes, num_pages, 0, v_scales, scale_mode, page_mode,
                     uniform_mode, block_table, nullptr, block_table_stride, nullptr, 1, block_table_rows,
                     page_range, n, ws_k, ws_v, ws_indices, ws_pages, apply_scale, stream);
}

ekv_status ekv_gather_prefill_elastic(ekv_ctx* c, const void* k_pages, const void* v_pages,
                                      long long v_page_stride_bytes, int num_pages, int num_v_slots,
                                      const float* v_scales, int scale_mode, const uint8_t* page_mode,
                                      int uniform_mode, const int32_t* block_table,
                                      const int32_t* v_block_table, int block_table_stride,
                                      const int32_t* boundaries, int has_base, int block_table_rows,
                                      const int32_t* page_range, int n, void* ws_k, void* ws_v,
                                      int32_t* ws_indices, int ws_pages, int apply_scale, void* stream) {
  if (!v_block_table) return EKV_ERR_INVALID_ARG;
  return gather_impl(c, k_pages, v_pages, v_page_stride_bytes, num_pages, num_v_slots, v_scales, scale_mode,
                     page_mode, uniform_mode, block_table, v_block_table, block_table_stride, boundaries,
                     has_base, block_table_rows, page_range, n, ws_k, ws_v, ws_indices, ws_pages, apply_scale,
                     stream);
}

namespace {

// Shared checks and launch of the page-mode transitions.
ekv_status transition(ekv_ctx* c, int op, void* v_pages, long long v_page_stride_bytes, int num_pages,
                      int num_slots, const int32_t* page_ids, const int32_t* src_loc, const int32_t* dst_loc,
                      int n, uint8_t* page_mode, float* scale_out, uint8_t* low, void* stream) {
  if (!c || n < 0) return EKV_ERR_INVALID_ARG;
  if (n == 0) return EKV_OK;
  const int Hkv = c->cfg.num_kv_heads, D = c->cfg.head_dim;
  if (!v_pages || !page_ids || !page_mode || num_pages < 1 || num_slots < 1) return EKV_ERR_INVALID_ARG;
  if (op < kToE4M3 || op > kPromote) return EKV_ERR_INVALID_ARG;
  if (op == kToE4M3 && !scale_out) return EKV_ERR_INVALID_ARG;
  if (op == kPromote && !low) return EKV_ERR_INVALID_ARG;
  if (low && !aligned16(low)) return EKV_ERR_INVALID_ARG;
  const long long n_elem = (long long)kPage * Hkv * D;
  if (v_page_stride_bytes < 2 * n_elem || (v_page_stride_bytes & 15) || !aligned16(v_pages))
    return EKV_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  c->last_stream = st;
  DemoteParams p;
  p.v_pages = static_cast<uint8_t*>(v_pages);
  p.v_page_stride = v_page_stride_bytes;
  p.num_pages = num_pages;
  p.page_ids = page_ids;
  p.page_mode = page_mode;
  p.scale_out = scale_out;
  p.low = low;
  p.src_loc = src_loc;
  p.dst_loc = dst_loc;
  p.num_slots = num_slots;
  p.Hkv = Hkv;
  p.D = D;
  p.err = c->err;
  if (launch_transition(p, op, n, c->num_sms, st) != cudaSuccess) return EKV_ERR_CUDA;
  note_launch(st, kAfterTransition);
  return EKV_OK;
}

}  // namespace

ekv_status ekv_demote_pages(ekv_ctx* c, void* v_pages, long long v_page_stride_bytes, int num_pages,
                            const int32_t* page_ids, int n, uint8_t* page_mode, float* scale_out,
                            void* stream) {
  return transition(c, kToE4M3, v_pages, v_page_stride_bytes, num_pages, num_pages, page_ids, nullptr, nullptr,
                    n, page_mode, scale_out, nullptr, stream);
}

ekv_status ekv_demote_pages_base(ekv_ctx* c, void* v_pages, long long v_page_stride_bytes, int num_pages,
                                 const int32_t* page_ids, int n, uint8_t* page_mode, void* low_out,
                                 void* stream) {
  return transition(c, kToBase, v_pages, v_page_stride_bytes, num_pages, num_pages, page_ids, nullptr, nullptr,
                    n, page_mode, nullptr, static_cast<uint8_t*>(low_out), stream);
}

ekv_status ekv_promote_pages(ekv_ctx* c, void* v_pages, long long v_page_stride_bytes, int num_pages,
                             const int32_t* page_ids, int n, uint8_t* page_mode, const void* low_in,
                             void* stream) {
  return transition(c, kPromote, v_pages, v_page_stride_bytes, num_pages, num_pages, page_ids, nullptr, nullptr,
                    n, page_mode, nullptr, static_cast<uint8_t*>(const_cast<void*>(low_in)), stream);
}

ekv_status ekv_transition_pages(ekv_ctx* c, int op, void* v_pages, long long v_page_stride_bytes, int num_slots,
                                int num_pages, const int32_t* page_ids, const int32_t* src_loc,
                                const int32_t* dst_loc, int n, uint8_t* page_mode, float* scale_out, void* low,
                                void* stream) {
  return transition(c, op, v_pages, v_page_stride_bytes, num_pages, num_slots, page_ids, src_loc, dst_loc, n,
                    page_mode, scale_out, static_cast<uint8_t*>(low), stream);
}

ekv_status ekv_append_kv(ekv_ctx* c, const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                         long long v_page_stride_bytes, int num_pages, const float* v_scales, int scale_mode,
                         const uint8_t* page_mode, int uniform_mode, const int32_t* block_table,
                         int block_table_stride, const int32_t* positions, int batch, void* stream) {
  if (!c || batch < 0) return EKV_ERR_INVALID_ARG;
  if (batch == 0) return EKV_OK;
  const int Hkv = c->cfg.num_kv_heads, D = c->cfg.head_dim;
  if (!k_new || !v_new || !k_pages || !v_pages || !block_table || !positions) return EKV_ERR_INVALID_ARG;
  if (num_pages < 1 || block_table_stride < 1) return EKV_ERR_INVALID_ARG;
  if (scale_mode != EKV_SCALE_PER_TENSOR && scale_mode != EKV_SCALE_PER_PAGE_HEAD) return EKV_ERR_INVALID_ARG;
  const int vmode = decode_vmode(page_mode, uniform_mode);
  if (vmode < 0) return EKV_ERR_INVALID_ARG;
  const long long n_elem = (long long)kPage * Hkv * D;
  if (v_page_stride_bytes < (vmode == kVE4M3 ? n_elem : 2 * n_elem) || (v_page_stride_bytes & 15))
    return EKV_ERR_INVALID_ARG;
  if (vmode == kVE4M3 && !v_scales) return EKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages))
    return EKV_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  c->last_stream = st;
  AppendParams p;
  p.k_new = static_cast<const __half*>(k_new);
  p.v_new = static_cast<const __half*>(v_new);
  p.k_pages = static_cast<__half*>(k_pages);
  p.v_pages = static_cast<uint8_t*>(v_pages);
  p.v_page_stride = v_page_stride_bytes;
  p.num_pages = num_pages;
  p.v_scales = v_scales;
  p.scale_mode = scale_mode;
  p.page_mode = page_mode;
  p.uniform_mode = uniform_mode;
  p.block_table = block_table;
  p.bt_stride = block_table_stride;
  p.positions = positions;
  p.Hkv = Hkv;
  p.D = D;
  p.err = c->err;
  if (launch_append(p, batch, st) != cudaSuccess) return EKV_ERR_CUDA;
  note_launch(st, kAfterAppend);
  return EKV_OK;
}

ekv_status ekv_prefill_attention(ekv_ctx* c, const void* q, const void* ws_k, const void* ws_v, int ws_pages,
                                 const int32_t* cu_seqlens, const int32_t* page_off, int n, int max_len,
                                 float sm_scale, void* out, float* lse, void* stream) {
  if (!c || n < 0 || max_len < 0) return EKV_ERR_INVALID_ARG;
  if (n == 0 || max_len == 0) return EKV_OK;
  if (!q || !ws_k || !ws_v || !cu_seqlens || !page_off || !out || ws_pages < 1) return EKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(ws_k) || !aligned16(ws_v) || !aligned16(out)) return EKV_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return EKV_ERR_INVALID_ARG;
  if (n > 65535) return EKV_ERR_UNSUPPORTED;
  const int Hq = c->cfg.num_q_heads, Hkv = c->cfg.num_kv_heads, D = c->cfg.head_dim;
  if (!(sm_scale > 0.f) || !isfinite(sm_scale)) sm_scale = 1.0f / sqrtf((float)D);
  DeviceGuard g(c->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  c->last_stream = st;
  PrefillParams p;
  p.q = static_cast<const __half*>(q);
  p.ws_k = static_cast<const __half*>(ws_k);
  p.ws_v = static_cast<const __half*>(ws_v);
  p.cu_seqlens = cu_seqlens;
  p.page_off = page_off;
  p.out = static_cast<__half*>(out);
  p.lse = lse;
  p.n = n;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.num_ws_pages = ws_pages;
  p.max_len = max_len;
  p.qscale = sm_scale * 1.4426950408889634f;
  p.err = c->err;
  const cudaError_t e = c->variant == 1 ? launch_prefill(p, D, max_len, st) : launch_prefill_tc05(p, D, max_len, st);
  if (e != cudaSuccess) return EKV_ERR_CUDA;
  note_launch(st, kAfterReader);
  return EKV_OK;
}

ekv_status ekv_get_error(ekv_ctx* c, int* code, int* detail) {
  if (!c) return EKV_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  cudaStream_t st = c->last_stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return EKV_ERR_CUDA;
  int h[4] = {0, 0, 0, 0};
  if (cudaMemcpyAsync(h, c->err, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(c->err, 0, sizeof(h), st) != cudaSuccess)
    return EKV_ERR_CUDA;
  // after a device error (a kernel may have wound down early) start the next call from
  // a clean plan buffer: no stale tickets. Only the context's stream is synchronised.
  if (cudaStreamSynchronize(st) != cudaSuccess) return EKV_ERR_CUDA;
  if (h[0] != 0 && (cudaMemsetAsync(c->plan, 0, kPlanInts * sizeof(int), st) != cudaSuccess ||
                    cudaStreamSynchronize(st) != cudaSuccess))
    return EKV_ERR_CUDA;
  if (code) *code = h[0];
  if (detail) *detail = h[1];
  return EKV_OK;
}

ekv_status ekv_profile_enable(ekv_ctx* c, int enable) {
  if (!c) return EKV_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (enable && c->ev.empty()) {
    c->ev.resize(2 * 8192);
    for (auto& e : c->ev)
      if (cudaEventCreate(&e) != cudaSuccess) return EKV_ERR_CUDA;
  }
  c->profiling = enable != 0;
  return EKV_OK;
}

ekv_status ekv_profile_read(ekv_ctx* c, double* split_ms, long long* launches) {
  if (!c) return EKV_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  double ms = 0.0;
  for (size_t i = 0; i < c->ev_used; ++i) {
    if (cudaEventSynchronize(c->ev[2 * i + 1]) != cudaSuccess) return EKV_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, c->ev[2 * i], c->ev[2 * i + 1]) != cudaSuccess) return EKV_ERR_CUDA;
    ms += t;
  }
  if (split_ms) *split_ms = ms;
  if (launches) *launches = (long long)c->ev_used;
  c->ev_used = 0;
  return EKV_OK;
}

ekv_status ekv_profile_launch_floor(ekv_ctx* c, int reps, void* stream, double* avg_ms) {
  if (!c || !avg_ms || reps < 1 || reps > 1024) return EKV_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  DecodeParams p{};
  p.batch = c->cfg.max_batch;
  const size_t smem = split_layout(p, c->cfg.head_dim, kVE4M3, kAlgoMma);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<cudaEvent_t> ev(2 * (size_t)reps, nullptr);
  ekv_status status = EKV_OK;
  for (auto& e : ev)
    if (cudaEventCreate(&e) != cudaSuccess) status = EKV_ERR_CUDA;
  double ms = 0.0;
  if (status == EKV_OK && (launch_floor(c->split_ctas, smem, st, reps, ev.data()) != cudaSuccess ||
                           cudaStreamSynchronize(st) != cudaSuccess))
    status = EKV_ERR_CUDA;
  for (int i = 0; status == EKV_OK && i < reps; ++i) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, ev[2 * i], ev[2 * i + 1]) != cudaSuccess) status = EKV_ERR_CUDA;
    ms += t;
  }
  for (auto& e : ev)
    if (e) cudaEventDestroy(e);
  if (status == EKV_OK) *avg_ms = ms / reps;
  return status;
}

#ifdef EKV_TEST_WAIT_TIMEOUT
// Test build only (libekv_waittest.so; not declared in ekv.h): the next `calls` decode
// calls (tensor-core consumer) make the first ring wait of CTA 0, warp 0 run out, so a
// test can check the timeout report and that the context is usable afterwards.
ekv_status ekv_test_inject_wait_timeout(int calls) {
  if (calls < 0) return EKV_ERR_INVALID_ARG;
  g_inject_timeout_calls = calls;
  return EKV_OK;
}
#endif

ekv_status ekv_query(ekv_ctx* c, int* num_sms, int* split_ctas) {
  if (!c) return EKV_ERR_INVALID_ARG;
  if (num_sms) *num_sms = c->num_sms;
  if (split_ctas) *split_ctas = c->split_ctas;
  return EKV_OK;
}

}  // extern "C"
