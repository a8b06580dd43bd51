// decode_simt.cu -- split-K paged decode with a CUDA-core consumer
// (FP32 FMAs), and the launch helpers shared by both consumers.
//
// What one launch computes (ElasticKV Sec. 3.2; knlp.io decode prefix over FP16 keys
// and FP8 values): for each sequence b and query head, online-softmax attention over
// the sequence's pages, split across CTAs, each CTA writing unnormalised partials
// (m, l, acc) that the last warp of each (sequence, KV head) combines (pipeline.cuh).
#include <mutex>
#include <set>
#include <utility>

#include "pipeline.cuh"

namespace ekv {

// ------------------------------------------------------------ CUDA-core consumer
// Lane layout for QK: lane = 8 * tg + c8 reads the 16-byte chunk c8 of each 64-column
// block of tokens tg, tg+4, tg+8, tg+12 (8 lanes share a token and reduce with three
// xor shuffles). For PV every lane owns D/32 consecutive columns of every token.
template <int D, int GP, int VMODE>
__device__ void consume_simt(const DecodeParams& p, uint8_t* stages, PageMeta* meta,
                             uint64_t* full, uint64_t* empty, const int* cu, int start,
                             int end, int b_first, int b_last, int per, float* pbuf_all) {
  using L = StageLayout<D, VMODE>;
  constexpr int DPL = D / 8;
  constexpr int VPL = D / 32;
  constexpr int KB = D / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = p.Hkv, NG = p.NG, G = p.G;
  const int h = warp % Hkv, grp = warp / Hkv;
  const int tg = lane >> 3, c8 = lane & 7;
  float* pbuf = pbuf_all + warp * (kPage * GP);
  const int k_sub = L::kKStage / NG, v_sub = L::kVStage / NG;

  for (int b = b_first; b <= b_last; ++b) {
    const int j0 = max(cu[b], start), j1 = min(cu[b + 1], end);
    if (j0 >= j1) continue;
    float qf[GP][DPL];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
#pragma unroll
      for (int kb = 0; kb < KB; ++kb) {
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (g < G)
          raw = __ldg(reinterpret_cast<const uint4*>(
              p.q + ((size_t)b * p.Hq + h * G + g) * D + kb * 64 + c8 * 8));
        const __half2* hv = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(hv[e]);
          qf[g][kb * 8 + 2 * e] = f.x * p.qscale;
          qf[g][kb * 8 + 2 * e + 1] = f.y * p.qscale;
        }
      }
    }
    float m[GP], l[GP], acc[GP][VPL];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int x = 0; x < VPL; ++x) acc[g][x] = 0.f;
    }
    const int r_begin = j0 - start, r_end = j1 - start;
    int r = r_begin + (((grp - r_begin) % NG) + NG) % NG;
    for (; r < r_end; r += NG) {
      const int si = r / NG;
      const int stage = si % L::kStages;
      const uint32_t ph = (uint32_t)(si / L::kStages) & 1u;
      if (!mbar_wait(&full[stage], ph)) {
        if (lane == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_TIMEOUT, blockIdx.x);
        return;
      }
      const PageMeta& mt = meta[stage * 8 + grp];
      if (!(mt.flags & kMetaSkip)) {
        const uint8_t* kp = stages + stage * L::kStageBytes + grp * k_sub;
        const uint8_t* vp = stages + stage * L::kStageBytes + L::kKStage + grp * v_sub;
        const int ntok = mt.ntok;
        const bool compact = VMODE == kVE4M3 || (VMODE == kVMixed && (mt.flags & kMetaCompact));
        const float vs = compact ? mt.scale[h] : 1.f;
        float s[4][GP];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = tg + 4 * i;
          float kf[DPL];
#pragma unroll
          for (int kb = 0; kb < KB; ++kb) {
            const uint4 raw = *reinterpret_cast<const uint4*>(
                kp + (kb * Hkv + h) * 2048 + swz128(t * 128 + c8 * 16));
            const __half2* hv = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __half22float2(hv[e]);
              kf[kb * 8 + 2 * e] = f.x;
              kf[kb * 8 + 2 * e + 1] = f.y;
            }
          }
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            float a = 0.f;
#pragma unroll
            for (int x = 0; x < DPL; ++x) a = fmaf(qf[g][x], kf[x], a);
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            s[i][g] = (t < ntok) ? a : -INFINITY;
          }
        }
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          float mx = fmaxf(fmaxf(s[0][g], s[1][g]), fmaxf(s[2][g], s[3][g]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(m[g], mx);
          const float alpha = exp2f(m[g] - mn);
          float ps = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float pv = exp2f(s[i][g] - mn);
            ps += pv;
            if (c8 == 0) pbuf[(tg + 4 * i) * GP + g] = pv * vs;
          }
          l[g] = l[g] * alpha + (c8 == 0 ? ps : 0.f);
#pragma unroll
          for (int x = 0; x < VPL; ++x) acc[g][x] *= alpha;
          m[g] = mn;
        }
        __syncwarp();
        for (int t = 0; t < ntok; ++t) {
          float vv[VPL];
          if (compact) {
            if (D == 128) {
              const uint32_t w4 = *reinterpret_cast<const uint32_t*>(
                  vp + h * (kPage * D) + swz128(t * 128 + lane * 4));
              const float2 a = e4m3x2_to_float2((uint16_t)(w4 & 0xffffu));
              const float2 c = e4m3x2_to_float2((uint16_t)(w4 >> 16));
              vv[0] = a.x; vv[1] = a.y; vv[2 % VPL] = c.x; vv[3 % VPL] = c.y;
            } else {
              const uint16_t w2 = *reinterpret_cast<const uint16_t*>(
                  vp + h * (kPage * D) + swz64(t * 64 + lane * 2));
              const float2 a = e4m3x2_to_float2(w2);
              vv[0] = a.x; vv[1 % VPL] = a.y;
            }
          } else {
            if (D == 128) {
              const int kb = lane >> 4;
              const uint2 w = *reinterpret_cast<const uint2*>(
                  vp + (kb * Hkv + h) * 2048 + swz128(t * 128 + (lane & 15) * 8));
              const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
              const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
              vv[0] = a.x; vv[1] = a.y; vv[2 % VPL] = c.x; vv[3 % VPL] = c.y;
            } else {
              const uint32_t w = *reinterpret_cast<const uint32_t*>(
                  vp + h * 2048 + swz128(t * 128 + lane * 4));
              const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w));
              vv[0] = a.x; vv[1 % VPL] = a.y;
            }
          }
          float pp[GP];
#pragma unroll
          for (int g = 0; g < GP; ++g) pp[g] = pbuf[t * GP + g];
#pragma unroll
          for (int g = 0; g < GP; ++g)
#pragma unroll
            for (int x = 0; x < VPL; ++x) acc[g][x] = fmaf(pp[g], vv[x], acc[g][x]);
        }
        __syncwarp();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    // partial record of (segment b, this CTA, page group grp) for this KV head's G heads
    const size_t R = (size_t)(b + blockIdx.x) * NG + grp;
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      if (g >= G) break;
      float ls = l[g];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
      float* dst = p.part_acc + (R * p.Hq + h * G + g) * D + lane * VPL;
      if (VPL == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(acc[g][0], acc[g][1 % VPL], acc[g][2 % VPL], acc[g][3 % VPL]);
      } else {
        *reinterpret_cast<float2*>(dst) = make_float2(acc[g][0], acc[g][1 % VPL]);
      }
      if (lane == 0) p.part_ml[R * p.Hq + h * G + g] = make_float2(m[g], ls);
    }
    finish_segment<D>(p, b, h, cu, per);
  }
}

// --------------------------------------------------------------------- the kernel
template <int D, int GP, int VMODE>
__global__ void __launch_bounds__(kThreads, 1)
decode_split_simt(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV8,
                  const __grid_constant__ CUtensorMap tmV16, const DecodeParams p) {
  using L = StageLayout<D, VMODE>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int warp_tot[kThreads / 32];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* stages = smem;
  PageMeta* meta = reinterpret_cast<PageMeta*>(smem + L::kMetaOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + L::kStages;
  int* cu = reinterpret_cast<int*>(smem + L::kCuOff);
  float* pbuf = reinterpret_cast<float*>(smem + L::kCuOff + (((p.batch + 1) * 4 + 15) & ~15));

  const int total = plan_pages(p, cu, warp_tot);
  const int per = total > 0 ? (total + (int)gridDim.x - 1) / (int)gridDim.x : 1;
  if (blockIdx.x == 0) write_empty_sequences(p);
  const int start = (int)blockIdx.x * per;
  const int end = min(total, start + per);
  if (start >= end) return;
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full[s], (uint32_t)p.NG);
      mbar_init(&empty[s], (uint32_t)kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const int b_first = upper_bound_i(cu, p.batch + 1, start) - 1;
  const int b_last = upper_bound_i(cu, p.batch + 1, end - 1) - 1;
  if ((threadIdx.x >> 5) == kConsumerWarps) {
    produce<D, VMODE>(p, &tmK, &tmV8, &tmV16, stages, meta, full, empty, cu, start, end);
  } else {
    consume_simt<D, GP, VMODE>(p, stages, meta, full, empty, cu, start, end, b_first, b_last, per, pbuf);
  }
}

// ------------------------------------------------------------------ launchers
// Opt the split kernels into large dynamic shared memory, once per (kernel, device).
cudaError_t set_smem_attr(const void* kern) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kern, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSplitSmemMax);
  if (e == cudaSuccess) done.insert({kern, dev});
  return e;
}

template <int D, int GP, int VMODE>
static cudaError_t launch_simt(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                               const DecodeParams& p, int grid, size_t smem, cudaStream_t st) {
  auto kern = decode_split_simt<D, GP, VMODE>;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(tk, t8, t16, p);
  return cudaGetLastError();
}

template <int D, int VMODE>
static cudaError_t dispatch_simt_g(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                                   const DecodeParams& p, int grid, size_t smem, cudaStream_t st) {
  if (p.G <= 1) return launch_simt<D, 1, VMODE>(tk, t8, t16, p, grid, smem, st);
  if (p.G <= 2) return launch_simt<D, 2, VMODE>(tk, t8, t16, p, grid, smem, st);
  if (p.G <= 4) return launch_simt<D, 4, VMODE>(tk, t8, t16, p, grid, smem, st);
  return launch_simt<D, 8, VMODE>(tk, t8, t16, p, grid, smem, st);
}

size_t split_smem_bytes(int D, int vmode, int algo, int batch) {
  int cu_off = 0;
  if (D == 128) {
    cu_off = vmode == kVE4M3 ? StageLayout<128, kVE4M3>::kCuOff
           : vmode == kVFP16 ? StageLayout<128, kVFP16>::kCuOff : StageLayout<128, kVMixed>::kCuOff;
  } else {
    cu_off = vmode == kVE4M3 ? StageLayout<64, kVE4M3>::kCuOff
           : vmode == kVFP16 ? StageLayout<64, kVFP16>::kCuOff : StageLayout<64, kVMixed>::kCuOff;
  }
  size_t bytes = 1024 + (size_t)cu_off + (((size_t)(batch + 1) * 4 + 15) & ~(size_t)15);
  if (algo == kAlgoSimt) bytes += (size_t)kConsumerWarps * kPage * 8 * 4;
  return bytes;
}

cudaError_t launch_split_simt(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                              const DecodeParams& p, int D, int vmode, int grid, cudaStream_t st) {
  const size_t smem = split_smem_bytes(D, vmode, kAlgoSimt, p.batch);
  if (D == 128) {
    if (vmode == kVE4M3) return dispatch_simt_g<128, kVE4M3>(tk, t8, t16, p, grid, smem, st);
    if (vmode == kVFP16) return dispatch_simt_g<128, kVFP16>(tk, t8, t16, p, grid, smem, st);
    return dispatch_simt_g<128, kVMixed>(tk, t8, t16, p, grid, smem, st);
  }
  if (vmode == kVE4M3) return dispatch_simt_g<64, kVE4M3>(tk, t8, t16, p, grid, smem, st);
  if (vmode == kVFP16) return dispatch_simt_g<64, kVFP16>(tk, t8, t16, p, grid, smem, st);
  return dispatch_simt_g<64, kVMixed>(tk, t8, t16, p, grid, smem, st);
}

}  // namespace ekv
