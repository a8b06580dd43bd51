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
__device__ void consume_simt(const DecodeParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV8,
                             const CUtensorMap* tmV16, uint8_t* smem, int start, int end, int b_first,
                             int b_last, int per) {
  using S = Slot<D, VMODE>;
  constexpr int DPL = D / 8;
  constexpr int VPL = D / 32;
  constexpr int KB = D / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = p.Hkv, G = p.G;
  const int h = warp % Hkv;
  const int v = (int)blockIdx.x * p.NG + warp / Hkv;    // this warp's range
  const int tg = lane >> 3, c8 = lane & 7;
  float* pbuf = reinterpret_cast<float*>(smem + p.pbuf_off) + warp * (kPage * GP);
  const int* cu = reinterpret_cast<const int*>(smem + p.cu_off);
  const WarpRing ring = warp_ring(p, smem, S::kBytes);
  const int n_range = end - start;
  const int n_my = n_range;
  const float tensor_scale =
      (VMODE != kVFP16 && p.scale_mode == EKV_SCALE_PER_TENSOR && p.v_scales) ? __ldg(p.v_scales) : 0.f;
  WarpMeta cur, nxt, nxt2;
  wm_ids<kElRuntime>(p, cu, start, n_my, lane, cur);
  wm_ids<kElRuntime>(p, cu, start, n_my, 32 + lane, nxt);
  wm_meta<VMODE, kElRuntime>(p, tensor_scale, h, cur);
  for (int kk = 0; kk < min(ring.nsl, n_my); ++kk)
    ring_issue<D, VMODE>(ring, kk % ring.nsl, h, __shfl_sync(0xffffffffu, cur.page, kk),
                         __shfl_sync(0xffffffffu, cur.vloc, kk), __shfl_sync(0xffffffffu, cur.flags, kk),
                         p.elastic != 0, tmK, tmV8, tmV16);
  wm_meta<VMODE, kElRuntime>(p, tensor_scale, h, nxt);
  wm_ids<kElRuntime>(p, cu, start, n_my, 64 + lane, nxt2);
  int k = 0;
  bool timed_out = false;

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
    bool seg_bad = false;                          // a page of this segment was skipped
    const int r_end = j1 - start;
    for (; k < r_end; ++k) {
      if ((k & 31) == 0 && k > 0) {
        cur = nxt;
        nxt = nxt2;
        wm_meta<VMODE, kElRuntime>(p, tensor_scale, h, nxt);
        wm_ids<kElRuntime>(p, cu, start, n_my, k + 64 + lane, nxt2);
      }
      const int s_idx = k % ring.nsl;
      if (!mbar_wait(&ring.full[s_idx], (uint32_t)(k / ring.nsl) & 1u)) {
        if (lane == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_TIMEOUT, blockIdx.x);
        for (int kk = k + 1; kk < min(k + ring.nsl, n_my); ++kk)
          mbar_wait(&ring.full[kk % ring.nsl], (uint32_t)(kk / ring.nsl) & 1u);
        timed_out = true;
        break;
      }
      const int mflags = __shfl_sync(0xffffffffu, cur.flags, k & 31);
      const int mntok = __shfl_sync(0xffffffffu, cur.ntok, k & 31);
      const float mscale = __shfl_sync(0xffffffffu, cur.scale, k & 31);
      seg_bad |= (mflags & kMetaSkip) != 0;
      if (!(mflags & kMetaSkip)) {
        const uint8_t* kp = ring.slots + (size_t)s_idx * S::kBytes;
        const uint8_t* vp = kp + S::kK;
        const int ntok = mntok;
        const bool compact = VMODE == kVE4M3 || (VMODE == kVMixed && (mflags & kMetaCompact));
        const bool base = VMODE == kVMixed && (mflags & kMetaBase);
        const float vs = compact ? mscale : 1.f;
        float s[4][GP];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = tg + 4 * i;
          float kf[DPL];
#pragma unroll
          for (int kb = 0; kb < KB; ++kb) {
            const uint4 raw = *reinterpret_cast<const uint4*>(
                kp + kb * 2048 + swz128(t * 128 + c8 * 16));
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
                  vp + swz128(t * 128 + lane * 4));
              const float2 a = e4m3x2_to_float2((uint16_t)(w4 & 0xffffu));
              const float2 c = e4m3x2_to_float2((uint16_t)(w4 >> 16));
              vv[0] = a.x; vv[1] = a.y; vv[2 % VPL] = c.x; vv[3 % VPL] = c.y;
            } else {
              const uint16_t w2 = *reinterpret_cast<const uint16_t*>(
                  vp + swz64(t * 64 + lane * 2));
              const float2 a = e4m3x2_to_float2(w2);
              vv[0] = a.x; vv[1 % VPL] = a.y;
            }
          } else if (base) {                        // high bytes, low bytes zero
            if (D == 128) {
              const uint32_t w4 = *reinterpret_cast<const uint32_t*>(vp + swz128(t * 128 + lane * 4));
              vv[0] = __half2float(__ushort_as_half((unsigned short)((w4 & 0xffu) << 8)));
              vv[1] = __half2float(__ushort_as_half((unsigned short)(w4 & 0xff00u)));
              vv[2 % VPL] = __half2float(__ushort_as_half((unsigned short)((w4 >> 8) & 0xff00u)));
              vv[3 % VPL] = __half2float(__ushort_as_half((unsigned short)((w4 >> 16) & 0xff00u)));
            } else {
              const uint16_t w2 = *reinterpret_cast<const uint16_t*>(vp + swz64(t * 64 + lane * 2));
              vv[0] = __half2float(__ushort_as_half((unsigned short)((w2 & 0xffu) << 8)));
              vv[1 % VPL] = __half2float(__ushort_as_half((unsigned short)(w2 & 0xff00u)));
            }
          } else {
            if (D == 128) {
              const int kb = lane >> 4;
              const uint2 w = *reinterpret_cast<const uint2*>(
                  vp + kb * 2048 + swz128(t * 128 + (lane & 15) * 8));
              const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
              const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
              vv[0] = a.x; vv[1] = a.y; vv[2 % VPL] = c.x; vv[3 % VPL] = c.y;
            } else {
              const uint32_t w = *reinterpret_cast<const uint32_t*>(
                  vp + swz128(t * 128 + lane * 4));
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
      // this consumer reads the slot while it computes: refill it afterwards
      fence_reads_before_refill();
      __syncwarp();
      const int kk = k + ring.nsl;
      if (kk < n_my) {
        const bool in_cur = (kk >> 5) == (k >> 5);
        const int pg = __shfl_sync(0xffffffffu, in_cur ? cur.page : nxt.page, kk & 31);
        const int fl = __shfl_sync(0xffffffffu, in_cur ? cur.flags : nxt.flags, kk & 31);
        const int vl = __shfl_sync(0xffffffffu, in_cur ? cur.vloc : nxt.vloc, kk & 31);
        ring_issue<D, VMODE>(ring, kk % ring.nsl, h, pg, vl, fl, p.elastic != 0, tmK, tmV8, tmV16);
      }
    }
    if (timed_out) break;
    // the finished output when this warp saw the whole sequence (no other range touches
    // it), else the partial record of (segment b, range v)
    const bool direct = !crosses_ctas(cu, b, start, end);
    const size_t R = (size_t)b + v;
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      if (g >= G) break;
      float ls = l[g];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
      if (seg_bad) ls = kBadRecord;
      if (direct) {
        const float inv = ls > 0.f ? 1.f / ls : 0.f;
        __half* o = p.out + ((size_t)b * p.Hq + h * G + g) * D + lane * VPL;
#pragma unroll
        for (int x = 0; x < VPL; x += 2)
          *reinterpret_cast<__half2*>(o + x) = __floats2half2_rn(acc[g][x] * inv, acc[g][(x + 1) % VPL] * inv);
        if (lane == 0 && p.lse)
          p.lse[(size_t)b * p.Hq + h * G + g] = ls > 0.f ? (m[g] + log2f(ls)) * 0.69314718055994531f : -INFINITY;
        continue;
      }
      float* dst = p.part_acc + (R * p.Hq + h * G + g) * D + lane * VPL;
      if (VPL == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(acc[g][0], acc[g][1 % VPL], acc[g][2 % VPL], acc[g][3 % VPL]);
      } else {
        *reinterpret_cast<float2*>(dst) = make_float2(acc[g][0], acc[g][1 % VPL]);
      }
      if (lane == 0) p.part_ml[R * p.Hq + h * G + g] = make_float2(m[g], ls);
    }
  }
  finish_warp<D>(p, cu, start, end, per, b_first, b_last, h, merge_buf(ring, S::kBytes));
}

// --------------------------------------------------------------------- the kernel
template <int D, int GP, int VMODE>
__global__ void __launch_bounds__(kThreads, 1)
decode_split_simt(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV8,
                  const __grid_constant__ CUtensorMap tmV16, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int warp_tot[kThreads / 32];
  uint8_t* smem = aligned_smem(smem_raw);
  int start, end, per, b_first, b_last;
  if (!split_prologue(p, smem, warp_tot, start, end, per, b_first, b_last)) return;
  consume_simt<D, GP, VMODE>(p, &tmK, &tmV8, &tmV16, smem, start, end, b_first, b_last, per);
}

// ------------------------------------------------------------------ launchers
// Opt a kernel into `bytes` of dynamic shared memory, once per (kernel, device).
cudaError_t set_smem_attr(const void* kern, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kern, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
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

// Shared-memory layout of a split launch: 8 rings of as many slots as fit next to the
// barriers (one per slot), the page prefix sums of `batch` sequences and (CUDA-core
// consumer) the probability buffer. Returns the dynamic smem bytes to request.
template <int D, int VMODE>
static size_t layout_for(DecodeParams& p, int algo) {
  using S = Slot<D, VMODE>;
  const size_t cu_bytes = ((size_t)(p.batch + 1) * 4 + 15) & ~(size_t)15;
  const size_t pbuf_bytes = algo == kAlgoSimt ? (size_t)kWarps * kPage * 8 * 4 : 0;
  const size_t fixed = 1024 + cu_bytes + pbuf_bytes;
  int nsl = (int)((kSplitSmemMax - fixed) / ((size_t)kWarps * (S::kBytes + 8)));
  nsl = nsl > kMaxSlots ? kMaxSlots : nsl;
  // At D = 128 the stream is fastest with 16-18 KiB in flight per warp, not with the most
  // that fits (measured per layer: FP16 pool 2 x 8 KiB slots 6.76 TB/s vs 3 slots 6.39 at
  // the pages' shape, 7.10 vs 6.69 on mixed lengths; E4M3 3 x 6 KiB vs 4: +0.2% at the
  // pages' shape, +0.6% at high concurrency; mixed pools 3 or 2 slots alike)
  if (D == 128 && VMODE == kVFP16 && nsl > 2) nsl = 2;
  if (D == 128 && VMODE == kVE4M3 && nsl > 3) nsl = 3;
  p.nsl = nsl;
  p.bar_off = kWarps * nsl * S::kBytes;
  p.cu_off = p.bar_off + kWarps * nsl * 8;
  p.pbuf_off = p.cu_off + (int)cu_bytes;
  return 1024 + (size_t)p.pbuf_off + pbuf_bytes;
}

size_t split_layout(DecodeParams& p, int D, int vmode, int algo) {
  if (D == 128) {
    if (vmode == kVE4M3) return layout_for<128, kVE4M3>(p, algo);
    if (vmode == kVFP16) return layout_for<128, kVFP16>(p, algo);
    return layout_for<128, kVMixed>(p, algo);
  }
  if (vmode == kVE4M3) return layout_for<64, kVE4M3>(p, algo);
  if (vmode == kVFP16) return layout_for<64, kVFP16>(p, algo);
  return layout_for<64, kVMixed>(p, algo);
}

cudaError_t launch_split_simt(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                              const DecodeParams& p, int D, int vmode, int grid, size_t smem, cudaStream_t st) {
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
