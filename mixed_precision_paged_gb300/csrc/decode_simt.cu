// decode_simt.cu -- split-K paged decode: device plan, TMA page pipeline, CUDA-core
// consumer, and the split merge.
//
// What one launch computes (ElasticKV Sec. 3.2; knlp.io decode prefix over FP16 keys
// and FP8 values): for each sequence b and query head, online-softmax attention over
// the sequence's pages, split across CTAs, each CTA writing unnormalised partials
// (m, l, acc) that decode_merge_kernel combines.
//
// Work split: the pages of all sequences form one stream (cu = page prefix sum,
// computed by every CTA from seq_lens); CTA c takes pages [c*per, (c+1)*per) of it,
// per = ceil(total / gridDim.x), so every CTA streams the same number of pages
// whatever the length mix. A CTA's range may cover several sequences (segments); it
// writes one partial record per (segment, page group) at record (b + c) * NG + group,
// which is unique because the CTAs that touch sequence b are exactly
// cu[b]/per .. (cu[b+1]-1)/per and those ranges of consecutive sequences only meet
// at one CTA.
//
// Pipeline: warp 8 is the producer. For each page it reads the block-table entry,
// the mode byte and the scales (32 pages at a time, one per lane), and issues one TMA
// box per (KV head, 64-element column block) of K and V into a stage; the boxes land
// 128B/64B-swizzled so that the consumers' 16-byte row reads are bank-conflict free.
// A stage holds 8 (page, KV head) slices: NG = 8 / H_kv consecutive pages. Consumer
// warp w handles KV head w % H_kv of the stage's page w / H_kv.
#include <mutex>
#include <set>
#include <utility>

#include "decode.cuh"

namespace ekv {

__device__ __forceinline__ int upper_bound_i(const int* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Block-wide prefix sum of pages per sequence into cu[0..B]; returns the total.
// Sequences with a length outside [0, bt_stride*16] count as empty and are reported
// (by CTA 0 only) and flagged so that the merge zeroes them.
__device__ int plan_pages(const DecodeParams& p, int* cu, int* warp_tot) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int kWarps = kThreads / 32;
  if (tid == 0) cu[0] = 0;
  int carry = 0;
  for (int base = 0; base < p.batch; base += kThreads) {
    const int b = base + tid;
    int np = 0;
    if (b < p.batch) {
      const int L = __ldg(p.seq_lens + b);
      if (L < 0 || L > p.bt_stride * kPage) {
        if (blockIdx.x == 0) {
          report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_SEQ_LEN, b);
          p.plan[kPlanBad + b] = 1;
        }
      } else {
        np = (L + kPage - 1) / kPage;
      }
    }
    int incl = np;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int woff = 0, chunk = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int t = warp_tot[w];
      woff += (w < warp) ? t : 0;
      chunk += t;
    }
    if (b < p.batch) cu[b + 1] = carry + woff + incl;
    carry += chunk;
    __syncthreads();
  }
  return carry;
}

// ------------------------------------------------------------------------ producer
template <int D, int VMODE>
__device__ void produce(const DecodeParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV8,
                        const CUtensorMap* tmV16, uint8_t* stages, PageMeta* meta,
                        uint64_t* full, uint64_t* empty, const int* cu, int start, int end) {
  using L = StageLayout<D, VMODE>;
  const int lane = threadIdx.x & 31;
  const int NG = p.NG, Hkv = p.Hkv;
  const int n_range = end - start;
  const int n_slots = (n_range + NG - 1) / NG * NG;
  const int k_sub = L::kKStage / NG;
  const int v_sub = L::kVStage / NG;
  const uint32_t k_bytes = kPage * Hkv * D * 2;
  const uint32_t v8_bytes = kPage * Hkv * D;
  const uint32_t v16_bytes = kPage * Hkv * D * 2;
  if (lane == 0) {
    tma_prefetch_desc(tmK);
    if (VMODE != kVFP16) tma_prefetch_desc(tmV8);
    if (VMODE != kVE4M3) tma_prefetch_desc(tmV16);
  }
  bool ok = true;
  int last_si = -1;
  for (int base = 0; base < n_slots && ok; base += 32) {
    const int r = base + lane;
    int page = 0, ntok = 0, flags = kMetaSkip;
    float sc[kMaxKvHeads];
#pragma unroll
    for (int h = 0; h < kMaxKvHeads; ++h) sc[h] = 1.f;
    if (r < n_range) {
      const int j = start + r;
      const int b = upper_bound_i(cu, p.batch + 1, j) - 1;
      const int lp = j - cu[b];
      page = __ldg(p.block_table + (size_t)b * p.bt_stride + lp);
      ntok = min(kPage, __ldg(p.seq_lens + b) - lp * kPage);
      flags = 0;
      if (page < 0 || page >= p.num_pages) {
        report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_ID, b);
        p.plan[kPlanBad + b] = 1;
        flags = kMetaSkip;
      } else {
        const int mode = VMODE == kVE4M3 ? 1 : (VMODE == kVFP16 ? 0 : (int)__ldg(p.page_mode + page));
        if (mode > 1) {
          report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_MODE, b);
          p.plan[kPlanBad + b] = 1;
          flags = kMetaSkip;
        } else if (mode == 1) {
          bool good = true;
          if (p.scale_mode == EKV_SCALE_PER_TENSOR) {
            const float s = __ldg(p.v_scales);
            good = scale_ok(s);
#pragma unroll
            for (int h = 0; h < kMaxKvHeads; ++h) sc[h] = s;
          } else {
#pragma unroll
            for (int h = 0; h < kMaxKvHeads; ++h) {
              if (h < Hkv) {
                sc[h] = __ldg(p.v_scales + (size_t)page * Hkv + h);
                good = good && scale_ok(sc[h]);
              }
            }
          }
          if (good) {
            flags = kMetaCompact;
          } else {
            report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_SCALE, b);
            p.plan[kPlanBad + b] = 1;
            flags = kMetaSkip;
          }
        }
      }
    }
    const int n_here = min(32, n_slots - base);
    for (int i = 0; i < n_here; ++i) {
      const int ri = base + i;
      const int si = ri / NG, sub = ri - si * NG;
      const int stage = si % L::kStages;
      const uint32_t ph = (uint32_t)(si / L::kStages) & 1u;
      if (sub == 0) {
        int w = 1;
        if (lane == 0) w = mbar_wait(&empty[stage], ph ^ 1u) ? 1 : 0;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          if (lane == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_TIMEOUT, blockIdx.x);
          ok = false;
          break;
        }
      }
      if (lane == i) {
        PageMeta& mt = meta[stage * 8 + sub];
        mt.page = page;
        mt.ntok = ntok;
        mt.flags = flags;
#pragma unroll
        for (int h = 0; h < kMaxKvHeads; ++h) mt.scale[h] = sc[h];
        if (flags & kMetaSkip) {
          mbar_arrive(&full[stage]);
        } else {
          const bool compact = (flags & kMetaCompact) != 0;
          mbar_arrive_expect_tx(&full[stage], k_bytes + (compact ? v8_bytes : v16_bytes));
          uint8_t* kd = stages + stage * L::kStageBytes + sub * k_sub;
          uint8_t* vd = stages + stage * L::kStageBytes + L::kKStage + sub * v_sub;
          for (int kb = 0; kb < D / 64; ++kb)
            for (int h = 0; h < Hkv; ++h)
              tma_load_4d(kd + (kb * Hkv + h) * 2048, tmK, kb * 64, h, 0, page, &full[stage]);
          if (compact) {
            for (int h = 0; h < Hkv; ++h)
              tma_load_4d(vd + h * (kPage * D), tmV8, 0, h, 0, page, &full[stage]);
          } else {
            for (int kb = 0; kb < D / 64; ++kb)
              for (int h = 0; h < Hkv; ++h)
                tma_load_4d(vd + (kb * Hkv + h) * 2048, tmV16, kb * 64, h, 0, page, &full[stage]);
          }
        }
      }
      __syncwarp();
      last_si = si;
    }
  }
  // No copy may still be landing in shared memory when the CTA exits: wait (bounded)
  // for the last fills. In normal operation the consumers already saw them complete.
  if (lane == 0 && last_si >= 0) {
    for (int si = max(0, last_si - L::kStages + 1); si <= last_si; ++si)
      mbar_wait(&full[si % L::kStages], (uint32_t)(si / L::kStages) & 1u);
  }
}

// ------------------------------------------------------------ CUDA-core consumer
// Lane layout for QK: lane = 8 * tg + c8 reads the 16-byte chunk c8 of each 64-column
// block of tokens tg, tg+4, tg+8, tg+12 (8 lanes share a token and reduce with three
// xor shuffles). For PV every lane owns D/32 consecutive columns of every token.
template <int D, int GP, int VMODE>
__device__ void consume_simt(const DecodeParams& p, uint8_t* stages, PageMeta* meta,
                             uint64_t* full, uint64_t* empty, const int* cu, int start,
                             int end, int b_first, int b_last, float* pbuf_all) {
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
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i <= p.batch; i += kThreads) p.plan[kPlanCu + i] = cu[i];
    if (threadIdx.x == 0) {
      p.plan[0] = per;
      p.plan[1] = total;
    }
  }
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
    consume_simt<D, GP, VMODE>(p, stages, meta, full, empty, cu, start, end, b_first, b_last, pbuf);
  }
}

// ------------------------------------------------------------------------ merge
// One CTA per sequence; warp w combines the records of query heads w, w+8, ...
//   M = max m_i,  L = sum l_i 2^(m_i - M),  out = sum acc_i 2^(m_i - M) / L,
//   lse = (M + log2 L) ln 2.
template <int D>
__global__ void __launch_bounds__(256)
decode_merge_kernel(const DecodeParams p) {
  constexpr int VPL = D / 32;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = p.plan[kPlanBad + b];
  __syncthreads();
  if (threadIdx.x == 0 && s_bad) p.plan[kPlanBad + b] = 0;
  const int per = p.plan[0];
  const int c_b = p.plan[kPlanCu + b], c_b1 = p.plan[kPlanCu + b + 1];
  const bool empty_seq = (c_b1 == c_b) || s_bad;
  const int NG = p.NG;
  int c0 = 0, nrec = 0;
  if (!empty_seq) {
    c0 = c_b / per;
    nrec = ((c_b1 - 1) / per - c0 + 1) * NG;
  }
  for (int hq = warp; hq < p.Hq; hq += 8) {
    __half* o = p.out + ((size_t)b * p.Hq + hq) * D + lane * VPL;
    if (empty_seq) {
#pragma unroll
      for (int x = 0; x < VPL; ++x) o[x] = __float2half(0.f);
      if (lane == 0 && p.lse) p.lse[(size_t)b * p.Hq + hq] = -INFINITY;
      continue;
    }
    float M = -INFINITY;
    for (int i = lane; i < nrec; i += 32) {
      const size_t R = (size_t)(b + c0 + i / NG) * NG + (i % NG);
      const float2 ml = p.part_ml[R * p.Hq + hq];
      if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float Ls = 0.f, acc[VPL];
#pragma unroll
    for (int x = 0; x < VPL; ++x) acc[x] = 0.f;
    for (int i = 0; i < nrec; ++i) {
      const size_t R = (size_t)(b + c0 + i / NG) * NG + (i % NG);
      const float2 ml = p.part_ml[R * p.Hq + hq];
      if (!(ml.y > 0.f)) continue;
      const float w = exp2f(ml.x - M);
      Ls = fmaf(w, ml.y, Ls);
      const float* src = p.part_acc + (R * p.Hq + hq) * D + lane * VPL;
      if (VPL == 4) {
        const float4 a = *reinterpret_cast<const float4*>(src);
        acc[0] = fmaf(w, a.x, acc[0]); acc[1 % VPL] = fmaf(w, a.y, acc[1 % VPL]);
        acc[2 % VPL] = fmaf(w, a.z, acc[2 % VPL]); acc[3 % VPL] = fmaf(w, a.w, acc[3 % VPL]);
      } else {
        const float2 a = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(w, a.x, acc[0]); acc[1 % VPL] = fmaf(w, a.y, acc[1 % VPL]);
      }
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    if (VPL == 4) {
      __half2 h01 = __floats2half2_rn(acc[0] * inv, acc[1 % VPL] * inv);
      __half2 h23 = __floats2half2_rn(acc[2 % VPL] * inv, acc[3 % VPL] * inv);
      uint2 st;
      st.x = *reinterpret_cast<uint32_t*>(&h01);
      st.y = *reinterpret_cast<uint32_t*>(&h23);
      *reinterpret_cast<uint2*>(o) = st;
    } else {
      __half2 h01 = __floats2half2_rn(acc[0] * inv, acc[1 % VPL] * inv);
      *reinterpret_cast<__half2*>(o) = h01;
    }
    if (lane == 0 && p.lse)
      p.lse[(size_t)b * p.Hq + hq] = Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
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

cudaError_t launch_merge(const DecodeParams& p, int D, cudaStream_t st) {
  if (p.batch == 0) return cudaSuccess;
  if (D == 128) decode_merge_kernel<128><<<p.batch, 256, 0, st>>>(p);
  else decode_merge_kernel<64><<<p.batch, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace ekv
