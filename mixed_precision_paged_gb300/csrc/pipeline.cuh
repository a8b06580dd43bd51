// pipeline.cuh -- the parts of the split-K decode that every consumer shares: the
// device-side plan (page prefix sum over seq_lens) and the TMA producer warp.
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
#pragma once

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

__device__ __forceinline__ void mark_bad(const DecodeParams& p, int b) {
  for (int h = 0; h < p.Hkv; ++h) p.plan[kPlanBad + b * kMaxKvHeads + h] = 1;
}

// Sequences with no pages (length 0, or a length the block table cannot hold) are
// touched by no CTA: CTA 0 writes their zero output and -inf lse.
__device__ __forceinline__ void write_empty_sequences(const DecodeParams& p) {
  const int n = p.Hq * p.D;
  for (int b = 0; b < p.batch; ++b) {
    const int L = __ldg(p.seq_lens + b);
    if (L > 0 && L <= p.bt_stride * kPage) continue;
    for (int i = threadIdx.x; i < n; i += blockDim.x) p.out[(size_t)b * n + i] = __float2half(0.f);
    if (p.lse)
      for (int i = threadIdx.x; i < p.Hq; i += blockDim.x) p.lse[(size_t)b * p.Hq + i] = -INFINITY;
  }
}

// Block-wide prefix sum of pages per sequence into cu[0..B]; returns the total.
// Sequences with a length outside [0, bt_stride*16] count as empty and are reported
// (by CTA 0 only) and flagged so that the merge zeroes them.
__device__ __forceinline__ int plan_pages(const DecodeParams& p, int* cu, int* warp_tot) {
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
        if (blockIdx.x == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_SEQ_LEN, b);
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
// Metadata of the page slot r of this CTA's range, one lane per slot.
struct SlotMeta {
  int page;
  int ntok;
  int flags;
  int b;
  float sc[kMaxKvHeads];
};

// Stage A: block-table entry of slot r (the load is consumed one batch later).
__device__ __forceinline__ void slot_ids(const DecodeParams& p, const int* cu, int start, int n_range, int r,
                                         SlotMeta& m) {
  m.page = 0;
  m.ntok = 0;
  m.flags = kMetaSkip;
  m.b = -1;
  if (r < n_range) {
    const int j = start + r;
    const int b = upper_bound_i(cu, p.batch + 1, j) - 1;
    const int lp = j - cu[b];
    m.b = b;
    m.page = __ldg(p.block_table + (size_t)b * p.bt_stride + lp);
    m.ntok = min(kPage, __ldg(p.seq_lens + b) - lp * kPage);
    m.flags = 0;
  }
}

// Stage B: checks, mode byte and scales of a slot whose page id is known.
template <int VMODE>
__device__ __forceinline__ void slot_meta(const DecodeParams& p, float tensor_scale, SlotMeta& m) {
#pragma unroll
  for (int h = 0; h < kMaxKvHeads; ++h) m.sc[h] = 1.f;
  if (m.b < 0) return;
  const int b = m.b, page = m.page;
  if (page < 0 || page >= p.num_pages) {
    report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_ID, b);
    mark_bad(p, b);
    m.flags = kMetaSkip;
    return;
  }
  const int mode = VMODE == kVE4M3 ? 1 : (VMODE == kVFP16 ? 0 : (int)__ldg(p.page_mode + page));
  if (mode > 1) {
    report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_MODE, b);
    mark_bad(p, b);
    m.flags = kMetaSkip;
    return;
  }
  if (mode == 0) return;
  bool good = true;
  if (p.scale_mode == EKV_SCALE_PER_TENSOR) {
    good = scale_ok(tensor_scale);
#pragma unroll
    for (int h = 0; h < kMaxKvHeads; ++h) m.sc[h] = tensor_scale;
  } else {
#pragma unroll
    for (int h = 0; h < kMaxKvHeads; ++h) {
      if (h < p.Hkv) {
        m.sc[h] = __ldg(p.v_scales + (size_t)page * p.Hkv + h);
        good = good && scale_ok(m.sc[h]);
      }
    }
  }
  if (good) {
    m.flags = kMetaCompact;
  } else {
    report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_SCALE, b);
    mark_bad(p, b);
    m.flags = kMetaSkip;
  }
}

// The producer walks its range 32 slots at a time, one slot per lane. Metadata is
// software-pipelined: while batch k is issued, the block-table entries of batch k+2
// and the mode bytes / scales of batch k+1 are already in flight, so no TMA issue
// waits on a dependent global load.
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
  const float tensor_scale =
      (VMODE != kVFP16 && p.scale_mode == EKV_SCALE_PER_TENSOR) ? __ldg(p.v_scales) : 1.f;
  SlotMeta cur, nxt, nxt2;
  slot_ids(p, cu, start, n_range, lane, cur);
  slot_ids(p, cu, start, n_range, 32 + lane, nxt);
  slot_meta<VMODE>(p, tensor_scale, cur);
  bool ok = true;
  int last_si = -1;
  for (int base = 0; base < n_slots && ok; base += 32) {
    slot_ids(p, cu, start, n_range, base + 64 + lane, nxt2);
    slot_meta<VMODE>(p, tensor_scale, nxt);
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
      // lane i publishes the slot's metadata and the expected bytes; then the warp's
      // lanes issue the page's TMA boxes in parallel, one box per lane
      const int pg = __shfl_sync(0xffffffffu, cur.page, i);
      const int fl = __shfl_sync(0xffffffffu, cur.flags, i);
      if (lane == i) {
        PageMeta& mt = meta[stage * 8 + sub];
        mt.page = cur.page;
        mt.ntok = cur.ntok;
        mt.flags = cur.flags;
#pragma unroll
        for (int h = 0; h < kMaxKvHeads; ++h) mt.scale[h] = cur.sc[h];
        if (cur.flags & kMetaSkip) {
          mbar_arrive(&full[stage]);
        } else {
          const bool compact = (cur.flags & kMetaCompact) != 0;
          mbar_arrive_expect_tx(&full[stage], k_bytes + (compact ? v8_bytes : v16_bytes));
        }
      }
      __syncwarp();
      if (!(fl & kMetaSkip)) {
        const bool compact = (fl & kMetaCompact) != 0;
        uint8_t* kd = stages + stage * L::kStageBytes + sub * k_sub;
        uint8_t* vd = stages + stage * L::kStageBytes + L::kKStage + sub * v_sub;
        const int nk = (D / 64) * Hkv;                      // K boxes: (column block, head)
        const int nv = compact ? Hkv : (D / 64) * Hkv;      // V boxes
        if (lane < nk) {
          const int kb = lane / Hkv, hh = lane - kb * Hkv;
          tma_load_4d(kd + lane * 2048, tmK, kb * 64, hh, 0, pg, &full[stage]);
        } else if (lane < nk + nv) {
          const int k = lane - nk;
          if (compact) {
            tma_load_4d(vd + k * (kPage * D), tmV8, 0, k, 0, pg, &full[stage]);
          } else {
            const int kb = k / Hkv, hh = k - kb * Hkv;
            tma_load_4d(vd + k * 2048, tmV16, kb * 64, hh, 0, pg, &full[stage]);
          }
        }
      }
      __syncwarp();
      last_si = si;
    }
    cur = nxt;
    nxt = nxt2;
  }
  // No copy may still be landing in shared memory when the CTA exits: wait (bounded)
  // for the last fills. In normal operation the consumers already saw them complete.
  if (lane == 0 && last_si >= 0) {
    for (int si = max(0, last_si - L::kStages + 1); si <= last_si; ++si)
      mbar_wait(&full[si % L::kStages], (uint32_t)(si / L::kStages) & 1u);
  }
}

// ------------------------------------------------------------------ fused merge
// Combine the partial records of sequence b for the G query heads of KV head h:
//   M = max m_i,  L = sum l_i 2^(m_i - M),  out = sum acc_i 2^(m_i - M) / L,
//   lse = (M + log2 L) ln 2.
// The warp's lanes split over (head, column block): 32/GP lanes per head read
// their columns of every record with independent loads, so a merge costs a few L2
// round trips whatever the record count. Records are read through L2 (ld.global.cg):
// other SMs wrote them in this launch.
template <int D>
__device__ void merge_heads(const DecodeParams& p, int b, int h, int c0, int n_cta, bool bad) {
  constexpr int kMaxDpl = D / 4;                     // columns per lane when G == 8
  const int lane = threadIdx.x & 31;
  const int G = p.G, NG = p.NG;
  const int GP = G <= 1 ? 1 : (G <= 2 ? 2 : (G <= 4 ? 4 : 8));
  const int lph = 32 / GP;                           // lanes per query head
  const int g = lane / lph, sub = lane - g * lph;
  const int dpl = D / lph;                           // columns per lane (2..32)
  const int d0 = sub * dpl;
  const bool active = g < G;
  const int hq = h * G + (active ? g : 0);
  const int nrec = n_cta * NG;
  const unsigned gmask = 0xffffffffu;
  __half* o = p.out + ((size_t)b * p.Hq + hq) * D + d0;
  if (bad) {
    if (active) {
#pragma unroll
      for (int x = 0; x < kMaxDpl; x += 2)
        if (x < dpl) *reinterpret_cast<__half2*>(o + x) = __floats2half2_rn(0.f, 0.f);
      if (sub == 0 && p.lse) p.lse[(size_t)b * p.Hq + hq] = -INFINITY;
    }
    return;
  }
  // pass 1: max of m over the records (lanes of a head split the records)
  float M = -INFINITY;
  for (int i = sub; i < nrec; i += lph) {
    const size_t R = (size_t)(b + c0 + i / NG) * NG + (i % NG);
    const float2 ml = __ldcg(p.part_ml + R * p.Hq + hq);
    if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
  for (int off = 1; off < lph; off <<= 1) M = fmaxf(M, __shfl_xor_sync(gmask, M, off));
  // pass 2: weights, L and the weighted column sums
  float acc[kMaxDpl];
#pragma unroll
  for (int x = 0; x < kMaxDpl; ++x) acc[x] = 0.f;
  float Ls = 0.f;
  for (int i0 = 0; i0 < nrec; i0 += lph) {
    float w = 0.f;
    {
      const int i = i0 + sub;
      if (i < nrec) {
        const size_t R = (size_t)(b + c0 + i / NG) * NG + (i % NG);
        const float2 ml = __ldcg(p.part_ml + R * p.Hq + hq);
        if (ml.y > 0.f) {
          w = exp2f(ml.x - M);
          Ls = fmaf(w, ml.y, Ls);
        }
      }
    }
    const int n_here = min(lph, nrec - i0);
    for (int j = 0; j < n_here; ++j) {
      const float wj = __shfl_sync(gmask, w, g * lph + j);
      if (wj == 0.f) continue;                       // uniform within the head's lanes
      const int i = i0 + j;
      const size_t R = (size_t)(b + c0 + i / NG) * NG + (i % NG);
      const float* src = p.part_acc + (R * p.Hq + hq) * D + d0;
#pragma unroll
      for (int x = 0; x < kMaxDpl; x += 2) {
        if (x < dpl) {
          const float2 a = __ldcg(reinterpret_cast<const float2*>(src + x));
          acc[x] = fmaf(wj, a.x, acc[x]);
          acc[x + 1] = fmaf(wj, a.y, acc[x + 1]);
        }
      }
    }
  }
  for (int off = 1; off < lph; off <<= 1) Ls += __shfl_xor_sync(gmask, Ls, off);
  if (!active) return;
  const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
  for (int x = 0; x < kMaxDpl; x += 2)
    if (x < dpl) *reinterpret_cast<__half2*>(o + x) = __floats2half2_rn(acc[x] * inv, acc[x + 1] * inv);
  if (sub == 0 && p.lse)
    p.lse[(size_t)b * p.Hq + hq] = Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
}

// Called by every consumer warp after it wrote its partial record of (segment b, KV
// head h): counts the record, and the warp that writes the last of the
// n_cta(b) * NG records of (b, h) merges them. No warp waits for another.
template <int D>
__device__ void finish_segment(const DecodeParams& p, int b, int h, const int* cu, int per) {
  const int lane = threadIdx.x & 31;
  const int c0 = cu[b] / per;
  const int n_cta = (cu[b + 1] - 1) / per - c0 + 1;
  const int expected = n_cta * p.NG;
  int* ticket = p.plan + kPlanTicket + b * kMaxKvHeads + h;
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    __threadfence();
    last = (atomicAdd(ticket, 1) == expected - 1) ? 1 : 0;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  int* badp = p.plan + kPlanBad + b * kMaxKvHeads + h;
  const bool bad = __ldcg(badp) != 0;
  merge_heads<D>(p, b, h, c0, n_cta, bad);
  __syncwarp();
  if (lane == 0) {
    *ticket = 0;
    if (bad) *badp = 0;
  }
}

}  // namespace ekv
