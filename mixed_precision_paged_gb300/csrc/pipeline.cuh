// pipeline.cuh -- the parts of the split-K decode that both consumers share: the
// device-side plan (page prefix sum over seq_lens), the per-warp TMA rings, the
// per-warp metadata prefetch and the fused split merge.
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
// Rings: warp w owns KV head h = w % Hkv and page group grp = w / Hkv (NG = 8 / Hkv
// groups): it handles the slices (page r, head h) of the CTA's pages r = grp, grp + NG,
// ... in order. Each warp keeps its own ring of `nsl` slots in shared memory and feeds
// it itself: lane 0 issues one TMA box for the K slice and one for the V slice,
// 128B/64B-swizzled so that the warp's 16-byte row reads are bank-conflict free. A bulk
// tensor copy stalls its issuing warp for about the same time whatever its size, so
// each slice is a single box. No warp waits for another, and a slot is refilled as soon
// as its owner has pulled the slice into registers.
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
// touched by no CTA: CTA 0 writes their zero output and -inf lse, reading the page
// prefix sums already in shared memory (no global loads on this path).
__device__ __forceinline__ void write_empty_sequences(const DecodeParams& p, const int* cu) {
  const int n = p.Hq * p.D;
  for (int b = 0; b < p.batch; ++b) {
    if (cu[b + 1] != cu[b]) continue;
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
  constexpr int kNW = kThreads / 32;
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
    for (int w = 0; w < kNW; ++w) {
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

// ----------------------------------------------------------- per-warp metadata
// Metadata of the warp's k-th page, one page per lane for 32 consecutive k.
struct WarpMeta {
  int page;
  int ntok;
  int flags;
  int b;
  float scale;
};

// Stage A: block-table entry of the warp's page k (consumed a batch later).
__device__ __forceinline__ void wm_ids(const DecodeParams& p, const int* cu, int start, int n_my, int grp, int k,
                                       WarpMeta& m) {
  m.page = 0;
  m.ntok = 0;
  m.flags = kMetaSkip;
  m.b = -1;
  m.scale = 1.f;
  if (k < n_my) {
    const int j = start + grp + k * p.NG;
    const int b = upper_bound_i(cu, p.batch + 1, j) - 1;
    const int lp = j - cu[b];
    m.b = b;
    m.page = __ldg(p.block_table + (size_t)b * p.bt_stride + lp);
    m.ntok = min(kPage, __ldg(p.seq_lens + b) - lp * kPage);
    m.flags = 0;
  }
}

// Stage B: checks, mode byte and the KV head's scale of a page whose id is known.
template <int VMODE>
__device__ __forceinline__ void wm_meta(const DecodeParams& p, float tensor_scale, int h, WarpMeta& m) {
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
  const float s = p.scale_mode == EKV_SCALE_PER_TENSOR ? tensor_scale
                                                         : __ldg(p.v_scales + (size_t)page * p.Hkv + h);
  if (scale_ok(s)) {
    m.flags = kMetaCompact;
    m.scale = s;
  } else {
    report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_SCALE, b);
    mark_bad(p, b);
    m.flags = kMetaSkip;
  }
}

// ------------------------------------------------------------------- warp rings
struct WarpRing {
  uint8_t* slots;       // this warp's nsl slots
  uint64_t* full;       // this warp's nsl barriers (one arrive + bytes per fill)
  int nsl;
};

__device__ __forceinline__ WarpRing warp_ring(const DecodeParams& p, uint8_t* smem, int slot_bytes) {
  const int warp = threadIdx.x >> 5;
  WarpRing r;
  r.slots = smem + (size_t)warp * p.nsl * slot_bytes;
  r.full = reinterpret_cast<uint64_t*>(smem + p.bar_off) + warp * p.nsl;
  r.nsl = p.nsl;
  return r;
}

// Fill the ring slot of page k (metadata page/flags broadcast by the caller). Lane 0
// arms the slot's barrier with the slice's bytes and issues one bulk tensor copy per
// tensor: K through the 5-D fp16 slice map, V through the E4M3 map (compact page) or
// the fp16 slice map (TARGET page). A skipped page only arrives on the barrier.
template <int D, int VMODE>
__device__ __forceinline__ void ring_issue(const WarpRing& ring, int k, int h, int page, int flags,
                                           const CUtensorMap* tmK, const CUtensorMap* tmV8,
                                           const CUtensorMap* tmV16) {
  using S = Slot<D, VMODE>;
  if ((threadIdx.x & 31) != 0) return;
  const int s = k % ring.nsl;
  uint64_t* bar = &ring.full[s];
  if (flags & kMetaSkip) {
    mbar_arrive(bar);
    return;
  }
  const bool compact = VMODE == kVE4M3 || (VMODE == kVMixed && (flags & kMetaCompact));
  uint8_t* dst = ring.slots + (size_t)s * S::kBytes;
  mbar_arrive_expect_tx(bar, S::kK + (compact ? kPage * D : kPage * D * 2));
  tma_load_5d(dst, tmK, 0, 0, 0, h, page, bar);
  if (compact) tma_load_4d(dst + S::kK, tmV8, 0, h, 0, page, bar);
  else tma_load_5d(dst + S::kK, tmV16, 0, 0, 0, h, page, bar);
}

// Order this warp's generic-proxy reads of a slot before the TMA (async-proxy) writes
// that refill it.
__device__ __forceinline__ void fence_reads_before_refill() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Common prologue of the split kernels: plan, this CTA's page range, barriers.
// Returns false when the CTA has no pages.
__device__ __forceinline__ bool split_prologue(const DecodeParams& p, uint8_t* smem, int* warp_tot, int& start,
                                               int& end, int& per, int& b_first, int& b_last) {
  int* cu = reinterpret_cast<int*>(smem + p.cu_off);
  const int total = plan_pages(p, cu, warp_tot);
  per = total > 0 ? (total + (int)gridDim.x - 1) / (int)gridDim.x : 1;
  if (blockIdx.x == 0) write_empty_sequences(p, cu);
  start = (int)blockIdx.x * per;
  end = min(total, start + per);
  if (start >= end) return false;
  if (threadIdx.x < kWarps * p.nsl) {
    mbar_init(reinterpret_cast<uint64_t*>(smem + p.bar_off) + threadIdx.x, 1);
    fence_barrier_init();
  }
  __syncthreads();
  b_first = upper_bound_i(cu, p.batch + 1, start) - 1;
  b_last = upper_bound_i(cu, p.batch + 1, end - 1) - 1;
  return true;
}

// Aligned dynamic shared memory of the split kernels.
__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* smem_raw) {
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  return smem_raw + pad;
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
