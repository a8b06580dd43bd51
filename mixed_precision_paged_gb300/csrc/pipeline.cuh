// pipeline.cuh -- the parts of the split-K decode that both consumers share: the
// device-side plan (page prefix sum over seq_lens), the per-warp TMA rings, the
// per-warp metadata prefetch and the fused split merge.
//
// Work split: the pages of all sequences form one stream (cu = page prefix sum,
// computed by every CTA from seq_lens), cut into gridDim.x * NG contiguous ranges of
// equal cost, a page costing 1 and each sequence start kSegmentCost more (page j of
// sequence b at position j + kSegmentCost * b; per = ceil(positions / ranges)), so every
// range takes about the same time whatever the length mix. Warp w of CTA c owns KV head h = w % Hkv and page group
// grp = w / Hkv (NG = 8 / Hkv groups) and streams range v = c * NG + grp: the warps of a
// KV head work on contiguous ranges, so a sequence that lies inside one range is
// finished by one warp with no merge at all. A range may cover several sequences
// (segments); a segment of a sequence that other ranges also touch becomes a partial
// record at index b + v, which is unique because the ranges that touch sequence b are
// consecutive (ranges_of) and those of consecutive sequences only meet at one range. Records are written without any synchronisation as segments end; the
// merges happen when a warp's stream ends (finish_warp).
//
// Rings: each warp handles the slices (page r, head h) of its range in order. Each warp
// keeps its own ring of `nsl` slots in shared memory and feeds
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

// Cost of starting a sequence in a page range, in pages: a segment's Q load, pipeline
// restart and end record (swept 1..3 on a 256-sequence mix and on 32 x 8K: 2 is best).
constexpr int kSegmentCost = 2;

// The first page whose cost-stream position j + kSegmentCost * b is >= x (total if none):
// b is the first sequence with cu[b + 1] + kSegmentCost * b > x.
__device__ __forceinline__ int page_at(const int* cu, int batch, int x) {
  int lo = 0, hi = batch;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid + 1] + kSegmentCost * mid <= x) lo = mid + 1; else hi = mid;
  }
  if (lo == batch) return cu[batch];
  return max(cu[lo], x - kSegmentCost * lo);
}

// The ranges that hold pages of sequence b (non-empty): v0 .. v0 + n - 1.
__device__ __forceinline__ void ranges_of(const int* cu, int b, int per, int& v0, int& n) {
  v0 = (cu[b] + kSegmentCost * b) / per;
  n = (cu[b + 1] - 1 + kSegmentCost * b) / per - v0 + 1;
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
// Sequences with a length outside [0, bt_stride*16] count as empty (CTA 0 writes their
// zero output) and are reported by CTA 0.
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
// Elastic-layout handling of the per-warp metadata and ring fills, fixed at compile
// time for the tensor-core consumer (the plain kernels carry none of it) or read from
// the launch parameters (CUDA-core consumer).
enum ElasticMode { kElNo = 0, kElYes = 1, kElRuntime = 2 };
template <int EL>
__device__ __forceinline__ bool is_elastic(const DecodeParams& p) {
  return EL == kElYes || (EL == kElRuntime && p.elastic != 0);
}

struct WarpMeta {
  int page;       // logical page: K rows, mode byte, scales
  int vloc;       // value coordinate: the page (plain) or its half-slot location (elastic)
  int lp;         // page index within its sequence
  int ntok;
  int flags;
  int b;
  float scale;
};

// Stage A: block-table entry of the warp's page k (consumed a batch later).
template <int EL>
__device__ __forceinline__ void wm_ids(const DecodeParams& p, const int* cu, int start, int n_my, int k,
                                       WarpMeta& m) {
  m.page = 0;
  m.vloc = 0;
  m.lp = 0;
  m.ntok = 0;
  m.flags = kMetaSkip;
  m.b = -1;
  m.scale = 1.f;
  if (k < n_my) {
    const int j = start + k;
    const int b = upper_bound_i(cu, p.batch + 1, j) - 1;
    const int lp = j - cu[b];
    m.b = b;
    m.lp = lp;
    m.page = __ldg(p.block_table + (size_t)b * p.bt_stride + lp);
    m.vloc = is_elastic<EL>(p) ? __ldg(p.v_block_table + (size_t)b * p.bt_stride + lp) : m.page;
    m.ntok = min(kPage, __ldg(p.seq_lens + b) - lp * kPage);
    m.flags = 0;
  }
}

// Stage B: checks, mode byte (TARGET / E4M3 / BASE) and, for an E4M3 page, the KV
// head's scale of a page whose id is known. A missing or bad scale skips the page.
template <int VMODE, int EL>
__device__ __forceinline__ void wm_meta(const DecodeParams& p, float tensor_scale, int h, WarpMeta& m) {
  if (m.b < 0) return;
  const int b = m.b, page = m.page;
  if (page < 0 || page >= p.num_pages) {
    report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_ID, b);
    m.flags = kMetaSkip;
    return;
  }
  int mode = VMODE == kVE4M3 ? 1 : (VMODE == kVFP16 ? 0 : p.uniform_mode);
  if (VMODE == kVMixed) {
    if (is_elastic<EL>(p) && p.boundaries) {         // TARGET-BASE-TARGET: no mode lookup
      const int b0 = __ldg(p.boundaries + 2 * b), b1 = __ldg(p.boundaries + 2 * b + 1);
      mode = (m.lp >= b0 && m.lp < b1) ? EKV_MODE_BASE : EKV_MODE_TARGET_FP16;
    } else if (p.page_mode) {
      mode = (int)__ldg(p.page_mode + page);
    }
  }
  if (is_elastic<EL>(p)) {                           // a location inside the value pool,
    const int v = m.vloc;                            // even for a TARGET page
    if (v < 0 || v >= 2 * p.num_v_slots || (mode == EKV_MODE_TARGET_FP16 && (v & 1))) {
      report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_ID, b);
      m.flags = kMetaSkip;
      return;
    }
  }
  if (mode > EKV_MODE_BASE) {
    report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_MODE, b);
    m.flags = kMetaSkip;
    return;
  }
  if (mode == EKV_MODE_TARGET_FP16) return;
  if (mode == EKV_MODE_BASE) {                       // no scale: shift and bitcast
    m.flags = kMetaBase;
    return;
  }
  const float s = !p.v_scales ? 0.f
                  : (p.scale_mode == EKV_SCALE_PER_TENSOR ? tensor_scale
                                                           : __ldg(p.v_scales + (size_t)page * p.Hkv + h));
  if (scale_ok(s)) {
    m.flags = kMetaCompact;
    m.scale = s;
  } else {
    report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_SCALE, b);
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

// The merge scratch of a warp: its ring, free once its stream has ended.
struct MergeBuf {
  uint8_t* buf;
  int bytes;
};

__device__ __forceinline__ MergeBuf merge_buf(const WarpRing& ring, int slot_bytes) {
  MergeBuf mb;
  mb.buf = ring.slots;
  mb.bytes = ring.nsl * slot_bytes;
  return mb;
}

// Fill ring slot s with page k (metadata page/flags broadcast by the caller; s = k mod
// nsl), from lane 0: arm the slot's barrier with the slice's bytes and issue one bulk
// tensor copy per tensor: K through the 5-D fp16 slice map, V through the byte map (E4M3
// or BASE page) or the fp16 slice map (TARGET page). A skipped page only arrives on the
// barrier.
template <int D, int VMODE>
__device__ __forceinline__ void ring_fill(const WarpRing& ring, int s, int h, int page, int vloc, int flags,
                                          bool elastic, const CUtensorMap* tmK, const CUtensorMap* tmV8,
                                          const CUtensorMap* tmV16) {
  using S = Slot<D, VMODE>;
  uint64_t* bar = &ring.full[s];
  if (flags & kMetaSkip) {
    mbar_arrive(bar);
    return;
  }
  // E4M3 and BASE pages both hold one byte per value: the same box
  const bool compact = VMODE == kVE4M3 || (VMODE == kVMixed && (flags & (kMetaCompact | kMetaBase)));
  uint8_t* dst = ring.slots + (size_t)s * S::kBytes;
  mbar_arrive_expect_tx(bar, S::kK + (compact ? kPage * D : kPage * D * 2));
  tma_load_5d(dst, tmK, 0, 0, 0, h, page, bar);
  if (elastic) {                                     // vloc = half-slot location
    if (compact) tma_load_5d(dst + S::kK, tmV8, 0, h, 0, vloc & 1, vloc >> 1, bar);
    else tma_load_5d(dst + S::kK, tmV16, 0, 0, 0, h, vloc >> 1, bar);
  } else {                                           // vloc = page
    if (compact) tma_load_4d(dst + S::kK, tmV8, 0, h, 0, vloc, bar);
    else tma_load_5d(dst + S::kK, tmV16, 0, 0, 0, h, vloc, bar);
  }
}

// ring_fill of slot s from the warp (lanes other than 0 return).
template <int D, int VMODE>
__device__ __forceinline__ void ring_issue(const WarpRing& ring, int s, int h, int page, int vloc, int flags,
                                           bool elastic, const CUtensorMap* tmK, const CUtensorMap* tmV8,
                                           const CUtensorMap* tmV16) {
  if ((threadIdx.x & 31) != 0) return;
  ring_fill<D, VMODE>(ring, s, h, page, vloc, flags, elastic, tmK, tmV8, tmV16);
}

// ring_fill of page k's slot (k mod nsl, computed by lane 0 alone).
template <int D, int VMODE>
__device__ __forceinline__ void ring_issue_page(const WarpRing& ring, int k, int h, int page, int vloc, int flags,
                                                bool elastic, const CUtensorMap* tmK, const CUtensorMap* tmV8,
                                                const CUtensorMap* tmV16) {
  if ((threadIdx.x & 31) != 0) return;
  ring_fill<D, VMODE>(ring, k % ring.nsl, h, page, vloc, flags, elastic, tmK, tmV8, tmV16);
}


// Common prologue of the split kernels: plan, this CTA's page range, barriers.
// Returns false when the CTA has no pages.
__device__ __forceinline__ bool split_prologue(const DecodeParams& p, uint8_t* smem, int* warp_tot, int& start,
                                               int& end, int& per, int& b_first, int& b_last) {
  int* cu = reinterpret_cast<int*>(smem + p.cu_off);
  const int total = plan_pages(p, cu, warp_tot);
  // ranges split the stream by cost: a page costs 1 and the start of a sequence (its Q
  // load and segment end) kSegmentCost more, so page j of sequence b sits at position
  // j + kSegmentCost * b of a stream of total + kSegmentCost * batch positions
  const int nv = (int)gridDim.x * p.NG;                // ranges: one per (CTA, page group)
  const int vtotal = total + kSegmentCost * p.batch;
  per = total > 0 ? (vtotal + nv - 1) / nv : 1;
  if (blockIdx.x == 0) {
    int mine = 0;
    for (int b = threadIdx.x; b < p.batch; b += blockDim.x) mine |= cu[b + 1] == cu[b];
    if (__syncthreads_or(mine)) {
      if (p.pdl) griddep_wait();                     // outputs only after the preceding kernel
      write_empty_sequences(p, cu);
    }
  }
  if (total == 0 || (int)blockIdx.x * p.NG * per >= vtotal) return false;   // the whole CTA is idle
  for (int i = threadIdx.x; i < kWarps * p.nsl; i += blockDim.x) {
    mbar_init(reinterpret_cast<uint64_t*>(smem + p.bar_off) + i, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // this warp's range (no CTA-wide barrier follows, so an idle warp may leave here)
  const int v = (int)blockIdx.x * p.NG + (int)(threadIdx.x >> 5) / p.Hkv;
  start = page_at(cu, p.batch, v * per);
  end = page_at(cu, p.batch, min(vtotal, (v + 1) * per));
  if (start >= end) return false;
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
// Partial results. A warp's result for (segment b, page group grp, KV head h) is
//   m = max score (log2 units), l = sum 2^(s - m), acc = sum 2^(s - m) v
// per query head. It is written as record b + v of range v, except when the warp saw
// the whole sequence (no other range touches it): then it writes
// the finished output directly. A warp that met a page it must skip (bad id, mode
// byte or scale) writes l = -1 instead: the merge turns that into a zero output and
// lse = -inf for the query heads of h.
constexpr float kBadRecord = -1.f;

// A merge job: the records rec0 .. rec0 + nrec - 1 of (sequence b, KV head h).
struct MergeJob {
  int b;
  int rec0;
  int nrec;
};

// Combine the records of each job, in one pass with a running maximum:
//   M = max m_i,  L = sum l_i 2^(m_i - M),  out = sum acc_i 2^(m_i - M) / L,
//   lse = (M + log2 L) ln 2.
// The records of consecutive jobs are staged together in `buf` (the warp's ring, idle
// once its stream has ended), up to kMaxSlots per wave: the acc blocks (G x D floats
// each, contiguous) by 16-byte cp.async copies spread over the lanes, the (m, l) pairs
// by plain loads, all issued before any is used. A wave costs one L2 round trip
// (freshly written records take ~2 us to come back), however many jobs and records it
// holds; a job longer than a wave continues in the next one. (A 1-D bulk copy per
// record would cost its issuing lane more than the round trip.) Lanes split over
// (query head, column block): 32/GP lanes per head, kDpl columns each. A record with
// l = 0 (a page group without tokens) contributes nothing; l < 0 marks a skipped page
// and zeroes the output of its job.
template <int D, int GP>
__device__ void merge_jobs(const DecodeParams& p, int h, const MergeJob* jobs, int nj, uint8_t* buf,
                           int buf_bytes) {
  constexpr int kLph = 32 / GP;                      // lanes per query head
  constexpr int kDpl = D / kLph;                     // columns per lane
  constexpr int kMaxSlots = 16;
  constexpr int kTables = kMaxSlots * 4 + kMaxSlots * 8 * 8;   // slot records, (m, l) pairs
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const int g = lane / kLph, sub = lane % kLph, d0 = sub * kDpl;
  const bool active = g < G;
  const int gl = active ? g : 0;
  const int rb = G * D * 4;                          // bytes of one record's acc block
  int* slot_rec = reinterpret_cast<int*>(buf);
  float2* slot_ml = reinterpret_cast<float2*>(buf + kMaxSlots * 4);   // [slot][8 heads]
  uint8_t* slot_acc = buf + kTables;
  int cap = (buf_bytes - kTables) / rb;
  cap = cap > kMaxSlots ? kMaxSlots : cap;
  if (cap < 1) {                                     // a ring smaller than one record: cannot happen
    if (lane == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_TIMEOUT, blockIdx.x);
    return;
  }
  float acc[kDpl];
  float M = -INFINITY, L = 0.f;
  bool bad = false;
  int j = 0, r = 0;                                  // next record to stage
  int cj = 0, cr = 0;                                // next record to combine
  while (j < nj) {
    // plan the wave (the same on every lane); lane 0 writes the slot table
    __syncwarp();                                    // the previous wave is consumed
    int ns = 0;
    while (j < nj && ns < cap) {
      if (lane == 0) slot_rec[ns] = jobs[j].rec0 + r;
      ++ns;
      if (++r == jobs[j].nrec) {
        ++j;
        r = 0;
      }
    }
    __syncwarp();
    for (int s = 0; s < ns; ++s) {
      const uint8_t* src = reinterpret_cast<const uint8_t*>(p.part_acc + ((size_t)slot_rec[s] * p.Hq + h * G) * D);
      for (int off = lane * 16; off < rb; off += 32 * 16) cp_async_16(slot_acc + s * rb + off, src + off);
    }
    float2 v[kMaxSlots * 8 / 32];
#pragma unroll
    for (int i = 0; i < kMaxSlots * 8 / 32; ++i) {
      const int q = lane + 32 * i;
      v[i] = q < ns * G ? __ldcg(p.part_ml + (size_t)slot_rec[q / G] * p.Hq + h * G + q % G)
                        : make_float2(-INFINITY, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kMaxSlots * 8 / 32; ++i) {
      const int q = lane + 32 * i;
      if (q < ns * G) slot_ml[(q / G) * 8 + q % G] = v[i];
    }
    cp_async_wait_all();
    __syncwarp();                                    // every lane's copies and pairs visible
    for (int s = 0; s < ns; ++s) {
      if (cr == 0) {
#pragma unroll
        for (int x = 0; x < kDpl; ++x) acc[x] = 0.f;
        M = -INFINITY;
        L = 0.f;
        bad = false;
      }
      const float2 ml = slot_ml[s * 8 + gl];
      bad |= ml.y < 0.f;
      if (ml.y > 0.f) {
        const float Mn = fmaxf(M, ml.x);
        const float sc = exp2f(M - Mn), w = exp2f(ml.x - Mn);
        L = fmaf(w, ml.y, L * sc);
        const float2* src = reinterpret_cast<const float2*>(slot_acc + s * rb) + (gl * D + d0) / 2;
#pragma unroll
        for (int x = 0; x < kDpl / 2; ++x) {
          const float2 a = src[x];
          acc[2 * x] = fmaf(w, a.x, acc[2 * x] * sc);
          acc[2 * x + 1] = fmaf(w, a.y, acc[2 * x + 1] * sc);
        }
        M = Mn;
      }
      if (++cr == jobs[cj].nrec) {                   // job cj complete: write its output
        if (active) {
          const int b = jobs[cj].b, hq = h * G + g;
          const float Lf = bad ? 0.f : L;
          const float inv = Lf > 0.f ? 1.f / Lf : 0.f;
          __half* o = p.out + ((size_t)b * p.Hq + hq) * D + d0;
#pragma unroll
          for (int x = 0; x < kDpl; x += 2)
            *reinterpret_cast<__half2*>(o + x) = __floats2half2_rn(acc[x] * inv, acc[x + 1] * inv);
          if (sub == 0 && p.lse)
            p.lse[(size_t)b * p.Hq + hq] = Lf > 0.f ? (M + log2f(Lf)) * 0.69314718055994531f : -INFINITY;
        }
        ++cj;
        cr = 0;
      }
    }
  }
}

template <int D>
__device__ void merge_run(const DecodeParams& p, int h, const MergeJob* jobs, int nj, const MergeBuf& mb) {
  if (nj == 0) return;
  const int G = p.G;
  if (G <= 1) merge_jobs<D, 1>(p, h, jobs, nj, mb.buf, mb.bytes);
  else if (G <= 2) merge_jobs<D, 2>(p, h, jobs, nj, mb.buf, mb.bytes);
  else if (G <= 4) merge_jobs<D, 4>(p, h, jobs, nj, mb.buf, mb.bytes);
  else merge_jobs<D, 8>(p, h, jobs, nj, mb.buf, mb.bytes);
}

// True when sequence b has pages outside the range [start, end).
__device__ __forceinline__ bool crosses_ctas(const int* cu, int b, int start, int end) {
  return cu[b] < start || cu[b + 1] > end;
}

// A warp's completion, after its stream ends (its records all written): the sequences
// that continue in other ranges (only the first and the last segment of a range can)
// take one ticket per warp for (b, h); the warp that takes the last of the n ranges'
// tickets merges (b, h) and resets the ticket. Mid-stream segment ends take no fence
// and no atomic: the tickets of the range's first segment are taken here too, which
// delays nothing, as its last records come from the range before, finishing at about
// the same time.
template <int D>
__device__ void finish_warp(const DecodeParams& p, const int* cu, int start, int end, int per, int b_first,
                            int b_last, int h, MergeBuf mb) {
  const int lane = threadIdx.x & 31;
  int cross_b[2] = {-1, -1};
  int n_cross = 0;
  if (cu[b_first] != cu[b_first + 1] && crosses_ctas(cu, b_first, start, end)) cross_b[n_cross++] = b_first;
  if (b_last != b_first && crosses_ctas(cu, b_last, start, end)) cross_b[n_cross++] = b_last;
  __syncwarp();
  unsigned last_mask = 0;
  if (lane == 0 && n_cross > 0) {
    fence_acq_rel_gpu();                               // release: the warp's records (ordered
                                                       // before lane 0 by the __syncwarp) first
    int old[2] = {0, 0};
    int* tk[2] = {nullptr, nullptr};
    for (int e = 0; e < n_cross; ++e) {
      tk[e] = p.plan + kPlanTicket + cross_b[e] * kMaxKvHeads + h;
      old[e] = atomicAdd(tk[e], 1);
    }
    for (int e = 0; e < n_cross; ++e) {
      int v0, n_ranges;
      ranges_of(cu, cross_b[e], per, v0, n_ranges);
      if (old[e] == n_ranges - 1) {
        last_mask |= 1u << e;
        *tk[e] = 0;
      }
    }
    if (last_mask) fence_acq_rel_gpu();                // acquire: the other ranges' records; the
                                                       // merge's __syncwarp orders the lanes' loads after it
  }
  last_mask = __shfl_sync(0xffffffffu, last_mask, 0);
  MergeJob jobs[2];
  int nj = 0;
  for (int e = 0; e < n_cross; ++e) {
    if (!(last_mask & (1u << e))) continue;
    const int b = cross_b[e];
    int v0, n_ranges;
    ranges_of(cu, b, per, v0, n_ranges);
    jobs[nj++] = MergeJob{b, b + v0, n_ranges};
  }
  merge_run<D>(p, h, jobs, nj, mb);
}

}  // namespace ekv
