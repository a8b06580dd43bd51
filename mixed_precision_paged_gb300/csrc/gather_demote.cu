// gather_demote.cu -- compact-prefill gather and TARGET -> compact demotion kernels.
//
// All are pure HBM streaming. Gather: one CTA per page, 16-byte vector loads issued
// all before the first store. Mode transitions (demotion to E4M3 or BASE, promotion):
// four persistent CTAs per SM, each with a ring of whole pages in shared memory.
#include "common.cuh"
#include "gather_demote.cuh"

namespace ekv {

// ------------------------------------------------------------------------ gather
// knlp.io "What changes in vLLM's prefill routing?": stored K16/V8 pages are copied
// into one bounded FP16 workspace; V8 is cast to FP16 (quantisation error kept).
// ws_k[w] = K page (bits); ws_v[w] = TARGET page (bits),
// fp16_rn(fp32_rn(E4M3(code) * s)) (fp16(E4M3(code)) when apply_scale == 0), or for a
// BASE page the fp16 word (byte << 8) (ElasticKV App. B.3; exact, no scale).
//
// One CTA per workspace page: every load of the page (K, then V or its codes and
// scales) is issued before the first store. Under a programmatic launch (p.pdl) the CTA
// signals its dependents at once and makes all those loads before griddepcontrol.wait,
// then writes the workspace after it: a gather that follows another gather (the chunks
// of one prefill admission) streams its pages in while the previous one drains.
constexpr int kGatherThreads = 256;
constexpr int kGatherVec = 8;                     // uint4 per thread: up to 32 KiB per fp16 page

__global__ void __launch_bounds__(kGatherThreads)
gather_kernel(const GatherParams p, const GatherRanges r) {
  if (p.pdl) griddep_launch_dependents();
  const int i = blockIdx.x;                       // page index within this launch
  int k = 0;
  while (k + 1 < r.n && r.off[k + 1] <= i) ++k;   // ranges are few (<= kMaxRanges)
  const int lp = r.first[k] + (i - r.off[k]);
  const int w = p.ws_base + i;
  const int page = __ldg(p.block_table + (size_t)r.seq[k] * p.bt_stride + lp);
  const int n_elem = kPage * p.Hkv * p.D;         // elements of one page
  uint4* wk = reinterpret_cast<uint4*>(p.ws_k + (size_t)w * n_elem);
  uint4* wv = reinterpret_cast<uint4*>(p.ws_v + (size_t)w * n_elem);
  const int nvec16 = n_elem * 2 / 16;             // uint4 per fp16 page
  const int nvec8 = n_elem / 16;                  // uint4 per byte page
  const int tid = threadIdx.x;
  int mode = 0;
  int detail = (page < 0 || page >= p.num_pages) ? EKV_DETAIL_PAGE_ID : EKV_DETAIL_NONE;
  int loc = 2 * page;                             // value location (half-slot index)
  if (detail == EKV_DETAIL_NONE) {
    if (p.v_block_table) {                        // pair-structured layout
      loc = __ldg(p.v_block_table + (size_t)r.seq[k] * p.bt_stride + lp);
      if (!p.has_base) {
        mode = EKV_MODE_TARGET_FP16;
      } else if (p.boundaries) {                  // TARGET-BASE-TARGET: no mode lookup
        const int b0 = __ldg(p.boundaries + 2 * r.seq[k]), b1 = __ldg(p.boundaries + 2 * r.seq[k] + 1);
        mode = (lp >= b0 && lp < b1) ? EKV_MODE_BASE : EKV_MODE_TARGET_FP16;
      } else {
        mode = p.page_mode ? (int)__ldg(p.page_mode + page) : p.uniform_mode;
      }
      // a TARGET page fills a whole slot (even location); a compact or BASE page one half
      if (loc < 0 || loc >= 2 * p.num_v_slots || (mode == EKV_MODE_TARGET_FP16 && (loc & 1)))
        detail = EKV_DETAIL_PAGE_ID;
    } else {
      mode = p.page_mode ? (int)__ldg(p.page_mode + page) : p.uniform_mode;
    }
    if (detail != EKV_DETAIL_NONE) {
    } else if (mode > EKV_MODE_BASE) {
      detail = EKV_DETAIL_PAGE_MODE;
    } else if (mode == EKV_MODE_COMPACT_E4M3 && p.apply_scale && !p.v_scales) {
      detail = EKV_DETAIL_SCALE;
    }
  }
  if (detail != EKV_DETAIL_NONE) {
    if (p.pdl) griddep_wait();                    // writes only after the preceding kernel
    if (tid == 0) {
      p.ws_indices[w] = w;
      report_error(p.err, EKV_ERR_DEVICE_CHECK, detail, w);
    }
    for (int v = tid; v < nvec16; v += kGatherThreads) {
      wk[v] = make_uint4(0, 0, 0, 0);
      wv[v] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  // loads: the K page, then the value page (a TARGET page at slot loc / 2; a compact or
  // BASE page in half loc % 2 of that slot) and, for codes, the KV heads' scales
  const uint4* sk = reinterpret_cast<const uint4*>(p.k_pages + (size_t)page * n_elem);
  const uint4* sv = reinterpret_cast<const uint4*>(p.v_pages + (size_t)(loc >> 1) * p.v_page_stride +
                                                   (size_t)(loc & 1) * n_elem);
  uint4 kb[kGatherVec], vb[kGatherVec];
#pragma unroll
  for (int u = 0; u < kGatherVec; ++u) {
    const int v = tid + u * kGatherThreads;
    if (v < nvec16) kb[u] = __ldg(sk + v);
  }
  const int nv = mode == EKV_MODE_TARGET_FP16 ? nvec16 : nvec8;
#pragma unroll
  for (int u = 0; u < kGatherVec; ++u) {
    const int v = tid + u * kGatherThreads;
    if (v < nv) vb[u] = __ldg(sv + v);
  }
  float sc[kGatherVec / 2];                       // E4M3: the scale of each code vector's head
#pragma unroll
  for (int u = 0; u < kGatherVec / 2; ++u) {
    const int v = tid + u * kGatherThreads;
    sc[u] = 1.f;
    if (mode == EKV_MODE_COMPACT_E4M3 && p.apply_scale && v < nvec8) {
      const int head = ((v * 16) / p.D) % p.Hkv;  // 16 codes of one head row (D >= 64)
      sc[u] = p.scale_mode == EKV_SCALE_PER_TENSOR ? __ldg(p.v_scales)
                                                   : __ldg(p.v_scales + (size_t)page * p.Hkv + head);
    }
  }
  if (p.pdl) griddep_wait();                      // the workspace is written after it
  if (tid == 0) p.ws_indices[w] = w;
#pragma unroll
  for (int u = 0; u < kGatherVec; ++u) {
    const int v = tid + u * kGatherThreads;
    if (v < nvec16) wk[v] = kb[u];
  }
  if (mode == EKV_MODE_TARGET_FP16) {             // bit copy
#pragma unroll
    for (int u = 0; u < kGatherVec; ++u) {
      const int v = tid + u * kGatherThreads;
      if (v < nvec16) wv[v] = vb[u];
    }
    return;
  }
  // E4M3 or BASE: 16 codes per uint4, all in one head row (D >= 64) -> 2 uint4 of fp16
#pragma unroll
  for (int u = 0; u < kGatherVec / 2; ++u) {
    const int v = tid + u * kGatherThreads;
    if (v >= nvec8) continue;
    const uint32_t words[4] = {vb[u].x, vb[u].y, vb[u].z, vb[u].w};
    uint32_t outw[8];
    if (mode == EKV_MODE_BASE) {                  // high byte in place, low byte zero
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        outw[2 * q] = __byte_perm(words[q], 0u, 0x1404);       // {0, b0, 0, b1}
        outw[2 * q + 1] = __byte_perm(words[q], 0u, 0x3424);   // {0, b2, 0, b3}
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint16_t two = (uint16_t)(words[q] >> (16 * hh));
          __half2 hv = e4m3x2_to_half2(two);
          if (p.apply_scale) {
            const float2 f = __half22float2(hv);
            hv = __halves2half2(__float2half_rn(__fmul_rn(f.x, sc[u])), __float2half_rn(__fmul_rn(f.y, sc[u])));
          }
          outw[q * 2 + hh] = *reinterpret_cast<uint32_t*>(&hv);
        }
      }
    }
    wv[2 * v] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
    wv[2 * v + 1] = make_uint4(outw[4], outw[5], outw[6], outw[7]);
  }
}

// ------------------------------------------------------------------------ transitions
// ElasticKV Sec. 3.4 "Transition protocols": synchronous, in place; a page reads in its
// new mode only after the kernel completes (stream order publishes data, scales and
// mode together).
//  kToE4M3 (TARGET -> compact): per KV head h, a = max|x|, s = a / 448 (IEEE fp32
//    divide; 1 when a == 0), code = E4M3_rn_satfinite(x / s). The quotient is the IEEE
//    one, computed by div_by_scale (reciprocal + one Markstein correction; checked
//    against __fdiv_rn).
//  kToBase (TARGET -> BASE, ElasticKV App. B.2): the high bytes of the fp16 values go
//    to the page's first half, the low bytes to the caller's backing row (if any).
//  kPromote (BASE -> TARGET, App. B.2): the fp16 words are rebuilt from the page's high
//    bytes and the backing's low bytes.
// Demotions skip (and report) a page holding NaN/inf and leave it TARGET.
//
// Streaming form: 4 CTAs per SM, each takes items blockIdx.x, blockIdx.x + grid, ...
// of page_ids. A CTA keeps S stages of 32 KiB worth (the FP16 page; for promotion the
// high bytes then the low bytes) in flight in a shared-memory ring, filled by 1-D bulk
// copies that thread 0 issues as soon as the page before it in that slot is in
// registers, so the next page streams in while the CTA works on this one. (Measured
// on 8,192 demotions: 4 CTAs x 48 KiB 6.3 TB/s, 3 x 64 KiB 6.1, 2 x 96 KiB 5.6,
// 1 x 192 KiB 4.3: the per-page work, not the depth of the ring, sets the pace.) Each
// thread holds its 8 x 16 B of the page in registers, so the page may be rewritten
// in place. Page ids and mode bytes of the next kChunk items are staged in shared
// memory by the whole CTA.
constexpr int kDemoteThreads = 256;
constexpr int kDemoteMaxStages = 8;
constexpr int kDemoteRingBytes = 48 * 1024;
constexpr int kDemoteChunk = 256;   // items staged at a time (small static smem: 4 CTAs per SM)

template <int OP>
__global__ void __launch_bounds__(kDemoteThreads, 4)
transition_kernel(const DemoteParams p, int n, int S) {
  constexpr int kMaxVec = 8;                      // 8 x 16 B x 256 = 32 KiB (H_kv*D <= 1024)
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kDemoteMaxStages];
  __shared__ int s_stage_page[kDemoteMaxStages];  // page in a slot, -1 = nothing to do
  __shared__ int s_stage_dst[kDemoteMaxStages];   // its destination location
  __shared__ int s_ids[kDemoteChunk];             // page of an item, -1 = skip it
  __shared__ int s_src[kDemoteChunk];             // its source and destination locations
  __shared__ int s_dst[kDemoteChunk];
  __shared__ unsigned int s_amax[kMaxKvHeads];
  __shared__ float s_scale[kMaxKvHeads];
  __shared__ float s_recip[kMaxKvHeads];
  __shared__ int s_nonfinite;
  const int tid = threadIdx.x, lane = tid & 31;
  const int grid = (int)gridDim.x;
  const int m = (n - (int)blockIdx.x + grid - 1) / grid;   // items of this CTA
  const int half_bytes = kPage * p.Hkv * p.D;     // one byte per value
  const int page_bytes = 2 * half_bytes;          // stage size
  const int nvec = page_bytes / 16;               // fp16 vectors of a page
  const int lanes_per_row = p.D / 8;              // 8 or 16: a row of one head
  // Vector v holds elements 8v .. 8v+7 of the page [16][H_kv][D], in KV head
  // (8v / D) mod H_kv. A thread's vectors are tid + 256u, 2048u elements apart, a
  // multiple of H_kv * D (<= 1024): they all lie in the same head.
  const int head = ((tid * 8) / p.D) % p.Hkv;
  const int want = OP == kPromote ? EKV_MODE_BASE : EKV_MODE_TARGET_FP16;

  // items k0 .. k0 + kChunk - 1 of this CTA: page id if valid and in the source mode,
  // with its source and destination value locations (half-slot indices)
  auto load_chunk = [&](int k0) {
    for (int t = tid; t < kDemoteChunk; t += kDemoteThreads) {
      const int k = k0 + t;
      int id = -1, src = 0, dst = 0;
      if (k < m) {
        const int i = (int)blockIdx.x + k * grid;
        const int page = __ldg(p.page_ids + i);
        if (page < 0 || page >= p.num_pages) {
          report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_ID, i);
        } else if (p.page_mode[page] == want) {   // else nothing to do
          src = p.src_loc ? __ldg(p.src_loc + i) : 2 * page;
          dst = p.dst_loc ? __ldg(p.dst_loc + i) : 2 * page;
          const int full = OP == kPromote ? dst : src;   // the location a TARGET page fills
          if (src < 0 || dst < 0 || src >= 2 * p.num_slots || dst >= 2 * p.num_slots || (full & 1))
            report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_ID, i);
          else
            id = page;
        }
      }
      s_ids[t] = id;
      s_src[t] = src;
      s_dst[t] = dst;
    }
  };
  // thread 0: slot k % S receives item k
  auto issue = [&](int k) {
    const int sl = k % S;
    const int page = s_ids[k % kDemoteChunk];
    const int src_loc = s_src[k % kDemoteChunk];
    s_stage_page[sl] = page;
    s_stage_dst[sl] = s_dst[k % kDemoteChunk];
    if (page < 0) {
      mbar_arrive(&full[sl]);
      return;
    }
    const uint8_t* src = p.v_pages + (size_t)(src_loc >> 1) * p.v_page_stride + (src_loc & 1) * half_bytes;
    mbar_arrive_expect_tx(&full[sl], (uint32_t)page_bytes);
    if (OP == kPromote) {
      const size_t i = (size_t)blockIdx.x + (size_t)k * grid;
      bulk_load(ring + sl * page_bytes, src, (uint32_t)half_bytes, &full[sl]);
      bulk_load(ring + sl * page_bytes + half_bytes, p.low + i * half_bytes, (uint32_t)half_bytes, &full[sl]);
    } else {
      bulk_load(ring + sl * page_bytes, src, (uint32_t)page_bytes, &full[sl]);
    }
  };

  if (tid < S) {
    mbar_init(&full[tid], 1);
    fence_barrier_init();
  }
  if (tid < kMaxKvHeads) s_amax[tid] = 0u;
  if (tid == 0) s_nonfinite = 0;
  load_chunk(0);
  __syncthreads();
  if (tid == 0)
    for (int k = 0; k < min(S, m); ++k) issue(k);

  for (int k = 0; k < m; ++k) {
    const int sl = k % S;
    const bool ok = mbar_wait(&full[sl], (uint32_t)(k / S) & 1u);
    const int page = s_stage_page[sl];
    const int dst_loc = s_stage_dst[sl];
    uint4 buf[kMaxVec];
    if (ok && page >= 0) {
      if (OP == kPromote) {
        // fp16 words 8v .. 8v+7 = (high byte << 8) | low byte
        const uint8_t* st = ring + sl * page_bytes;
#pragma unroll
        for (int u = 0; u < kMaxVec; ++u) {
          const int v = tid + u * kDemoteThreads;
          if (v < nvec) {
            const uint2 hb = *reinterpret_cast<const uint2*>(st + 8 * v);
            const uint2 lb = *reinterpret_cast<const uint2*>(st + half_bytes + 8 * v);
            buf[u] = make_uint4(__byte_perm(lb.x, hb.x, 0x5140), __byte_perm(lb.x, hb.x, 0x7362),
                                __byte_perm(lb.y, hb.y, 0x5140), __byte_perm(lb.y, hb.y, 0x7362));
          }
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(ring + sl * page_bytes);
        // every vector of this thread lies in KV head `head`: reduce locally first,
        // fp16 magnitudes compared as unsigned 16-bit pairs (NaN/inf >= 0x7c00)
        unsigned int mx2 = 0u;
#pragma unroll
        for (int u = 0; u < kMaxVec; ++u) {
          const int v = tid + u * kDemoteThreads;
          if (v < nvec) {
            buf[u] = src[v];
            mx2 = __vmaxu2(mx2, __vmaxu2(buf[u].x & 0x7fff7fffu, buf[u].y & 0x7fff7fffu));
            mx2 = __vmaxu2(mx2, __vmaxu2(buf[u].z & 0x7fff7fffu, buf[u].w & 0x7fff7fffu));
          }
        }
        unsigned int mx = max(mx2 & 0xffffu, mx2 >> 16);
        for (int off = 1; off < lanes_per_row; off <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if ((lane % lanes_per_row) == 0 && tid < nvec) atomicMax(&s_amax[head], mx);
      }
    }
    const int kn = k + S;                          // the item that refills this slot
    if (kn < m && kn % kDemoteChunk == 0) {        // block-uniform
      __syncthreads();                             // every read of the old chunk is done
      load_chunk(kn);
    }
    // the slot is in registers (or unused): refill it; a timed-out wait ends the CTA
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_TIMEOUT, blockIdx.x);
        for (int kk = k; kk < min(k + S, m); ++kk)     // this CTA's copies still in flight
          mbar_wait(&full[kk % S], (uint32_t)(kk / S) & 1u);
      }
      return;
    }
    if (tid == 0 && kn < m) {
      fence_reads_before_refill();
      issue(kn);
    }
    if (page < 0) continue;                        // block-uniform
    // a demotion writes the half at dst_loc; a promotion the slot of dst_loc (even)
    uint8_t* base = p.v_pages + (size_t)(dst_loc >> 1) * p.v_page_stride + (dst_loc & 1) * half_bytes;
    if (OP == kPromote) {
      uint4* dst = reinterpret_cast<uint4*>(base);
#pragma unroll
      for (int u = 0; u < kMaxVec; ++u) {
        const int v = tid + u * kDemoteThreads;
        if (v < nvec) dst[v] = buf[u];
      }
      __syncthreads();
      if (tid == 0) p.page_mode[page] = EKV_MODE_TARGET_FP16;
      continue;
    }
    if (tid < p.Hkv) {
      const unsigned int bits = s_amax[tid];
      s_amax[tid] = 0u;
      if (bits >= 0x7c00u) {
        s_nonfinite = 1;
      } else if (OP == kToE4M3) {
        const float a = __half2float(__ushort_as_half((unsigned short)bits));
        const float sc = a == 0.f ? 1.f : __fdiv_rn(a, 448.f);
        s_scale[tid] = sc;
        s_recip[tid] = __frcp_rn(sc);
      }
    }
    __syncthreads();
    const bool skip = s_nonfinite != 0;
    if (!skip && OP == kToE4M3) {
      const float s = s_scale[head], rs = s_recip[head];
#pragma unroll
      for (int u = 0; u < kMaxVec; ++u) {
        const int v = tid + u * kDemoteThreads;
        if (v >= nvec) break;
        const uint32_t w[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
        uint32_t packed[2];
#pragma unroll
        for (int q = 0; q < 4; q += 2) {
          const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w[q]));
          const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w[q + 1]));
          const uint16_t lo = float2_to_e4m3x2(div_by_scale(a.x, s, rs), div_by_scale(a.y, s, rs));
          const uint16_t hi = float2_to_e4m3x2(div_by_scale(b.x, s, rs), div_by_scale(b.y, s, rs));
          packed[q / 2] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        *reinterpret_cast<uint2*>(base + (size_t)v * 8) = make_uint2(packed[0], packed[1]);
      }
      if (tid < p.Hkv) p.scale_out[(size_t)page * p.Hkv + tid] = s_scale[tid];
    }
    if (!skip && OP == kToBase) {
      uint8_t* low = p.low ? p.low + ((size_t)blockIdx.x + (size_t)k * grid) * half_bytes : nullptr;
#pragma unroll
      for (int u = 0; u < kMaxVec; ++u) {
        const int v = tid + u * kDemoteThreads;
        if (v >= nvec) break;
        const uint4 w = buf[u];                    // 8 fp16 words: bytes (low, high) each
        *reinterpret_cast<uint2*>(base + (size_t)v * 8) =
            make_uint2(__byte_perm(w.x, w.y, 0x7531), __byte_perm(w.z, w.w, 0x7531));
        if (low)
          *reinterpret_cast<uint2*>(low + (size_t)v * 8) =
              make_uint2(__byte_perm(w.x, w.y, 0x6420), __byte_perm(w.z, w.w, 0x6420));
      }
    }
    __syncthreads();                               // s_nonfinite and the scales are read
    if (tid == 0) {
      if (skip) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_NONFINITE_PAGE, page);
      else p.page_mode[page] = OP == kToBase ? EKV_MODE_BASE : EKV_MODE_COMPACT_E4M3;
      s_nonfinite = 0;
    }
  }
}

cudaError_t set_smem_attr(const void* kern, int bytes);

template <int OP>
static cudaError_t launch_op(const DemoteParams& p, int n, int num_sms, cudaStream_t st) {
  const int page_bytes = kPage * p.Hkv * p.D * 2;
  int S = kDemoteRingBytes / page_bytes;
  S = S > kDemoteMaxStages ? kDemoteMaxStages : S;
  const int grid = n < 4 * num_sms ? n : 4 * num_sms;
  auto kern = transition_kernel<OP>;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern), kDemoteRingBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kDemoteThreads, (size_t)S * page_bytes, st>>>(p, n, S);
  return cudaGetLastError();
}

cudaError_t launch_transition(const DemoteParams& p, int op, int n, int num_sms, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (op == kToBase) return launch_op<kToBase>(p, n, num_sms, st);
  if (op == kPromote) return launch_op<kPromote>(p, n, num_sms, st);
  return launch_op<kToE4M3>(p, n, num_sms, st);
}

// ------------------------------------------------------------------------ writer
// knlp.io "Asymmetric K16/V8 KV cache" (implementation checks: cache writer "K
// bit-exact, V within FP8 noise"): the new token t = positions[b] of sequence b goes to
// row t % 16 of page block_table[b][t / 16]; K as its fp16 bits, V in the page's mode:
// fp16 bits (TARGET), E4M3_rn_satfinite(x / s) with the page's existing scale (compact;
// IEEE quotient), or the high bytes (BASE). One CTA per sequence, one 16-byte vector of
// 8 values per thread. A bad position, page id or mode byte writes nothing; a KV head
// whose scale is missing or not positive finite keeps its old bytes. All reported.
__global__ void __launch_bounds__(128)
append_kernel(const AppendParams p) {
  // three dependent global round trips: the position, the page id, then the mode byte and
  // the scale together; the new row (which depends on neither) is loaded first
  const int b = blockIdx.x, tid = threadIdx.x;
  const int row_elems = p.Hkv * p.D;
  const int v = tid;                              // vector of 8 values
  const bool mine = 8 * v < row_elems;
  uint4 kx = make_uint4(0u, 0u, 0u, 0u), vx = kx;
  if (mine) {
    kx = __ldg(reinterpret_cast<const uint4*>(p.k_new + (size_t)b * row_elems) + v);
    vx = __ldg(reinterpret_cast<const uint4*>(p.v_new + (size_t)b * row_elems) + v);
  }
  const int t = __ldg(p.positions + b);
  if (t < 0) return;
  if (t >= p.bt_stride * kPage) {
    if (tid == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_SEQ_LEN, b);
    return;
  }
  const int page = __ldg(p.block_table + (size_t)b * p.bt_stride + t / kPage);
  if (page < 0 || page >= p.num_pages) {
    if (tid == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_ID, b);
    return;
  }
  const int head = mine ? (8 * v) / p.D : 0;
  const int mode = p.page_mode ? (int)__ldg(p.page_mode + page) : p.uniform_mode;
  const float s = !p.v_scales ? 0.f
                  : (p.scale_mode == EKV_SCALE_PER_TENSOR ? __ldg(p.v_scales)
                                                           : __ldg(p.v_scales + (size_t)page * p.Hkv + head));
  if (mode > EKV_MODE_BASE) {
    if (tid == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_MODE, b);
    return;
  }
  if (!mine) return;
  const int row = t % kPage;
  reinterpret_cast<uint4*>(p.k_pages + ((size_t)page * kPage + row) * row_elems)[v] = kx;
  uint8_t* vpage = p.v_pages + (size_t)page * p.v_page_stride;
  if (mode == EKV_MODE_TARGET_FP16) {
    reinterpret_cast<uint4*>(vpage + (size_t)row * row_elems * 2)[v] = vx;
    return;
  }
  uint2* dst = reinterpret_cast<uint2*>(vpage + (size_t)row * row_elems) + v;
  if (mode == EKV_MODE_BASE) {                    // high byte of each fp16 word
    *dst = make_uint2(__byte_perm(vx.x, vx.y, 0x7531), __byte_perm(vx.z, vx.w, 0x7531));
    return;
  }
  if (!scale_ok(s)) {
    report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_SCALE, b);
    return;
  }
  const uint32_t w[4] = {vx.x, vx.y, vx.z, vx.w};
  uint32_t packed[2];
#pragma unroll
  for (int q = 0; q < 4; q += 2) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w[q]));
    const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&w[q + 1]));
    const uint16_t lo = float2_to_e4m3x2(__fdiv_rn(a.x, s), __fdiv_rn(a.y, s));
    const uint16_t hi = float2_to_e4m3x2(__fdiv_rn(c.x, s), __fdiv_rn(c.y, s));
    packed[q / 2] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  *dst = make_uint2(packed[0], packed[1]);
}

cudaError_t launch_append(const AppendParams& p, int batch, cudaStream_t st) {
  if (batch <= 0) return cudaSuccess;
  append_kernel<<<batch, 128, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gather(const GatherParams& p, const GatherRanges& r, int pages, cudaStream_t st) {
  if (pages <= 0) return cudaSuccess;
  if (!p.pdl) {
    gather_kernel<<<pages, kGatherThreads, 0, st>>>(p, r);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pages);
  cfg.blockDim = dim3(kGatherThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_kernel, p, r);
}

}  // namespace ekv
