// gather_demote.cu -- compact-prefill gather and TARGET -> compact demotion kernels.
//
// Both are pure HBM streaming: one CTA per page, 16-byte vector loads issued all
// before the first use (8 KiB..32 KiB in flight per CTA, several CTAs per SM).
#include "common.cuh"
#include "gather_demote.cuh"

namespace ekv {

// ------------------------------------------------------------------------ gather
// knlp.io "What changes in vLLM's prefill routing?": stored K16/V8 pages are copied
// into one bounded FP16 workspace; V8 is cast to FP16 (quantisation error kept).
// ws_k[w] = K page (bits); ws_v[w] = TARGET page (bits) or
// fp16_rn(fp32_rn(E4M3(code) * s)) (fp16(E4M3(code)) when apply_scale == 0).
__global__ void __launch_bounds__(256)
gather_kernel(const GatherParams p, const GatherRanges r) {
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
  const int tid = threadIdx.x;
  if (tid == 0) p.ws_indices[w] = w;
  int mode = 0;
  bool bad = page < 0 || page >= p.num_pages;
  if (!bad) {
    mode = p.page_mode ? (int)__ldg(p.page_mode + page) : p.uniform_mode;
    if (mode > 1) bad = true;
  }
  if (bad) {
    if (tid == 0)
      report_error(p.err, EKV_ERR_DEVICE_CHECK, mode > 1 ? EKV_DETAIL_PAGE_MODE : EKV_DETAIL_PAGE_ID, w);
    for (int v = tid; v < nvec16; v += 256) {
      wk[v] = make_uint4(0, 0, 0, 0);
      wv[v] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  // K: bit copy
  const uint4* sk = reinterpret_cast<const uint4*>(p.k_pages + (size_t)page * n_elem);
  constexpr int kVecPerThread = 8;                // up to 32 KiB per page
  {
    uint4 buf[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int v = tid + u * 256;
      if (v < nvec16) buf[u] = __ldg(sk + v);
    }
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int v = tid + u * 256;
      if (v < nvec16) wk[v] = buf[u];
    }
  }
  const uint8_t* vsrc = p.v_pages + (size_t)page * p.v_page_stride;
  if (mode == 0) {
    const uint4* sv = reinterpret_cast<const uint4*>(vsrc);
    uint4 buf[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int v = tid + u * 256;
      if (v < nvec16) buf[u] = __ldg(sv + v);
    }
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int v = tid + u * 256;
      if (v < nvec16) wv[v] = buf[u];
    }
    return;
  }
  // compact: 16 codes per uint4, all in one head row (D >= 64)
  const int nvec8 = n_elem / 16;
  const uint4* sv = reinterpret_cast<const uint4*>(vsrc);
  constexpr int kCodeVecPerThread = 4;            // up to 16 KiB of codes
  uint4 buf[kCodeVecPerThread];
#pragma unroll
  for (int u = 0; u < kCodeVecPerThread; ++u) {
    const int v = tid + u * 256;
    if (v < nvec8) buf[u] = __ldg(sv + v);
  }
#pragma unroll
  for (int u = 0; u < kCodeVecPerThread; ++u) {
    const int v = tid + u * 256;
    if (v >= nvec8) continue;
    const int head = ((v * 16) / p.D) % p.Hkv;
    float s = 1.f;
    if (p.apply_scale)
      s = p.scale_mode == EKV_SCALE_PER_TENSOR ? __ldg(p.v_scales) : __ldg(p.v_scales + (size_t)page * p.Hkv + head);
    const uint32_t words[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
    uint32_t outw[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint16_t two = (uint16_t)(words[q] >> (16 * hh));
        __half2 hv = e4m3x2_to_half2(two);
        if (p.apply_scale) {
          const float2 f = __half22float2(hv);
          hv = __halves2half2(__float2half_rn(__fmul_rn(f.x, s)), __float2half_rn(__fmul_rn(f.y, s)));
        }
        outw[q * 2 + hh] = *reinterpret_cast<uint32_t*>(&hv);
      }
    }
    wv[2 * v] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
    wv[2 * v + 1] = make_uint4(outw[4], outw[5], outw[6], outw[7]);
  }
}

// ------------------------------------------------------------------------ demote
// ElasticKV Sec. 3.4: synchronous in-place demotion; the page reads as compact only
// after the kernel completes (stream order publishes codes, scales and mode together).
// Per KV head h: a = max|x|, s = a / 448 (IEEE fp32 divide; 1 when a == 0),
// code = E4M3_rn_satfinite(x / s). The quotient is the IEEE one, computed by
// div_by_scale (reciprocal + one Markstein correction; checked against __fdiv_rn).
// The whole FP16 page is loaded into registers before the first barrier, so the
// codes may overwrite the page's first half.
__global__ void __launch_bounds__(256, 4)
demote_kernel(const DemoteParams p) {
  constexpr int kMaxVec = 8;                      // 8 x 16 B x 256 = 32 KiB (H_kv*D <= 1024)
  __shared__ unsigned int s_amax[kMaxKvHeads];
  __shared__ float s_scale[kMaxKvHeads];
  __shared__ float s_recip[kMaxKvHeads];
  __shared__ int s_nonfinite;
  const int tid = threadIdx.x, lane = tid & 31;
  const int page = __ldg(p.page_ids + blockIdx.x);
  if (page < 0 || page >= p.num_pages) {
    if (tid == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_ID, blockIdx.x);
    return;
  }
  if (p.page_mode[page] != EKV_MODE_TARGET_FP16) return;      // already compact: skip
  if (tid < kMaxKvHeads) s_amax[tid] = 0u;
  if (tid == 0) s_nonfinite = 0;
  __syncthreads();
  const int n_elem = kPage * p.Hkv * p.D;
  const int nvec = n_elem / 8;                    // 8 fp16 per uint4
  const int lanes_per_row = p.D / 8;              // 8 or 16: a row of one head
  uint8_t* base = p.v_pages + (size_t)page * p.v_page_stride;
  const uint4* src = reinterpret_cast<const uint4*>(base);
  uint4 buf[kMaxVec];
#pragma unroll
  for (int u = 0; u < kMaxVec; ++u) {
    const int v = tid + u * 256;
    if (v < nvec) buf[u] = src[v];
  }
#pragma unroll
  for (int u = 0; u < kMaxVec; ++u) {
    const int v = tid + u * 256;
    if (u * 256 >= nvec) break;                   // block-uniform
    unsigned int mx = 0u;
    if (v < nvec) {
      const uint32_t w[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        mx = max(mx, w[q] & 0x7fffu);
        mx = max(mx, (w[q] >> 16) & 0x7fffu);
      }
    }
    // fp16 magnitudes compare as unsigned integers; NaN/inf are >= 0x7c00
    for (int off = 1; off < lanes_per_row; off <<= 1)
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (v < nvec && (lane % lanes_per_row) == 0) {
      const int head = ((v * 8) / p.D) % p.Hkv;
      atomicMax(&s_amax[head], mx);
    }
  }
  __syncthreads();
  if (tid < p.Hkv) {
    const unsigned int bits = s_amax[tid];
    if (bits >= 0x7c00u) {
      s_nonfinite = 1;
    } else {
      const float a = __half2float(__ushort_as_half((unsigned short)bits));
      const float sc = a == 0.f ? 1.f : __fdiv_rn(a, 448.f);
      s_scale[tid] = sc;
      s_recip[tid] = __frcp_rn(sc);
    }
  }
  __syncthreads();
  if (s_nonfinite) {
    if (tid == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_NONFINITE_PAGE, page);
    return;
  }
#pragma unroll
  for (int u = 0; u < kMaxVec; ++u) {
    const int v = tid + u * 256;
    if (v >= nvec) break;
    const int head = ((v * 8) / p.D) % p.Hkv;
    const float s = s_scale[head], rs = s_recip[head];
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
  __syncthreads();
  if (tid < p.Hkv) p.scale_out[(size_t)page * p.Hkv + tid] = s_scale[tid];
  __threadfence();
  __syncthreads();
  if (tid == 0) p.page_mode[page] = EKV_MODE_COMPACT_E4M3;
}

cudaError_t launch_gather(const GatherParams& p, const GatherRanges& r, int pages, cudaStream_t st) {
  if (pages <= 0) return cudaSuccess;
  gather_kernel<<<pages, 256, 0, st>>>(p, r);
  return cudaGetLastError();
}

cudaError_t launch_demote(const DemoteParams& p, int n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  demote_kernel<<<n, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace ekv
