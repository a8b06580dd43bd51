// decode_mma.cu -- tensor-core consumer of the split-K paged decode.
//
// Same pipeline and partial records as the CUDA-core consumer (pipeline.cuh); the
// per-(page, KV head) tiles are multiplied with mma.sync.m16n8k16 (f16 x f16 -> f32):
//
//   QK:  S^T[t][g] = sum_d K[t][d] Q[g][d]    M = 16 tokens, N = 8 query heads of the
//        KV head's GQA group (G <= 8, zero-padded), K = D in steps of 16.
//        A = K rows via ldmatrix from the swizzled TMA box; B = Q, held in registers.
//   PV:  O^T[d][g] = sum_t V^T[d][t] P^T[t][g] M = 16 rows of d, N = 8, K = 16 tokens.
//        B = P^T from the QK accumulators (one movmatrix per 8 tokens); A = V^T:
//        E4M3 rows through ldmatrix.trans on byte pairs + byte permute + an exact
//        E4M3 -> f16 convert in registers (the compact page is never materialised,
//        ElasticKV Sec. 3.2 / knlp.io fused V8 load); FP16 rows through 32-bit loads
//        and a byte permute.
//
// The d rows of the PV tile are permuted: m-tile i, row r holds d = 16i + 2r and row
// r + 8 holds d = 16i + 2r + 1, so each lane's E4M3 bytes come from one ldmatrix.trans
// element. The records are written back in natural d order.
//
// Scores are scaled in fp32 after the QK product (Q stays exact in f16); P is rounded
// to f16 for the PV product and the running sum l accumulates the rounded values, so
// the normalisation matches the weights actually applied. A compact page's value scale
// is applied in fp32 to that page's PV product (acc += s * (P V8)), except for the
// uniform per-tensor case where it is applied once to the partial record.
#include <mutex>
#include <set>
#include <utility>

#include "pipeline.cuh"

namespace ekv {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ uint32_t e4m3_pair_to_h2(uint32_t two_codes) {
  return h2_bits(e4m3x2_to_half2((uint16_t)two_codes));
}

// A fragment (V^T rows d, cols = tokens) of one m-tile from one ldmatrix.trans
// register of E4M3 byte pairs: bytes {V[t][d], V[t][d+1], V[t+1][d], V[t+1][d+1]}.
__device__ __forceinline__ void e4m3_rows(uint32_t reg, uint32_t& row_d, uint32_t& row_d1) {
  const uint32_t x = __byte_perm(reg, 0u, 0x3120);   // {V[t][d], V[t+1][d], V[t][d+1], V[t+1][d+1]}
  row_d = e4m3_pair_to_h2(x & 0xffffu);
  row_d1 = e4m3_pair_to_h2(x >> 16);
}

template <int D, int VMODE>
__device__ void consume_mma(const DecodeParams& p, uint8_t* stages, PageMeta* meta, uint64_t* full,
                            uint64_t* empty, const int* cu, int start, int end, int b_first, int b_last, int per) {
  using L = StageLayout<D, VMODE>;
  constexpr int KS = D / 16;   // k-steps of QK
  constexpr int MT = D / 16;   // m-tiles of PV
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = p.Hkv, NG = p.NG, G = p.G;
  const int h = warp % Hkv, grp = warp / Hkv;
  const int q4 = lane & 3, r8 = lane >> 2;          // fragment coordinates
  const int k_sub = L::kKStage / NG, v_sub = L::kVStage / NG;
  const bool uniform_scale = VMODE == kVE4M3 && p.scale_mode == EKV_SCALE_PER_TENSOR;
  // ldmatrix row address pattern (token, 16-byte chunk offset) of this lane
  const int lm_t = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int lm_c = lane >> 4;

  for (int b = b_first; b <= b_last; ++b) {
    const int j0 = max(cu[b], start), j1 = min(cu[b + 1], end);
    if (j0 >= j1) continue;
    // B fragments of Q^T: lane holds Q[g = r8][16s + 2q4 (+1)] and [16s + 8 + 2q4 (+1)]
    uint32_t qb[KS][2];
    {
      const bool gv = r8 < G;
      const __half* qrow = p.q + ((size_t)b * p.Hq + h * G + (gv ? r8 : 0)) * D;
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        qb[s][0] = gv ? __ldg(reinterpret_cast<const unsigned int*>(qrow + 16 * s + 2 * q4)) : 0u;
        qb[s][1] = gv ? __ldg(reinterpret_cast<const unsigned int*>(qrow + 16 * s + 8 + 2 * q4)) : 0u;
      }
    }
    float acc[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;           // running max of g = 2q4, 2q4 + 1
    float l0 = 0.f, l1 = 0.f;                       // this lane's share of the sums
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
      const int flags = mt.flags;
      const int ntok = mt.ntok;
      const bool compact = VMODE == kVE4M3 || (VMODE == kVMixed && (flags & kMetaCompact));
      const bool skip = (flags & kMetaSkip) != 0;
      const float vs = (compact && !uniform_scale) ? mt.scale[h] : 1.f;
      // Pull this (page, head) slice into registers and free the stage at once, so
      // that the producer can refill it while the tiles are multiplied: K as QK A
      // fragments, V as raw rows (E4M3: ldmatrix.trans byte pairs; FP16: 32-bit words).
      uint32_t kf[KS][4];
      uint32_t vr[MT][4];
      if (!skip) {
        const uint32_t kp = smem_u32(stages + stage * L::kStageBytes + grp * k_sub);
        const uint32_t vp = smem_u32(stages + stage * L::kStageBytes + L::kKStage + grp * v_sub);
#pragma unroll
        for (int s = 0; s < KS; ++s) {
          const int kb = s >> 2, c = 2 * (s & 3) + lm_c;
          ldsm_x4(kp + (kb * Hkv + h) * 2048 + swz128(lm_t * 128 + c * 16), kf[s][0], kf[s][1], kf[s][2], kf[s][3]);
        }
        if (compact) {
          const uint32_t vbox = vp + h * (kPage * D);
#pragma unroll
          for (int j = 0; j < MT / 2; ++j) {
            const int c = 2 * j + lm_c;
            const uint32_t off = D == 128 ? swz128(lm_t * 128 + c * 16) : swz64(lm_t * 64 + c * 16);
            ldsm_x4_trans(vbox + off, vr[j][0], vr[j][1], vr[j][2], vr[j][3]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < MT; ++i) {
            const int d = 16 * i + 2 * r8;
            const uint32_t box = vp + ((d >> 6) * Hkv + h) * 2048;
            const uint32_t col = (d & 63) * 2;
            const int t0 = 2 * q4;
            vr[i][0] = lds_u32(box + swz128(t0 * 128 + col));
            vr[i][1] = lds_u32(box + swz128((t0 + 1) * 128 + col));
            vr[i][2] = lds_u32(box + swz128((t0 + 8) * 128 + col));
            vr[i][3] = lds_u32(box + swz128((t0 + 9) * 128 + col));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (!skip) {
        // ---- QK on the tensor cores: two independent accumulation chains
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        float sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < KS; ++s) {
          if (s & 1) mma_f16(sd, kf[s][0], kf[s][1], kf[s][2], kf[s][3], qb[s][0], qb[s][1]);
          else mma_f16(sc, kf[s][0], kf[s][1], kf[s][2], kf[s][3], qb[s][0], qb[s][1]);
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) sc[x] += sd[x];
        // rows r8 and r8 + 8 (tokens), cols 2q4, 2q4 + 1 (query heads)
        const bool v_lo = r8 < ntok, v_hi = r8 + 8 < ntok;
        const float s00 = v_lo ? sc[0] * p.qscale : -INFINITY;
        const float s01 = v_lo ? sc[1] * p.qscale : -INFINITY;
        const float s10 = v_hi ? sc[2] * p.qscale : -INFINITY;
        const float s11 = v_hi ? sc[3] * p.qscale : -INFINITY;
        float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const __half2 plo = __floats2half2_rn(exp2f(s00 - mn0), exp2f(s01 - mn1));   // token r8
        const __half2 phi = __floats2half2_rn(exp2f(s10 - mn0), exp2f(s11 - mn1));   // token r8+8
        if (__any_sync(0xffffffffu, (mn0 > m0) || (mn1 > m1))) {
          const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
          l0 *= al0;
          l1 *= al1;
#pragma unroll
          for (int i = 0; i < MT; ++i) {
            acc[i][0] *= al0; acc[i][2] *= al0;
            acc[i][1] *= al1; acc[i][3] *= al1;
          }
          m0 = mn0;
          m1 = mn1;
        }
        {
          const float2 a = __half22float2(plo), c = __half22float2(phi);
          l0 += a.x + c.x;
          l1 += a.y + c.y;
        }
        // B fragments of P^T: transpose the 8x8 (token, head) blocks
        const uint32_t pb0 = movmatrix_trans(h2_bits(plo));   // tokens 0..7
        const uint32_t pb1 = movmatrix_trans(h2_bits(phi));   // tokens 8..15

        // ---- PV on the tensor cores
        // token masks of the A fragments: tokens 2q4, 2q4+1 (a0..a3), +8 (a4..a7)
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (ntok < kPage) {
          mlo = (2 * q4 < ntok ? 0x0000ffffu : 0u) | (2 * q4 + 1 < ntok ? 0xffff0000u : 0u);
          mhi = (2 * q4 + 8 < ntok ? 0x0000ffffu : 0u) | (2 * q4 + 9 < ntok ? 0xffff0000u : 0u);
        }
        const bool scaled = compact && !uniform_scale;
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          uint32_t a0, a1, a2, a3;
          if (compact) {
            const uint32_t* rr = vr[i >> 1];
            e4m3_rows(rr[(i & 1) * 2], a0, a1);
            e4m3_rows(rr[(i & 1) * 2 + 1], a2, a3);
          } else {
            a0 = __byte_perm(vr[i][0], vr[i][1], 0x5410);
            a1 = __byte_perm(vr[i][0], vr[i][1], 0x7632);
            a2 = __byte_perm(vr[i][2], vr[i][3], 0x5410);
            a3 = __byte_perm(vr[i][2], vr[i][3], 0x7632);
          }
          a0 &= mlo; a1 &= mlo; a2 &= mhi; a3 &= mhi;
          if (scaled) {
            // per-page scale in fp32 on this page's product
            float t4[4] = {0.f, 0.f, 0.f, 0.f};
            mma_f16(t4, a0, a1, a2, a3, pb0, pb1);
            acc[i][0] = fmaf(vs, t4[0], acc[i][0]);
            acc[i][1] = fmaf(vs, t4[1], acc[i][1]);
            acc[i][2] = fmaf(vs, t4[2], acc[i][2]);
            acc[i][3] = fmaf(vs, t4[3], acc[i][3]);
          } else {
            mma_f16(acc[i], a0, a1, a2, a3, pb0, pb1);
          }
        }
      }
    }
    // ---- partial record (natural d order)
    float lt0 = l0, lt1 = l1;
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
    }
    const float us = uniform_scale ? __ldg(p.v_scales) : 1.f;
    const size_t R = (size_t)(b + blockIdx.x) * NG + grp;
    const int g0 = 2 * q4, g1 = 2 * q4 + 1;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      const int d = 16 * i + 2 * r8;
      if (g0 < G)
        *reinterpret_cast<float2*>(p.part_acc + (R * p.Hq + h * G + g0) * D + d) =
            make_float2(acc[i][0] * us, acc[i][2] * us);
      if (g1 < G)
        *reinterpret_cast<float2*>(p.part_acc + (R * p.Hq + h * G + g1) * D + d) =
            make_float2(acc[i][1] * us, acc[i][3] * us);
    }
    if (r8 == 0) {
      if (g0 < G) p.part_ml[R * p.Hq + h * G + g0] = make_float2(m0, lt0);
      if (g1 < G) p.part_ml[R * p.Hq + h * G + g1] = make_float2(m1, lt1);
    }
    finish_segment<D>(p, b, h, cu, per);
  }
}

template <int D, int VMODE>
__global__ void __launch_bounds__(kThreads, 1)
decode_split_mma(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV8,
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
    consume_mma<D, VMODE>(p, stages, meta, full, empty, cu, start, end, b_first, b_last, per);
  }
}

template <int D, int VMODE>
static cudaError_t launch_mma(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                              const DecodeParams& p, int grid, cudaStream_t st) {
  auto kern = decode_split_mma<D, VMODE>;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  const size_t smem = split_smem_bytes(D, VMODE, kAlgoMma, p.batch);
  kern<<<grid, kThreads, smem, st>>>(tk, t8, t16, p);
  return cudaGetLastError();
}

cudaError_t launch_split_mma(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                             const DecodeParams& p, int D, int vmode, int grid, cudaStream_t st) {
  if (D == 128) {
    if (vmode == kVE4M3) return launch_mma<128, kVE4M3>(tk, t8, t16, p, grid, st);
    if (vmode == kVFP16) return launch_mma<128, kVFP16>(tk, t8, t16, p, grid, st);
    return launch_mma<128, kVMixed>(tk, t8, t16, p, grid, st);
  }
  if (vmode == kVE4M3) return launch_mma<64, kVE4M3>(tk, t8, t16, p, grid, st);
  if (vmode == kVFP16) return launch_mma<64, kVFP16>(tk, t8, t16, p, grid, st);
  return launch_mma<64, kVMixed>(tk, t8, t16, p, grid, st);
}

}  // namespace ekv
