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

// 2^x with the MUFU approximation (flush-to-zero; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ uint32_t e4m3_pair_to_h2(uint32_t two_codes) {
  return h2_bits(e4m3x2_to_half2((uint16_t)two_codes));
}

// The same for a BASE page: each byte is the high byte of an fp16 value whose low
// byte is zero (ElasticKV App. B.3, shift-and-bitcast): the byte permute alone places
// V[t][d], V[t+1][d] (and V[t][d+1], V[t+1][d+1]) in the high halves.
__device__ __forceinline__ void base_rows(uint32_t reg, uint32_t& row_d, uint32_t& row_d1) {
  row_d = __byte_perm(reg, 0u, 0x2404);    // {0, V[t][d], 0, V[t+1][d]}
  row_d1 = __byte_perm(reg, 0u, 0x3414);   // {0, V[t][d+1], 0, V[t+1][d+1]}
}

// A fragment (V^T rows d, cols = tokens) of one m-tile from one ldmatrix.trans
// register of E4M3 byte pairs: bytes {V[t][d], V[t][d+1], V[t+1][d], V[t+1][d+1]}.
__device__ __forceinline__ void e4m3_rows(uint32_t reg, uint32_t& row_d, uint32_t& row_d1) {
  const uint32_t x = __byte_perm(reg, 0u, 0x3120);   // {V[t][d], V[t+1][d], V[t][d+1], V[t+1][d+1]}
  row_d = e4m3_pair_to_h2(x & 0xffffu);
  row_d1 = e4m3_pair_to_h2(x >> 16);
}

// Growth of the running max (log2 units) that triggers a re-base (the weights stay < 256).
constexpr float kRebase = 8.f;
// Pages before a segment's end at which the next sequence's query rows are prefetched.
constexpr int kQPrefetch = 4;

template <int D, int VMODE, int EL>
__device__ void consume_mma(const DecodeParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV8,
                            const CUtensorMap* tmV16, uint8_t* smem, int start, int end, int b_first,
                            int b_last, int per) {
  using S = Slot<D, VMODE>;
  constexpr int KS = D / 16;   // k-steps of QK
  constexpr int MT = D / 16;   // m-tiles of PV
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = p.Hkv, G = p.G;
  const int h = warp % Hkv;
  const int v = (int)blockIdx.x * p.NG + warp / Hkv;    // this warp's range
  const int q4 = lane & 3, r8 = lane >> 2;          // fragment coordinates
  const bool uniform_scale = VMODE == kVE4M3 && p.scale_mode == EKV_SCALE_PER_TENSOR;
  // ldmatrix row address pattern (token, 16-byte chunk offset) of this lane
  const int lm_t = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int lm_c = lane >> 4;
  const int* cu = reinterpret_cast<const int*>(smem + p.cu_off);
  const WarpRing ring = warp_ring(p, smem, S::kBytes);
  const int n_range = end - start;
  const int n_my = n_range;                          // this warp's pages

  // metadata of the warp's pages, 32 per batch, one per lane: cur = batch of k,
  // nxt = next batch (mode bytes / scales in flight), nxt2 = the one after (ids in flight)
  const float tensor_scale =
      (VMODE != kVFP16 && p.scale_mode == EKV_SCALE_PER_TENSOR && p.v_scales) ? __ldg(p.v_scales) : 0.f;
#ifdef EKV_TEST_WAIT_TIMEOUT
  // test build only: 16 bytes more than any copy delivers on slot 0's first phase
  if (p.inject_timeout && blockIdx.x == 0 && warp == 0 && lane == 0 && n_my > 0) mbar_expect_tx(&ring.full[0], 16);
#endif
  WarpMeta cur, nxt, nxt2;
  wm_ids<EL>(p, cu, start, n_my, lane, cur);
  wm_ids<EL>(p, cu, start, n_my, 32 + lane, nxt);
  wm_meta<VMODE, EL>(p, tensor_scale, h, cur);
  // prime the ring; under a programmatic launch the fills before the wait stop at the
  // first page that is the last of its sequence (the cache writer, when it is the
  // preceding kernel, is writing that page's new token row)
  const int n0 = min(ring.nsl, n_my);
  const int n_pre = p.pdl ? min(n0, cu[b_first + 1] - 1 - start) : n0;
  auto prime = [&](int kk) {
    ring_issue<D, VMODE>(ring, kk, h, __shfl_sync(0xffffffffu, cur.page, kk),   // slot kk (kk < nsl)
                         EL == kElYes ? __shfl_sync(0xffffffffu, cur.vloc, kk) : __shfl_sync(0xffffffffu, cur.page, kk),
                         __shfl_sync(0xffffffffu, cur.flags, kk), EL == kElYes, tmK, tmV8, tmV16);
  };
  for (int kk = 0; kk < n_pre; ++kk) prime(kk);
  wm_meta<VMODE, EL>(p, tensor_scale, h, nxt);
  wm_ids<EL>(p, cu, start, n_my, 64 + lane, nxt2);
  if (p.pdl) {
    griddep_wait();
    for (int kk = n_pre; kk < n0; ++kk) prime(kk);
  }
  // Two orders of the per-page steps, chosen per pool by measurement (the per-page chain
  // is latency-bound, and its instruction order moves the stream rate by several percent).
  // Uniform E4M3 pool (kLate): QK, sums, V conversion, then the refill of the slot, whose
  // index lane 0 derives from the page. Other pools: QK issued, refill at once (its issue
  // overlaps the products), then sums and conversion, with the slot tracked incrementally.
  // Per layer on one box the second order gives mixed +10%, TARGET/BASE +11%, FP16 +1.5%,
  // and uniform E4M3 -2.4%, so E4M3 keeps the first.
  constexpr bool kLate = VMODE == kVE4M3;
  int k = 0;                                        // next page of this warp
  int s_idx = 0;                                    // its ring slot (k mod nsl) ...
  uint32_t phase = 0;                               // ... and that slot's fill parity
  bool timed_out = false;

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
    bool seg_bad = false;                           // a page of this segment was skipped
    const int r_end = j1 - start;
    for (; k < r_end; ++k) {
      // a few pages before this segment ends, the next sequence's query rows of this KV
      // head (G x D fp16, one 128-byte line per lane) are pulled into L1, so that the
      // next segment starts without a trip to memory
      if (k == r_end - kQPrefetch && b < b_last && lane * 64 < G * D) {
        const __half* qn = p.q + ((size_t)(b + 1) * p.Hq + h * G) * D + lane * 64;
        asm volatile("prefetch.global.L1 [%0];" ::"l"(qn));
      }
      if ((k & 31) == 0 && k > 0) {                 // next metadata batch
        cur = nxt;
        nxt = nxt2;
        wm_meta<VMODE, EL>(p, tensor_scale, h, nxt);
        wm_ids<EL>(p, cu, start, n_my, k + 64 + lane, nxt2);
      }
      const int slot = kLate ? k % ring.nsl : s_idx;
      if (!mbar_wait(&ring.full[slot], kLate ? (uint32_t)(k / ring.nsl) & 1u : phase)) {
        if (lane == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_TIMEOUT, blockIdx.x);
        // drain this warp's other fills in flight (bounded), then stop
        for (int kk = k + 1; kk < min(k + ring.nsl, n_my); ++kk)
          mbar_wait(&ring.full[kk % ring.nsl], (uint32_t)(kk / ring.nsl) & 1u);
        timed_out = true;
        break;
      }
      const int flags = __shfl_sync(0xffffffffu, cur.flags, k & 31);
      const int ntok = __shfl_sync(0xffffffffu, cur.ntok, k & 31);
      const float pscale = __shfl_sync(0xffffffffu, cur.scale, k & 31);
      const bool compact = VMODE == kVE4M3 || (VMODE == kVMixed && (flags & kMetaCompact));
      const bool base = VMODE == kVMixed && (flags & kMetaBase);
      const bool bytes8 = compact || base;          // one byte per value: E4M3 or BASE
      const bool skip = (flags & kMetaSkip) != 0;
      seg_bad |= skip;
      const float vs = (compact && !uniform_scale) ? pscale : 1.f;
      // Pull this (page, head) slice into registers and refill its slot at once, so
      // that the next fill is in flight while the tiles are multiplied: K as QK A
      // fragments, V as raw rows (E4M3: ldmatrix.trans byte pairs; FP16: 32-bit words).
      uint32_t kf[KS][4];
      uint32_t vr[MT][4];
      if (!skip) {
        const uint32_t kp = smem_u32(ring.slots + (size_t)slot * S::kBytes);
        const uint32_t vp = kp + S::kK;
#pragma unroll
        for (int s = 0; s < KS; ++s) {
          const int kb = s >> 2, c = 2 * (s & 3) + lm_c;
          ldsm_x4(kp + kb * 2048 + swz128(lm_t * 128 + c * 16), kf[s][0], kf[s][1], kf[s][2], kf[s][3]);
        }
        if (bytes8) {
          const uint32_t vbox = vp;
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
            const uint32_t box = vp + (d >> 6) * 2048;
            const uint32_t col = (d & 63) * 2;
            const int t0 = 2 * q4;
            vr[i][0] = lds_u32(box + swz128(t0 * 128 + col));
            vr[i][1] = lds_u32(box + swz128((t0 + 1) * 128 + col));
            vr[i][2] = lds_u32(box + swz128((t0 + 8) * 128 + col));
            vr[i][3] = lds_u32(box + swz128((t0 + 9) * 128 + col));
          }
        }
      }
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t va[MT][4];
      if constexpr (kLate) {
        // ---- QK on the tensor cores (four independent accumulation chains), and the V
        // rows turned into PV A fragments: after this the slot's data lives in registers
        if (!skip) {
          float sx[3][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
          for (int s = 0; s < KS; ++s) {
            float (&acc4)[4] = (s & 3) == 0 ? sc : sx[(s & 3) - 1];
            mma_f16(acc4, kf[s][0], kf[s][1], kf[s][2], kf[s][3], qb[s][0], qb[s][1]);
          }
#pragma unroll
          for (int x = 0; x < 4; ++x) sc[x] += (sx[0][x] + sx[1][x]) + sx[2][x];
#pragma unroll
          for (int i = 0; i < MT; ++i) {
            if (compact) {
              const uint32_t* rr = vr[i >> 1];
              e4m3_rows(rr[(i & 1) * 2], va[i][0], va[i][1]);
              e4m3_rows(rr[(i & 1) * 2 + 1], va[i][2], va[i][3]);
            } else if (base) {
              const uint32_t* rr = vr[i >> 1];
              base_rows(rr[(i & 1) * 2], va[i][0], va[i][1]);
              base_rows(rr[(i & 1) * 2 + 1], va[i][2], va[i][3]);
            } else {
              va[i][0] = __byte_perm(vr[i][0], vr[i][1], 0x5410);
              va[i][1] = __byte_perm(vr[i][0], vr[i][1], 0x7632);
              va[i][2] = __byte_perm(vr[i][2], vr[i][3], 0x5410);
              va[i][3] = __byte_perm(vr[i][2], vr[i][3], 0x7632);
            }
          }
        }
        // the slice is consumed from shared memory: refill the slot with page k + nsl
        fence_reads_before_refill();
        __syncwarp();
        {
          const int kk = k + ring.nsl;
          if (kk < n_my) {
            const bool in_cur = (kk >> 5) == (k >> 5);
            const int pg = __shfl_sync(0xffffffffu, in_cur ? cur.page : nxt.page, kk & 31);
            const int fl = __shfl_sync(0xffffffffu, in_cur ? cur.flags : nxt.flags, kk & 31);
            const int vl = EL == kElYes ? __shfl_sync(0xffffffffu, in_cur ? cur.vloc : nxt.vloc, kk & 31) : pg;
            ring_issue_page<D, VMODE>(ring, kk, h, pg, vl, fl, EL == kElYes, tmK, tmV8, tmV16);
          }
        }
      } else {
        // ---- QK on the tensor cores (four independent accumulation chains), issued before
        // the slot's refill so that the refill's issue overlaps their latency
        float sx[3][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (!skip) {
#pragma unroll
          for (int s = 0; s < KS; ++s) {
            float (&acc4)[4] = (s & 3) == 0 ? sc : sx[(s & 3) - 1];
            mma_f16(acc4, kf[s][0], kf[s][1], kf[s][2], kf[s][3], qb[s][0], qb[s][1]);
          }
        }
        // the slice is consumed from shared memory (it is in registers): refill the slot
        // with page k + nsl
        fence_reads_before_refill();
        __syncwarp();
        {
          const int kk = k + ring.nsl;
          if (kk < n_my) {
            const bool in_cur = (kk >> 5) == (k >> 5);
            const int pg = __shfl_sync(0xffffffffu, in_cur ? cur.page : nxt.page, kk & 31);
            const int fl = __shfl_sync(0xffffffffu, in_cur ? cur.flags : nxt.flags, kk & 31);
            const int vl = EL == kElYes ? __shfl_sync(0xffffffffu, in_cur ? cur.vloc : nxt.vloc, kk & 31) : pg;
            ring_issue<D, VMODE>(ring, s_idx, h, pg, vl, fl, EL == kElYes, tmK, tmV8, tmV16);
          }
        }
        // ---- the QK sums, and the V rows turned into PV A fragments
        if (!skip) {
#pragma unroll
          for (int x = 0; x < 4; ++x) sc[x] += (sx[0][x] + sx[1][x]) + sx[2][x];
#pragma unroll
          for (int i = 0; i < MT; ++i) {
            if (compact) {
              const uint32_t* rr = vr[i >> 1];
              e4m3_rows(rr[(i & 1) * 2], va[i][0], va[i][1]);
              e4m3_rows(rr[(i & 1) * 2 + 1], va[i][2], va[i][3]);
            } else if (base) {
              const uint32_t* rr = vr[i >> 1];
              base_rows(rr[(i & 1) * 2], va[i][0], va[i][1]);
              base_rows(rr[(i & 1) * 2 + 1], va[i][2], va[i][3]);
            } else {
              va[i][0] = __byte_perm(vr[i][0], vr[i][1], 0x5410);
              va[i][1] = __byte_perm(vr[i][0], vr[i][1], 0x7632);
              va[i][2] = __byte_perm(vr[i][2], vr[i][3], 0x5410);
              va[i][3] = __byte_perm(vr[i][2], vr[i][3], 0x7632);
            }
          }
        }
      }
      if (!skip) {
        // rows r8 and r8 + 8 (tokens), cols 2q4, 2q4 + 1 (query heads)
        const bool v_lo = r8 < ntok, v_hi = r8 + 8 < ntok;
        const float s00 = v_lo ? sc[0] * p.qscale : -INFINITY;
        const float s01 = v_lo ? sc[1] * p.qscale : -INFINITY;
        const float s10 = v_hi ? sc[2] * p.qscale : -INFINITY;
        const float s11 = v_hi ? sc[3] * p.qscale : -INFINITY;
        // Running max, re-based lazily: only when a score exceeds the reference m by more
        // than kRebase (log2 units) is the page's max reduced over the warp and O, l
        // rescaled, so the weights 2^(s - m) stay below 2^kRebase (exact in fp16's range;
        // any reference gives the same normalised result). The first page of a segment
        // (m = -inf) always re-bases.
        float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
        if (__any_sync(0xffffffffu, (mx0 > m0 + kRebase) || (mx1 > m1 + kRebase))) {
#pragma unroll
          for (int o = 4; o <= 16; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
          }
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
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
        const __half2 plo = __floats2half2_rn(ex2(s00 - m0), ex2(s01 - m1));   // token r8
        const __half2 phi = __floats2half2_rn(ex2(s10 - m0), ex2(s11 - m1));   // token r8+8
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
          uint32_t a0 = va[i][0], a1 = va[i][1], a2 = va[i][2], a3 = va[i][3];
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
      if (++s_idx == ring.nsl) {
        s_idx = 0;
        phase ^= 1u;
      }
    }
    if (timed_out) break;
    // ---- segment end (natural d order): the finished output when this warp saw the
    // whole sequence (no other range touches it), else a partial record
    float lt0 = l0, lt1 = l1;
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
    }
    const float us = uniform_scale ? __ldg(p.v_scales) : 1.f;
    const int g0 = 2 * q4, g1 = 2 * q4 + 1;
    if (seg_bad) lt0 = lt1 = kBadRecord;
    if (!crosses_ctas(cu, b, start, end)) {
      const float i0 = lt0 > 0.f ? us / lt0 : 0.f, i1 = lt1 > 0.f ? us / lt1 : 0.f;
      __half* ob = p.out + ((size_t)b * p.Hq + h * G) * D;
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const int d = 16 * i + 2 * r8;
        if (g0 < G)
          *reinterpret_cast<__half2*>(ob + g0 * D + d) = __floats2half2_rn(acc[i][0] * i0, acc[i][2] * i0);
        if (g1 < G)
          *reinterpret_cast<__half2*>(ob + g1 * D + d) = __floats2half2_rn(acc[i][1] * i1, acc[i][3] * i1);
      }
      if (r8 == 0 && p.lse) {
        float* lb = p.lse + (size_t)b * p.Hq + h * G;
        if (g0 < G) lb[g0] = lt0 > 0.f ? (m0 + log2f(lt0)) * 0.69314718055994531f : -INFINITY;
        if (g1 < G) lb[g1] = lt1 > 0.f ? (m1 + log2f(lt1)) * 0.69314718055994531f : -INFINITY;
      }
      continue;
    }
    const size_t R = (size_t)b + v;
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
  }
  finish_warp<D>(p, cu, start, end, per, b_first, b_last, h, merge_buf(ring, S::kBytes));
}

template <int D, int VMODE, int EL>
__global__ void __launch_bounds__(kThreads, 1)
decode_split_mma(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV8,
                 const __grid_constant__ CUtensorMap tmV16, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int warp_tot[kThreads / 32];
  uint8_t* smem = aligned_smem(smem_raw);
  int start, end, per, b_first, b_last;
  if (p.pdl) griddep_launch_dependents();          // the next call may take this SM when it frees
  if (!split_prologue(p, smem, warp_tot, start, end, per, b_first, b_last)) return;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmK);
    if (VMODE != kVFP16) tma_prefetch_desc(&tmV8);
    if (VMODE != kVE4M3) tma_prefetch_desc(&tmV16);
  }
  consume_mma<D, VMODE, EL>(p, &tmK, &tmV8, &tmV16, smem, start, end, b_first, b_last, per);
}

template <int D, int VMODE, int EL>
static cudaError_t launch_mma(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                              const DecodeParams& p, int grid, size_t smem, cudaStream_t st) {
  auto kern = decode_split_mma<D, VMODE, EL>;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  if (!p.pdl) {
    kern<<<grid, kThreads, smem, st>>>(tk, t8, t16, p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, t8, t16, p);
}

template <int D>
static cudaError_t launch_mma_d(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                                const DecodeParams& p, int vmode, int grid, size_t smem, cudaStream_t st) {
  if (p.elastic) {              // the elastic layout: the native FP16 path or the mixed one
    if (vmode == kVFP16) return launch_mma<D, kVFP16, kElYes>(tk, t8, t16, p, grid, smem, st);
    return launch_mma<D, kVMixed, kElYes>(tk, t8, t16, p, grid, smem, st);
  }
  if (vmode == kVE4M3) return launch_mma<D, kVE4M3, kElNo>(tk, t8, t16, p, grid, smem, st);
  if (vmode == kVFP16) return launch_mma<D, kVFP16, kElNo>(tk, t8, t16, p, grid, smem, st);
  return launch_mma<D, kVMixed, kElNo>(tk, t8, t16, p, grid, smem, st);
}

cudaError_t launch_split_mma(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                             const DecodeParams& p, int D, int vmode, int grid, size_t smem, cudaStream_t st) {
  return D == 128 ? launch_mma_d<128>(tk, t8, t16, p, vmode, grid, smem, st)
                  : launch_mma_d<64>(tk, t8, t16, p, vmode, grid, smem, st);
}

}  // namespace ekv
