// prefill_tc05.cu -- FP16 causal prefill over the gathered workspace on the fifth-
// generation tensor cores (tcgen05 MMA, tensor-memory accumulators, TMA loads).
//
// knlp.io "Asymmetric K16/V8 KV cache", "What changes in vLLM's prefill routing?": after
// the gather has cast the stored K16/V8 pages into the bounded FP16 workspace, a native
// FP16 prefill runs over it (FP16 query, key and value; causal; whole prompts, no cached
// prefix). Prompt i's queries are rows cu_seqlens[i] .. of q; its keys and values are
// workspace pages page_off[i], page_off[i] + 1, ... ([W][16][Hkv][D]).
//
// One CTA computes 256 query rows (two tiles of 128, the MMA's M) of one query head
// against the key/value blocks of 64 tokens of its KV head up to the diagonal:
//   warp 0       TMA producer: K and V blocks into a ring of NS stages, in the order the
//                MMA warp uses them (K0, K1, V0, K2, V1, K3, ...); zeroes the value rows
//                past the prompt in the last block, so that P = 0 never meets a NaN;
//   warp 1       MMA issuer (one thread): S_t,j = Q_t K_j^T (SS form, both K-major) into
//                tensor memory, O_t += P_t,j V_j (TS form: P from tensor memory, V
//                N-major in shared memory);
//   warp 2       allocates and frees the 512 tensor-memory columns;
//   warps 4..7   softmax of query tile 0, warps 8..11 of tile 1 (thread = query row):
//                load the tile's Q rows into shared memory, then per key block read S,
//                mask the diagonal, update the running max, write P = exp2(S' - m) as
//                fp16 over the first half of S's own columns, and at the end normalise
//                O and write out and lse.
// Tensor memory, tile t: S/P buffers (64 columns each, alternating by key block) at
// 256t and 256t + 64, O (D fp32 columns) at 256t + 128. The S of block j + 2 overwrites
// P of block j only after the MMA warp has seen O += P_j V_j complete. Every mbarrier is
// waited phase by phase (a parity wait is only defined within one phase of the barrier):
// the softmax warps see each O += P V of their tile before handing over the next P.
// The running max is re-based lazily: O and l are rescaled only when a row's max grows by
// more than 2^8 (the exponentials stay <= 256, exact to fp16's relative precision), so
// most blocks touch O not at all. l sums the fp32 exponentials.
// Every wait is bounded (1 s): a timeout is reported and every role winds down.
#include "common.cuh"
#include "pool_maps.h"
#include "prefill.cuh"
#include "tc05.cuh"

namespace ekv {

namespace {

constexpr int kQRows = 128;                 // rows of a query tile (MMA M)
constexpr int kKB = 64;                     // keys per K / V block
constexpr int kTThreads = 384;
constexpr float kRebase = 8.f;              // log2 growth of the max that forces a rescale

template <int D>
struct TcCfg {
  static constexpr int NB = D / 64;                  // 128-byte slabs of a row
  static constexpr int QB = kQRows * D * 2;          // bytes of a query tile
  static constexpr int IB = kKB * D * 2;             // bytes of a K or V block
  static constexpr int NS = D == 128 ? 10 : 16;      // ring stages
};

template <int NS>
struct TcBars {
  uint64_t q_full;               // 256 arrivals: both tiles' Q rows in shared memory
  uint64_t v_fixed;              // last value block with its rows past the prompt zeroed
  uint64_t mma_final;            // every MMA issued has completed
  uint64_t kv_full[NS];          // TMA bytes landed
  uint64_t kv_empty[NS];         // the MMAs reading the stage have completed
  uint64_t s_full[2][2];         // [tile][buffer]: S written
  uint64_t p_full[2][2];         // [tile][buffer]: P written, S read (128 arrivals)
  uint64_t pv_done[2];           // [tile]: O += P V of the block completed
  uint32_t tmem_base;
  int abort;
};

template <int D>
constexpr int tc_smem_bytes() {
  return 1024 + 2 * TcCfg<D>::QB + TcCfg<D>::NS * TcCfg<D>::IB + (int)sizeof(TcBars<TcCfg<D>::NS>);
}

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && (*abort || globaltimer_ns() - t0 > kWaitTimeoutNs)) return false;
  }
}

__device__ __forceinline__ void give_up(int* err, volatile int* abort) {
  if (!*abort) report_error(err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_TIMEOUT, -1);
  *abort = 1;
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kTThreads, 1)
prefill_tc05_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                    const PrefillParams p, int nqb) {
  using C = TcCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t sm_raw[];
  // ---- which 256 query rows: heavier query blocks first, then prompt, then query head
  const int HqN = p.Hq * p.n;
  const int qb = nqb - 1 - (int)(blockIdx.x / HqN);
  const int i = (int)(blockIdx.x % HqN) / p.Hq, hq = (int)(blockIdx.x % p.Hq);
  const int row0 = __ldg(p.cu_seqlens + i);
  const int len = __ldg(p.cu_seqlens + i + 1) - row0;
  if (qb == nqb - 1 && threadIdx.x == 0 && len > p.max_len)        // reported, rows cut there
    report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_SEQ_LEN, i);
  const int L = min(len, p.max_len);
  const int q0 = qb * 2 * kQRows;
  if (q0 >= L) return;
  const int h = hq / p.G;
  const int pg0 = __ldg(p.page_off + i);
  if (pg0 < 0 || pg0 + (L + kPage - 1) / kPage > p.num_ws_pages) {
    if (threadIdx.x == 0 && qb == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_ID, i);
    return;
  }
  // key blocks of 64 each tile needs: up to its last row's diagonal, and not past the prompt
  const int nkb = (L + kKB - 1) / kKB;
  const int nt0 = min(q0 / kKB + 2, nkb);
  const int nt1 = q0 + kQRows < L ? min(q0 / kKB + 4, nkb) : 0;
  const int n = max(nt0, nt1);
  const int zr = L - (n - 1) * kKB;          // value rows >= zr of the last block are zeroed

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;                                     // [2][NB][128 rows][128 B]
  uint8_t* sKV = base + 2 * C::QB;                        // [NS][NB][64 rows][128 B]
  TcBars<NS>* bars = reinterpret_cast<TcBars<NS>*>(sKV + NS * C::IB);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 2 * kQRows);
    mbar_init(&bars->v_fixed, 1);
    mbar_init(&bars->mma_final, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&bars->s_full[t][b], 1);
        mbar_init(&bars->p_full[t][b], kQRows);
      }
      mbar_init(&bars->pv_done[t], 1);
    }
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 2) tc05::tmem_alloc(&bars->tmem_base, 512);
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const int tok0 = pg0 * kPage;
    int u = 0;
    auto issue = [&](int is_v, int j) -> bool {
      const int s = u % NS;
      if (u >= NS) {
        bool ok = wait_bar(&bars->kv_empty[s], ((u / NS) - 1) & 1, abort);
        if (!__all_sync(0xffffffffu, ok)) return false;
      }
      uint8_t* dst = sKV + s * C::IB;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->kv_full[s], C::IB);
        tma_load_4d(dst, is_v ? &tv : &tk, 0, tok0 + j * kKB, 0, h, &bars->kv_full[s]);
      }
      if (is_v && j == n - 1 && zr < kKB) {
        bool ok = wait_bar(&bars->kv_full[s], (u / NS) & 1, abort);
        if (!__all_sync(0xffffffffu, ok)) return false;
        const int per_slab = (kKB - zr) * 8;               // 16-byte chunks past the prompt
        for (int e = lane; e < per_slab * C::NB; e += 32) {
          const int slab = e / per_slab, rem = e % per_slab;
          *reinterpret_cast<uint4*>(dst + slab * kKB * 128 + (zr + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->v_fixed);
      }
      ++u;
      return true;
    };
    bool ok = issue(0, 0);
    if (ok && n > 1) ok = issue(0, 1);
    for (int j = 0; ok && j < n; ++j) {
      ok = issue(1, j);
      if (ok && j + 2 < n) ok = issue(0, j + 2);
    }
    if (!ok && lane == 0) give_up(p.err, abort);
    // the copies still in flight land before the CTA can exit
    for (int v = u > NS ? u - NS : 0; v < u; ++v) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bars->kv_full[v % NS], (v / NS) & 1) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = tc05::idesc_f16_f32(kQRows, kKB, false);
      constexpr uint32_t idO = tc05::idesc_f16_f32(kQRows, D, true);
      const int nt[2] = {nt0, nt1};
      const uint32_t q_addr = smem_u32(sQ), kv_addr = smem_u32(sKV);
      int u = 0;
      bool ok = wait_bar(&bars->q_full, 0, abort);
      // wait for item u; returns its shared address (0 on a failed wait)
      auto take = [&](bool fixed) -> uint32_t {
        const int s = u % NS;
        const bool got = fixed ? wait_bar(&bars->v_fixed, 0, abort) : wait_bar(&bars->kv_full[s], (u / NS) & 1, abort);
        if (!got) return 0u;
        tc05::fence_after_sync();
        return kv_addr + s * C::IB;
      };
      auto release = [&]() { tc05::commit(&bars->kv_empty[u % NS]); ++u; };
      auto issue_s = [&](int t, int j, uint32_t kaddr) {
        const uint32_t d = tbase + t * 256 + (j & 1) * kKB;
        const uint32_t qa = q_addr + t * C::QB;
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc05::mma_ss(d, tc05::sdesc_sw128(qa + (k >> 2) * (kQRows * 128) + (k & 3) * 32, 16, 1024),
                       tc05::sdesc_sw128(kaddr + (k >> 2) * (kKB * 128) + (k & 3) * 32, 16, 1024), idS, k > 0);
        tc05::commit(&bars->s_full[t][j & 1]);
      };
      // prologue: S of key blocks 0 and 1 for both tiles
      for (int j = 0; ok && j < 2 && j < n; ++j) {
        const uint32_t ka = take(false);
        ok = ka != 0u;
        if (!ok) break;
        for (int t = 0; t < 2; ++t)
          if (j < nt[t]) issue_s(t, j, ka);
        release();
      }
      for (int j = 0; ok && j < n; ++j) {
        const uint32_t va = take(j == n - 1 && zr < kKB);
        ok = va != 0u;
        if (!ok) break;
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= nt[t]) continue;
          ok = wait_bar(&bars->p_full[t][j & 1], (j >> 1) & 1, abort);
          if (!ok) break;
          tc05::fence_after_sync();
          const uint32_t pa = tbase + t * 256 + (j & 1) * kKB;
#pragma unroll
          for (int k = 0; k < kKB / 16; ++k)
            tc05::mma_ts(tbase + t * 256 + 128, pa + 8 * k,
                         tc05::sdesc_sw128(va + k * 2048, kKB * 128, 1024), idO, j > 0 || k > 0);
          tc05::commit(&bars->pv_done[t]);
        }
        if (!ok) break;
        release();
        if (j + 2 < n) {
          const uint32_t ka = take(false);
          ok = ka != 0u;
          for (int t = 0; t < 2 && ok; ++t) {
            if (j + 2 >= nt[t]) continue;
            // P of block j (the buffer S of block j + 2 lands in) has been consumed
            ok = wait_bar(&bars->pv_done[t], j & 1, abort);
            if (ok) {
              tc05::fence_after_sync();
              issue_s(t, j + 2, ka);
            }
          }
          if (!ok) break;
          release();
        }
      }
      if (!ok) give_up(p.err, abort);
      tc05::commit(&bars->mma_final);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bars->mma_final, 0) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------- softmax, tile t
    const int t = (warp - 4) >> 2, r = threadIdx.x - 128 - t * kQRows;
    const uint32_t lanebase = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int prow = q0 + t * kQRows + r;                 // this thread's query position
    const int nmine = t == 0 ? nt0 : nt1;
    // Q row -> shared memory in the 128B-swizzled K-major layout (zeros past the prompt)
    {
      uint8_t* dst = sQ + t * C::QB + r * 128;
      const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)(row0 + prow) * p.Hq + hq) * D);
      const bool valid = nmine > 0 && prow < L;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(dst + (c >> 3) * (kQRows * 128) + (((c & 7) ^ (r & 7)) << 4)) = v;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&bars->q_full);
    }
    const float qs = p.qscale;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    const uint32_t t_o = tbase + t * 256 + 128 + lanebase;
    for (int j = 0; j < nmine; ++j) {
      const uint32_t t_s = tbase + t * 256 + (j & 1) * kKB + lanebase;
      ok = __all_sync(0xffffffffu, wait_bar(&bars->s_full[t][j & 1], (j >> 1) & 1, abort));
      if (!ok) break;
      tc05::fence_after_sync();
      float x[kKB];
      {
        uint32_t a[32], b[32];
        tc05::ld32(t_s, a);
        tc05::ld32(t_s + 32, b);
        tc05::wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(a[c]);
          x[32 + c] = __uint_as_float(b[c]);
        }
      }
      const int k0 = j * kKB;
      if (k0 + kKB - 1 > q0 + t * kQRows) {               // the block reaches past some row
#pragma unroll
        for (int c = 0; c < kKB; ++c)
          if (k0 + c > prow) x[c] = -INFINITY;
      }
      float mx = x[0];
#pragma unroll
      for (int c = 1; c < kKB; ++c) mx = fmaxf(mx, x[c]);
      const float m_new = fmaxf(m_ref, mx * qs);
      const bool need = m_new > m_ref + kRebase;
      // O += P V of block j - 1 is awaited once per block j >= 1 (here, or before P is
      // handed over): a parity wait is only defined while the barrier is at most one
      // phase away, so no pv_done phase may be skipped
      bool pv_seen = j == 0;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2f(m_ref - m_new) : 1.f;
        if (j > 0) {                                       // O holds blocks < j: rescale it
          ok = __all_sync(0xffffffffu, wait_bar(&bars->pv_done[t], (j - 1) & 1, abort));
          if (!ok) break;
          pv_seen = true;
          tc05::fence_after_sync();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tc05::ld32(t_o + 32 * c, o);
            tc05::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc05::st32(t_o + 32 * c, o);
          }
        }
        l *= alpha;
        if (need) m_ref = m_new;
      }
      const float nm = -m_ref;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2f(fmaf(x[2 * c], qs, nm)), p1 = ex2f(fmaf(x[2 * c + 1], qs, nm));
        l += p0 + p1;
        pk[c] = pack_half2(p0, p1);
      }
      tc05::st32(t_s, pk);
      tc05::wait_st();
      if (!pv_seen) {
        ok = __all_sync(0xffffffffu, wait_bar(&bars->pv_done[t], (j - 1) & 1, abort));
        if (!ok) break;
      }
      tc05::fence_before_sync();
      mbar_arrive(&bars->p_full[t][j & 1]);
    }
    if (!ok && lane == 0) give_up(p.err, abort);
    if (ok && nmine > 0) {
      ok = __all_sync(0xffffffffu, wait_bar(&bars->pv_done[t], (nmine - 1) & 1, abort));
      if (!ok && lane == 0) give_up(p.err, abort);
    }
    if (ok && nmine > 0) {
      tc05::fence_after_sync();
      const float inv = 1.f / l;
      __half* dst = p.out + ((size_t)(row0 + prow) * p.Hq + hq) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc05::ld32(t_o + 32 * c, o);
        tc05::wait_ld();
        if (prow < L) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 w;
            w.x = pack_half2(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
            w.y = pack_half2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
            w.z = pack_half2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
            w.w = pack_half2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + 32 * c + 8 * e) = w;
          }
        }
      }
      if (prow < L && p.lse) p.lse[(size_t)(row0 + prow) * p.Hq + hq] = (m_ref + log2f(l)) * 0.69314718055994531f;
    }
  }
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc05::fence_after_sync();
    tc05::tmem_free(tbase, 512);
  }
}

// 4-D view (d mod 64, token, d / 64, KV head) of the workspace [W][16][Hkv][D] fp16; the
// box {64, 64, D/64, 1} lands one key/value block as [D/64][64 rows][128 B], 128B swizzle.
static bool encode_ws_map(CUtensorMap* tm, const void* base, int D, int Hkv, int num_pages) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {64, (cuuint64_t)num_pages * kPage, (cuuint64_t)(D / 64), (cuuint64_t)Hkv};
  cuuint64_t strides[3] = {(cuuint64_t)Hkv * D * 2, 128, (cuuint64_t)D * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)kKB, (cuuint32_t)(D / 64), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t set_smem_attr(const void* kern, int bytes);

template <int D>
static cudaError_t launch_tc05_d(const PrefillParams& p, int max_len, cudaStream_t st) {
  CUtensorMap tk, tv;
  if (!encode_ws_map(&tk, p.ws_k, D, p.Hkv, p.num_ws_pages) || !encode_ws_map(&tv, p.ws_v, D, p.Hkv, p.num_ws_pages))
    return cudaErrorInvalidValue;
  const int smem = tc_smem_bytes<D>();
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(prefill_tc05_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  const int nqb = (max_len + 2 * kQRows - 1) / (2 * kQRows);
  const long long grid = (long long)nqb * p.Hq * p.n;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  prefill_tc05_kernel<D><<<(unsigned)grid, kTThreads, smem, st>>>(tk, tv, p, nqb);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tc05(const PrefillParams& p, int D, int max_len, cudaStream_t st) {
  if (p.n <= 0 || max_len <= 0) return cudaSuccess;
  return D == 128 ? launch_tc05_d<128>(p, max_len, st) : launch_tc05_d<64>(p, max_len, st);
}

}  // namespace ekv
