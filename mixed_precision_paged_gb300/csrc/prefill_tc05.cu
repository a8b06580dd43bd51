// prefill_tc05.cu -- FP16 causal prefill over the gathered workspace on the fifth-
// generation tensor cores (tcgen05 MMA, tensor-memory accumulators, TMA loads).
//
// knlp.io "Asymmetric K16/V8 KV cache", "What changes in vLLM's prefill routing?": after
// the gather has cast the stored K16/V8 pages into the bounded FP16 workspace, a native
// FP16 prefill runs over it (FP16 query, key and value; causal; whole prompts, no cached
// prefix). Prompt i's queries are rows cu_seqlens[i] .. of q; its keys and values are
// workspace pages page_off[i], page_off[i] + 1, ... ([W][16][Hkv][D]).
//
// Work item = 256 query rows (two tiles of 128, the MMA's M) of one query head against
// the key/value blocks of 128 tokens of its KV head up to the diagonal. The kernel is
// persistent: one CTA per SM takes the items in a fixed order (heavier query blocks
// first, dealt in a snake over the CTAs), keeps its barriers and tensor memory across
// them, and overlaps one item's epilogue with the next item's loads and first S.
//   warp 0       TMA producer: per item, each active query tile once the tile's previous
//                rows have been read by their last S (one box when the 128 rows end inside
//                q; else rows by plain loads, zeros past the prompt), then K and V blocks
//                into a ring of NS stages in the order the MMA warp uses them (K0, V0,
//                K1, V1, ...); zeroes the value rows past the prompt in an item's last
//                block, so that P = 0 never meets a NaN;
//   warp 1       MMA issuer (one thread): S_t = Q_t K_j^T (SS form, both K-major) and
//                O_t += P_t V_j (TS form: P from tensor memory, V N-major in shared
//                memory), tiles interleaved so that one tile's softmax overlaps the other
//                tile's MMAs; an item's first O_t += P V waits until the softmax has read
//                the previous item's O_t out;
//   warp 2       allocates and frees the 512 tensor-memory columns;
//   warps 4..7   softmax of query tile 0, warps 8..11 of tile 1 (thread = query row):
//                per key block read S (a max pass and an exponential pass over 32-column
//                chunks), mask the diagonal block, update the running max, write
//                P = exp2(S' - m) as fp16 over the first half of S's columns, and at the
//                end of an item normalise O and write out and lse.
// Tensor memory, tile t: S/P at 256t (128 columns), O at 256t + 128 (D fp32 columns).
// The MMA warp issues S of block j + 1 over P of block j right behind O += P_j V_j (the
// tensor core runs one thread's MMAs in issue order, so P_j is read before S_{j+1}
// overwrites it); the commit that signals S_{j+1} arrives only when every earlier MMA,
// O += P_j V_j included, has completed, so the softmax of block j + 1 may rescale O at
// any time before it hands over P.
// The instruction stream of the MMA warp is the scarce resource: one tcgen05.mma or
// tcgen05.commit issues every ~45 cycles per SM whatever its size, so the MMAs are the
// largest the tensor memory allows (N = 128 for S, N = D for O) and their descriptors are
// one 32-bit add from a precomputed base.
// The running max is re-based lazily: O and l are rescaled only when a row's max grows by
// more than 2^8 (the exponentials stay <= 256, exact to fp16's relative precision), so
// most blocks touch O not at all. l sums the fp32 exponentials. The softmax is bound by
// its instruction count, so the causal mask is a separate instance of each pass, run only
// on the diagonal block.
// Every mbarrier is waited phase by phase (a parity wait is only defined within one phase
// of the barrier); every wait is bounded (1 s): a timeout is reported and every role
// winds down.
#include "common.cuh"
#include "pool_maps.h"
#include "prefill.cuh"
#include "tc05.cuh"

namespace ekv {

namespace {

constexpr int kQRows = 128;                 // rows of a query tile (MMA M)
constexpr int kKB = 128;                    // keys per K / V block (S's N)
constexpr int kTThreads = 384;
constexpr float kRebase = 8.f;              // log2 growth of the max that forces a rescale

template <int D>
struct TcCfg {
  static constexpr int NB = D / 64;                  // 128-byte slabs of a row
  static constexpr int QB = kQRows * D * 2;          // bytes of a query tile
  static constexpr int IB = kKB * D * 2;             // bytes of a K or V block
  static constexpr int NS = D == 128 ? 5 : 12;       // ring stages
};

template <int NS>
struct TcBars {
  uint64_t q_full[2];            // [tile]: the tile's query rows of its next work item landed
  uint64_t q_empty[2];           // [tile]: an item's last S has read the tile's query rows
  uint64_t v_raw;                // a last value block reaching past its prompt landed (producer)
  uint64_t mma_final;            // every MMA issued has completed
  uint64_t kv_full[NS];          // TMA bytes landed (a last value block: and its tail zeroed)
  uint64_t kv_empty[NS];         // the MMAs reading the stage have completed
  uint64_t s_full[2];            // [tile]: S of the next block written
  uint64_t p_full[2];            // [tile]: P written, S read (one arrival per softmax warp)
  uint64_t pv_done[2];           // [tile]: a work item's last O += P V completed
  uint64_t o_free[2];            // [tile]: an item's O read out (one arrival per softmax warp)
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

// max of three (one instruction on sm_100+)
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (d0, d1) = (a0, a1) * (b0, b1) + (c0, c1), one packed FP32 instruction
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// (a0, a1) += (b0, b1), one packed FP32 instruction
__device__ __forceinline__ void fadd2(float& a0, float& a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb;\n\t"
      "mov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\t"
      "add.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Warp-wide store of 16 columns (thread t: lane base + t).
__device__ __forceinline__ void tst16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Warp-wide load of 16 columns (thread t: lane base + t).
__device__ __forceinline__ void tld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// The S row of one 128-key block, read from tensor memory into registers once: with
// MASK, keys k0 + col after the query prow become -inf. Returns the row max (raw score).
template <bool MASK>
__device__ __forceinline__ float row_in_regs(uint32_t t_s, int k0, int prow, uint32_t (&a)[4][32]) {
  tc05::ld32(t_s, a[0]);
  tc05::ld32(t_s + 32, a[1]);
  tc05::ld32(t_s + 64, a[2]);
  tc05::ld32(t_s + 96, a[3]);
  tc05::wait_ld();
  float mg[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (MASK) {
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (k0 + 32 * c + e > prow) a[c][e] = __float_as_uint(-INFINITY);
    }
    float m8[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t* y = a[c] + 8 * g;
      m8[g] = fmaxf(max3f(max3f(__uint_as_float(y[0]), __uint_as_float(y[1]), __uint_as_float(y[2])),
                          __uint_as_float(y[3]), __uint_as_float(y[4])),
                    max3f(__uint_as_float(y[5]), __uint_as_float(y[6]), __uint_as_float(y[7])));
    }
    mg[c] = max3f(m8[0], m8[1], fmaxf(m8[2], m8[3]));
  }
  return max3f(mg[0], mg[1], fmaxf(mg[2], mg[3]));
}

// P = exp2(S * qs + nm) of the row held in registers, as fp16 pairs over the first 64
// tensor-memory columns of the block (S is no longer read there); returns the sum of the
// fp32 exponentials.
__device__ __forceinline__ float row_exp_store(uint32_t t_s, float qs, float nm, uint32_t (&a)[4][32]) {
  float la[4] = {0.f, 0.f, 0.f, 0.f}, lb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float a0, a1;
      ffma2(a0, a1, __uint_as_float(a[c][2 * e]), __uint_as_float(a[c][2 * e + 1]), qs, qs, nm, nm);
      const float p0 = ex2f(a0), p1 = ex2f(a1);
      fadd2(la[e & 3], lb[e & 3], p0, p1);
      a[c][e] = pack_half2(p0, p1);                 // a[c][2e], a[c][2e + 1] already read
    }
    tst16(t_s + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(&a[c][0]));
  }
  fadd2(la[0], lb[0], la[2], lb[2]);
  fadd2(la[1], lb[1], la[3], lb[3]);
  return (la[0] + la[1]) + (lb[0] + lb[1]);
}

}  // namespace

// One work item: 256 query rows (two tiles of 128) of one query head of one prompt.
struct WorkItem {
  int row0, L, q0, hq, h, pg0;
  int nt0, nt1, n;     // key blocks of tile 0 / tile 1 / either
  int zr;              // value rows >= zr of the last block lie past the prompt
  bool valid;
};

// Work item w: heavier query blocks first (w / (Hq n) counts the query blocks down), then
// prompt, then query head. Every role of a CTA computes the same items; with `report` the
// prompt's errors are recorded (once per prompt: at its last / first query block).
__device__ __forceinline__ WorkItem work_item(const PrefillParams& p, int nqb, int w, bool report) {
  WorkItem it;
  const int HqN = p.Hq * p.n;
  const int qb = nqb - 1 - w / HqN;
  const int i = (w % HqN) / p.Hq;
  it.hq = w % p.Hq;
  it.row0 = __ldg(p.cu_seqlens + i);
  const int len = __ldg(p.cu_seqlens + i + 1) - it.row0;
  if (report && qb == nqb - 1 && len > p.max_len)              // reported, rows cut there
    report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_SEQ_LEN, i);
  it.L = min(len, p.max_len);
  it.q0 = qb * 2 * kQRows;
  it.h = it.hq / p.G;
  it.pg0 = __ldg(p.page_off + i);
  it.valid = it.q0 < it.L;
  if (it.valid && (it.pg0 < 0 || it.pg0 + (it.L + kPage - 1) / kPage > p.num_ws_pages)) {
    if (report && qb == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_ID, i);
    it.valid = false;
  }
  // key blocks each tile needs: up to its own (diagonal) block, and not past the prompt
  const int nkb = (it.L + kKB - 1) / kKB;
  it.nt0 = min(it.q0 / kKB + 1, nkb);
  it.nt1 = it.q0 + kQRows < it.L ? min(it.q0 / kKB + 2, nkb) : 0;
  it.n = max(it.nt0, it.nt1);
  it.zr = it.L - (it.n - 1) * kKB;
  return it;
}

// The r-th work item of this CTA: items are dealt in rounds of gridDim.x, alternately
// forwards and backwards (a snake), which balances a list sorted from heavy to light about
// as well as greedy assignment. An index >= the item count means no r-th item.
__device__ __forceinline__ int item_index(int r) {
  const int g = (int)gridDim.x, c = (int)blockIdx.x;
  return r * g + ((r & 1) ? g - 1 - c : c);
}

template <int D>
__global__ void __launch_bounds__(kTThreads, 1)
prefill_tc05_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tq, const PrefillParams p, int nqb) {
  using C = TcCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t sm_raw[];
  const int W = nqb * p.Hq * p.n;                         // work items
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;                                     // [2][NB][128 rows][128 B]
  uint8_t* sKV = base + 2 * C::QB;                        // [NS][NB][128 rows][128 B]
  TcBars<NS>* bars = reinterpret_cast<TcBars<NS>*>(sKV + NS * C::IB);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->q_empty[t], 1);
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], kQRows / 32);
      mbar_init(&bars->pv_done[t], 1);
      mbar_init(&bars->o_free[t], kQRows / 32);
    }
    mbar_init(&bars->v_raw, 1);
    mbar_init(&bars->mma_final, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
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
    const int T = __ldg(p.cu_seqlens + p.n);               // rows of q
    int stage = 0, u = 0;
    uint32_t phase = 0, rawc = 0;
    uint32_t ql[2] = {0u, 0u};                             // query tiles loaded, per tile
    bool ok = true;
    for (int r = 0; ok && item_index(r) < W; ++r) {
      const WorkItem it = work_item(p, nqb, item_index(r), lane == 0);
      if (!it.valid) continue;
      // The item's query tiles, each once the tile's previous rows have been read by their
      // last S. One TMA box when the 128 rows end inside q (rows past the prompt then
      // belong to the next prompt: they are computed, never stored); else rows by plain
      // loads with zeros past the prompt.
      for (int t = 0; t < 2 && ok; ++t) {
        if ((t == 0 ? it.nt0 : it.nt1) == 0) continue;
        if (ql[t] > 0) {
          ok = __all_sync(0xffffffffu, wait_bar(&bars->q_empty[t], (ql[t] - 1u) & 1u, abort));
          if (!ok) break;
        }
        const int rq = it.row0 + it.q0 + t * kQRows;
        uint8_t* dq = sQ + t * C::QB;
        if (rq + kQRows <= T) {
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars->q_full[t], C::QB);
            tma_load_4d(dq, &tq, 0, rq, 0, it.hq, &bars->q_full[t]);
          }
        } else {
          for (int e = lane; e < kQRows * (D / 8); e += 32) {
            const int rr = e / (D / 8), c = e % (D / 8);
            const bool valid = it.q0 + t * kQRows + rr < it.L;
            const uint4 v = valid ? __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)(rq + rr) * p.Hq + it.hq) * D) + c)
                                  : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(dq + (c >> 3) * (kQRows * 128) + rr * 128 + (((c & 7) ^ (rr & 7)) << 4)) = v;
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->q_full[t]);
        }
        ++ql[t];
      }
      if (!ok) break;
      const int tok0 = it.pg0 * kPage;
      for (int j = 0; ok && j < it.n; ++j) {
        for (int is_v = 0; is_v < 2; ++is_v) {
          if (u >= NS) {                                    // the stage's previous item consumed
            ok = __all_sync(0xffffffffu, wait_bar(&bars->kv_empty[stage], phase ^ 1u, abort));
            if (!ok) break;
          }
          uint8_t* dst = sKV + stage * C::IB;
          if (is_v && j == it.n - 1 && it.zr < kKB) {
            // the last value block reaches past the prompt: it lands on v_raw, its rows past
            // the prompt are zeroed (so that P = 0 never meets a NaN), then the stage is
            // published on kv_full by a plain arrival
            if (lane == 0) {
              mbar_arrive_expect_tx(&bars->v_raw, C::IB);
              tma_load_4d(dst, &tv, 0, tok0 + j * kKB, 0, it.h, &bars->v_raw);
            }
            ok = __all_sync(0xffffffffu, wait_bar(&bars->v_raw, rawc & 1u, abort));
            ++rawc;
            if (!ok) break;
            const int per_slab = (kKB - it.zr) * 8;         // 16-byte chunks past the prompt
            for (int e = lane; e < per_slab * C::NB; e += 32) {
              const int slab = e / per_slab, rem = e % per_slab;
              *reinterpret_cast<uint4*>(dst + slab * kKB * 128 + (it.zr + rem / 8) * 128 + (rem % 8) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->kv_full[stage]);
          } else if (lane == 0) {
            mbar_arrive_expect_tx(&bars->kv_full[stage], C::IB);
            tma_load_4d(dst, is_v ? &tv : &tk, 0, tok0 + j * kKB, 0, it.h, &bars->kv_full[stage]);
          }
          ++u;
          if (++stage == NS) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    if (!ok && lane == 0) give_up(p.err, abort);
    // the copies still in flight land before the CTA can exit
    for (int v = u > NS ? u - NS : 0; v < u; ++v) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bars->kv_full[v % NS], (v / NS) & 1) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
    for (int t = 0; t < 2; ++t) {
      if (ql[t] == 0) continue;
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bars->q_full[t], (ql[t] - 1u) & 1u) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    // The whole warp runs the control flow and computes the descriptors (warp-uniform
    // values); one elected lane issues each group of MMAs and commits.
    constexpr uint32_t idS = tc05::idesc_f16_f32(kQRows, kKB, false);
    constexpr uint32_t idO = tc05::idesc_f16_f32(kQRows, D, true);
    constexpr uint32_t HI = tc05::sdesc_hi(1024);          // 8-row groups 1024 B apart
    // descriptor low words: Q tile 0, K-major and V (N-major) views of ring stage 0
    const uint32_t q_lo = tc05::sdesc_lo(smem_u32(sQ), 16);
    const uint32_t k_lo = tc05::sdesc_lo(smem_u32(sKV), 16);
    const uint32_t v_lo = tc05::sdesc_lo(smem_u32(sKV), kKB * 128);
    // ring cursors of the K items (2j) and the V items (2j + 1) of each work item
    int ks = 0, vs = 1;
    uint32_t kp = 0, vp = 0;
    // phases taken so far: q_full[t], p_full[t]; items with an O of tile t (o_free phases)
    uint32_t qc[2] = {0u, 0u}, pc[2] = {0u, 0u}, oc[2] = {0u, 0u};
    auto adv2 = [&](int& s, uint32_t& ph) {
      s += 2;
      if (s >= NS) {
        s -= NS;
        ph ^= 1u;
      }
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_bar(bar, parity, abort));
    };
    auto issue_s = [&](int t) {                            // S_t = Q_t K^T from stage ks
      const uint32_t qa = q_lo + t * (C::QB >> 4), ka = k_lo + ks * (C::IB >> 4);
      const uint32_t d = tbase + t * 256;
      if (tc05::elect_one()) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc05::mma_ss(d, tc05::sdesc_join(qa + (((k >> 2) * (kQRows * 128) + (k & 3) * 32) >> 4), HI),
                       tc05::sdesc_join(ka + (((k >> 2) * (kKB * 128) + (k & 3) * 32) >> 4), HI), idS, k > 0);
        tc05::commit(&bars->s_full[t]);
      }
      __syncwarp();
    };
    auto commit_one = [&](uint64_t* bar) {
      if (tc05::elect_one()) tc05::commit(bar);
      __syncwarp();
    };
    bool ok = true;
    for (int r = 0; ok && item_index(r) < W; ++r) {
      const WorkItem it = work_item(p, nqb, item_index(r), false);
      if (!it.valid) continue;
      const int nt[2] = {it.nt0, it.nt1}, n = it.n;
      ok = wait_all(&bars->kv_full[ks], kp);
      // S of the first block for each active tile, once its query rows are in. The tile's
      // S columns hold the previous item's last P until its O += P V, issued before, has
      // read it (one thread's MMAs run in issue order).
      for (int t = 0; t < 2 && ok; ++t) {
        if (nt[t] == 0) continue;
        ok = wait_all(&bars->q_full[t], qc[t] & 1u);
        ++qc[t];
        if (!ok) break;
        tc05::fence_after_sync();
        issue_s(t);
        if (nt[t] == 1) commit_one(&bars->q_empty[t]);    // the tile's last S of the item
      }
      if (!ok) break;
      commit_one(&bars->kv_empty[ks]);
      adv2(ks, kp);
      for (int j = 0; ok && j < n; ++j) {
        ok = wait_all(&bars->kv_full[vs], vp);
        if (!ok) break;
        tc05::fence_after_sync();
        const uint32_t va = v_lo + vs * (C::IB >> 4);
        bool k_ready = false;
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= nt[t]) continue;
          // O_t += P_t V_j once the softmax has written P (and, for the first block, once
          // the previous item's O_t has been read out: this product overwrites it)
          ok = wait_all(&bars->p_full[t], pc[t] & 1u);
          ++pc[t];
          if (ok && j == 0 && oc[t] > 0) ok = wait_all(&bars->o_free[t], (oc[t] - 1u) & 1u);
          if (!ok) break;
          tc05::fence_after_sync();
          const uint32_t pa = tbase + t * 256, od = tbase + t * 256 + 128;
          const bool acc0 = j > 0;
          if (tc05::elect_one()) {
#pragma unroll
            for (int k = 0; k < kKB / 16; ++k)
              tc05::mma_ts(od, pa + 8 * k, tc05::sdesc_join(va + k * (2048 >> 4), HI), idO, acc0 || k > 0);
            if (j + 1 == nt[t]) tc05::commit(&bars->pv_done[t]);   // the item's last O_t += P V
          }
          __syncwarp();
          if (j + 1 < nt[t]) {
            // S_t of block j + 1 overwrites P_t. It is issued at once, behind O_t += P_t V_j:
            // the tensor core runs the MMAs of this thread in issue order, so P_t is read
            // before it is overwritten, and the commit after S_t (s_full) arrives only
            // once every MMA issued before it, O_t += P_t V_j included, has completed.
            ok = k_ready || wait_all(&bars->kv_full[ks], kp);
            if (!ok) break;
            k_ready = true;
            tc05::fence_after_sync();
            issue_s(t);
            if (j + 2 == nt[t]) commit_one(&bars->q_empty[t]);   // the tile's last S of the item
          }
        }
        if (!ok) break;
        commit_one(&bars->kv_empty[vs]);
        adv2(vs, vp);
        if (j + 1 < n) {
          commit_one(&bars->kv_empty[ks]);
          adv2(ks, kp);
        }
      }
      for (int t = 0; t < 2; ++t)
        if (nt[t] > 0) ++oc[t];
    }
    if (!ok && lane == 0) give_up(p.err, abort);
    commit_one(&bars->mma_final);
    if (lane == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bars->mma_final, 0) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------- softmax, tile t
    const int t = (warp - 4) >> 2, r = threadIdx.x - 128 - t * kQRows;
    const uint32_t lanebase = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float qs = p.qscale;
    const uint32_t t_s = tbase + t * 256 + lanebase, t_o = tbase + t * 256 + 128 + lanebase;
    uint32_t sc = 0, pvc = 0;                              // phases taken: s_full, pv_done
    bool ok = true;
    for (int ri = 0; ok && item_index(ri) < W; ++ri) {
      const WorkItem it = work_item(p, nqb, item_index(ri), false);
      const int nmine = !it.valid ? 0 : (t == 0 ? it.nt0 : it.nt1);
      if (nmine == 0) continue;
      const int prow = it.q0 + t * kQRows + r;             // this thread's query position
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < nmine; ++j) {
        // S of block j is ready; O += P V of block j - 1 has completed too (the commit that
        // signals S was issued after it)
        ok = __all_sync(0xffffffffu, wait_bar(&bars->s_full[t], sc & 1u, abort));
        ++sc;
        if (!ok) break;
        tc05::fence_after_sync();
        const int k0 = j * kKB;
        const bool diag = k0 + kKB - 1 > it.q0 + t * kQRows;   // the block reaches past some row
        uint32_t sv[4][32];
        const float mx = diag ? row_in_regs<true>(t_s, k0, prow, sv) : row_in_regs<false>(t_s, k0, prow, sv);
        const float m_new = fmaxf(m_ref, mx * qs);
        const bool need = m_new > m_ref + kRebase;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2f(m_ref - m_new) : 1.f;
          // O holds blocks < j, all complete (S of this block was committed after them)
          if (j > 0) {
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {
              uint32_t o[16];
              tld16(t_o + 16 * c, o);
              tc05::wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tst16(t_o + 16 * c, o);
            }
          }
          l *= alpha;
          if (need) m_ref = m_new;
        }
        l += row_exp_store(t_s, qs, -m_ref, sv);
        tc05::wait_st();
        tc05::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[t]);      // one arrival per warp
      }
      if (!ok) break;
      // the item's last O += P V (its commit covers every earlier MMA)
      ok = __all_sync(0xffffffffu, wait_bar(&bars->pv_done[t], pvc & 1u, abort));
      ++pvc;
      if (!ok) break;
      tc05::fence_after_sync();
      const float inv = 1.f / l;
      __half* dst = p.out + ((size_t)(it.row0 + prow) * p.Hq + it.hq) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc05::ld32(t_o + 32 * c, o);
        tc05::wait_ld();
        if (c == D / 32 - 1) {                             // O read out: the next item may overwrite it
          tc05::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->o_free[t]);
        }
        if (prow < it.L) {
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
      if (prow < it.L && p.lse)
        p.lse[(size_t)(it.row0 + prow) * p.Hq + it.hq] = (m_ref + log2f(l)) * 0.69314718055994531f;
    }
    if (!ok && lane == 0) give_up(p.err, abort);
  }
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc05::fence_after_sync();
    tc05::tmem_free(tbase, 512);
  }
}

// 4-D view (d mod 64, row, d / 64, head) of an fp16 [rows][heads][D] array; the box
// {64, 128, D/64, 1} lands 128 rows of one head as [D/64][128 rows][128 B], 128B swizzle:
// a key/value block of the workspace ([W][16][Hkv][D], rows = W * 16) or a query tile.
static bool encode_rows_map(CUtensorMap* tm, const void* base, int D, int heads, cuuint64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {64, rows, (cuuint64_t)(D / 64), (cuuint64_t)heads};
  cuuint64_t strides[3] = {(cuuint64_t)heads * D * 2, 128, (cuuint64_t)D * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)kKB, (cuuint32_t)(D / 64), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t set_smem_attr(const void* kern, int bytes);

template <int D>
static cudaError_t launch_tc05_d(const PrefillParams& p, int max_len, cudaStream_t st) {
  CUtensorMap tk, tv, tq;
  const cuuint64_t ws_rows = (cuuint64_t)p.num_ws_pages * kPage;
  // The query rows: the host does not know T = cu_seqlens[n], so the map spans every row
  // index a prompt can have (the device checks bound the boxes: a box is issued only for
  // 128 rows inside one prompt, so it never reads past q's T rows).
  const cuuint64_t q_rows = 0x7fffffffull;
  if (!encode_rows_map(&tk, p.ws_k, D, p.Hkv, ws_rows) || !encode_rows_map(&tv, p.ws_v, D, p.Hkv, ws_rows) ||
      !encode_rows_map(&tq, p.q, D, p.Hq, q_rows))
    return cudaErrorInvalidValue;
  const int smem = tc_smem_bytes<D>();
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(prefill_tc05_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  const int nqb = (max_len + 2 * kQRows - 1) / (2 * kQRows);
  const long long items = (long long)nqb * p.Hq * p.n;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = (int)(items < sms ? items : sms);        // persistent: one CTA per SM
  prefill_tc05_kernel<D><<<grid, kTThreads, smem, st>>>(tk, tv, tq, p, nqb);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tc05(const PrefillParams& p, int D, int max_len, cudaStream_t st) {
  if (p.n <= 0 || max_len <= 0) return cudaSuccess;
  return D == 128 ? launch_tc05_d<128>(p, max_len, st) : launch_tc05_d<64>(p, max_len, st);
}

}  // namespace ekv
