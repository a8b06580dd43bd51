// prefill_mma.cu -- FP16 causal prefill of whole prompts over the gathered workspace.
//
// knlp.io "Asymmetric K16/V8 KV cache", "What changes in vLLM's prefill routing?": after
// the gather has cast the stored K16/V8 pages into the bounded FP16 workspace, a native
// FP16 prefill runs over it (FP16 query, key and value; causal; whole prompts, no cached
// prefix). Prompt i owns workspace pages page_off[i], page_off[i] + 1, ... in the
// gather's [W][16][H_kv][D] layout; its queries are rows cu_seqlens[i] .. of q.
//
// Flash-attention form on mma.sync.m16n8k16 (f16 x f16 -> f32): a CTA takes 64 query
// rows of one query head (4 warps x 16 rows) and walks the KV head's key/value blocks
// of 64 tokens up to the diagonal. K and V tiles are staged in shared memory by 16-byte
// cp.async copies (double-buffered, the 16-byte chunks XOR-swizzled by row so that
// ldmatrix over 8 rows is bank-conflict free; tokens past the prompt are zero-filled).
// S = Q K^T with Q fragments held in registers and K^T fragments by ldmatrix; online
// softmax in the log2 domain; the f16-rounded P goes straight from the S accumulators
// into the A fragments of O += P V (V fragments by ldmatrix.trans); l accumulates the
// rounded P. CTAs with more work (later query blocks) are launched first.
#include "common.cuh"
#include "prefill.cuh"

namespace ekv {

namespace {

constexpr int kBM = 64;        // query rows per CTA
constexpr int kBN = 64;        // keys per block
constexpr int kPThreads = 128;

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 16-byte copy global -> shared, zero-filled when `valid` is false (no bytes read)
__device__ __forceinline__ void cp16z(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16 : 0)
               : "memory");
}

// byte offset of (row, 16-byte chunk c) in a tile of rows of D fp16, chunks XOR-swizzled
template <int D>
__device__ __forceinline__ uint32_t tile_off(int row, int c) {
  return (uint32_t)(row * D * 2 + ((c ^ (row & 7)) << 4));
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kPThreads)
prefill_kernel(const PrefillParams p) {
  constexpr int KS = D / 16;                   // k-steps of QK
  constexpr int NT = D / 8;                    // n-tiles of O
  constexpr int CPR = D / 8;                   // 16-byte chunks per row
  constexpr int kTile = kBN * D * 2;           // bytes of one K or V tile
  extern __shared__ __align__(128) uint8_t sm[];
  const int i = blockIdx.z, hq = blockIdx.y;
  const int row0 = __ldg(p.cu_seqlens + i);
  const int len = __ldg(p.cu_seqlens + i + 1) - row0;
  const int q0 = ((int)gridDim.x - 1 - (int)blockIdx.x) * kBM;   // heavier blocks first
  if (blockIdx.x == 0 && threadIdx.x == 0 && len > p.max_len)     // reported, rows cut there
    report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_SEQ_LEN, i);
  const int L = min(len, p.max_len);
  if (q0 >= L) return;
  const int h = hq / p.G;
  const int pg0 = __ldg(p.page_off + i);
  const int npages = (L + kPage - 1) / kPage;
  if (pg0 < 0 || pg0 + npages > p.num_ws_pages) {
    if (threadIdx.x == 0 && q0 == 0) report_error(p.err, EKV_ERR_DEVICE_CHECK, EKV_DETAIL_PAGE_ID, i);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, qd = lane & 3;
  const uint32_t sbase = smem_u32(sm);          // [buf][K tile | V tile]

  // K/V tile j -> buffer b: 64 rows x CPR chunks for K and for V, 2 * CPR / 2 per thread
  auto load_tile = [&](int j, int b) {
    const uint32_t kdst = sbase + b * 2 * kTile, vdst = kdst + kTile;
#pragma unroll
    for (int u = 0; u < kBN * CPR / kPThreads; ++u) {
      const int e = tid + u * kPThreads;
      const int row = e / CPR, c = e % CPR;
      const int t = j * kBN + row;
      const bool ok = t < L;
      const size_t src = ok ? (((size_t)(pg0 + t / kPage) * kPage + (t % kPage)) * p.Hkv + h) * D + c * 8 : 0;
      cp16z(kdst + tile_off<D>(row, c), p.ws_k + src, ok);
      cp16z(vdst + tile_off<D>(row, c), p.ws_v + src, ok);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  const int nblk = (min(q0 + kBM, L) + kBN - 1) / kBN;
  load_tile(0, 0);

  // Q fragments of this warp's 16 rows (rows past the prompt read row 0: never written)
  const int qa_row = q0 + warp * 16 + r, qb_row = qa_row + 8;
  const __half* qr0 = p.q + ((size_t)(row0 + (qa_row < L ? qa_row : 0)) * p.Hq + hq) * D;
  const __half* qr1 = p.q + ((size_t)(row0 + (qb_row < L ? qb_row : 0)) * p.Hq + hq) * D;
  uint32_t qf[KS][4];
#pragma unroll
  for (int s = 0; s < KS; ++s) {
    qf[s][0] = __ldg(reinterpret_cast<const uint32_t*>(qr0 + 16 * s + 2 * qd));
    qf[s][1] = __ldg(reinterpret_cast<const uint32_t*>(qr1 + 16 * s + 2 * qd));
    qf[s][2] = __ldg(reinterpret_cast<const uint32_t*>(qr0 + 16 * s + 8 + 2 * qd));
    qf[s][3] = __ldg(reinterpret_cast<const uint32_t*>(qr1 + 16 * s + 8 + 2 * qd));
  }
  float o[NT][4];
#pragma unroll
  for (int x = 0; x < NT; ++x) o[x][0] = o[x][1] = o[x][2] = o[x][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  // ldmatrix lane roles
  const int lm_mat = lane >> 3, lm_row = lane & 7;

  for (int j = 0; j < nblk; ++j) {
    if (j + 1 < nblk) {
      load_tile(j + 1, (j + 1) & 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const uint32_t kt = sbase + (j & 1) * 2 * kTile, vt = kt + kTile;
    // ---- S = Q K^T: 8 n-tiles of 8 keys, KS k-steps
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ks += 2) {
        uint32_t b0, b1, b2, b3;                 // k-steps ks and ks + 1 of n-tile nt
        ldsm4(kt + tile_off<D>(nt * 8 + lm_row, 2 * ks + lm_mat), b0, b1, b2, b3);
        mma16816(s[nt], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
        mma16816(s[nt], qf[ks + 1][0], qf[ks + 1][1], qf[ks + 1][2], qf[ks + 1][3], b2, b3);
      }
    }
    // ---- scale, causal mask (keys after the query, or past the prompt), online softmax
    const bool diag = j * kBN + kBN - 1 > q0 + warp * 16;   // some key may follow some row
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int key = j * kBN + nt * 8 + 2 * qd;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v0 = s[nt][e] * p.qscale, v1 = s[nt][2 + e] * p.qscale;
        if (diag) {
          if (key + e > qa_row) v0 = -INFINITY;
          if (key + e > qb_row) v1 = -INFINITY;
        }
        s[nt][e] = v0;
        s[nt][2 + e] = v1;
        mx0 = fmaxf(mx0, v0);
        mx1 = fmaxf(mx1, v1);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = ex2f(m0 - mn0), al1 = ex2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    l0 *= al0;
    l1 *= al1;
#pragma unroll
    for (int x = 0; x < NT; ++x) {
      o[x][0] *= al0;
      o[x][1] *= al0;
      o[x][2] *= al1;
      o[x][3] *= al1;
    }
    // P (f16) as A fragments, 16 keys per k-step; l sums the rounded values
    uint32_t pa[4][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int nt = 2 * kk + half;
        const __half2 lo = __floats2half2_rn(ex2f(s[nt][0] - mn0), ex2f(s[nt][1] - mn0));
        const __half2 hi = __floats2half2_rn(ex2f(s[nt][2] - mn1), ex2f(s[nt][3] - mn1));
        const float2 lf = __half22float2(lo), hf = __half22float2(hi);
        l0 += lf.x + lf.y;
        l1 += hf.x + hf.y;
        pa[kk][half * 2 + 0] = *reinterpret_cast<const uint32_t*>(&lo);
        pa[kk][half * 2 + 1] = *reinterpret_cast<const uint32_t*>(&hi);
      }
    }
    // ---- O += P V: NT n-tiles of 8 d, 4 k-steps of 16 keys
#pragma unroll
    for (int nt = 0; nt < NT; nt += 2) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t b0, b1, b2, b3;                 // n-tiles nt and nt + 1, keys 16kk .. 16kk+15
        ldsm4t(vt + tile_off<D>(kk * 16 + (lm_mat & 1) * 8 + lm_row, nt + (lm_mat >> 1)), b0, b1, b2, b3);
        mma16816(o[nt], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
        mma16816(o[nt + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
      }
    }
    __syncthreads();                             // the buffer is refilled next iteration
  }
  // ---- normalise and write the rows of the prompt
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float i0 = 1.f / l0, i1 = 1.f / l1;
  if (qa_row < L) {
    __half* dst = p.out + ((size_t)(row0 + qa_row) * p.Hq + hq) * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<__half2*>(dst + nt * 8 + 2 * qd) = __floats2half2_rn(o[nt][0] * i0, o[nt][1] * i0);
    if (qd == 0 && p.lse) p.lse[(size_t)(row0 + qa_row) * p.Hq + hq] = (m0 + log2f(l0)) * 0.69314718055994531f;
  }
  if (qb_row < L) {
    __half* dst = p.out + ((size_t)(row0 + qb_row) * p.Hq + hq) * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<__half2*>(dst + nt * 8 + 2 * qd) = __floats2half2_rn(o[nt][2] * i1, o[nt][3] * i1);
    if (qd == 0 && p.lse) p.lse[(size_t)(row0 + qb_row) * p.Hq + hq] = (m1 + log2f(l1)) * 0.69314718055994531f;
  }
}

cudaError_t set_smem_attr(const void* kern, int bytes);

cudaError_t launch_prefill(const PrefillParams& p, int D, int max_len, cudaStream_t st) {
  if (p.n <= 0 || max_len <= 0) return cudaSuccess;
  const dim3 grid((max_len + kBM - 1) / kBM, p.Hq, p.n);
  if (D == 128) {
    const int smem = 2 * 2 * kBN * 128 * 2;
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(prefill_kernel<128>), smem);
    if (e != cudaSuccess) return e;
    prefill_kernel<128><<<grid, kPThreads, smem, st>>>(p);
  } else {
    const int smem = 2 * 2 * kBN * 64 * 2;
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(prefill_kernel<64>), smem);
    if (e != cudaSuccess) return e;
    prefill_kernel<64><<<grid, kPThreads, smem, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace ekv
