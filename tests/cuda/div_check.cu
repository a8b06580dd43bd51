// Exhaustive check of div_by_scale (common.cuh) against __fdiv_rn over the demotion
// domain: every scale s = fp32_rn(a / 448) for a a positive finite fp16 value (s = 1
// for a = 0), every finite fp16 x with |x| <= a. Prints the number of bit
// mismatches of the quotient.
#include <cstdio>
#include <cuda_fp16.h>

#include "../../mixed_precision_paged_gb300/csrc/common.cuh"

__global__ void check(unsigned long long* mismatches, unsigned int* first) {
  const unsigned short abits = (unsigned short)blockIdx.x;                // 0x0000 .. 0x7bff
  const float a = __half2float(__ushort_as_half(abits));
  const float s = a == 0.f ? 1.f : __fdiv_rn(a, 448.f);                  // the kernel's rule
  const float r = __frcp_rn(s);
  unsigned long long bad = 0;
  for (unsigned int xb = threadIdx.x; xb < 0x10000u; xb += blockDim.x) {
    const unsigned short mag = (unsigned short)(xb & 0x7fffu);
    if (mag > abits) continue;                                             // |x| <= a (and finite)
    const float x = __half2float(__ushort_as_half((unsigned short)xb));
    const float ref = __fdiv_rn(x, s);
    const float got = ekv::div_by_scale(x, s, r);
    if (__float_as_uint(ref) != __float_as_uint(got)) {
      ++bad;
      atomicCAS(first, 0u, ((unsigned int)abits << 16) | xb | 0x80000000u);
    }
  }
  if (bad) atomicAdd(mismatches, bad);
}

int main() {
  unsigned long long* d_m;
  unsigned int* d_f;
  cudaMalloc(&d_m, sizeof(*d_m));
  cudaMalloc(&d_f, sizeof(*d_f));
  cudaMemset(d_m, 0, sizeof(*d_m));
  cudaMemset(d_f, 0, sizeof(*d_f));
  check<<<0x7c00, 256>>>(d_m, d_f);
  cudaError_t e = cudaDeviceSynchronize();
  unsigned long long m = ~0ull;
  unsigned int f = 0;
  cudaMemcpy(&m, d_m, sizeof(m), cudaMemcpyDeviceToHost);
  cudaMemcpy(&f, d_f, sizeof(f), cudaMemcpyDeviceToHost);
  printf("status %d mismatches %llu first %08x\n", (int)e, m, f);
  return (e == cudaSuccess && m == 0) ? 0 : 1;
}
