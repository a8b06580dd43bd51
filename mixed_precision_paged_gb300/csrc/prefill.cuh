// prefill.cuh -- parameters and launchers of the FP16 causal prefill over the gathered
// workspace (knlp.io "Asymmetric K16/V8 KV cache", "What changes in vLLM's prefill
// routing?"): prompt i's queries are rows cu_seqlens[i] .. of q [T][Hq][D]; its keys and
// values are workspace pages page_off[i], page_off[i] + 1, ... of [W][16][Hkv][D] fp16.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ekv {

struct PrefillParams {
  const __half* q;             // [T][Hq][D]
  const __half* ws_k;          // [W][16][Hkv][D]
  const __half* ws_v;
  const int32_t* cu_seqlens;   // [n + 1]
  const int32_t* page_off;     // [n]
  __half* out;                 // [T][Hq][D]
  float* lse;                  // [T][Hq] or null
  int n, Hq, Hkv, G, num_ws_pages;
  int max_len;                 // rows past it are neither read as keys nor written
  float qscale;                // sm_scale * log2(e)
  int* err;
};

// Legacy warp-level MMA form (mma.sync): 64 query rows per CTA.
cudaError_t launch_prefill(const PrefillParams& p, int D, int max_len, cudaStream_t st);

// Fifth-generation tensor-core form (tcgen05, TMEM accumulators, TMA loads): 256 query
// rows per CTA. Builds its own tensor maps of the workspace.
cudaError_t launch_prefill_tc05(const PrefillParams& p, int D, int max_len, cudaStream_t st);

}  // namespace ekv
