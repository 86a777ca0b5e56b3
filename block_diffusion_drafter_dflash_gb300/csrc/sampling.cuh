// Stochastic lossless verification and inverse-CDF sampling over the
// vocabulary (sampling.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace dflash {

// One draw: the distribution max(0, p_t - p_d) (pd != nullptr) or p_t, each
// softmax(logits / T) of a logits row with its (max, sum) statistics in the
// log2 domain; the drawn id goes to *out.
struct DrawSel {
  const float* pt;
  const float* pd;
  float2 mst, msd;
  int32_t* out;
};

// 8192-logit chunks of a row of `vocab` logits.
int sampling_chunks(int vocab);
// Scratch of `rows` logits rows and `draws` draws.
size_t sampling_workspace_bytes(int rows, int draws, int vocab);

// B requests, g = block size: drafter logits [B][g-1][V], target logits
// [B][g][V], drafts [B][g-1], uniforms u_accept [B][g-1] and u_sample [B].
cudaError_t verify_sampled_launch(const float* draft_logits, const float* target_logits, const int32_t* drafts,
                                  const float* u_accept, const float* u_sample, int B, int g, int V,
                                  float temperature, int32_t* accept_len, int32_t* out_tokens,
                                  int32_t* next_anchor, void* ws, int* launches, cudaStream_t s);

// tokens[r] = inverse-CDF draw with uniform u[r] from softmax(logits[r] / T).
cudaError_t sample_tokens_launch(const float* logits, int rows, int V, float temperature, const float* u,
                                 int32_t* tokens, void* ws, int* launches, cudaStream_t s);

}  // namespace dflash
