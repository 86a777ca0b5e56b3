// Forward attention of a packed training sequence (packed_attention.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace dflash {

// Operand layout of one call, carved from the caller's workspace.
struct PackedPlan {
  int N, block;
  int S;                  // context tokens of the sequence (may be 0)
  int Sa;                 // max(S, 1): rows of each context slab as laid out
  int nq, nkv, hd, S8, g8, splits;
  int32_t* status;        // bounded-wait status word (DFLASH_ERR_TIMEOUT on expiry)
  int32_t* ctx_len;       // [N] the anchors: context keys each block sees
  float* qf;              // [N][nq][block][hd]
  __nv_bfloat16* kc;      // [nkv][2][Sa][hd]
  __nv_bfloat16* vc;      // [nkv][2][hd][S8]
  __nv_bfloat16* kb;      // [N][nkv][2][block][hd]
  __nv_bfloat16* vb;      // [N][nkv][2][hd][g8]
  float* opart;           // split partials
  float2* ml;
};

int packed_splits(int N, int S, int nkv, int sms);
size_t packed_workspace_bytes(int N, int block, int S, int nq, int nkv, int hd, int sms);
PackedPlan packed_plan(void* ws, int N, int block, int S, int nq, int nkv, int hd, int sms);
// Pack, split-KV tensor-core attention with a shared context, fp32 merge.
cudaError_t packed_attention_run(const PackedPlan& pl, int dtype_f32, const void* q, const void* kc, const void* vc,
                                 const void* kb, const void* vb, const int32_t* anchors_dev, float* out, int sms,
                                 int* launches, cudaStream_t s);

}  // namespace dflash
