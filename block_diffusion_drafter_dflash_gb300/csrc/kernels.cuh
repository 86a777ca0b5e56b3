// Launchers of the non-GEMM kernels of the draft cycle.
#pragma once

#include "common.cuh"

namespace dflash {

// ---------------------------------------------------------------- attention
// Block queries of one draft layer against [context K/V of the cache ; block K/V]
// (no mask: every block row sees all context and the whole block).
// K/V are stored as planes of the model dtype, index [..][plane][pos][hd]:
// fp32 one plane; bf16 block K/V hi and lo planes, the bf16 cache `kvp`
// planes (hi and lo, or one rounded value).
struct AttnParams {
  const float* q;       // [B][nq][block][hd] fp32 (RoPE applied)
  const void* kb;       // [B][nkv][planes][block][hd]  (RoPE applied)
  const void* vb;       // [B][nkv][planes][block][hd]; bf16 models: [B][nkv][planes][hd][pad8(block)]
  const void* kc;       // cache K [B][layers][nkv][kvp][cap][hd]
  const void* vc;       // cache V (bf16 models: [B][layers][nkv][kvp][hd][pad8(cap)])
  const int32_t* ctx_len;
  int layer, layers, cap;
  int kvp;              // planes of the cache (fp32 models: 1)
  int B, nq, nkv, hd, block;
  int chunk;            // keys per split (context + block keys counted together)
  int splits;
  int ctx_shared;       // 1: every request reads request 0's context slab (packed training blocks of one sequence)
  float* opart;         // [B][nq][block][splits][hd] unnormalised partial outputs
  float2* ml;           // [B][nq][block][splits] (running max, running sum)
  void* out;            // [B*block][nq*hd]: the W_O GEMM's activation operand
  size_t out_plane;     // elements between its hi and lo planes
  float scale;          // 1/sqrt(hd)
};

namespace attn_tc { struct Maps; }

// fp32 models: CUDA-core split-KV attention and the merge of the splits.
template <typename T> cudaError_t attention_launch(const AttnParams& p, cudaStream_t s);
// bf16 models: tensor-core split-KV attention (tensor maps of the K/V cache and
// of the block K/V, see attn_tc.cuh) and the merge; V is stored hd-major.
cudaError_t attention_bf16_launch(const AttnParams& p, const attn_tc::Maps& maps, int32_t* status, cudaStream_t s,
                                  bool out_f32 = false);
// Tensor maps of the bf16 attention: K cache [slabs*cap][hd], V cache
// [slabs*hd][cap] (row pitch cap_pitch) with B*layers*nkv*kvp slabs, block K
// [slabs*block][hd], block V [slabs*hd][block] (row pitch block_pitch) with
// B*nkv*2 slabs; 64 x rows boxes, 128-byte swizzle.
bool encode_attention_maps(attn_tc::Maps* m, const void* kc, const void* vc, const void* kb, const void* vb, int B,
                           int layers, int nkv, int hd, int cap, int cap_pitch, int kvp, int block, int block_pitch);
// Shared-memory opt-in of the tensor-core split-KV attention kernel for head size hd.
cudaError_t attention_tc_prepare(int hd);
// One-time per-device setup (shared-memory opt-in) for up to `rows` query rows.
template <typename T> cudaError_t attention_prepare(int rows, int hd);
int attention_max_rows();   // largest (nq/nkv)*block the kernel accepts

// ---------------------------------------------------------------- elementwise
// x[row] = E[token(row)], token = anchor[b] at block position 0 else mask_id;
// u[row] = RMSNorm(x[row]) * g.  Also zeroes `zero_n` ints at `zero_ptr`.
// An anchor outside [0, vocab) sets DFLASH_ERR_INVALID_ARG in `status`.
// Outputs written as GEMM activation operands (`plane` = elements between the
// hi and lo planes of a bf16 model; unused for fp32).
// Also fills rope[row][hd/2] = (cos, sin) of position ctx_len[b] + k.
template <typename T>
cudaError_t embed_norm_launch(const T* embed, const int32_t* anchor, int mask_id, int vocab, int B, int block, int D,
                              const T* g, float eps, float* x, T* u, size_t plane, int* zero_ptr, int zero_n,
                              int32_t* status, const int32_t* ctx_len, const double* inv_freq, int hd, float2* rope,
                              cudaStream_t s);

// u[row] = RMSNorm(x[row]) * g for `rows` rows.
template <typename T>
cudaError_t rmsnorm_launch(const float* x, const T* g, float eps, int rows, int D, T* u, size_t plane, cudaStream_t s);

// Final norm of the mask rows only (block position >= 1), compacted to
// hm[b*(block-1) + k-1]; zeroes the argmax slots of those rows.
template <typename T>
cudaError_t final_norm_launch(const float* x, const T* g, float eps, int B, int block, int D, T* hm, size_t plane,
                              unsigned long long* slots, cudaStream_t s);

// H_t[row] = RMSNorm(y[row]) * g_c for rows with rowinfo[row].x >= 0, 0 otherwise;
// rope[row][hd/2] = (cos, sin) of the row's position; with xf, H_t also in fp32.
template <typename T>
cudaError_t fuse_norm_launch(const float* y, const T* g, float eps, const int2* rowinfo, int rows, int D, T* ht,
                             size_t plane, const double* inv_freq, int hd, float2* rope, cudaStream_t s,
                             float* xf = nullptr);

// Input-fusion context rows: causal attention of each injected row (request,
// position p) over its request's cached keys 0..p of layer `layer`; q fp32
// [rows][nq*hd] (RoPE applied), output the W_O GEMM operand [rows][nq*hd]
// (planes `out_plane` apart; zero for padding rows).
template <typename T>
cudaError_t ctx_attention_launch(const float* q, const T* kc, const T* vc, const int2* rowinfo, int rows, int layer,
                                 int layers, int nq, int nkv, int hd, int cap, int vpitch, int kvp, float scale,
                                 T* out, size_t out_plane, cudaStream_t s);

// QK-norm models: per-head RMSNorm (gain g [hd], epsilon eps) then RoPE, in
// place, of the block queries q (fp32 [B][nq][block][hd]) and block keys kb
// (planes [B][nkv][plane][block][hd]) of one layer, (cos, sin) from
// rope[b*block + k][hd/2] ...
template <typename T>
cudaError_t qknorm_block_launch(float* q, T* kb, const T* g_q, const T* g_k, int B, int block, int nq, int nkv, int hd,
                                float eps, const float2* rope, cudaStream_t s);
// ... and of the injected context keys of one layer in the cache
// ([b][layer][kvh][plane][cap][hd], kvp planes) at the rows of rowinfo,
// rope[row][hd/2].
template <typename T>
cudaError_t qknorm_cache_launch(T* kc, const int2* rowinfo, int rows, int layer, int layers, int nkv, int hd, int cap,
                                int kvp, const T* g_k, float eps, const float2* rope, cudaStream_t s);

// Row -> (request, position) map of an injection and the ctx_len update;
// with `rope`, also rope[row][hd/2] = (cos, sin) of the row's position.
cudaError_t inject_prep_launch(const int32_t* n_new, int32_t* ctx_len, int B, int max_rows, int cap,
                               int2* rowinfo, int* zero_ptr, int zero_n, int32_t* status, cudaStream_t s,
                               const double* inv_freq = nullptr, int hd = 0, float2* rope = nullptr);

// drafts[row] = index packed in slots[row].
cudaError_t argmax_finalize_launch(const unsigned long long* slots, int rows, int32_t* drafts, cudaStream_t s);

// Synthetic target of the benchmark (see dflash_synthetic_target).
cudaError_t synthetic_target_launch(const int32_t* draft, const uint8_t* match, const int32_t* off,
                                    const int32_t* bonus, int npat, long long* pidx, const int32_t* tau,
                                    long long* tau_sum, int B, int g, int V, int32_t* y, cudaStream_t s);

// Greedy verification, one warp per request.
// One CTA whose bounded wait on an mbarrier that never completes runs out
// after `budget_cycles` SM cycles and sets DFLASH_ERR_TIMEOUT in `status`.
cudaError_t wait_selftest_launch(long long budget_cycles, int32_t* status, cudaStream_t s);
cudaError_t verify_launch(const int32_t* draft, const int32_t* target, int B, int block, int32_t* accept_len,
                          int32_t* out_tokens, int32_t* next_anchor, cudaStream_t s);

}  // namespace dflash
