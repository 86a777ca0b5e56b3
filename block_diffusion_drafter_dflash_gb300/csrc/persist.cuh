// Persistent phase-program kernel of the bf16 drafter at small batch: the
// description one launch runs (see persist.cu for the design).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "attn_tc.cuh"
#include "kernels.cuh"

namespace dflash {

constexpr int kPRows = 16;         // token rows one launch serves (one MMA column block per plane)
constexpr int kPMaxPhases = 56;    // 5 per draft layer + the LM head (+ fusion, injection)
constexpr int kPMaxSeg = 64;
constexpr int kPXMaps = 6;
constexpr int kPAttnRows = 64;     // query rows of one (request, kv head) group: 4 warps x 16
constexpr int kPMaxStages = 10;

enum : int { kPhGemm = 0, kPhAttn = 1 };   // an attention phase ends with the merge of its key chunks
// epilogue of a projection phase
enum : int {
  kEpFuse = 0,   // y = acc: planes of y * gain, per-tile sums of y^2 (context fusion)
  kEpInject,     // context K/V into the cache (EpiInject), scaled by 1/rms
  kEpQKV,        // block Q/K/V (EpiQKV), scaled by 1/rms
  kEpResid,      // x += acc: planes of x * gain, per-tile sums of x^2 (W_O, W_D)
  kEpSwiGLU,     // silu(gate) * up (EpiSwiGLU), scaled by 1/rms
  kEpLM          // argmax (and optional logits) of the mask rows, scaled by 1/rms
};

struct PPhase {
  int kind, epi;
  int kw;          // K columns per iteration (one ring stage): 64, or 128 for narrow phases
  int kb;          // kw-column blocks of K
  int tiles;       // 128-feature output tiles
  int seg0, nseg;  // weight segments: seg[seg0 .. seg0+nseg), tile_begin relative to the phase
  int xmap;        // activation tensor map
  int planes;      // activation planes (1: exact bf16 input, 2: hi/lo pair)
  int prow;        // map rows from plane 0 to plane 1
  int scaled;      // multiply the accumulator of row m by 1/rms(row m) before the epilogue
  int layer;       // draft layer of an attention phase
  const __nv_bfloat16* gain;  // kEpFuse / kEpResid: gain of the RMSNorm that reads the planes written
  int mrows;       // token rows of the phase (the injected rows for the fusion and injection phases)
  const float* ssq_in;        // scaled phases: sums of squares of the normed input
  __nv_bfloat16* u_out;       // kEpFuse / kEpResid: planes written ([2][16][D], u_plane apart)
  float* ssq_out;             // kEpFuse / kEpResid: their per-tile sums of squares [D/128][16]
};

struct PParams {
  CUtensorMap xmap[kPXMaps];   // activation maps: 64 x 16 boxes, 128-byte swizzle
  const CUtensorMap* wmaps;    // weight maps of the model (device memory)
  int nphase;
  int M;                       // token rows of the drafter pass (<= 16)
  int D;                       // hidden size (RMSNorm width)
  float eps;
  int stages;                  // ring depth
  float* x;                    // residual stream [M][D] fp32 (nullptr when no phase keeps one)
  __nv_bfloat16* u;            // default planes of kEpFuse / kEpResid: [2][16][D]
  size_t u_plane;              // elements between the hi and lo planes of u (and of every u_out)
  float* ssq;                  // default [D/128][16] sums of squares of the last normed input
  float* partial;              // [grid][2][16][128] stream-K partial tiles
  int* tickets;                // [largest tile count] stream-K tickets, zero at launch
  unsigned int* bar;           // grid barrier counter, zero at launch (follows tickets)
  int* gcnt;                   // [layers][B][nkv] finished attention chunks, zero at launch (follows bar)
  int32_t* status;
  EpiQKV<__nv_bfloat16> qkv;
  EpiSwiGLU<__nv_bfloat16> swiglu;
  EpiInject<__nv_bfloat16> inject;
  unsigned long long* slots;   // [16] argmax slots, zero at launch
  float* logits;               // [B][block-1][vocab] or nullptr
  int32_t* drafts;             // [B][block-1] or nullptr
  int vocab, block;
  AttnParams attn;             // layer taken from the phase; opart/ml/out/splits = chunk partials, output
  attn_tc::Maps amaps;         // tensor maps of the K/V cache and the block K/V
  unsigned long long* trace;    // optional timestamps [grid][kPMaxPhases][18] (see persist.cu) or nullptr
  PPhase ph[kPMaxPhases];
  GemmSeg seg[kPMaxSeg];
};

// Ring depth and dynamic shared memory of the kernel for head size hd.
int persist_stages(int hd);
size_t persist_smem(int stages, int hd);
// Grid = one CTA per SM; cooperative (all CTAs co-resident).
cudaError_t persist_launch(const PParams& p, int grid, int hd, cudaStream_t s);
cudaError_t persist_prepare(int hd);

// Draft prologue: x[row] = E[token], planes of x * g_in (u), per-tile sums of
// x^2 (ssq), RoPE table of the row's position, zeroed slots / tickets /
// barrier (`nzero` ints at `zero`).
cudaError_t persist_draft_prep_launch(const __nv_bfloat16* embed, const int32_t* anchor, int mask_id, int vocab,
                                      int B, int block, int D, const __nv_bfloat16* g, float* x, __nv_bfloat16* u,
                                      size_t u_plane, float* ssq, unsigned long long* slots, int* zero, int nzero,
                                      int32_t* status, const int32_t* ctx_len, const double* inv_freq, int hd,
                                      float2* rope, cudaStream_t s);

}  // namespace dflash
