// Forward attention of a packed training sequence (paper §4.2: the anchor
// blocks sampled from one sequence are concatenated and run in one pass under
// a sparse mask; explainer "Training Rehearses the Same Masked Blocks Used at
// Runtime", Figure 4).  Block n, anchored at position a_n, attends to the
// sequence's injected context keys 0 .. a_n - 1 and to its own block rows,
// bidirectionally, and to nothing of another block.
//
// That is the drafter's block attention with one "request" per block whose
// context length is its anchor position and whose context is the sequence's
// (shared by every block), so it runs on the same tensor-core split-KV
// attention (attn_tc.cuh, attention_tc.cu) with ctx_shared set.  A packing
// kernel first brings the caller's token-major tensors into that kernel's
// operand layout: queries fp32 [N][nq][block][hd]; keys and values as hi/lo
// bf16 planes (lo = 0 for bf16 inputs; fp32 inputs keep fp32-level
// precision), keys [..][plane][pos][hd], values head-dim-major
// [..][plane][hd][pos, padded to 8 with zeros].  No mask is materialised.
#include <cuda.h>

#include <algorithm>

#include "attn_tc.cuh"
#include "common.cuh"
#include "gemm.cuh"
#include "kernels.cuh"
#include "packed_attention.cuh"

namespace dflash {
namespace {

template <typename T>
__device__ __forceinline__ void split_store(__nv_bfloat16* dst, size_t plane, size_t i, T v) {
  put_act(dst, plane, i, to_f32(v));   // hi at i, lo (the rounding residual) at plane + i
}

// One thread per output element of each region (grid-stride).
template <typename T>
__global__ void __launch_bounds__(256) pack_kernel(PackedPlan pl, const T* q, const T* kc, const T* vc, const T* kb,
                                                   const T* vb, const int32_t* anchors_src) {
  griddep_wait();   // an earlier call may still read this workspace
  griddep_trigger();
  const int N = pl.N, g = pl.block, S = pl.S, Sa = pl.Sa, nq = pl.nq, nkv = pl.nkv, hd = pl.hd, S8 = pl.S8,
            g8 = pl.g8;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t t0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  // queries [N][g][nq][hd] -> fp32 [N][nq][g][hd]
  const size_t nq_el = (size_t)N * g * nq * hd;
  for (size_t e = t0; e < nq_el; e += stride) {
    const int d = (int)(e % hd);
    size_t r = e / hd;
    const int h = (int)(r % nq);
    r /= nq;
    const int k = (int)(r % g), n = (int)(r / g);
    pl.qf[(((size_t)n * nq + h) * g + k) * hd + d] = to_f32(q[e]);
  }
  // context keys [S][nkv][hd] -> planes [nkv][2][Sa][hd]
  const size_t kc_el = (size_t)S * nkv * hd;
  for (size_t e = t0; e < kc_el; e += stride) {
    const int d = (int)(e % hd);
    const size_t r = e / hd;
    const int h = (int)(r % nkv), pos = (int)(r / nkv);
    split_store(pl.kc, (size_t)Sa * hd, ((size_t)h * 2 * Sa + pos) * hd + d, kc[e]);
  }
  // context values -> planes [nkv][2][hd][S8], columns S..S8-1 zero
  const size_t vc_el = (size_t)nkv * hd * S8;
  for (size_t e = t0; e < vc_el; e += stride) {
    const int pos = (int)(e % S8);
    const size_t r = e / S8;
    const int d = (int)(r % hd), h = (int)(r / hd);
    const float v = pos < S ? to_f32(vc[((size_t)pos * nkv + h) * hd + d]) : 0.f;
    put_act(pl.vc, (size_t)hd * S8, ((size_t)h * 2 * hd + d) * S8 + pos, v);
  }
  // block keys [N][g][nkv][hd] -> planes [N][nkv][2][g][hd]
  const size_t kb_el = (size_t)N * g * nkv * hd;
  for (size_t e = t0; e < kb_el; e += stride) {
    const int d = (int)(e % hd);
    size_t r = e / hd;
    const int h = (int)(r % nkv);
    r /= nkv;
    const int k = (int)(r % g), n = (int)(r / g);
    split_store(pl.kb, (size_t)g * hd, (((size_t)n * nkv + h) * 2 * g + k) * hd + d, kb[e]);
  }
  // block values -> planes [N][nkv][2][hd][g8], columns g..g8-1 zero
  const size_t vb_el = (size_t)N * nkv * hd * g8;
  for (size_t e = t0; e < vb_el; e += stride) {
    const int k = (int)(e % g8);
    size_t r = e / g8;
    const int d = (int)(r % hd);
    r /= hd;
    const int h = (int)(r % nkv), n = (int)(r / nkv);
    const float v = k < g ? to_f32(vb[(((size_t)n * g + k) * nkv + h) * hd + d]) : 0.f;
    put_act(pl.vb, (size_t)hd * g8, (((size_t)n * nkv + h) * 2 * hd + d) * g8 + k, v);
  }
  if (t0 == 0) {   // one thread: the status word, and the anchors (an anchor outside the sequence is clamped and flagged)
    int32_t st = 0;
    for (int n = 0; n < N; ++n) {
      int a = anchors_src[n];
      if (a < 0 || a > S) {
        st = DFLASH_ERR_INVALID_ARG;
        a = a < 0 ? 0 : S;
      }
      pl.ctx_len[n] = a;
    }
    *pl.status = st;
  }
}

size_t al(size_t v) { return (v + 255) & ~(size_t)255; }
int pad8i(int v) { return (v + 7) & ~7; }

}  // namespace

int packed_splits(int N, int S, int nkv, int sms) {
  const int tiles = (S + attn_tc::kKeys - 1) / attn_tc::kKeys + 1;
  const int groups = std::max(1, N * nkv);
  return std::max(1, std::min(tiles, (4 * sms + groups - 1) / groups));
}

size_t packed_workspace_bytes(int N, int block, int S, int nq, int nkv, int hd, int sms) {
  const int splits = packed_splits(N, S, nkv, sms);
  const size_t rows = (size_t)N * nq * block;
  const int Sa = std::max(S, 1);
  return al(4) + al(4 * (size_t)N) + al(4 * (size_t)N * nq * block * hd) + al(2 * 2 * (size_t)nkv * Sa * hd) +
         al(2 * 2 * (size_t)nkv * hd * pad8i(Sa)) + al(2 * 2 * (size_t)N * nkv * block * hd) +
         al(2 * 2 * (size_t)N * nkv * hd * pad8i(block)) + al(4 * rows * splits * hd) + al(8 * rows * splits);
}

PackedPlan packed_plan(void* ws, int N, int block, int S, int nq, int nkv, int hd, int sms) {
  PackedPlan p{};
  p.N = N;
  p.block = block;
  p.S = S;
  p.Sa = std::max(S, 1);
  p.nq = nq;
  p.nkv = nkv;
  p.hd = hd;
  p.S8 = pad8i(p.Sa);
  p.g8 = pad8i(block);
  p.splits = packed_splits(N, S, nkv, sms);
  char* c = static_cast<char*>(ws);
  auto take = [&](size_t bytes) {
    char* r = c;
    c += al(bytes);
    return r;
  };
  p.status = reinterpret_cast<int32_t*>(take(4));
  p.ctx_len = reinterpret_cast<int32_t*>(take(4 * (size_t)N));
  p.qf = reinterpret_cast<float*>(take(4 * (size_t)N * nq * block * hd));
  p.kc = reinterpret_cast<__nv_bfloat16*>(take(2 * 2 * (size_t)nkv * p.Sa * hd));
  p.vc = reinterpret_cast<__nv_bfloat16*>(take(2 * 2 * (size_t)nkv * hd * p.S8));
  p.kb = reinterpret_cast<__nv_bfloat16*>(take(2 * 2 * (size_t)N * nkv * block * hd));
  p.vb = reinterpret_cast<__nv_bfloat16*>(take(2 * 2 * (size_t)N * nkv * hd * p.g8));
  const size_t rows = (size_t)N * nq * block;
  p.opart = reinterpret_cast<float*>(take(4 * rows * p.splits * hd));
  p.ml = reinterpret_cast<float2*>(take(8 * rows * p.splits));
  return p;
}

cudaError_t packed_attention_run(const PackedPlan& pl, int dtype_f32, const void* q, const void* kc, const void* vc,
                                 const void* kb, const void* vb, const int32_t* anchors_dev, float* out, int sms,
                                 int* launches, cudaStream_t s) {
  *launches = 0;
  const size_t work = std::max<size_t>({(size_t)pl.N * pl.block * pl.nq * pl.hd, (size_t)pl.nkv * pl.hd * pl.S8,
                                        (size_t)pl.N * pl.nkv * pl.hd * pl.g8});
  const int grid = (int)std::min<size_t>((work + 255) / 256, (size_t)sms * 8);
  cudaError_t e;
  if (dtype_f32)
    e = launch_pdl(pack_kernel<float>, dim3(grid), dim3(256), 0, s, pl, static_cast<const float*>(q),
                   static_cast<const float*>(kc), static_cast<const float*>(vc), static_cast<const float*>(kb),
                   static_cast<const float*>(vb), anchors_dev);
  else
    e = launch_pdl(pack_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s, pl, static_cast<const __nv_bfloat16*>(q),
                   static_cast<const __nv_bfloat16*>(kc), static_cast<const __nv_bfloat16*>(vc),
                   static_cast<const __nv_bfloat16*>(kb), static_cast<const __nv_bfloat16*>(vb), anchors_dev);
  if (e != cudaSuccess) return e;
  ++*launches;
  // tensor maps: the context as one slab per (kv head, plane), the blocks' own
  // keys and values with N slabs each (64-column boxes, 128-byte swizzle)
  attn_tc::Maps maps;
  if (!encode_activation_map(&maps.kc, pl.kc, pl.hd, pl.nkv * 2 * pl.Sa, pl.hd, attn_tc::kKeys) ||
      !encode_activation_map(&maps.vc, pl.vc, pl.Sa, pl.nkv * 2 * pl.hd, pl.S8, pl.hd) ||
      !encode_activation_map(&maps.kb, pl.kb, pl.hd, pl.N * pl.nkv * 2 * pl.block, pl.hd, attn_tc::kKeys) ||
      !encode_activation_map(&maps.vb, pl.vb, pl.block, pl.N * pl.nkv * 2 * pl.hd, pl.g8, pl.hd))
    return cudaErrorInvalidValue;
  AttnParams ap{};
  ap.q = pl.qf;
  ap.kb = pl.kb;
  ap.vb = pl.vb;
  ap.kc = pl.kc;
  ap.vc = pl.vc;
  ap.ctx_len = pl.ctx_len;
  ap.layer = 0;
  ap.layers = 1;
  ap.cap = pl.Sa;
  ap.kvp = 2;   // the packed context keeps hi and lo planes
  ap.B = pl.N;
  ap.nq = pl.nq;
  ap.nkv = pl.nkv;
  ap.hd = pl.hd;
  ap.block = pl.block;
  ap.splits = pl.splits;
  ap.ctx_shared = 1;
  ap.opart = pl.opart;
  ap.ml = pl.ml;
  ap.out = out;
  ap.out_plane = 0;
  ap.scale = 1.0f / sqrtf((float)pl.hd);
  e = attention_bf16_launch(ap, maps, pl.status, s, true);
  if (e != cudaSuccess) return e;
  *launches += 2;
  return cudaSuccess;
}

}  // namespace dflash
