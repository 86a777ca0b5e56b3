// Causal attention of context rows for the input-fusion ablation (paper
// §5.5.5: target features enter once, at the input, and every draft layer
// processes the context positions; the DFlash mask's context rows are causal,
// j <= i).  Each injected row (request b, position p) of layer `layer`
// attends to its request's cached keys 0..p — the earlier context and the
// rows of this injection up to itself, all written to the cache by the
// layer's K/V projection just before.
//
// One warp per (row, query head), on the CUDA cores: the lanes take 32 keys
// at a time (lane j scores key k0 + j against the query, held in shared
// memory), the warp keeps the running max and sum (base-2 exponent, scores
// pre-scaled by log2(e)/sqrt(hd)), and lane l accumulates output dimensions
// l, l+32, ... over the chunk's keys.  Keys and values are read as stored:
// fp32, or the kvp bf16 planes (values head-dim-major) of bf16 models.
#include "common.cuh"
#include "kernels.cuh"

namespace dflash {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <typename T, int HD>
__global__ void __launch_bounds__(128) ctx_attn_kernel(const float* q, const T* kc, const T* vc, const int2* rowinfo,
                                                       int rows, int layer, int layers, int nq, int nkv, int cap,
                                                       int vpitch, int kvp, float qscale, T* out, size_t out_plane) {
  griddep_wait();   // the K/V projection of this layer has written the cache
  griddep_trigger();
  constexpr int E = HD / 32;
  __shared__ float qs[4][HD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * 4 + warp;
  if (w >= rows * nq) return;
  const int row = w / nq, h = w - row * nq;
  const int2 ri = rowinfo[row];
  T* dst = out;
  const size_t obase = (size_t)row * nq * HD + (size_t)h * HD;
  if (ri.x < 0) {   // a padding row: a zero operand row
#pragma unroll
    for (int e = 0; e < E; ++e) put_act(dst, out_plane, obase + lane + 32 * e, 0.f);
    return;
  }
  const int b = ri.x, pos = ri.y, kvh = h / (nq / nkv);
  constexpr bool bf16 = ActPlanes<T>::n == 2;
  const size_t slab = ((size_t)b * layers + layer) * nkv + kvh;
  const T* kb = kc + slab * kvp * (size_t)cap * HD;                  // [plane][cap][HD]
  const size_t kplane = (size_t)cap * HD;
  const T* vb = bf16 ? vc + slab * kvp * (size_t)HD * vpitch         // [plane][HD][vpitch]
                     : vc + slab * (size_t)cap * HD;                 // [cap][HD]
  const size_t vplane = bf16 ? (size_t)HD * vpitch : 0;
#pragma unroll
  for (int e = 0; e < E; ++e) qs[warp][lane + 32 * e] = q[obase + lane + 32 * e] * qscale;
  __syncwarp();
  float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int k0 = 0; k0 <= pos; k0 += 32) {
    const int key = k0 + lane;
    float sc = -INFINITY;
    if (key <= pos) {
      float a = 0.f;
      const size_t kr = (size_t)key * HD;
#pragma unroll 8
      for (int d = 0; d < HD; ++d) a += qs[warp][d] * get_kv(kb, kplane, kr + d, kvp);
      sc = a;
    }
    float mx = sc;
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float mn = fmaxf(m, mx);
    const float alpha = m == -INFINITY ? 0.f : exp2f(m - mn);
    const float p = key <= pos ? exp2f(sc - mn) : 0.f;
    float ps = p;
    for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    l = l * alpha + ps;
    m = mn;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= alpha;
    const int nk = min(32, pos + 1 - k0);
    for (int j = 0; j < nk; ++j) {
      const float pj = __shfl_sync(0xffffffffu, p, j);
      const int kj = k0 + j;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int d = lane + 32 * e;
        const float v = bf16 ? get_kv(vb, vplane, (size_t)d * vpitch + kj, kvp)
                             : get_kv(vb, vplane, (size_t)kj * HD + d, kvp);
        acc[e] += pj * v;
      }
    }
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int e = 0; e < E; ++e) put_act(dst, out_plane, obase + lane + 32 * e, acc[e] * inv);
}

}  // namespace

template <typename T>
cudaError_t ctx_attention_launch(const float* q, const T* kc, const T* vc, const int2* rowinfo, int rows, int layer,
                                 int layers, int nq, int nkv, int hd, int cap, int vpitch, int kvp, float scale,
                                 T* out, size_t out_plane, cudaStream_t s) {
  const int warps = rows * nq;
  if (warps == 0) return cudaSuccess;
  const float qscale = scale * kLog2e;
  if (hd == 64)
    return launch_pdl(ctx_attn_kernel<T, 64>, dim3((warps + 3) / 4), dim3(128), 0, s, q, kc, vc, rowinfo, rows, layer,
                      layers, nq, nkv, cap, vpitch, kvp, qscale, out, out_plane);
  return launch_pdl(ctx_attn_kernel<T, 128>, dim3((warps + 3) / 4), dim3(128), 0, s, q, kc, vc, rowinfo, rows, layer,
                    layers, nq, nkv, cap, vpitch, kvp, qscale, out, out_plane);
}

template cudaError_t ctx_attention_launch<float>(const float*, const float*, const float*, const int2*, int, int, int,
                                                 int, int, int, int, int, int, float, float*, size_t, cudaStream_t);
template cudaError_t ctx_attention_launch<__nv_bfloat16>(const float*, const __nv_bfloat16*, const __nv_bfloat16*,
                                                         const int2*, int, int, int, int, int, int, int, int, int,
                                                         float, __nv_bfloat16*, size_t, cudaStream_t);

}  // namespace dflash
