// Non-causal block attention of the drafter (split-KV, online softmax): the
// CUDA-core kernels of fp32 models and the merge of the splits (all models).
//
// For request b and kv head h the query rows are the (nq/nkv) query heads of
// the group times the block positions; the keys are the request's injected
// context K (cache) followed by the block's own K.  No mask is needed: under
// the DFlash mask a block row sees every context position and every block
// position.  The key range is cut into splits; each CTA keeps a running max,
// a running sum and an unnormalised output per row, and a second kernel merges
// the splits exactly (log-sum-exp rescaling).
#include <cfloat>
#include <type_traits>

#include "kernels.cuh"

namespace dflash {

// tensor-core split kernel for bf16 models (attention_tc.cu)
cudaError_t attention_tc_prepare(int hd);
cudaError_t attention_tc_split_launch(const AttnParams& p, const attn_tc::Maps& maps, int32_t* status, cudaStream_t s);

namespace {

constexpr int kAttnThreads = 128;
constexpr int kKeyTile = 32;
constexpr int kMaxRows = 128;

__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T>
__global__ void __launch_bounds__(kAttnThreads) attn_split_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ float sm[];
  griddep_wait();
  griddep_trigger();
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = p.nq / p.nkv, rows = G * p.block, hd = p.hd;
  const int c = p.ctx_len[b];
  const int total = c + p.block;
  const int j0 = split * p.chunk, j1 = min(total, j0 + p.chunk);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = kAttnThreads / 32;

  float* Qs = sm;                       // [rows][hd]
  float* Os = Qs + rows * hd;           // [rows][hd]
  float* Ks = Os + rows * hd;           // [kKeyTile][hd+1]
  float* Vs = Ks + kKeyTile * (hd + 1); // [kKeyTile][hd]
  float* Ms = Vs + kKeyTile * hd;       // [rows]
  float* Ls = Ms + rows;                // [rows]

  const float* q = p.q;
  for (int e = threadIdx.x; e < rows * hd; e += kAttnThreads) {
    int r = e / hd, d = e - r * hd, g = r / p.block, k = r - g * p.block;
    int qh = kvh * G + g;
    Qs[e] = q[(((size_t)b * p.nq + qh) * p.block + k) * hd + d] * p.scale;
    Os[e] = 0.f;
  }
  for (int r = threadIdx.x; r < rows; r += kAttnThreads) {
    Ms[r] = -FLT_MAX;
    Ls[r] = 0.f;
  }

  const float* kc = static_cast<const float*>(p.kc) + (((size_t)b * p.layers + p.layer) * p.nkv + kvh) * p.cap * hd;
  const float* vc = static_cast<const float*>(p.vc) + (((size_t)b * p.layers + p.layer) * p.nkv + kvh) * p.cap * hd;
  const float* kb = static_cast<const float*>(p.kb) + ((size_t)b * p.nkv + kvh) * p.block * hd;
  const float* vb = static_cast<const float*>(p.vb) + ((size_t)b * p.nkv + kvh) * p.block * hd;

  for (int jt = j0; jt < j1; jt += kKeyTile) {
    const int n = min(kKeyTile, j1 - jt);
    __syncthreads();
    for (int e = threadIdx.x; e < n * hd; e += kAttnThreads) {
      int jj = e / hd, d = e - jj * hd, j = jt + jj;
      float kv, vv;
      if (j < c) {
        kv = kc[(size_t)j * hd + d];
        vv = vc[(size_t)j * hd + d];
      } else {
        kv = kb[(size_t)(j - c) * hd + d];
        vv = vb[(size_t)(j - c) * hd + d];
      }
      Ks[jj * (hd + 1) + d] = kv;
      Vs[jj * hd + d] = vv;
    }
    __syncthreads();
    for (int r = warp; r < rows; r += nwarps) {
      float s = -FLT_MAX;
      if (lane < n) {
        s = 0.f;
        const float* qr = Qs + r * hd;
        const float* kr = Ks + lane * (hd + 1);
        for (int d = 0; d < hd; ++d) s = fmaf(qr[d], kr[d], s);
      }
      const float m_old = Ms[r];
      const float m_new = fmaxf(m_old, warp_max(s));
      const float pj = lane < n ? __expf(s - m_new) : 0.f;
      const float alpha = __expf(m_old - m_new);
      const float lsum = warp_sum(pj);
      for (int d = lane; d < hd; d += 32) {
        float acc = Os[r * hd + d] * alpha;
        for (int j = 0; j < n; ++j) acc = fmaf(__shfl_sync(0xffffffffu, pj, j), Vs[j * hd + d], acc);
        Os[r * hd + d] = acc;
      }
      __syncwarp();
      if (lane == 0) {
        Ms[r] = m_new;
        Ls[r] = Ls[r] * alpha + lsum;
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < rows * hd; e += kAttnThreads) {
    int r = e / hd, d = e - r * hd, g = r / p.block, k = r - g * p.block;
    size_t row = (((size_t)b * p.nq + kvh * G + g) * p.block + k) * p.splits + split;
    p.opart[row * hd + d] = Os[e];
    if (d == 0) p.ml[row] = make_float2(Ms[r], Ls[r]);
  }
}

// One CTA of 128 threads per (request, query head, block position): merge the
// splits.  The per-split (max, sum) pairs are read in parallel and reduced in
// shared memory; each thread then adds one output dimension over all splits.
template <typename T>
__global__ void __launch_bounds__(128) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ float w[];                 // [splits] weights, then 8 floats of scratch
  float* red = w + p.splits;
  griddep_wait();
  griddep_trigger();
  const int row = blockIdx.x;                  // ((b*nq + qh)*block + k)
  const int k = row % p.block, qh = (row / p.block) % p.nq, b = row / (p.block * p.nq);
  const float2* ml = p.ml + (size_t)row * p.splits;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float mx = -FLT_MAX;
  for (int sp = threadIdx.x; sp < p.splits; sp += blockDim.x) {
    const float2 v = ml[sp];
    w[sp] = v.y > 0.f ? v.x : -FLT_MAX;
    mx = fmaxf(mx, w[sp]);
  }
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  float l = 0.f;
  for (int sp = threadIdx.x; sp < p.splits; sp += blockDim.x) {
    const float2 v = ml[sp];
    const float e = v.y > 0.f ? __expf(v.x - M) : 0.f;
    w[sp] = e;
    l += e * v.y;
  }
  for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if (lane == 0) red[4 + warp] = l;
  __syncthreads();
  const float inv = 1.f / ((red[4] + red[5]) + (red[6] + red[7]));
  const int d = threadIdx.x;
  if (d >= p.hd) return;
  const float* src = p.opart + (size_t)row * p.splits * p.hd + d;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  int sp = 0;
  for (; sp + 4 <= p.splits; sp += 4) {
    a0 += w[sp] * src[(size_t)sp * p.hd];
    a1 += w[sp + 1] * src[(size_t)(sp + 1) * p.hd];
    a2 += w[sp + 2] * src[(size_t)(sp + 2) * p.hd];
    a3 += w[sp + 3] * src[(size_t)(sp + 3) * p.hd];
  }
  for (; sp < p.splits; ++sp) a0 += w[sp] * src[(size_t)sp * p.hd];
  T* out = static_cast<T*>(p.out);
  const size_t base = ((size_t)b * p.block + k) * p.nq * p.hd + (size_t)qh * p.hd;
  put_act(out, p.out_plane, base + d, ((a0 + a1) + (a2 + a3)) * inv);
}

size_t attn_smem_bytes(int rows, int hd) {
  return sizeof(float) * ((size_t)2 * rows * hd + kKeyTile * (hd + 1) + (size_t)kKeyTile * hd + 2 * rows);
}

}  // namespace

int attention_max_rows() { return kMaxRows; }

template <typename T>
cudaError_t attention_prepare(int rows, int hd) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) return attention_tc_prepare(hd);
  return cudaFuncSetAttribute(attn_split_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)attn_smem_bytes(rows, hd));
}

cudaError_t attention_bf16_launch(const AttnParams& p, const attn_tc::Maps& maps, int32_t* status, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  cudaError_t e = attention_tc_split_launch(p, maps, status, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_combine_kernel<__nv_bfloat16>, dim3(p.B * p.nq * p.block), dim3(128),
                    (p.splits + 8) * sizeof(float), s, p);
}

template <typename T>
cudaError_t attention_launch(const AttnParams& p, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  if constexpr (std::is_same<T, __nv_bfloat16>::value) return cudaErrorInvalidValue;   // attention_bf16_launch
  const int rows = (p.nq / p.nkv) * p.block;
  cudaError_t e = launch_pdl(attn_split_kernel<T>, dim3(p.splits, p.nkv, p.B), dim3(kAttnThreads),
                             attn_smem_bytes(rows, p.hd), s, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_combine_kernel<T>, dim3(p.B * p.nq * p.block), dim3(128), (p.splits + 8) * sizeof(float), s,
                    p);
}

template cudaError_t attention_prepare<float>(int, int);
template cudaError_t attention_prepare<__nv_bfloat16>(int, int);
template cudaError_t attention_launch<float>(const AttnParams&, cudaStream_t);
template cudaError_t attention_launch<__nv_bfloat16>(const AttnParams&, cudaStream_t);

}  // namespace dflash
