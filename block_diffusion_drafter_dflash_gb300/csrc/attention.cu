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

// Merge of the key splits: one warp per (request, query head, block
// position) row, four rows per CTA of 128 threads.  Lane s holds split s's
// (max, sum) and weight (32 splits at a time, broadcast by shuffles); lane l
// owns output elements [E*l, E*l + E), E = hd / 32, read as one vector per
// split.  Splits with weight 0 (no keys) are not read.
template <typename T>
__global__ void __launch_bounds__(128) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  griddep_wait();
  griddep_trigger();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);   // ((b*nq + qh)*block + k)
  if (row >= p.B * p.nq * p.block) return;
  const int k = row % p.block, qh = (row / p.block) % p.nq, b = row / (p.block * p.nq);
  const float2* ml = p.ml + (size_t)row * p.splits;
  float M = -FLT_MAX;
  for (int sp = lane; sp < p.splits; sp += 32) {
    const float2 v = ml[sp];
    if (v.y > 0.f) M = fmaxf(M, v.x);
  }
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const int E = p.hd >> 5;   // 2 or 4
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, l = 0.f;
  const float* src = p.opart + (size_t)row * p.splits * p.hd + E * lane;
  for (int s0 = 0; s0 < p.splits; s0 += 32) {
    float wgt = 0.f;
    if (s0 + lane < p.splits) {
      const float2 v = ml[s0 + lane];
      wgt = v.y > 0.f ? __expf(v.x - M) : 0.f;
      l += wgt * v.y;
    }
    const int n = min(32, p.splits - s0);
    for (int u0 = 0; u0 < n; u0 += 8) {   // eight splits' vectors in flight before any is used
      float wu[8];
      float4 x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        wu[j] = __shfl_sync(0xffffffffu, wgt, (u0 + j) & 31);
        if (u0 + j >= n) wu[j] = 0.f;
        const float* sv = src + (size_t)(s0 + u0 + j) * p.hd;
        x[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (wu[j] != 0.f) {   // the same for every lane
          if (E == 4) {
            x[j] = *reinterpret_cast<const float4*>(sv);
          } else {
            const float2 y = *reinterpret_cast<const float2*>(sv);
            x[j].x = y.x;
            x[j].y = y.y;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc[0] += wu[j] * x[j].x;
        acc[1] += wu[j] * x[j].y;
        acc[2] += wu[j] * x[j].z;
        acc[3] += wu[j] * x[j].w;
      }
    }
  }
  for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  const float inv = 1.f / l;
  T* out = static_cast<T*>(p.out);
  const size_t base = ((size_t)b * p.block + k) * p.nq * p.hd + (size_t)qh * p.hd + E * lane;
  for (int e = 0; e < E; ++e) put_act(out, p.out_plane, base + e, acc[e] * inv);
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

cudaError_t attention_bf16_launch(const AttnParams& p, const attn_tc::Maps& maps, int32_t* status, cudaStream_t s,
                                  bool out_f32) {
  if (p.B <= 0) return cudaSuccess;
  cudaError_t e = attention_tc_split_launch(p, maps, status, s);
  if (e != cudaSuccess) return e;
  // the merge writes the W_O GEMM's bf16 hi/lo operand planes, or fp32 rows
  if (out_f32)
    return launch_pdl(attn_combine_kernel<float>, dim3((p.B * p.nq * p.block + 3) / 4), dim3(128), 0, s, p);
  return launch_pdl(attn_combine_kernel<__nv_bfloat16>, dim3((p.B * p.nq * p.block + 3) / 4), dim3(128), 0, s, p);
}

template <typename T>
cudaError_t attention_launch(const AttnParams& p, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  if constexpr (std::is_same<T, __nv_bfloat16>::value) return cudaErrorInvalidValue;   // attention_bf16_launch
  const int rows = (p.nq / p.nkv) * p.block;
  cudaError_t e = launch_pdl(attn_split_kernel<T>, dim3(p.splits, p.nkv, p.B), dim3(kAttnThreads),
                             attn_smem_bytes(rows, p.hd), s, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_combine_kernel<T>, dim3((p.B * p.nq * p.block + 3) / 4), dim3(128), 0, s, p);
}

template cudaError_t attention_prepare<float>(int, int);
template cudaError_t attention_prepare<__nv_bfloat16>(int, int);
template cudaError_t attention_launch<float>(const AttnParams&, cudaStream_t);
template cudaError_t attention_launch<__nv_bfloat16>(const AttnParams&, cudaStream_t);

}  // namespace dflash
