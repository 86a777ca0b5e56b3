// Row-wise kernels of the draft cycle: embedding gather, RMSNorms, the
// injection row map, argmax read-out and greedy verification.
#include "kernels.cuh"
#include "ptx.cuh"

namespace dflash {

namespace {

constexpr int kRowThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
  return t;
}

// Each row kernel keeps its row in registers: thread t holds float4s
// t, t+256, ... (at most kMaxV4 of them, so D <= 4*256*kMaxV4), all loads are
// issued before the first use, and the row is read once.
constexpr int kMaxV4 = 8;

struct RowRegs {
  float4 v[kMaxV4];
};

// ss = sum of squares of the row held in r (nv float4s in the row)
__device__ __forceinline__ float row_sumsq(const RowRegs& r, int nv) {
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxV4; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    if (idx < nv) ss += r.v[i].x * r.v[i].x + r.v[i].y * r.v[i].y + r.v[i].z * r.v[i].z + r.v[i].w * r.v[i].w;
  }
  return ss;
}

// u = x * rsqrt(mean(x^2) + eps) * g for a row held in registers; u is a GEMM
// activation operand (planes `plane` elements apart).
// With `xf`, the normed row is also stored in fp32 (a residual stream that
// starts at the normed value: the context rows of the input-fusion path).
template <typename T>
__device__ __forceinline__ void norm_store(const RowRegs& r, const T* g, float eps, int D, T* u, size_t plane,
                                           float* red, float* xf = nullptr) {
  const int nv = D >> 2;
  const float rs = rsqrtf(block_sum(row_sumsq(r, nv), red) / (float)D + eps);
#pragma unroll
  for (int i = 0; i < kMaxV4; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    if (idx < nv) {
      const float4 gg = load4(g + 4 * idx);
      const float4 x = r.v[i];
      const float4 o = make_float4(x.x * rs * gg.x, x.y * rs * gg.y, x.z * rs * gg.z, x.w * rs * gg.w);
      put_act4(u, plane, 4 * (size_t)idx, o);
      if (xf) *reinterpret_cast<float4*>(xf + 4 * (size_t)idx) = o;
    }
  }
}

template <typename T>
__device__ __forceinline__ void load_row(const T* x, int D, RowRegs& r) {
  const int nv = D >> 2;
#pragma unroll
  for (int i = 0; i < kMaxV4; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    if (idx < nv) r.v[i] = load4(x + 4 * idx);
  }
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) embed_norm_kernel(const T* embed, const int32_t* anchor, int mask_id,
                                                                 int vocab, int block, int D, const T* g, float eps,
                                                                 float* x, T* u, size_t plane, int* zero_ptr,
                                                                 int zero_n, int32_t* status, const int32_t* ctx_len,
                                                                 const double* inv_freq, int hd, float2* rope) {
  __shared__ float red[32];
  griddep_wait();
  griddep_trigger();
  const int row = blockIdx.x, b = row / block, k = row - b * block;
  if (zero_ptr)
    for (int i = row * blockDim.x + threadIdx.x; i < zero_n; i += gridDim.x * blockDim.x) zero_ptr[i] = 0;
  const int pos = ctx_len[b] + k;
  for (int i = threadIdx.x; i < (hd >> 1); i += blockDim.x) {
    float sn, cs;
    rope_sincos(pos, inv_freq, i, &sn, &cs);
    rope[(size_t)row * (hd >> 1) + i] = make_float2(cs, sn);
  }
  int tok = k == 0 ? anchor[b] : mask_id;
  if (tok < 0 || tok >= vocab) {  // an anchor outside the vocabulary: flag it, read row 0
    if (threadIdx.x == 0) report_status(status, DFLASH_ERR_INVALID_ARG);
    tok = 0;
  }
  RowRegs r;
  load_row(embed + (size_t)tok * D, D, r);
  float* xr = x + (size_t)row * D;
#pragma unroll
  for (int i = 0; i < kMaxV4; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    if (idx < (D >> 2)) *reinterpret_cast<float4*>(xr + 4 * idx) = r.v[i];
  }
  norm_store(r, g, eps, D, u + (size_t)row * D, plane, red);
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_kernel(const float* x, const T* g, float eps, int D, T* u,
                                                              size_t plane) {
  __shared__ float red[32];
  griddep_wait();
  griddep_trigger();
  RowRegs r;
  load_row(x + (size_t)blockIdx.x * D, D, r);
  norm_store(r, g, eps, D, u + (size_t)blockIdx.x * D, plane, red);
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) final_norm_kernel(const float* x, const T* g, float eps, int block,
                                                                 int D, T* hm, size_t plane,
                                                                 unsigned long long* slots) {
  __shared__ float red[32];
  griddep_wait();
  griddep_trigger();
  const int r = blockIdx.x;                   // compact mask-row index
  const int b = r / (block - 1), k = r - b * (block - 1) + 1;
  if (threadIdx.x == 0) slots[r] = 0ull;
  RowRegs v;
  load_row(x + ((size_t)b * block + k) * D, D, v);
  norm_store(v, g, eps, D, hm + (size_t)r * D, plane, red);
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) fuse_norm_kernel(const float* y, const T* g, float eps,
                                                                const int2* rowinfo, int D, T* ht, size_t plane,
                                                                const double* inv_freq, int hd, float2* rope,
                                                                float* xf) {
  __shared__ float red[32];
  griddep_wait();
  griddep_trigger();
  const int row = blockIdx.x;
  {
    const int pos = max(rowinfo[row].y, 0);
    for (int i = threadIdx.x; i < (hd >> 1); i += blockDim.x) {
      float sn, cs;
      rope_sincos(pos, inv_freq, i, &sn, &cs);
      rope[(size_t)row * (hd >> 1) + i] = make_float2(cs, sn);
    }
  }
  if (rowinfo[row].x < 0) {
    for (int i = threadIdx.x; i < (D >> 2); i += blockDim.x) {
      put_act4(ht, plane, (size_t)row * D + 4 * i, make_float4(0.f, 0.f, 0.f, 0.f));
      if (xf) *reinterpret_cast<float4*>(xf + (size_t)row * D + 4 * i) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  RowRegs r;
  load_row(y + (size_t)row * D, D, r);
  norm_store(r, g, eps, D, ht + (size_t)row * D, plane, red, xf ? xf + (size_t)row * D : nullptr);
}

// One CTA: exclusive scan of n_new, per-row (request, position), ctx_len
// update; with `rope`, also the (cos, sin) table of every row's position.
__global__ void __launch_bounds__(1024) inject_prep_kernel(const int32_t* n_new, int32_t* ctx_len, int B,
                                                           int max_rows, int cap, int2* rowinfo, int* zero_ptr,
                                                           int zero_n, int32_t* status, const double* inv_freq,
                                                           int hd, float2* rope) {
  extern __shared__ int sh[];  // [B] offsets, [B] base positions, [B] accepted counts
  int* off = sh;
  int* base = sh + B;
  int* cnt = sh + 2 * B;
  griddep_wait();
  griddep_trigger();
  for (int i = threadIdx.x; i < zero_n; i += blockDim.x) zero_ptr[i] = 0;
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      int n = n_new[b];
      if (n < 0) n = 0;
      int c = ctx_len[b];
      int fit = n;
      if (c + fit > cap) {
        fit = max(0, cap - c);
        report_status(status, DFLASH_ERR_CAPACITY);
      }
      if (acc + n > max_rows) {  // rows beyond the launch are dropped
        report_status(status, DFLASH_ERR_CAPACITY);
        n = max(0, max_rows - acc);
        fit = min(fit, n);
      }
      off[b] = acc;
      base[b] = c;
      cnt[b] = fit;
      acc += n;
      ctx_len[b] = c + fit;
    }
  }
  __syncthreads();
  for (int r = threadIdx.x; r < max_rows; r += blockDim.x) {
    int2 ri = make_int2(-1, -1);
    // the request owning row r: last b with off[b] <= r
    int lo = 0, hi = B - 1, own = -1;
    while (lo <= hi) {
      int mid = (lo + hi) >> 1;
      if (off[mid] <= r) {
        own = mid;
        lo = mid + 1;
      } else {
        hi = mid - 1;
      }
    }
    if (own >= 0) {
      int j = r - off[own];
      if (j < cnt[own]) ri = make_int2(own, base[own] + j);
    }
    rowinfo[r] = ri;
  }
  if (rope) {
    __syncthreads();   // rowinfo of every row written by this CTA
    const int half = hd >> 1;
    for (int e = threadIdx.x; e < max_rows * half; e += blockDim.x) {
      const int r = e / half, i = e - r * half;
      float sn, cs;
      rope_sincos(max(rowinfo[r].y, 0), inv_freq, i, &sn, &cs);
      rope[e] = make_float2(cs, sn);
    }
  }
}

__global__ void argmax_finalize_kernel(const unsigned long long* slots, int rows, int32_t* drafts) {
  griddep_wait();
  griddep_trigger();
  int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r < rows) drafts[r] = unpack_argmax_index(slots[r]);
}

// One warp per request: n = leading positions where d_{k+1} == y_k.
__global__ void verify_kernel(const int32_t* draft, const int32_t* target, int B, int block, int32_t* accept_len,
                              int32_t* out_tokens, int32_t* next_anchor) {
  griddep_wait();
  griddep_trigger();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= B) return;
  const int nd = block - 1;
  const int32_t* d = draft + (size_t)b * nd;
  const int32_t* y = target + (size_t)b * block;
  const bool mismatch = lane < nd && d[lane] != y[lane];
  const unsigned bad = __ballot_sync(0xffffffffu, mismatch);
  const int n = bad ? __ffs(bad) - 1 : nd;
  const int yn = y[n];
  int32_t* out = out_tokens + (size_t)b * block;
  if (lane < block) out[lane] = lane < n ? d[lane] : (lane == n ? yn : -1);
  if (lane == 0) {
    accept_len[b] = n + 1;
    next_anchor[b] = yn;
  }
}

// Synthetic target for benchmarks and tests (one CTA): pattern p = *pidx,
// y[b][k] = match ? d : (d + 1 + off) mod V for k < g-1, y[b][g-1] = bonus;
// adds the previous verification's accepted lengths to *tau_sum; advances p.
__global__ void __launch_bounds__(1024) synthetic_target_kernel(const int32_t* draft, const uint8_t* match,
                                                                const int32_t* off, const int32_t* bonus, int npat,
                                                                long long* pidx, const int32_t* tau,
                                                                long long* tau_sum, int B, int g, int V, int32_t* y) {
  griddep_wait();
  griddep_trigger();
  __shared__ long long sp;
  if (threadIdx.x == 0) sp = *pidx;
  __syncthreads();
  const long long p = sp;
  const int nd = g - 1;
  for (int e = threadIdx.x; e < B * g; e += blockDim.x) {
    const int b = e / g, k = e - b * g;
    int v;
    if (k < nd) {
      const size_t i = ((size_t)p * B + b) * nd + k;
      const long long d = draft[(size_t)b * nd + k];
      v = match[i] ? (int)d : (int)((d + 1 + off[i]) % V);
    } else {
      v = bonus[(size_t)p * B + b];
    }
    y[e] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (tau && tau_sum) {
      long long t = 0;
      for (int b = 0; b < B; ++b) t += tau[b];
      *tau_sum += t;
    }
    *pidx = (p + 1) % npat;
  }
}

// QK-norm then RoPE of one head vector held by a warp: lane l holds
// elements l, l + 32, ... (E = hd/32 of them), so each rotate-half pair
// (d, d + hd/2) sits in one lane (elements e and e + E/2).
template <int E>
__device__ __forceinline__ void qknorm_rope_vec(float* v, const float* g, float eps, int hd, const float2* rope_row) {
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) ss += v[e] * v[e];
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float r = rsqrtf(ss / (float)hd + eps);
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] *= r * g[e];
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int e = 0; e < E / 2; ++e) {
    const float2 cs = rope_row[lane + 32 * e];   // (cos, sin) of pair i = lane + 32 e
    const float a = v[e], b = v[e + E / 2];
    v[e] = a * cs.x - b * cs.y;
    v[e + E / 2] = b * cs.x + a * cs.y;
  }
}

// Block queries (fp32 [b][head][k][hd]) and block keys (T planes
// [b][kvh][plane][k][hd]) of one layer: one warp per head vector.
template <typename T, int E>
__global__ void __launch_bounds__(256) qknorm_block_kernel(float* q, T* kb, const T* g_q, const T* g_k, int B, int block,
                                                           int nq, int nkv, float eps, const float2* rope) {
  griddep_wait();   // the projection that wrote q and kb has finished
  griddep_trigger();
  const int hd = 32 * E, half = hd / 2;
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int nqv = B * nq * block, nkvv = B * nkv * block;
  if (w >= nqv + nkvv) return;
  const bool is_q = w < nqv;
  const int idx = is_q ? w : w - nqv;
  const int nh = is_q ? nq : nkv;
  const int b = idx / (nh * block), rem = idx - b * nh * block, h = rem / block, k = rem - h * block;
  const T* gain = is_q ? g_q : g_k;
  float v[E], g[E];
#pragma unroll
  for (int e = 0; e < E; ++e) g[e] = to_f32(gain[lane + 32 * e]);
  const size_t plane = (size_t)block * hd;
  const size_t base = is_q ? (((size_t)b * nq + h) * block + k) * hd
                           : (((size_t)b * nkv + h) * ActPlanes<T>::n * block + k) * hd;
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = is_q ? q[base + lane + 32 * e] : get_act(kb, plane, base + lane + 32 * e);
  qknorm_rope_vec<E>(v, g, eps, hd, rope + (size_t)(b * block + k) * half);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (is_q)
      q[base + lane + 32 * e] = v[e];
    else
      put_act(kb, plane, base + lane + 32 * e, v[e]);
  }
}

// Injected context keys of layer `layer` in the cache (kvp T planes
// [b][layer][kvh][plane][cap][hd]) for the rows of rowinfo: one warp per
// (row, kv head); padding rows are skipped.
template <typename T, int E>
__global__ void __launch_bounds__(256) qknorm_cache_kernel(T* kc, const int2* rowinfo, int rows, int layer, int layers,
                                                           int nkv, int cap, int kvp, const T* g_k, float eps,
                                                           const float2* rope) {
  griddep_wait();   // the injection projection (or the previous layer's pass) has finished
  griddep_trigger();
  const int hd = 32 * E, half = hd / 2;
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= rows * nkv) return;
  const int row = w / nkv, h = w - row * nkv;
  const int2 ri = rowinfo[row];
  if (ri.x < 0) return;
  float v[E], g[E];
#pragma unroll
  for (int e = 0; e < E; ++e) g[e] = to_f32(g_k[lane + 32 * e]);
  const size_t plane = (size_t)cap * hd;
  const size_t base = ((((size_t)ri.x * layers + layer) * nkv + h) * kvp * cap + ri.y) * hd;
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = get_kv(kc, plane, base + lane + 32 * e, kvp);
  qknorm_rope_vec<E>(v, g, eps, hd, rope + (size_t)row * half);
#pragma unroll
  for (int e = 0; e < E; ++e) put_kv(kc, plane, base + lane + 32 * e, v[e], kvp);
}

}  // namespace

template <typename T>
cudaError_t qknorm_block_launch(float* q, T* kb, const T* g_q, const T* g_k, int B, int block, int nq, int nkv, int hd,
                                float eps, const float2* rope, cudaStream_t s) {
  const int n = B * (nq + nkv) * block;
  if (n == 0) return cudaSuccess;
  if (hd == 64)
    return launch_pdl(qknorm_block_kernel<T, 2>, dim3((n + 7) / 8), dim3(256), 0, s, q, kb, g_q, g_k, B, block, nq, nkv,
                      eps, rope);
  return launch_pdl(qknorm_block_kernel<T, 4>, dim3((n + 7) / 8), dim3(256), 0, s, q, kb, g_q, g_k, B, block, nq, nkv,
                    eps, rope);
}

template <typename T>
cudaError_t qknorm_cache_launch(T* kc, const int2* rowinfo, int rows, int layer, int layers, int nkv, int hd, int cap,
                                int kvp, const T* g_k, float eps, const float2* rope, cudaStream_t s) {
  const int n = rows * nkv;
  if (n == 0) return cudaSuccess;
  if (hd == 64)
    return launch_pdl(qknorm_cache_kernel<T, 2>, dim3((n + 7) / 8), dim3(256), 0, s, kc, rowinfo, rows, layer, layers,
                      nkv, cap, kvp, g_k, eps, rope);
  return launch_pdl(qknorm_cache_kernel<T, 4>, dim3((n + 7) / 8), dim3(256), 0, s, kc, rowinfo, rows, layer, layers, nkv,
                    cap, kvp, g_k, eps, rope);
}

cudaError_t synthetic_target_launch(const int32_t* draft, const uint8_t* match, const int32_t* off,
                                    const int32_t* bonus, int npat, long long* pidx, const int32_t* tau,
                                    long long* tau_sum, int B, int g, int V, int32_t* y, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  return launch_pdl(synthetic_target_kernel, dim3(1), dim3(1024), 0, s, draft, match, off, bonus, npat, pidx, tau,
                    tau_sum, B, g, V, y);
}

template <typename T>
cudaError_t embed_norm_launch(const T* embed, const int32_t* anchor, int mask_id, int vocab, int B, int block, int D,
                              const T* g, float eps, float* x, T* u, size_t plane, int* zero_ptr, int zero_n,
                              int32_t* status, const int32_t* ctx_len, const double* inv_freq, int hd, float2* rope,
                              cudaStream_t s) {
  if (B * block == 0) return cudaSuccess;
  return launch_pdl(embed_norm_kernel<T>, dim3(B * block), dim3(kRowThreads), 0, s, embed, anchor, mask_id, vocab, block,
                    D, g, eps, x, u, plane, zero_ptr, zero_n, status, ctx_len, inv_freq, hd, rope);
}

template <typename T>
cudaError_t rmsnorm_launch(const float* x, const T* g, float eps, int rows, int D, T* u, size_t plane, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  return launch_pdl(rmsnorm_kernel<T>, dim3(rows), dim3(kRowThreads), 0, s, x, g, eps, D, u, plane);
}

template <typename T>
cudaError_t final_norm_launch(const float* x, const T* g, float eps, int B, int block, int D, T* hm, size_t plane,
                              unsigned long long* slots, cudaStream_t s) {
  if (B * (block - 1) == 0) return cudaSuccess;
  return launch_pdl(final_norm_kernel<T>, dim3(B * (block - 1)), dim3(kRowThreads), 0, s, x, g, eps, block, D, hm, plane,
                    slots);
}

template <typename T>
cudaError_t fuse_norm_launch(const float* y, const T* g, float eps, const int2* rowinfo, int rows, int D, T* ht,
                             size_t plane, const double* inv_freq, int hd, float2* rope, cudaStream_t s, float* xf) {
  if (rows == 0) return cudaSuccess;
  return launch_pdl(fuse_norm_kernel<T>, dim3(rows), dim3(kRowThreads), 0, s, y, g, eps, rowinfo, D, ht, plane,
                    inv_freq, hd, rope, xf);
}

cudaError_t inject_prep_launch(const int32_t* n_new, int32_t* ctx_len, int B, int max_rows, int cap, int2* rowinfo,
                               int* zero_ptr, int zero_n, int32_t* status, cudaStream_t s, const double* inv_freq,
                               int hd, float2* rope) {
  return launch_pdl(inject_prep_kernel, dim3(1), dim3(1024), 3 * B * sizeof(int), s, n_new, ctx_len, B, max_rows, cap,
                    rowinfo, zero_ptr, zero_n, status, inv_freq, hd, rope);
}

cudaError_t argmax_finalize_launch(const unsigned long long* slots, int rows, int32_t* drafts, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  return launch_pdl(argmax_finalize_kernel, dim3((rows + 255) / 256), dim3(256), 0, s, slots, rows, drafts);
}

cudaError_t verify_launch(const int32_t* draft, const int32_t* target, int B, int block, int32_t* accept_len,
                          int32_t* out_tokens, int32_t* next_anchor, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  const int warps = 4;
  return launch_pdl(verify_kernel, dim3((B + warps - 1) / warps), dim3(32 * warps), 0, s, draft, target, B, block,
                    accept_len, out_tokens, next_anchor);
}

#define DFLASH_EW_INST(T)                                                                                        \
  template cudaError_t embed_norm_launch<T>(const T*, const int32_t*, int, int, int, int, int, const T*, float,     \
                                            float*, T*, size_t, int*, int, int32_t*, const int32_t*,              \
                                            const double*, int, float2*, cudaStream_t);                          \
  template cudaError_t rmsnorm_launch<T>(const float*, const T*, float, int, int, T*, size_t, cudaStream_t);      \
  template cudaError_t final_norm_launch<T>(const float*, const T*, float, int, int, int, T*, size_t,              \
                                            unsigned long long*, cudaStream_t);                                   \
  template cudaError_t fuse_norm_launch<T>(const float*, const T*, float, const int2*, int, int, T*, size_t,      \
                                           const double*, int, float2*, cudaStream_t, float*);                    \
  template cudaError_t qknorm_block_launch<T>(float*, T*, const T*, const T*, int, int, int, int, int, float,      \
                                              const float2*, cudaStream_t);                                       \
  template cudaError_t qknorm_cache_launch<T>(T*, const int2*, int, int, int, int, int, int, int, const T*, float, \
                                              const float2*, cudaStream_t);

DFLASH_EW_INST(float)
DFLASH_EW_INST(__nv_bfloat16)

// Self-test of the bounded waits: one thread waits on a shared-memory
// mbarrier that nothing ever arrives on, with the same bounded wait the
// pipelines use; when `budget` SM cycles have passed it sets
// DFLASH_ERR_TIMEOUT in the status word and the kernel returns.
__global__ void wait_selftest_kernel(long long budget, int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    (void)ptx::mbar_wait(&bar, 0, budget, status);
  }
}

cudaError_t wait_selftest_launch(long long budget_cycles, int32_t* status, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(budget_cycles, status);
  return cudaGetLastError();
}

}  // namespace dflash
