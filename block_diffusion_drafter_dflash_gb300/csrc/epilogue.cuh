// GEMM epilogues of the draft cycle.  Each one consumes a finished fp32 output
// tile held in shared memory, feature-major: tile[n * ld + m] for the 128
// output features n of global tile `gtile` and the token rows m0 .. m0+mc-1.
// Every thread of the CTA calls the functor; consecutive threads take
// consecutive features so that global stores are coalesced.
#pragma once

#include "common.cuh"

namespace dflash {

// Y[row][gtile*128 + n] = acc  (fp32; the fusion projection before its RMSNorm)
struct EpiStoreF32 {
  float* y;
  int ldy;
  __device__ __forceinline__ void operator()(const float* t, int ld, int m0, int mc, int gtile, const GemmSeg&,
                                             int) const {
    for (int idx = threadIdx.x; idx < mc * kTileN; idx += blockDim.x) {
      int m = idx / kTileN, n = idx % kTileN;
      y[(size_t)(m0 + m) * ldy + (size_t)gtile * kTileN + n] = t[n * ld + m];
    }
  }
};

// x[row][feature] += acc  (fp32 residual stream; W_O and W_D outputs).
// Thread n owns feature n of a group of rows: the residual values of 8 rows
// are loaded before any is stored, so the loads overlap.
struct EpiResidual {
  float* x;
  int ldx;
  __device__ __forceinline__ void operator()(const float* t, int ld, int m0, int mc, int gtile, const GemmSeg&,
                                             int) const {
    const int n = threadIdx.x & (kTileN - 1), step = blockDim.x / kTileN;
    float* col = x + (size_t)gtile * kTileN + n;
    for (int mb = threadIdx.x / kTileN; mb < mc; mb += 8 * step) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = mb + j * step;
        if (m < mc) v[j] = col[(size_t)(m0 + m) * ldx];
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = mb + j * step;
        if (m < mc) col[(size_t)(m0 + m) * ldx] = v[j] + t[n * ld + m];
      }
    }
  }
};

// a[row][j] = silu(gate_j) * up_j for a paired (W_G, W_U) tile: features
// 0..63 of the tile are gate rows 64t.., features 64..127 the matching up rows.
// `a` is the next GEMM's activation operand (planes `plane` elements apart).
template <typename T>
struct EpiSwiGLU {
  T* a;
  int lda;
  size_t plane;
  __device__ __forceinline__ void operator()(const float* t, int ld, int m0, int mc, int, const GemmSeg&,
                                             int tis) const {
    for (int idx = threadIdx.x; idx < mc * kHalfN; idx += blockDim.x) {
      int m = idx / kHalfN, c = idx % kHalfN;
      float g = t[c * ld + m], u = t[(c + kHalfN) * ld + m];
      float s = g / (1.0f + __expf(-g));
      put_act(a, plane, (size_t)(m0 + m) * lda + (size_t)tis * kHalfN + c, s * u);
    }
  }
};

// Rotate-half RoPE of feature n of a tile holding whole heads of size hd.
__device__ __forceinline__ float rope_apply(const float* t, int ld, int m, int n, int d, int hd, int pos,
                                           const double* inv_freq) {
  const int half = hd >> 1;
  const float v = t[n * ld + m];
  const int i = d < half ? d : d - half;
  const int pn = d < half ? n + half : n - half;
  const float p = t[pn * ld + m];
  float s, c;
  rope_sincos(pos, inv_freq, i, &s, &c);
  return d < half ? v * c - p * s : v * c + p * s;
}

// Block Q/K/V of one draft layer: tag 0 = Q, 1 = K, 2 = V.  Row = b*block + k
// sits at position ctx_len[b] + k; Q and K get RoPE.  Outputs are fp32,
// head-major [b][head][k][hd].
struct EpiQKV {
  float* q;
  float* kb;
  float* vb;
  const int32_t* ctx_len;
  const double* inv_freq;
  int block, nq, nkv, hd;
  __device__ __forceinline__ void operator()(const float* t, int ld, int m0, int mc, int, const GemmSeg& sg,
                                             int tis) const {
    const int tag = sg.tag;
    float* dst = tag == 0 ? q : (tag == 1 ? kb : vb);
    const int nh = tag == 0 ? nq : nkv;
    for (int idx = threadIdx.x; idx < mc * kTileN; idx += blockDim.x) {
      int m = idx / kTileN, n = idx % kTileN;
      int row = m0 + m, b = row / block, k = row - b * block;
      int feat = tis * kTileN + n, head = feat / hd, d = feat - head * hd;
      float v = tag == 2 ? t[n * ld + m] : rope_apply(t, ld, m, n, d, hd, __ldg(ctx_len + b) + k, inv_freq);
      dst[(((size_t)b * nh + head) * block + k) * hd + d] = v;
    }
  }
};

// Context K/V injection: tag = 2*layer + (0: K, 1: V).  rowinfo[row] =
// (request, position) or (-1, -1) for padding rows.  Writes the cache
// [b][layer][kvh][pos][hd] (fp32); K gets RoPE at its absolute position.
struct EpiInject {
  float* kc;
  float* vc;
  const int2* rowinfo;
  const double* inv_freq;
  int layers, nkv, hd, cap;
  __device__ __forceinline__ void operator()(const float* t, int ld, int m0, int mc, int, const GemmSeg& sg,
                                             int tis) const {
    const int layer = sg.tag >> 1, is_v = sg.tag & 1;
    float* dst = is_v ? vc : kc;
    for (int idx = threadIdx.x; idx < mc * kTileN; idx += blockDim.x) {
      int m = idx / kTileN, n = idx % kTileN;
      int2 ri = __ldg(rowinfo + m0 + m);
      if (ri.x < 0) continue;
      int feat = tis * kTileN + n, head = feat / hd, d = feat - head * hd;
      float v = is_v ? t[n * ld + m] : rope_apply(t, ld, m, n, d, hd, ri.y, inv_freq);
      dst[((((size_t)ri.x * layers + layer) * nkv + head) * cap + ri.y) * hd + d] = v;
    }
  }
};

// LM head: optional fp32 logits, and a packed (value, lowest index) atomicMax
// per row into slots[row] (zeroed beforehand).
struct EpiArgmax {
  unsigned long long* slots;
  float* logits;  // [rows][vocab] or nullptr
  int vocab;
  __device__ __forceinline__ void operator()(const float* t, int ld, int m0, int mc, int gtile, const GemmSeg&,
                                             int) const {
    if (logits) {
      for (int idx = threadIdx.x; idx < mc * kTileN; idx += blockDim.x) {
        int m = idx / kTileN, n = idx % kTileN;
        logits[(size_t)(m0 + m) * vocab + (size_t)gtile * kTileN + n] = t[n * ld + m];
      }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int m = warp; m < mc; m += nw) {
      unsigned long long best = 0ull;
      for (int n = lane; n < kTileN; n += 32) {
        unsigned long long k = pack_argmax(t[n * ld + m], gtile * kTileN + n);
        best = k > best ? k : best;
      }
      for (int o = 16; o; o >>= 1) {
        unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
      if (lane == 0) atomicMax(slots + m0 + m, best);
    }
  }
};

}  // namespace dflash
