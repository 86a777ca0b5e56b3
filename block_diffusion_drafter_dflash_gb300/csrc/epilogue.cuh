// GEMM epilogues of the draft cycle.  Each one consumes a finished fp32 output
// tile held in shared memory, feature-major: tile[n * ld + m] for the 128
// output features n of global tile `gtile` and the token rows m0 .. m0+mc-1.
// Threads tid = 0 .. nth-1 (a multiple of 128) call the functor together;
// consecutive threads take consecutive features so that global stores are
// coalesced (consecutive rows where the destination is feature-major: the
// hd-major V of bf16 models).
#pragma once

#include "common.cuh"

namespace dflash {

// Y[row][gtile*128 + n] = acc  (fp32; the fusion projection before its RMSNorm)
struct EpiStoreF32 {
  float* y;
  int ldy;
  __device__ __forceinline__ void operator()(const float* t, int ld, int m0, int mc, int gtile, const GemmSeg&,
                                             int, int tid, int nth) const {
    for (int idx = tid; idx < mc * kTileN; idx += nth) {
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
                                             int, int tid, int nth) const {
    const int n = tid & (kTileN - 1), step = nth / kTileN;
    float* col = x + (size_t)gtile * kTileN + n;
    for (int mb = tid / kTileN; mb < mc; mb += 8 * step) {
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
                                             int tis, int tid, int nth) const {
    for (int idx = tid; idx < mc * kHalfN; idx += nth) {
      int m = idx / kHalfN, c = idx % kHalfN;
      float g = t[c * ld + m], u = t[(c + kHalfN) * ld + m];
      float s = g / (1.0f + __expf(-g));
      put_act(a, plane, (size_t)(m0 + m) * lda + (size_t)tis * kHalfN + c, s * u);
    }
  }
};

// RoPE in the Q/K/V and injection epilogues is rotate-half: feature d < hd/2
// pairs with d + hd/2 of the same head (both in the same 128-feature tile),
// x' = x cos - x_partner sin for the first half, x cos + x_partner sin for the
// second, with (cos, sin) of the row's position from a per-row table.  With
// no table (rope == nullptr: QK-norm models, whose norm comes before RoPE and
// needs a whole head) the values are stored unrotated for qknorm_rope.

// Block Q/K/V of one draft layer: tag 0 = Q, 1 = K, 2 = V.  Row = b*block + k
// sits at position ctx_len[b] + k, whose RoPE (cos, sin) table rope[row][hd/2]
// was filled by the embedding kernel; Q and K get RoPE.  Q is fp32
// [b][head][k][hd]; K and V are stored like the context cache: K as
// [b][head][plane][k][hd] of T (two bf16 planes hi, lo for bf16 models); V
// likewise for fp32 models, hd-major [b][head][plane][hd][vpitch] for bf16
// models (vpitch = block rounded up to 8).
template <typename T>
struct EpiQKV {
  float* q;
  T* kb;
  T* vb;
  const float2* rope;
  int block, nq, nkv, hd;
  int vpitch;
  // thread n owns feature n of the tile; the RoPE entries of 8 rows are
  // loaded before any store so that their loads overlap
  __device__ __forceinline__ void operator()(const float* t, int ld, int m0, int mc, int, const GemmSeg& sg,
                                             int tis, int tid, int nth) const {
    const int tag = sg.tag;
    T* dkv = tag == 1 ? kb : vb;
    const int nh = tag == 0 ? nq : nkv, half = hd >> 1;
    const int planes = ActPlanes<T>::n;
    if (tag == 2 && planes == 2) {   // bf16 V, hd-major: consecutive threads take consecutive rows
      if (mc <= 0) return;
      const int hsh = 31 - __clz(hd);   // hd is a power of two
      const int fstep = nth / mc, mstep = nth - fstep * mc;
      int f = tid / mc, m = tid - f * mc;   // element tid, tid + nth, ... of the [feature][row] tile
      while (f < kTileN) {
        const int row = m0 + m, b = row / block, k = row - b * block;
        const int feat = tis * kTileN + f, head = feat >> hsh, d = feat & (hd - 1);
        put_act(dkv, (size_t)hd * vpitch, (((size_t)b * nh + head) * 2 * hd + d) * vpitch + k, t[f * ld + m]);
        f += fstep;
        m += mstep;
        if (m >= mc) {
          m -= mc;
          ++f;
        }
      }
      return;
    }
    const int n = tid & (kTileN - 1), step = nth / kTileN;
    const int hsh = 31 - __clz(hd);   // hd is a power of two
    const int feat = tis * kTileN + n, head = feat >> hsh, d = feat & (hd - 1);
    const int i = d < half ? d : d - half;
    const int pn = d < half ? n + half : n - half;
    for (int mb = tid / kTileN; mb < mc; mb += 8 * step) {
      float2 sc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = mb + j * step;
        sc[j] = (rope && tag != 2 && m < mc) ? __ldg(rope + (size_t)(m0 + m) * half + i) : make_float2(1.f, 0.f);
      }
      int b = (m0 + mb) / block, k = m0 + mb - b * block;   // (request, block position) of row m0 + mb
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = mb + j * step;
        if (m >= mc) break;
        if (j > 0) {   // the next row, `step` further on
          k += step;
          while (k >= block) {
            k -= block;
            ++b;
          }
        }
        const float v = t[n * ld + m], pv = t[pn * ld + m];
        const float r = tag == 2 ? v : (d < half ? v * sc[j].x - pv * sc[j].y : v * sc[j].x + pv * sc[j].y);
        if (tag == 0)
          q[(((size_t)b * nh + head) * block + k) * hd + d] = r;
        else
          put_act(dkv, (size_t)block * hd, (((size_t)b * nh + head) * planes * block + k) * hd + d, r);
      }
    }
  }
};

// Context K/V injection: tag = 2*layer + (0: K, 1: V).  rowinfo[row] =
// (request, position) or (-1, -1) for padding rows; rope[row][hd/2] = (cos,
// sin) at that position.  Writes the cache [b][layer][kvh][plane][pos][hd] of
// T (fp32 one plane; bf16 two planes hi, lo) — for bf16 models V hd-major,
// [b][layer][kvh][plane][hd][vpitch] (vpitch = capacity rounded up to 8);
// K gets RoPE at its position.
template <typename T>
struct EpiInject {
  T* kc;
  T* vc;
  const int2* rowinfo;
  const float2* rope;
  int layers, nkv, hd, cap;
  int vpitch;
  int kvp;   // bf16 planes of each cached value (2: hi and lo, 1: rounded); 1 for fp32 caches
  __device__ __forceinline__ void operator()(const float* t, int ld, int m0, int mc, int, const GemmSeg& sg,
                                             int tis, int tid, int nth) const {
    const int layer = sg.tag >> 1, is_v = sg.tag & 1, half = hd >> 1;
    T* dst = is_v ? vc : kc;
    const int planes = kvp;
    if (is_v && ActPlanes<T>::n == 2) {
      // bf16 V is hd-major: consecutive threads take consecutive rows
      // (positions) of one feature, so that a warp's stores are contiguous
      if (mc <= 0) return;
      const int hsh = 31 - __clz(hd);   // hd is a power of two
      const int fstep = nth / mc, mstep = nth - fstep * mc;
      int f = tid / mc, m = tid - f * mc;   // element tid, tid + nth, ... of the [feature][row] tile
      while (f < kTileN) {
        const int2 ri = __ldg(rowinfo + m0 + m);
        if (ri.x >= 0) {
          const int feat = tis * kTileN + f, head = feat >> hsh, d = feat & (hd - 1);
          put_kv(dst, (size_t)hd * vpitch,
                 ((((size_t)ri.x * layers + layer) * nkv + head) * planes * hd + d) * vpitch + ri.y, t[f * ld + m],
                 planes);
        }
        f += fstep;
        m += mstep;
        if (m >= mc) {
          m -= mc;
          ++f;
        }
      }
      return;
    }
    const int n = tid & (kTileN - 1), step = nth / kTileN;
    const int hsh = 31 - __clz(hd);   // hd is a power of two
    const int feat = tis * kTileN + n, head = feat >> hsh, d = feat & (hd - 1);
    const int i = d < half ? d : d - half;
    const int pn = d < half ? n + half : n - half;
    for (int mb = tid / kTileN; mb < mc; mb += 8 * step) {
      int2 ri[8];
      float2 sc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = mb + j * step;
        ri[j] = m < mc ? __ldg(rowinfo + m0 + m) : make_int2(-1, -1);
        sc[j] = (rope && !is_v && m < mc) ? __ldg(rope + (size_t)(m0 + m) * half + i) : make_float2(1.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = mb + j * step;
        if (m >= mc) break;
        if (ri[j].x < 0) continue;
        const float v = t[n * ld + m], pv = t[pn * ld + m];
        const float r = is_v ? v : (d < half ? v * sc[j].x - pv * sc[j].y : v * sc[j].x + pv * sc[j].y);
        put_kv(dst, (size_t)cap * hd,
               ((((size_t)ri[j].x * layers + layer) * nkv + head) * planes * cap + ri[j].y) * hd + d, r, planes);
      }
    }
  }
};

// Query projection of injected context rows (input-fusion path): y[row][f]
// fp32 with RoPE at the row's position (rope[row][hd/2], as filled with the
// injection's row map); rows keep the injection's packed order.
struct EpiRowsRope {
  float* y;
  int ldy;
  const float2* rope;
  int hd;
  __device__ __forceinline__ void operator()(const float* t, int ld, int m0, int mc, int gtile, const GemmSeg&,
                                             int, int tid, int nth) const {
    const int n = tid & (kTileN - 1), step = nth / kTileN, half = hd >> 1;
    const int feat = gtile * kTileN + n, d = feat & (hd - 1);
    const int i = d < half ? d : d - half;
    const int pn = d < half ? n + half : n - half;
    for (int m = tid / kTileN; m < mc; m += step) {
      const float2 sc = __ldg(rope + (size_t)(m0 + m) * half + i);
      const float v = t[n * ld + m], pv = t[pn * ld + m];
      y[(size_t)(m0 + m) * ldy + feat] = d < half ? v * sc.x - pv * sc.y : v * sc.x + pv * sc.y;
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
                                             int, int tid, int nth) const {
    if (logits) {
      for (int idx = tid; idx < mc * kTileN; idx += nth) {
        int m = idx / kTileN, n = idx % kTileN;
        logits[(size_t)(m0 + m) * vocab + (size_t)gtile * kTileN + n] = t[n * ld + m];
      }
    }
    const int lane = tid & 31, warp = tid >> 5, nw = nth >> 5;
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
