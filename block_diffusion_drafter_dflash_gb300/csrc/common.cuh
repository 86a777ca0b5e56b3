// Shared device/host definitions of the DFlash draft-cycle library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflash.h"

namespace dflash {

constexpr int kTileN = 128;      // output features per GEMM tile (two 64-row halves)
constexpr int kHalfN = 64;
constexpr int kMaxSeg = 16;      // weight matrices one GEMM launch may read
constexpr int kMaxBlock = 32;    // largest block_size (a warp per request in verify)

// ---------------------------------------------------------------- scalar types
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// ---------------------------------------------------------------- device status
// First device-detected error wins; later ones are dropped.
__device__ __forceinline__ void report_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// ---------------------------------------------------------------- RoPE
// Rotate-half RoPE angle for pair index i at integer position `pos`:
// pos * theta^(-2i/hd).  The product and its reduction to [-pi, pi] are done
// in double so that positions in the tens of thousands keep full fp32
// accuracy in the final sin/cos.
__device__ __forceinline__ void rope_sincos(int pos, const double* inv_freq, int i, float* s, float* c) {
  const double two_pi = 6.283185307179586476925286766559;
  double a = (double)pos * inv_freq[i];
  double k = rint(a * (1.0 / two_pi));
  float r = (float)fma(-k, two_pi, a);
  sincosf(r, s, c);
}

// ---------------------------------------------------------------- argmax packing
// Orderable 64-bit key: larger float first, then LOWER index (ties -> lowest id).
__device__ __forceinline__ unsigned long long pack_argmax(float v, int idx) {
  unsigned int b = __float_as_uint(v);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)b << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned int)idx);
}
__device__ __forceinline__ int unpack_argmax_index(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (unsigned int)(k & 0xFFFFFFFFull));
}

// ---------------------------------------------------------------- GEMM problem
// Y[m, n] = sum_k X[m, k] W[n, k] over a list of weight segments.  Each
// 128-feature output tile is assembled from two 64-row halves:
//   unpaired segment, tile t: rows [128t, 128t+64) and [128t+64, 128t+128) of w0
//   paired segment,   tile t: rows [64t, 64t+64) of w0 and of w1
// (paired tiles put a SwiGLU gate half next to its up half).
struct GemmSeg {
  const void* w0;
  const void* w1;
  int tiles;       // 128-feature output tiles in this segment
  int tile_begin;  // first global tile index of this segment
  int paired;
  int tag;         // meaning chosen by the epilogue (Q/K/V, layer, ...)
};

struct GemmProblem {
  const void* x;   // activations [M][K], row stride ldx elements
  int ldx;
  int M;
  int K;
  int nseg;
  int total_tiles;
  int splits;          // split-K factor (1 = none)
  int kblocks_per_split;   // in units of 64 columns of K
  float* partial;      // [splits][M][total_tiles*128] when splits > 1
  int* counters;       // [token tiles][total_tiles], zero between launches
  GemmSeg seg[kMaxSeg];
};

__host__ __device__ __forceinline__ int find_seg(const GemmProblem& p, int tile) {
  int s = 0;
  while (s + 1 < p.nseg && tile >= p.seg[s + 1].tile_begin) ++s;
  return s;
}

// First weight row of half `h` of tile `t` within segment `sg`, and its base.
__host__ __device__ __forceinline__ const void* half_base(const GemmSeg& sg, int h) {
  return (sg.paired && h) ? sg.w1 : sg.w0;
}
__host__ __device__ __forceinline__ int half_first_row(const GemmSeg& sg, int t, int h) {
  return sg.paired ? kHalfN * t : kTileN * t + kHalfN * h;
}

}  // namespace dflash
