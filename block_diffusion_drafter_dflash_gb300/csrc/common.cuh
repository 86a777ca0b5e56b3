// Shared device/host definitions of the DFlash draft-cycle library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/dflash.h"

namespace dflash {

constexpr int kTileN = 128;      // output features per GEMM tile (two 64-row halves)
constexpr int kHalfN = 64;
constexpr int kMaxSeg = 16;      // weight matrices one GEMM launch may read
constexpr int kMaxBlock = 32;    // largest block_size (a warp per request in verify)

// ---------------------------------------------------------------- dependent launches
// Kernels of the cycle are launched with programmatic dependent launch: a
// kernel may become resident while its predecessor drains, prefetch what does
// not depend on it (weights), and must call griddep_wait() before it reads or
// writes anything an earlier kernel of the stream touches.  griddep_trigger()
// lets the successor launch once every CTA of this grid has started.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Experiment switches (ring depths, split factors, plan logging) are read
// from the environment only when DFLASH_DEBUG=1: a normal process never has
// its plans changed by a stray variable.  Returns the variable or nullptr.
inline const char* debug_env(const char* name) {
  static const bool on = [] {
    const char* d = getenv("DFLASH_DEBUG");
    return d && strcmp(d, "1") == 0;
  }();
  return on ? getenv(name) : nullptr;
}

inline bool pdl_enabled() {
  static int on = -1;
  if (on < 0) {
    const char* e = getenv("DFLASH_PDL");
    on = (e && strcmp(e, "0") == 0) ? 0 : 1;
  }
  return on == 1;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- scalar types
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// ---------------------------------------------------------------- activations
// Every tensor handed from one step of the cycle to the next is kept at fp32
// precision.  fp32 models store it as fp32 (one plane).  bf16 models store
// each value v as two bf16 planes, hi = bf16(v) and lo = bf16(v - hi), which
// the tensor cores consume as two operands against the same (exact) bf16
// weights: hi*W + lo*W carries ~16 significant bits of v instead of 8.
template <typename T> struct ActPlanes;
template <> struct ActPlanes<float> { static constexpr int n = 1; };
template <> struct ActPlanes<__nv_bfloat16> { static constexpr int n = 2; };

__device__ __forceinline__ void put_act(float* base, size_t /*plane*/, size_t i, float v) { base[i] = v; }
__device__ __forceinline__ void put_act(__nv_bfloat16* base, size_t plane, size_t i, float v) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  base[i] = hi;
  base[plane + i] = __float2bfloat16_rn(v - __bfloat162float(hi));
}
// One cached context K/V value: the hi and lo bf16 planes (kvp = 2) or the
// value rounded to one bf16 (kvp = 1); fp32 caches keep the value.
__device__ __forceinline__ void put_kv(float* base, size_t /*plane*/, size_t i, float v, int /*kvp*/) { base[i] = v; }
__device__ __forceinline__ void put_kv(__nv_bfloat16* base, size_t plane, size_t i, float v, int kvp) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  base[i] = hi;
  if (kvp == 2) base[plane + i] = __float2bfloat16_rn(v - __bfloat162float(hi));
}
// four consecutive values (i a multiple of 4)
__device__ __forceinline__ void put_act4(float* base, size_t /*plane*/, size_t i, float4 v) {
  *reinterpret_cast<float4*>(base + i) = v;
}
__device__ __forceinline__ void put_act4(__nv_bfloat16* base, size_t plane, size_t i, float4 v) {
  __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
  float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
  __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - f0.x, v.y - f0.y), l1 = __floats2bfloat162_rn(v.z - f1.x, v.w - f1.y);
  uint2 hi, lo;
  hi.x = *reinterpret_cast<uint32_t*>(&h0);
  hi.y = *reinterpret_cast<uint32_t*>(&h1);
  lo.x = *reinterpret_cast<uint32_t*>(&l0);
  lo.y = *reinterpret_cast<uint32_t*>(&l1);
  *reinterpret_cast<uint2*>(base + i) = hi;
  *reinterpret_cast<uint2*>(base + plane + i) = lo;
}
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  uint2 r = *reinterpret_cast<const uint2*>(p);
  float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&r.x));
  float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&r.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float get_act(const float* base, size_t /*plane*/, size_t i) { return base[i]; }
__device__ __forceinline__ float get_act(const __nv_bfloat16* base, size_t plane, size_t i) {
  return __bfloat162float(base[i]) + __bfloat162float(base[plane + i]);
}
// a cached context K/V value of `kvp` planes (see put_kv)
__device__ __forceinline__ float get_kv(const float* base, size_t /*plane*/, size_t i, int /*kvp*/) { return base[i]; }
__device__ __forceinline__ float get_kv(const __nv_bfloat16* base, size_t plane, size_t i, int kvp) {
  return kvp == 2 ? get_act(base, plane, i) : __bfloat162float(base[i]);
}

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
  int map0, map1;  // tensor-map indices of w0 / w1 (tensor-core path)
  int tiles;       // 128-feature output tiles in this segment
  int tile_begin;  // first global tile index of this segment
  int paired;
  int tag;         // meaning chosen by the epilogue (Q/K/V, layer, ...)
  int tw;          // persistent kernel: features per tile (128 or 256; paired: 128 gate + 128 up)
};

struct GemmProblem {
  const void* x;   // activations: `planes` planes of [M][K], row stride ldx elements
  int ldx;
  int planes;          // 1, or 2 for a hi/lo bf16 pair
  size_t plane_stride; // elements from plane 0 to plane 1 (a multiple of ldx)
  int M;
  int K;
  int nseg;
  int total_tiles;
  int splits;          // split-K factor (1 = none)
  int kblocks_per_split;   // in units of 64 columns of K
  int stages;          // shared-memory pipeline depth (tensor-core path)
  float* partial;      // [splits][M][total_tiles*128] when splits > 1
  int* counters;       // [token tiles][total_tiles], zero between launches
  const void* wmaps;   // device array of weight tensor maps (tensor-core path)
  int32_t* status;     // device status word
  unsigned long long* trace;   // per-CTA timestamps (8 per CTA) or nullptr
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
