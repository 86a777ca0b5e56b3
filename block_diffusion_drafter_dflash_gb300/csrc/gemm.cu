// Projection GEMMs of the draft cycle: Y = X W^T with a fused epilogue.
//
// CUDA-core kernel: a CTA owns one 128-feature output tile, 16 token rows and
// one split of K.  Weights and activations are staged through shared memory
// in 32-column slices and accumulated in fp32.  With split-K each split writes
// an fp32 partial tile to scratch; the last CTA of a tile (counted with an
// atomic ticket, no waiting) adds the partials in split order — so results do
// not depend on scheduling — and runs the epilogue.
#include <algorithm>
#include <type_traits>

#include "gemm.cuh"

namespace dflash {

namespace {

constexpr int kSimtBM = 16;
constexpr int kSimtBK = 32;
constexpr int kSimtThreads = 256;

template <typename T, class Epi>
__global__ void __launch_bounds__(kSimtThreads) gemm_simt_kernel(const __grid_constant__ GemmProblem p,
                                                                 const __grid_constant__ Epi epi) {
  __shared__ float sw[kTileN][kSimtBK + 1];
  __shared__ float sx[kSimtBM][kSimtBK + 1];
  __shared__ float st[kTileN * (kSimtBM + 1)];
  __shared__ int s_last;

  const int gtile = blockIdx.x, split = blockIdx.y, mt = blockIdx.z;
  const int m0 = mt * kSimtBM;
  const int mc = min(kSimtBM, p.M - m0);
  const int si = find_seg(p, gtile);
  const GemmSeg& sg = p.seg[si];
  const int tis = gtile - sg.tile_begin;
  const int tid = threadIdx.x, n = tid & (kTileN - 1), mh = tid >> 7;
  const int k_begin = split * p.kblocks_per_split * 64;
  const int k_end = min(p.K, k_begin + p.kblocks_per_split * 64);
  const T* X = static_cast<const T*>(p.x);
  griddep_wait();
  griddep_trigger();

  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;

  for (int k0 = k_begin; k0 < k_end; k0 += kSimtBK) {
    for (int e = tid; e < kTileN * kSimtBK; e += kSimtThreads) {
      int r = e / kSimtBK, kk = e % kSimtBK, h = r / kHalfN;
      const T* wb = static_cast<const T*>(half_base(sg, h));
      int row = half_first_row(sg, tis, h) + (r & (kHalfN - 1));
      sw[r][kk] = to_f32(wb[(size_t)row * p.K + k0 + kk]);
    }
    for (int e = tid; e < kSimtBM * kSimtBK; e += kSimtThreads) {
      int m = e / kSimtBK, kk = e % kSimtBK;
      float v = 0.f;
      if (m < mc)
        for (int pl = 0; pl < p.planes; ++pl) v += to_f32(X[pl * p.plane_stride + (size_t)(m0 + m) * p.ldx + k0 + kk]);
      sx[m][kk] = v;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kSimtBK; ++kk) {
      float w = sw[n][kk];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, sx[mh * 8 + i][kk], acc[i]);
    }
    __syncthreads();
  }

  const int ld = kSimtBM + 1;
  if (p.splits == 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) st[n * ld + mh * 8 + i] = acc[i];
  } else {
    const size_t ntot = (size_t)p.total_tiles * kTileN;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int m = mh * 8 + i;
      if (m < mc) p.partial[((size_t)split * p.M + m0 + m) * ntot + (size_t)gtile * kTileN + n] = acc[i];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      int* c = p.counters + mt * p.total_tiles + gtile;
      int old = atomicAdd(c, 1);
      s_last = old == p.splits - 1;
      if (s_last) *c = 0;  // ready for the next launch
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int m = mh * 8 + i;
      float s = 0.f;
      if (m < mc)
        for (int sp = 0; sp < p.splits; ++sp)
          s += __ldcg(p.partial + ((size_t)sp * p.M + m0 + m) * ntot + (size_t)gtile * kTileN + n);
      st[n * ld + m] = s;
    }
  }
  __syncthreads();
  epi(st, ld, m0, mc, gtile, sg, tis, threadIdx.x, blockDim.x);
}

}  // namespace

GemmPlan plan_gemm(int dtype, int M, int K, int tiles, int sms, int tc, int planes) {
  if (dtype == DFLASH_DTYPE_BF16 && tc) return plan_gemm_tc(M, K, tiles, sms, planes);
  GemmPlan g{};
  g.tc = 0;
  g.planes = planes;
  g.bm = kSimtBM;
  g.token_tiles = (M + kSimtBM - 1) / kSimtBM;
  const int kblocks = K / 64;
  const long ctas = (long)tiles * g.token_tiles;
  int splits = (int)std::max(1L, std::min<long>((2L * sms + ctas - 1) / ctas, 16L));
  splits = std::min(splits, std::max(1, kblocks));
  g.kblocks_per_split = (kblocks + splits - 1) / splits;
  g.splits = (kblocks + g.kblocks_per_split - 1) / g.kblocks_per_split;
  g.partial_floats = g.splits > 1 ? (size_t)g.splits * M * tiles * kTileN : 0;
  g.counters = g.splits > 1 ? g.token_tiles * tiles : 0;
  return g;
}

void apply_plan(GemmProblem& p, const GemmPlan& plan, float* partial, int* counters) {
  p.splits = plan.splits;
  p.kblocks_per_split = plan.kblocks_per_split;
  p.stages = plan.stages;
  p.partial = partial;
  p.counters = counters;
}

template <typename T, class Epi>
cudaError_t gemm_launch(const GemmProblem& p, const GemmPlan& plan, const Epi& epi, cudaStream_t s) {
  if (p.M <= 0 || p.total_tiles <= 0) return cudaSuccess;
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    if (plan.tc) return gemm_tc_launch<Epi>(p, plan, epi, s);
  }
  dim3 grid(p.total_tiles, plan.splits, plan.token_tiles);
  return launch_pdl(gemm_simt_kernel<T, Epi>, grid, dim3(kSimtThreads), 0, s, p, epi);
}

#define DFLASH_GEMM_INST(T)                                                                            \
  template cudaError_t gemm_launch<T, EpiStoreF32>(const GemmProblem&, const GemmPlan&, const EpiStoreF32&, \
                                                   cudaStream_t);                                       \
  template cudaError_t gemm_launch<T, EpiResidual>(const GemmProblem&, const GemmPlan&, const EpiResidual&, \
                                                   cudaStream_t);                                       \
  template cudaError_t gemm_launch<T, EpiSwiGLU<T>>(const GemmProblem&, const GemmPlan&,                 \
                                                    const EpiSwiGLU<T>&, cudaStream_t);                 \
  template cudaError_t gemm_launch<T, EpiQKV<T>>(const GemmProblem&, const GemmPlan&, const EpiQKV<T>&,  \
                                                 cudaStream_t);                                         \
  template cudaError_t gemm_launch<T, EpiInject<T>>(const GemmProblem&, const GemmPlan&,                 \
                                                    const EpiInject<T>&, cudaStream_t);                 \
  template cudaError_t gemm_launch<T, EpiArgmax>(const GemmProblem&, const GemmPlan&, const EpiArgmax&,  \
                                                 cudaStream_t);                                         \
  template cudaError_t gemm_launch<T, EpiRowsRope>(const GemmProblem&, const GemmPlan&, const EpiRowsRope&, \
                                                   cudaStream_t);

DFLASH_GEMM_INST(float)
DFLASH_GEMM_INST(__nv_bfloat16)

}  // namespace dflash
