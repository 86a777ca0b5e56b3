// Tensor-core block attention for bf16 drafters, at fp32-level precision.
//
// One thread-block cluster of kCluster CTAs per (request, kv head).  The
// request's keys — its context K/V followed by the block's own K/V — are cut
// into kCluster contiguous chunks, one per CTA; every CTA runs the whole
// query group (the nq/nkv heads times the block rows, one warp per 16 rows)
// over its chunk (attn_core.cuh), then the cluster merges the partial (max,
// sum, output) rows through distributed shared memory: CTA r finalises rows
// r, r+kCluster, ...  No global scratch, no second kernel, and the chunking
// adapts to each request's own context length.
#include <cooperative_groups.h>

#include <cfloat>
#include <cstdlib>

#include "attn_core.cuh"

namespace dflash {

namespace cg = cooperative_groups;

namespace {

using attn::kKeys;
using attn::kNegBig;
constexpr int kStages = 3;      // cp.async ring depth

template <int HD, int NW, int CL>
struct ClusterCfg {
  static constexpr int kCluster = CL;                         // CTAs per (request, kv head)
  static constexpr int kThreads = NW * 32;
  static constexpr int kRows = NW * 16;                        // query rows (padded)
  static constexpr int kRing = kStages * attn::TileCfg<HD>::kStageB;
  static constexpr int kMerge = kRows * HD * 4 + 2 * kRows * 4;  // o, m, l of every row
  static constexpr int kSmem = kRing > kMerge ? kRing : kMerge;
};

struct CtaSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

template <int HD, int NW, int CL>
__global__ void __launch_bounds__(NW * 32) attn_cluster_kernel(const __grid_constant__ AttnParams p) {
  using C = ClusterCfg<HD, NW, CL>;
  constexpr int kCluster = CL;
  extern __shared__ __align__(128) uint8_t sm[];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();

  griddep_wait();
  griddep_trigger();
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int G = p.nq / p.nkv, rows = G * p.block;
  const int c = p.ctx_len[b];
  const int total = c + p.block;
  const int per = (total + kCluster - 1) / kCluster;
  const int chunk = (per + kKeys - 1) / kKeys * kKeys;
  const int j0 = rank * chunk, j1 = min(total, j0 + chunk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  attn::AttnAcc<HD> acc;
  attn::attn_chunk<HD, NW, kStages>(p, b, kvh, c, j0, j1, sm, tid, CtaSync{}, acc);

  // ---- publish this CTA's partial rows: o (unnormalised), m, l
  const int r_lo = warp * 16 + g, r_hi = r_lo + 8;
  float* os = reinterpret_cast<float*>(sm);              // [kRows][HD]
  float* ms = os + C::kRows * HD;                        // [kRows]
  float* ls = ms + C::kRows;                             // [kRows]
#pragma unroll
  for (int nb = 0; nb < HD / 8; ++nb) {
    *reinterpret_cast<float2*>(os + r_lo * HD + nb * 8 + 2 * t) = make_float2(acc.o[nb][0], acc.o[nb][1]);
    *reinterpret_cast<float2*>(os + r_hi * HD + nb * 8 + 2 * t) = make_float2(acc.o[nb][2], acc.o[nb][3]);
  }
  if (t == 0) {
    ms[r_lo] = acc.m_a;
    ms[r_hi] = acc.m_b;
    ls[r_lo] = acc.l_a;
    ls[r_hi] = acc.l_b;
  }
  cluster.sync();

  // ---- merge: CTA `rank` finalises rows rank, rank + kCluster, ...
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  for (int r = rank + warp * kCluster; r < rows; r += NW * kCluster) {
    float mr[kCluster], lr[kCluster];
    float M = kNegBig;
#pragma unroll
    for (int q = 0; q < kCluster; ++q) {
      mr[q] = *cluster.map_shared_rank(ms + r, q);
      lr[q] = *cluster.map_shared_rank(ls + r, q);
      if (lr[q] > 0.f) M = fmaxf(M, mr[q]);
    }
    float L = 0.f;
#pragma unroll
    for (int q = 0; q < kCluster; ++q) {
      mr[q] = lr[q] > 0.f ? exp2f(mr[q] - M) : 0.f;     // weight of rank q
      L += mr[q] * lr[q];
    }
    const float inv = 1.f / L;
    const int gh = r / p.block, k = r - gh * p.block;
    const size_t obase = ((size_t)b * p.block + k) * p.nq * HD + (size_t)(kvh * G + gh) * HD;
    for (int d = lane; d < HD; d += 32) {
      float a = 0.f;
#pragma unroll
      for (int q = 0; q < kCluster; ++q)
        if (mr[q] != 0.f) a += mr[q] * *cluster.map_shared_rank(os + r * HD + d, q);
      put_act(out, p.out_plane, obase + d, a * inv);
    }
  }
  cluster.sync();                             // keep every CTA's partials alive until all reads are done
}

template <int HD, int NW, int CL>
cudaError_t launch_one(const AttnParams& p, cudaStream_t s) {
  using C = ClusterCfg<HD, NW, CL>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, p.nkv, p.B);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<HD, NW, CL>, p);
}

template <int HD, int NW, int CL>
cudaError_t prepare_one() {
  cudaError_t e = cudaFuncSetAttribute(attn_cluster_kernel<HD, NW, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       ClusterCfg<HD, NW, CL>::kSmem);
  if (e == cudaSuccess && CL > 8)
    e = cudaFuncSetAttribute(attn_cluster_kernel<HD, NW, CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <int HD, int CL>
cudaError_t prepare_hd() {
  cudaError_t e;
  if ((e = prepare_one<HD, 1, CL>()) || (e = prepare_one<HD, 2, CL>()) || (e = prepare_one<HD, 4, CL>()) ||
      (e = prepare_one<HD, 8, CL>()))
    return e;
  return cudaSuccess;
}

template <int HD, int CL>
cudaError_t launch_hd(const AttnParams& p, cudaStream_t s) {
  const int rows = (p.nq / p.nkv) * p.block;
  const int nw = rows <= 16 ? 1 : rows <= 32 ? 2 : rows <= 64 ? 4 : 8;
  switch (nw) {
    case 1: return launch_one<HD, 1, CL>(p, s);
    case 2: return launch_one<HD, 2, CL>(p, s);
    case 4: return launch_one<HD, 4, CL>(p, s);
    default: return launch_one<HD, 8, CL>(p, s);
  }
}

int cluster_choice(const AttnParams& p) {
  static const char* env = getenv("DFLASH_ATTN_CLUSTER");
  if (env) return atoi(env) == 16 ? 16 : 8;
  // 16-CTA clusters when 8-CTA ones would leave most SMs idle
  return (long)p.B * p.nkv * 8 < 152 ? 16 : 8;
}

}  // namespace

cudaError_t attention_mma_prepare(int hd) {
  cudaError_t e;
  if (hd == 128) {
    if ((e = prepare_hd<128, 8>()) || (e = prepare_hd<128, 16>())) return e;
  } else {
    if ((e = prepare_hd<64, 8>()) || (e = prepare_hd<64, 16>())) return e;
  }
  return cudaSuccess;
}

// Whole attention of one layer (no separate merge kernel).
cudaError_t attention_mma_launch(const AttnParams& p, cudaStream_t s) {
  const bool big = cluster_choice(p) == 16;
  if (p.hd == 128) return big ? launch_hd<128, 16>(p, s) : launch_hd<128, 8>(p, s);
  return big ? launch_hd<64, 16>(p, s) : launch_hd<64, 8>(p, s);
}

}  // namespace dflash
