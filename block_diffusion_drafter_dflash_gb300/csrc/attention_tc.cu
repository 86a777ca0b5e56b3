// Split-KV block attention of bf16 drafters on the tensor cores (tcgen05).
//
// One CTA of 256 threads per (split, kv head, request): the request's keys —
// its context in 128-key tiles, then one tile of the block's own keys — are
// cut into `splits` ranges of whole tiles; the CTA runs the group's query rows
// (64 per pass) over its range (attn_tc.cuh; the two warps of each TMEM lane
// quarter split a tile's keys and output columns, since at one CTA per SM the
// per-tile chain of read-back, softmax and P stores is the time) and writes
// unnormalised partial rows plus their (max, sum); attn_combine_kernel
// (attention.cu) merges the splits.  Maxima are written in natural-log units,
// as the merge expects.
#include <cuda.h>

#include "attn_tc.cuh"
#include "gemm.cuh"

namespace dflash {

namespace {

constexpr float kLn2 = 0.6931471805599453f;

constexpr int kSplitThreads = 256;

template <int HD>
struct SplitSmem {
  // operand tiles, barriers, the TMEM address slot, then 256 floats of
  // row max / sum exchange between the two warps of a lane quarter
  static constexpr size_t kXch = attn_tc::Cfg<HD>::kBytes + sizeof(attn_tc::Bars) + 16;
  static constexpr size_t kBytes = 1024 + kXch + 256 * sizeof(float);
  static constexpr int kTmem = attn_tc::Cfg<HD>::kTmemCols <= 256 ? 256 : 512;
};

struct CtaSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

template <int HD>
__global__ void __launch_bounds__(kSplitThreads, 1) attn_tc_split_kernel(const __grid_constant__ AttnParams p,
                                                               const __grid_constant__ attn_tc::Maps maps,
                                                               int32_t* status) {
  using C = attn_tc::Cfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  attn_tc::Bars* bars = reinterpret_cast<attn_tc::Bars*>(sm + C::kBytes);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 1);
  float* xch = reinterpret_cast<float*>(sm + SplitSmem<HD>::kXch);
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;

  if (tid == 0) {
    attn_tc::init_bars(bars);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&maps.kc);
    ptx::prefetch_tmap(&maps.vc);
    ptx::prefetch_tmap(&maps.kb);
    ptx::prefetch_tmap(&maps.vb);
  }
  if (tid < 32) ptx::tmem_alloc(tslot, SplitSmem<HD>::kTmem);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;
  griddep_wait();
  griddep_trigger();

  const int G = p.nq / p.nkv, rows = G * p.block, passes = (rows + 63) / 64;
  const int c = p.ctx_len[b];
  const int nct = (c + attn_tc::kKeys - 1) / attn_tc::kKeys, T = nct + 1;
  const int t0 = (int)((long long)split * T / p.splits), t1 = (int)((long long)(split + 1) * T / p.splits);
  // partial row of query row r of the group: ((b*nq + qh)*block + k)*splits + split
  auto prow = [&](int r) {
    const int gh = r / p.block, k = r - gh * p.block;
    return ((size_t)(b * p.nq + kvh * G + gh) * p.block + k) * p.splits + split;
  };
  int uses = 0;
  bool ok = true;
  for (int pass = 0; pass < passes && ok; ++pass) {
    if (t0 >= t1) {   // no keys here: an empty partial (weight 0 in the merge)
      for (int e = tid; e < 64 * HD; e += kSplitThreads) {
        const int r = 64 * pass + e / HD;
        if (r < rows) p.opart[prow(r) * HD + e % HD] = 0.f;
      }
      for (int i = tid; i < 64; i += kSplitThreads)
        if (64 * pass + i < rows) p.ml[prow(64 * pass + i)] = make_float2(-3.0e38f, 0.f);
      continue;
    }
    auto out = [&](int r, int d0, const float* v) {
      float* dst = p.opart + prow(r) * HD + d0;
#pragma unroll
      for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    };
    auto done = [&](int r, float m_log2, float l) { p.ml[prow(r)] = make_float2(m_log2 * kLn2, l); };
    ok = attn_tc::run<HD, kSplitThreads>(p, maps, b, kvh, pass, t0, t1, nct, c, sm, tmem, bars, uses, tid, CtaSync{},
                                         status, out, done, xch);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (tid < 32) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, SplitSmem<HD>::kTmem);
  }
}

template <int HD>
cudaError_t launch_hd(const AttnParams& p, const attn_tc::Maps& maps, int32_t* status, cudaStream_t s) {
  return launch_pdl(attn_tc_split_kernel<HD>, dim3(p.splits, p.nkv, p.B), dim3(kSplitThreads), SplitSmem<HD>::kBytes, s, p,
                    maps, status);
}

}  // namespace

cudaError_t attention_tc_prepare(int hd) {
  if (hd == 64)
    return cudaFuncSetAttribute(attn_tc_split_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)SplitSmem<64>::kBytes);
  return cudaFuncSetAttribute(attn_tc_split_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)SplitSmem<128>::kBytes);
}

cudaError_t attention_tc_split_launch(const AttnParams& p, const attn_tc::Maps& maps, int32_t* status,
                                      cudaStream_t s) {
  return p.hd == 64 ? launch_hd<64>(p, maps, status, s) : launch_hd<128>(p, maps, status, s);
}

bool encode_attention_maps(attn_tc::Maps* m, const void* kc, const void* vc, const void* kb, const void* vb, int B,
                           int layers, int nkv, int hd, int cap, int cap_pitch, int kvp, int block, int block_pitch) {
  const int slabs_c = B * layers * nkv * kvp, slabs_b = B * nkv * 2;
  return encode_activation_map(&m->kc, kc, hd, slabs_c * cap, hd, attn_tc::kKeys) &&
         encode_activation_map(&m->vc, vc, cap, slabs_c * hd, cap_pitch, hd) &&
         encode_activation_map(&m->kb, kb, hd, slabs_b * block, hd, attn_tc::kKeys) &&
         encode_activation_map(&m->vb, vb, block, slabs_b * hd, block_pitch, hd);
}

}  // namespace dflash
