// Tensor-core block attention for bf16 drafters, at fp32-level precision.
//
// Same work split as the CUDA-core kernel (one CTA per request, kv head and
// key split; one warp per 16 query rows of the kv head's group), but the two
// products run on mma.sync m16n8k16 with each fp32 operand carried as a
// bf16 pair x = hi + lo:
//     S = Q K^T ~ Qhi Khi^T + Qhi Klo^T + Qlo Khi^T
//     O = P V   ~ Phi Vhi  + Phi Vlo  + Plo Vhi
// (the dropped lo*lo term is ~2^-16 relative).  K and V tiles of 32 keys are
// staged as fp32 with cp.async (double buffer), split into hi/lo bf16 tiles
// in shared memory (XOR-swizzled 16-byte chunks so ldmatrix is conflict
// free), and consumed with ldmatrix / ldmatrix.trans.  Softmax is online in
// the log2 domain (Q is pre-scaled by log2(e)/sqrt(hd)); partial (o, m, l)
// per split are merged by attn_combine_kernel.
#include <cfloat>

#include "kernels.cuh"

namespace dflash {

namespace {

constexpr int kKeys = 32;              // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegBig = -1.0e30f;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// pack two floats into a bf16x2 register (low half = first)
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
// hi/lo split of a float pair
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = pack_bf16(a - hf.x, b - hf.y);
}

__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// byte offset of 16-byte chunk `ch` of row `r` in a [rows][HD] bf16 tile
template <int HD>
__device__ __forceinline__ int swz(int r, int ch) {
  return r * (HD * 2) + ((ch ^ (r & 7)) << 4);
}

template <int HD, int NW>
struct MmaCfg {
  static constexpr int kThreads = NW * 32;
  static constexpr int kStageF = kKeys * HD;                  // floats per K (or V) staging tile
  static constexpr int kTileB = kKeys * HD * 2;               // bytes per bf16 tile
  static constexpr int kSmem = 2 * 2 * kStageF * 4 + 4 * kTileB;   // 2 stages x (K,V) fp32 + Khi,Klo,Vhi,Vlo
};

template <int HD, int NW>
__global__ void __launch_bounds__(NW * 32) attn_mma_kernel(const __grid_constant__ AttnParams p) {
  using C = MmaCfg<HD, NW>;
  extern __shared__ __align__(128) uint8_t sm[];
  float* stage = reinterpret_cast<float*>(sm);                     // [2][K,V][kKeys][HD]
  uint8_t* khi = sm + 2 * 2 * C::kStageF * 4;
  uint8_t* klo = khi + C::kTileB;
  uint8_t* vhi = klo + C::kTileB;
  uint8_t* vlo = vhi + C::kTileB;

  griddep_wait();
  griddep_trigger();
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = p.nq / p.nkv, rows = G * p.block;
  const int c = p.ctx_len[b];
  const int total = c + p.block;
  const int j0 = split * p.chunk, j1 = min(total, j0 + p.chunk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  const float* kc = p.kc + (((size_t)b * p.layers + p.layer) * p.nkv + kvh) * p.cap * HD;
  const float* vc = p.vc + (((size_t)b * p.layers + p.layer) * p.nkv + kvh) * p.cap * HD;
  const float* kb = p.kb + ((size_t)b * p.nkv + kvh) * p.block * HD;
  const float* vb = p.vb + ((size_t)b * p.nkv + kvh) * p.block * HD;

  // issue the fp32 loads of key tile starting at jt into staging buffer `buf`
  auto load_tile = [&](int jt, int buf) {
    float* ks = stage + (size_t)buf * 2 * C::kStageF;
    float* vs = ks + C::kStageF;
    constexpr int chunks = kKeys * HD / 4;   // 16-byte chunks per tile
    for (int e = tid; e < chunks; e += C::kThreads) {
      const int r = e / (HD / 4), col = (e % (HD / 4)) * 4;
      const int j = jt + r;
      const bool valid = j < j1;
      const float* ksrc = kc;
      const float* vsrc = vc;
      if (valid) {
        ksrc = j < c ? kc + (size_t)j * HD + col : kb + (size_t)(j - c) * HD + col;
        vsrc = j < c ? vc + (size_t)j * HD + col : vb + (size_t)(j - c) * HD + col;
      }
      cp_async16(ks + r * HD + col, ksrc, valid);
      cp_async16(vs + r * HD + col, vsrc, valid);
    }
    cp_async_commit();
  };

  // ---- Q fragments (hi/lo), scaled into the log2 domain
  const int r_lo = warp * 16 + g, r_hi = r_lo + 8;
  const float qscale = p.scale * kLog2e;
  auto q_row = [&](int r) -> const float* {
    if (r >= rows) return nullptr;
    const int gh = r / p.block, k = r - gh * p.block;
    return p.q + (((size_t)b * p.nq + kvh * G + gh) * p.block + k) * HD;
  };
  const float* qa = q_row(r_lo);
  const float* qb = q_row(r_hi);
  uint32_t qh[HD / 16][4], ql[HD / 16][4];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const int c0 = kk * 16 + 2 * t, c1 = c0 + 8;
    float2 x0 = qa ? *reinterpret_cast<const float2*>(qa + c0) : make_float2(0.f, 0.f);
    float2 x1 = qb ? *reinterpret_cast<const float2*>(qb + c0) : make_float2(0.f, 0.f);
    float2 x2 = qa ? *reinterpret_cast<const float2*>(qa + c1) : make_float2(0.f, 0.f);
    float2 x3 = qb ? *reinterpret_cast<const float2*>(qb + c1) : make_float2(0.f, 0.f);
    split2(x0.x * qscale, x0.y * qscale, qh[kk][0], ql[kk][0]);
    split2(x1.x * qscale, x1.y * qscale, qh[kk][1], ql[kk][1]);
    split2(x2.x * qscale, x2.y * qscale, qh[kk][2], ql[kk][2]);
    split2(x3.x * qscale, x3.y * qscale, qh[kk][3], ql[kk][3]);
  }

  float o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = kNegBig, m_b = kNegBig, l_a = 0.f, l_b = 0.f;

  const int ntiles = j0 < j1 ? (j1 - j0 + kKeys - 1) / kKeys : 0;
  if (ntiles > 0) load_tile(j0, 0);
  for (int it = 0; it < ntiles; ++it) {
    const int jt = j0 + it * kKeys;
    cp_async_wait_all();
    __syncthreads();                          // staging[it&1] landed; hi/lo tiles free
    if (it + 1 < ntiles) load_tile(jt + kKeys, (it + 1) & 1);
    {   // split the staged fp32 tile into hi/lo bf16 tiles
      const float* ks = stage + (size_t)(it & 1) * 2 * C::kStageF;
      const float* vs = ks + C::kStageF;
      for (int e = tid; e < kKeys * HD / 4; e += C::kThreads) {
        const int r = e / (HD / 4), col = (e % (HD / 4)) * 4;
        const int off = swz<HD>(r, col >> 3) + (col & 7) * 2;
        float4 kv = *reinterpret_cast<const float4*>(ks + r * HD + col);
        float4 vv = *reinterpret_cast<const float4*>(vs + r * HD + col);
        uint32_t h0, l0, h1, l1;
        split2(kv.x, kv.y, h0, l0);
        split2(kv.z, kv.w, h1, l1);
        *reinterpret_cast<uint2*>(khi + off) = make_uint2(h0, h1);
        *reinterpret_cast<uint2*>(klo + off) = make_uint2(l0, l1);
        split2(vv.x, vv.y, h0, l0);
        split2(vv.z, vv.w, h1, l1);
        *reinterpret_cast<uint2*>(vhi + off) = make_uint2(h0, h1);
        *reinterpret_cast<uint2*>(vlo + off) = make_uint2(l0, l1);
      }
    }
    __syncthreads();

    // ---- S = Q K^T for this warp's 16 rows x 32 keys (4 n-blocks of 8 keys)
    float s[4][4];
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
    const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {          // keys 16jp .. 16jp+15
        const int key = 16 * jp + rr + 8 * (mi >> 1);
        const int off = swz<HD>(key, 2 * kk + (mi & 1));
        uint32_t bh[4], bl[4];
        ldsm_x4(smem_addr(khi + off), bh);
        ldsm_x4(smem_addr(klo + off), bl);
        mma16816(s[2 * jp], qh[kk], bh[0], bh[1]);
        mma16816(s[2 * jp], qh[kk], bl[0], bl[1]);
        mma16816(s[2 * jp], ql[kk], bh[0], bh[1]);
        mma16816(s[2 * jp + 1], qh[kk], bh[2], bh[3]);
        mma16816(s[2 * jp + 1], qh[kk], bl[2], bl[3]);
        mma16816(s[2 * jp + 1], ql[kk], bh[2], bh[3]);
      }
    }
    // ---- mask keys past the split's end, online softmax (log2 domain)
    float mx_a = kNegBig, mx_b = kNegBig;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      const int k0 = jt + nb * 8 + 2 * t;
      if (k0 >= j1) s[nb][0] = s[nb][2] = kNegBig;
      if (k0 + 1 >= j1) s[nb][1] = s[nb][3] = kNegBig;
      mx_a = fmaxf(mx_a, fmaxf(s[nb][0], s[nb][1]));
      mx_b = fmaxf(mx_b, fmaxf(s[nb][2], s[nb][3]));
    }
#pragma unroll
    for (int sh = 1; sh <= 2; sh <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, sh));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, sh));
    }
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float al_a = exp2f(m_a - mn_a), al_b = exp2f(m_b - mn_b);
    m_a = mn_a;
    m_b = mn_b;
    l_a *= al_a;
    l_b *= al_b;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      o[i][0] *= al_a;
      o[i][1] *= al_a;
      o[i][2] *= al_b;
      o[i][3] *= al_b;
    }
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      s[nb][0] = exp2f(s[nb][0] - m_a);
      s[nb][1] = exp2f(s[nb][1] - m_a);
      s[nb][2] = exp2f(s[nb][2] - m_b);
      s[nb][3] = exp2f(s[nb][3] - m_b);
      l_a += s[nb][0] + s[nb][1];
      l_b += s[nb][2] + s[nb][3];
    }
    // ---- O += P V (two k-steps of 16 keys)
#pragma unroll
    for (int jp = 0; jp < 2; ++jp) {
      uint32_t ph[4], pl[4];
      split2(s[2 * jp][0], s[2 * jp][1], ph[0], pl[0]);
      split2(s[2 * jp][2], s[2 * jp][3], ph[1], pl[1]);
      split2(s[2 * jp + 1][0], s[2 * jp + 1][1], ph[2], pl[2]);
      split2(s[2 * jp + 1][2], s[2 * jp + 1][3], ph[3], pl[3]);
      const int key = 16 * jp + rr + 8 * (mi & 1);
#pragma unroll
      for (int h = 0; h < HD / 16; ++h) {       // hd 16h .. 16h+15
        const int off = swz<HD>(key, 2 * h + (mi >> 1));
        uint32_t bh[4], bl[4];
        ldsm_x4_t(smem_addr(vhi + off), bh);
        ldsm_x4_t(smem_addr(vlo + off), bl);
        mma16816(o[2 * h], ph, bh[0], bh[1]);
        mma16816(o[2 * h], ph, bl[0], bl[1]);
        mma16816(o[2 * h], pl, bh[0], bh[1]);
        mma16816(o[2 * h + 1], ph, bh[2], bh[3]);
        mma16816(o[2 * h + 1], ph, bl[2], bl[3]);
        mma16816(o[2 * h + 1], pl, bh[2], bh[3]);
      }
    }
  }

  // ---- partial results: unnormalised o, running max (natural log units), sum
#pragma unroll
  for (int sh = 1; sh <= 2; sh <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, sh);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, sh);
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? r_hi : r_lo;
    if (r >= rows) continue;
    const int gh = r / p.block, k = r - gh * p.block;
    const size_t row = (((size_t)b * p.nq + kvh * G + gh) * p.block + k) * p.splits + split;
    const float m = half ? m_b : m_a, l = half ? l_b : l_a;
#pragma unroll
    for (int nb = 0; nb < HD / 8; ++nb)
      *reinterpret_cast<float2*>(p.opart + row * HD + nb * 8 + 2 * t) =
          half ? make_float2(o[nb][2], o[nb][3]) : make_float2(o[nb][0], o[nb][1]);
    if (t == 0) p.ml[row] = make_float2(ntiles > 0 ? m * kLn2 : -FLT_MAX, ntiles > 0 ? l : 0.f);
  }
}

template <int HD, int NW>
cudaError_t launch_one(const AttnParams& p, cudaStream_t s) {
  using C = MmaCfg<HD, NW>;
  return launch_pdl(attn_mma_kernel<HD, NW>, dim3(p.splits, p.nkv, p.B), dim3(C::kThreads), C::kSmem, s, p);
}

template <int HD, int NW>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(attn_mma_kernel<HD, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              MmaCfg<HD, NW>::kSmem);
}

}  // namespace

int attention_mma_key_tile() { return kKeys; }

cudaError_t attention_mma_prepare(int hd) {
  cudaError_t e = cudaSuccess;
  if (hd == 128) {
    if ((e = prepare_one<128, 1>()) || (e = prepare_one<128, 2>()) || (e = prepare_one<128, 4>()) ||
        (e = prepare_one<128, 8>()))
      return e;
  } else {
    if ((e = prepare_one<64, 1>()) || (e = prepare_one<64, 2>()) || (e = prepare_one<64, 4>()) ||
        (e = prepare_one<64, 8>()))
      return e;
  }
  return e;
}

cudaError_t attention_mma_split_launch(const AttnParams& p, cudaStream_t s) {
  const int rows = (p.nq / p.nkv) * p.block;
  const int nw = rows <= 16 ? 1 : rows <= 32 ? 2 : rows <= 64 ? 4 : 8;
  if (p.hd == 128) {
    switch (nw) {
      case 1: return launch_one<128, 1>(p, s);
      case 2: return launch_one<128, 2>(p, s);
      case 4: return launch_one<128, 4>(p, s);
      default: return launch_one<128, 8>(p, s);
    }
  }
  switch (nw) {
    case 1: return launch_one<64, 1>(p, s);
    case 2: return launch_one<64, 2>(p, s);
    case 4: return launch_one<64, 4>(p, s);
    default: return launch_one<64, 8>(p, s);
  }
}

}  // namespace dflash
