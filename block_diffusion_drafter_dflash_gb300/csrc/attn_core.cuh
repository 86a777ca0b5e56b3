// Tensor-core block attention core for bf16 drafters, at fp32-level precision:
// one (request, kv head) group's whole query block against a contiguous chunk
// of its keys, with an online softmax.  Used by the cluster attention kernel
// (partials merged through distributed shared memory) and by the persistent
// draft kernel (partials merged through global memory).
//
// K and V are stored as two bf16 planes, x = hi + lo (context cache and block
// alike), so both products run on mma.sync m16n8k16 as three bf16 products:
//     S = Q K^T ~ Qhi Khi^T + Qhi Klo^T + Qlo Khi^T
//     O = P V   ~ Phi Vhi  + Phi Vlo  + Plo Vhi
// (the dropped lo*lo term is ~2^-16 relative).  Tiles of 32 keys of the four
// planes stream through a STAGES-deep cp.async ring straight into
// XOR-swizzled shared memory (16-byte chunks; ldmatrix conflict free).
// Softmax runs in the log2 domain (Q is pre-scaled by log2(e)/sqrt(hd)).
// Key order: the request's context keys 0..c-1, then its block keys.
#pragma once

#include "kernels.cuh"

namespace dflash {
namespace attn {

constexpr int kKeys = 32;       // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -1.0e30f;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// byte offset of 16-byte chunk `ch` of row `r` in a [rows][HD] bf16 tile
template <int HD>
__device__ __forceinline__ int swz(int r, int ch) {
  return r * (HD * 2) + ((ch ^ (r & 7)) << 4);
}

template <int HD>
struct TileCfg {
  static constexpr int kTileB = kKeys * HD * 2;   // one bf16 plane tile
  static constexpr int kStageB = 4 * kTileB;      // Khi, Klo, Vhi, Vlo
};

// Running state of one thread: its two query rows (g and g+8 of the warp's
// 16) and the HD/8 output fragments.
template <int HD>
struct AttnAcc {
  float o[HD / 8][4];
  float m_a, m_b, l_a, l_b;
};

// Keys [j0, j1) of group (b, kvh) for the NW*16 query rows of the group
// (row r = head-in-group * block + k); thread `tid` of NW*32 participating
// threads; `sync()` is a barrier over exactly those threads.  On return `acc`
// holds the unnormalised output, the running max and the (quad-reduced) sum
// of this thread's rows; the ring is free again.
template <int HD, int NW, int STAGES, class Sync>
__device__ __forceinline__ void attn_chunk(const AttnParams& p, int b, int kvh, int c, int j0, int j1, uint8_t* sm,
                                           int tid, Sync sync, AttnAcc<HD>& acc) {
  using C = TileCfg<HD>;
  constexpr int kThreads = NW * 32;
  const int G = p.nq / p.nkv, rows = G * p.block;
  const int ntiles = j0 < j1 ? (j1 - j0 + kKeys - 1) / kKeys : 0;
  const int lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  const size_t cplane = (size_t)p.cap * HD, bplane = (size_t)p.block * HD;
  const __nv_bfloat16* kc =
      static_cast<const __nv_bfloat16*>(p.kc) + (((size_t)b * p.layers + p.layer) * p.nkv + kvh) * 2 * cplane;
  const __nv_bfloat16* vc =
      static_cast<const __nv_bfloat16*>(p.vc) + (((size_t)b * p.layers + p.layer) * p.nkv + kvh) * 2 * cplane;
  const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(p.kb) + ((size_t)b * p.nkv + kvh) * 2 * bplane;
  const __nv_bfloat16* vb = static_cast<const __nv_bfloat16*>(p.vb) + ((size_t)b * p.nkv + kvh) * 2 * bplane;

  // tile it -> ring stage it % STAGES: the four planes, 16-byte chunks
  auto load_tile = [&](int it) {
    if (it < ntiles) {
      const int jt = j0 + it * kKeys;
      const uint32_t base = smem_addr(sm + (it % STAGES) * C::kStageB);
      constexpr int cpr = HD * 2 / 16;   // chunks per row
      for (int e = tid; e < 4 * kKeys * cpr; e += kThreads) {
        const int pl = e / (kKeys * cpr), rem = e - pl * kKeys * cpr;
        const int r = rem / cpr, ch = rem - r * cpr;
        const int j = jt + r;
        const bool valid = j < j1;
        const bool is_v = pl >= 2, lo = pl & 1;
        const __nv_bfloat16* src = is_v ? vc : kc;
        if (valid) {
          if (j < c)
            src = (is_v ? vc : kc) + lo * cplane + (size_t)j * HD + ch * 8;
          else
            src = (is_v ? vb : kb) + lo * bplane + (size_t)(j - c) * HD + ch * 8;
        }
        cp_async16(base + pl * C::kTileB + swz<HD>(r, ch), src, valid);
      }
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
    // L2 loads: in the persistent kernel Q was written by other CTAs of the same launch
    float2 x0 = qa ? __ldcg(reinterpret_cast<const float2*>(qa + c0)) : make_float2(0.f, 0.f);
    float2 x1 = qb ? __ldcg(reinterpret_cast<const float2*>(qb + c0)) : make_float2(0.f, 0.f);
    float2 x2 = qa ? __ldcg(reinterpret_cast<const float2*>(qa + c1)) : make_float2(0.f, 0.f);
    float2 x3 = qb ? __ldcg(reinterpret_cast<const float2*>(qb + c1)) : make_float2(0.f, 0.f);
    split2(x0.x * qscale, x0.y * qscale, qh[kk][0], ql[kk][0]);
    split2(x1.x * qscale, x1.y * qscale, qh[kk][1], ql[kk][1]);
    split2(x2.x * qscale, x2.y * qscale, qh[kk][2], ql[kk][2]);
    split2(x3.x * qscale, x3.y * qscale, qh[kk][3], ql[kk][3]);
  }

  float(&o)[HD / 8][4] = acc.o;
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = kNegBig, m_b = kNegBig, l_a = 0.f, l_b = 0.f;

#pragma unroll
  for (int i = 0; i < STAGES - 1; ++i) load_tile(i);
  const int mi = lane >> 3, rr = lane & 7;
  for (int it = 0; it < ntiles; ++it) {
    const int jt = j0 + it * kKeys;
    cp_async_wait<STAGES - 2>();
    sync();                                   // tile it landed; stage (it-1) free for tile it+STAGES-1
    load_tile(it + STAGES - 1);
    const uint8_t* st = sm + (it % STAGES) * C::kStageB;
    const uint8_t *khi = st, *klo = st + C::kTileB, *vhi = st + 2 * C::kTileB, *vlo = st + 3 * C::kTileB;

    // ---- S = Q K^T for this warp's 16 rows x 32 keys (4 n-blocks of 8 keys)
    float s[4][4];
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
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
    // ---- mask keys past the chunk, online softmax (log2 domain)
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
  cp_async_wait<0>();
  sync();                                     // every tile consumed: the ring is free
#pragma unroll
  for (int sh = 1; sh <= 2; sh <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, sh);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, sh);
  }
  acc.m_a = ntiles > 0 ? m_a : kNegBig;
  acc.m_b = ntiles > 0 ? m_b : kNegBig;
  acc.l_a = ntiles > 0 ? l_a : 0.f;
  acc.l_b = ntiles > 0 ? l_b : 0.f;
}

}  // namespace attn
}  // namespace dflash
