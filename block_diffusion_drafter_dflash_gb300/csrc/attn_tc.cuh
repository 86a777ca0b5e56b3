// Tensor-core (tcgen05) block attention for bf16 drafters at fp32-level
// precision: one (request, kv head) group's query rows against a range of
// 128-key tiles of its keys, online softmax, unnormalised output.  Used by the
// split-KV attention kernel (attention_tc.cu) and by the persistent drafter
// kernel (persist.cu).
//
// Operands.  Every value v is carried as two bf16 parts hi + lo.  The MMA's A
// operand holds, in each 32-row quarter of its 128 rows, the hi parts of 16
// query rows followed by their lo parts; its B operand stacks the hi plane of
// the keys over their lo plane (N = 2 x 128 keys).  One instruction (a
// tcgen05.mma costs about the same for any N up to 256) thus gives all four
// products, and summed over a row's hi and lo accumulator rows and over a
// key's hi and lo accumulator columns,
//     S = (Qhi + Qlo)(Khi + Klo)^T
// (the same for O = P V with P in A and [Vhi; Vlo] in B, N = 2 hd).  A query
// row's two accumulator rows sit in one warp's TMEM lanes, 16 apart, so each
// of the four warps reads back its own 16 rows and adds the halves with one
// shuffle.  Scores are in the log2 domain (Q is pre-scaled by
// log2(e)/sqrt(hd)).
//
// A cache of one rounded bf16 per value (kvp = 1) gives its tiles' keys and
// values one plane: N = 128 keys for S and N = hd for that tile's P V; the
// block tile keeps both planes, and its lo-plane product goes to the O lo
// columns, which then hold nothing else.
//
// Keys.  A group's keys are its context keys 0..c-1 (cache) in tiles of 128,
// then one tile of its block keys.  With ctx_shared every request reads the
// context slab of request 0 (its own length c): the blocks of one packed
// training sequence share that sequence's context.  K is stored key-major
// ([pos][hd]) and V hd-major ([hd][pos]), so that both products read their B
// operand K-major;
// tiles arrive by TMA (128-byte swizzle).  Keys past the valid ones read
// finite values (the cache is zeroed at creation; past the tensor end TMA
// fills zeros) and get probability exactly 0 (score -inf).
//
// Softmax.  The running row max is only raised when a tile's max exceeds it
// by more than 8 (log2 units), so the unnormalised output in TMEM is rescaled
// rarely; probabilities stay below 2^8, well inside fp32 and bf16 range.
#pragma once

#include <cuda.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace dflash {
namespace attn_tc {

constexpr int kKeys = 128;                 // keys per tile (MMA N of Q K^T)
constexpr int kTile16 = 128 * 128;         // one 128-row x 128-byte operand tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -1.0e30f;
constexpr float kLazy = 8.0f;              // raise the running max only beyond this margin
constexpr long long kBudget = 200000000LL;

// Tensor maps of one launch: K cache, V cache (hd-major), block K, block V (hd-major).
struct Maps {
  CUtensorMap kc, vc, kb, vb;
};

// Shared memory (1024-byte aligned base): Q A-tile per 64 columns of hd;
// K B-tiles [hd/64][plane] (the two planes of a column block adjacent, one
// 256-row operand); V B-tiles [key half][plane] (hd rows x 64 keys each, the
// planes adjacent); P A-tiles [key half].  Tensor memory: S in columns
// [0, 256) (Khi keys, then Klo keys), O in [256, 256 + 2 hd).
template <int HD>
struct Cfg {
  static constexpr int kSub = HD / 64;                       // 64-column blocks of hd
  static constexpr int kQ = kSub * kTile16;
  static constexpr int kK = 2 * kSub * kTile16;
  static constexpr int kVHalf = HD * 128;                    // hd rows x 64 keys
  static constexpr int kV = 2 * 2 * kVHalf;
  static constexpr int kP = 2 * kTile16;
  static constexpr int kOffK = kQ, kOffV = kOffK + kK, kOffP = kOffV + kV;
  static constexpr int kBytes = kOffP + kP;
  static constexpr int kTmemCols = 2 * kKeys + 2 * HD;       // S then O, both planes
  static constexpr uint32_t kKBytes = 2u * kSub * kTile16;   // TMA bytes of a K tile
  static constexpr uint32_t kVBytes = 2u * 2 * kVHalf;       // TMA bytes of a V tile
};

struct Bars {
  uint64_t kfull, vfull, sdone, odone;
};

__device__ __forceinline__ void init_bars(Bars* b) {
  ptx::mbar_init(&b->kfull, 1);
  ptx::mbar_init(&b->vfull, 1);
  ptx::mbar_init(&b->sdone, 1);
  ptx::mbar_init(&b->odone, 1);
}

// A-tile row of query row i (0..63) of a pass: quarter i/16, hi part at +0, lo at +16
__device__ __forceinline__ int a_row(int i, int lo) { return 32 * (i >> 4) + 16 * lo + (i & 15); }
// byte offset of 16-byte chunk `ch` of row `r` in a 128-byte-swizzled K-major tile
__device__ __forceinline__ int sw(int r, int ch) { return r * 128 + ((ch ^ (r & 7)) << 4); }

__device__ __forceinline__ uint4 pack8(const float* v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
  __nv_bfloat162 c = __floats2bfloat162_rn(v[4], v[5]), d = __floats2bfloat162_rn(v[6], v[7]);
  return make_uint4(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b),
                    *reinterpret_cast<uint32_t*>(&c), *reinterpret_cast<uint32_t*>(&d));
}
// hi/lo parts of 8 values as two 16-byte chunks
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
  float h[8], l[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
    l[j] = v[j] - h[j];
  }
  hi = pack8(h);
  lo = pack8(l);
}

// Q rows [64*pass, 64*pass+64) of group (b, kvh) into the A tiles, scaled into
// the log2 domain; rows past the group's rows are zero.  NT threads (128 or
// 256), each with 64*HD/(8*NT) chunks of 8 values: every load is issued before
// the first store, so the whole tile costs one memory round trip.  In two
// halves: stage_q_load issues the loads, stage_q_store converts and stores, so
// that other work can be issued while the loads are in flight.
template <int HD, int NT>
struct QRegs {
  static constexpr int kPer = 64 * (HD / 8) / NT;   // 8-value chunks per thread
  float4 x[kPer][2];
};

template <int HD, int NT>
__device__ __forceinline__ void stage_q_load(const AttnParams& p, int b, int kvh, int pass, int tid, QRegs<HD, NT>& qr) {
  constexpr int kPer = QRegs<HD, NT>::kPer;
  const int G = p.nq / p.nkv, rows = G * p.block;
  float4(&x)[kPer][2] = qr.x;
  // thread tid's chunks lie in rows r0, r0 + kRowStep, ...: (head, block
  // position) of each follows from the previous one without a division
  constexpr int kRowStep = NT / (HD / 8);
  const int c8 = tid % (HD / 8), r0 = 64 * pass + tid / (HD / 8);
  int gh = r0 / p.block, k = r0 - gh * p.block;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int r = r0 + kRowStep * u;
    if (u > 0) {
      k += kRowStep;
      while (k >= p.block) {
        k -= p.block;
        ++gh;
      }
    }
    if (r < rows) {
      const float* src = p.q + (((size_t)b * p.nq + kvh * G + gh) * p.block + k) * HD + 8 * c8;
      x[u][0] = __ldcg(reinterpret_cast<const float4*>(src));
      x[u][1] = __ldcg(reinterpret_cast<const float4*>(src + 4));
    } else {
      x[u][0] = x[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

template <int HD, int NT>
__device__ __forceinline__ void stage_q_store(const AttnParams& p, uint8_t* sm, int tid, const QRegs<HD, NT>& qr) {
  constexpr int kPer = QRegs<HD, NT>::kPer;
  const float qscale = p.scale * kLog2e;
  const float4(&x)[kPer][2] = qr.x;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid + NT * u, i = e / (HD / 8), c8 = e - i * (HD / 8), s = c8 >> 3, ch = c8 & 7;
    const float v[8] = {x[u][0].x * qscale, x[u][0].y * qscale, x[u][0].z * qscale, x[u][0].w * qscale,
                        x[u][1].x * qscale, x[u][1].y * qscale, x[u][1].z * qscale, x[u][1].w * qscale};
    uint4 hi, lo;
    split8(v, hi, lo);
    uint8_t* q = sm + s * kTile16;
    *reinterpret_cast<uint4*>(q + sw(a_row(i, 0), ch)) = hi;
    *reinterpret_cast<uint4*>(q + sw(a_row(i, 1), ch)) = lo;
  }
}

// Planes of tile t: the cache's for a context tile, two for the block tile.
__device__ __forceinline__ int tile_planes(const AttnParams& p, int t, int nct) { return t < nct ? p.kvp : 2; }

// Warm the descriptor cache for the attention's tensor maps (one thread).
__device__ __forceinline__ void prefetch_maps(const Maps& m) {
  ptx::prefetch_tmap(&m.kc);
  ptx::prefetch_tmap(&m.vc);
  ptx::prefetch_tmap(&m.kb);
  ptx::prefetch_tmap(&m.vb);
}

// TMA of tile t of group (b, kvh) of layer p.layer: context keys [128t, 128t+128)
// for t < nct, else the block's keys.  Issued by one thread.
template <int HD>
__device__ void load_k(const AttnParams& p, const Maps& m, int b, int kvh, int t, int nct, uint8_t* sm, Bars* bars) {
  using C = Cfg<HD>;
  uint8_t* kt = sm + C::kOffK;
  const int bc = p.ctx_shared ? 0 : b;   // the context slab
  const int np = tile_planes(p, t, nct);
  ptx::mbar_arrive_expect_tx(&bars->kfull, np * (C::kKBytes / 2));
  for (int pl = 0; pl < np; ++pl)
    for (int s = 0; s < C::kSub; ++s) {
      uint8_t* dst = kt + (s * 2 + pl) * kTile16;
      if (t < nct) {
        const int row = ((((bc * p.layers + p.layer) * p.nkv + kvh) * p.kvp + pl) * p.cap) + kKeys * t;
        ptx::tma_load_2d(dst, &m.kc, &bars->kfull, 64 * s, row, ptx::policy_evict_first());
      } else {
        const int row = ((b * p.nkv + kvh) * 2 + pl) * p.block;
        ptx::tma_load_2d(dst, &m.kb, &bars->kfull, 64 * s, row, ptx::policy_evict_last());
      }
    }
}

template <int HD>
__device__ void load_v(const AttnParams& p, const Maps& m, int b, int kvh, int t, int nct, uint8_t* sm, Bars* bars) {
  using C = Cfg<HD>;
  uint8_t* vt = sm + C::kOffV;
  const int bc = p.ctx_shared ? 0 : b;   // the context slab
  const int np = tile_planes(p, t, nct);
  ptx::mbar_arrive_expect_tx(&bars->vfull, np * (C::kVBytes / 2));
  for (int pl = 0; pl < np; ++pl)
    for (int h = 0; h < 2; ++h) {
      uint8_t* dst = vt + (h * 2 + pl) * C::kVHalf;
      if (t < nct) {
        const int row = (((bc * p.layers + p.layer) * p.nkv + kvh) * p.kvp + pl) * HD;
        ptx::tma_load_2d(dst, &m.vc, &bars->vfull, kKeys * t + 64 * h, row, ptx::policy_evict_first());
      } else {
        const int row = ((b * p.nkv + kvh) * 2 + pl) * HD;
        ptx::tma_load_2d(dst, &m.vb, &bars->vfull, 64 * h, row, ptx::policy_evict_last());
      }
    }
}

// One item: query rows of pass `pass` of group (b, kvh) against tiles [t0, t1)
// (nct context tiles of the c context keys, then the block tile).  NT participating threads (tid
// 0..NT-1).  Warp w reads TMEM lanes 32(w%4)..32(w%4)+31, which must be its
// own lane quarter.  With NT = 256 the two warps of a lane quarter split the
// work of their 16 query rows: warp w < 4 takes keys 0..31 and 64..95 of every
// tile, warp w+4 keys 32..63 and 96..127, and they halve the output columns;
// the row maxima and sums go through `xch` (256 floats of shared memory).
// Thread 0 issues the TMA loads and the MMAs.  `uses` counts the tiles this
// CTA ran before (mbarrier phases).  On return out(row, d0, v32) has
// received, for every valid row of the pass, its unnormalised output in
// chunks of 32 columns, and done(row, m_log2, l) its running max and sum.
// Optional `stamps` (globaltimer): [0] Q staged, [1] the first tile's scores
// ready, [2] the last P V done, [3] output written, [4] the first V tile in
// shared memory, [5] the first P tile stored.  Returns false on a timeout.
template <int HD, int NT, class Sync, class Out, class Done>
__device__ bool run(const AttnParams& p, const Maps& m, int b, int kvh, int pass, int t0, int t1, int nct, int c,
                    uint8_t* sm, uint32_t tmem, Bars* bars, int& uses, int tid, Sync sync, int32_t* status, Out out,
                    Done done, float* xch = nullptr, unsigned long long* stamps = nullptr) {
  static_assert(NT == 128 || NT == 256, "128 or 256 threads");
  using C = Cfg<HD>;
  constexpr int NP = NT / 128;        // warps per lane quarter
  constexpr int KC = 64 / NP;         // keys of each 64-key half that one lane keeps
  constexpr int DC = HD / NP;         // output columns one warp reads back
  const int lane = tid & 31, w = tid >> 5, q4 = w & 3, part = w >> 2;
  const int G = p.nq / p.nkv, rows = G * p.block;
  const uint32_t lanes = static_cast<uint32_t>(q4 * 32) << 16;
  const uint32_t tS = tmem + lanes, tO = tmem + lanes + 2 * kKeys;   // this warp's lanes
  const uint32_t idS2 = ptx::idesc_bf16_f32(128, 2 * kKeys), idO2 = ptx::idesc_bf16_f32(128, 2 * HD);
  const uint32_t idS1 = ptx::idesc_bf16_f32(128, kKeys), idO1 = ptx::idesc_bf16_f32(128, HD);
  // O columns a rescale touches: the lo half holds only the block tile's
  // product when the cache has one plane, and that tile comes last
  const int ocols = (p.kvp == 2 ? 2 * HD : HD) / NP;
  const int i = 16 * q4 + (lane & 15);   // query row of the pass held by this lane (hi part if lane < 16)
  bool ok = true;

  // the first tile's K while the Q loads are in flight; its V once the
  // scores are issued (it is needed only after the softmax)
  {
    QRegs<HD, NT> qr;
    stage_q_load<HD, NT>(p, b, kvh, pass, tid, qr);
    if (tid == 0 && t0 < t1) load_k<HD>(p, m, b, kvh, t0, nct, sm, bars);
    stage_q_store<HD, NT>(p, sm, tid, qr);
  }
  ptx::fence_proxy_async_shared();
  sync();
  if (stamps && tid == 0) stamps[0] = ptx::globaltimer();

  float m_used = kNegInf, l_sum = 0.f;
  for (int t = t0; t < t1; ++t) {
    const uint32_t par = static_cast<uint32_t>(uses + (t - t0)) & 1u;
    const int nk = t < nct ? min(kKeys, c - kKeys * t) : p.block;   // valid keys of the tile
    const int np = tile_planes(p, t, nct);
    // ---- S = Q K^T (thread 0), then the K buffer is free for the next tile
    if (tid == 0) {
      ok = ptx::mbar_wait(&bars->kfull, par, kBudget, status);
      if (ok) {
        ptx::tc_fence_after();
        for (int s = 0; s < C::kSub; ++s)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = ptx::smem_desc_sw128(sm + s * kTile16) + 2 * k;
            const uint64_t bd = ptx::smem_desc_sw128(sm + C::kOffK + s * 2 * kTile16) + 2 * k;
            ptx::mma_bf16(tmem, ad, bd, np == 2 ? idS2 : idS1, (s | k) != 0 ? 1u : 0u);
          }
        ptx::mma_commit(&bars->sdone);
        if (t > t0) {   // the V buffer is free once the previous P V is done
          ok = ptx::mbar_wait(&bars->odone, par ^ 1u, kBudget, status);
          if (ok) load_v<HD>(p, m, b, kvh, t, nct, sm, bars);
        } else {
          load_v<HD>(p, m, b, kvh, t, nct, sm, bars);
        }
      }
    }
    ok = ptx::mbar_wait(&bars->sdone, par, kBudget, status) && ok;
    ptx::tc_fence_after();
    if (stamps && tid == 0 && t == t0) stamps[1] = ptx::globaltimer();
    if (tid == 0 && ok && t + 1 < t1) load_k<HD>(p, m, b, kvh, t + 1, nct, sm, bars);

    // ---- softmax of this warp's 16 rows: lanes l and l+16 hold a row's hi and
    // lo accumulator rows; lane l < 16 keeps keys of the first 64-key half,
    // lane l+16 of the second, and each sends the partner the half it does not
    // keep (one shuffle a key).  This warp's keys: KC per half from KC*part.
    const int half = lane >> 4;
    float pv[KC];
    if (np == 2) {
#pragma unroll
      for (int c0 = 0; c0 < KC; c0 += 16) {
        const int cc = KC * part + c0;
        float v[64];   // [Khi keys cc.., Klo keys cc.., Khi keys 64+cc.., Klo keys 64+cc..]
        ptx::tmem_ld16x4(tS + cc, tS + kKeys + cc, tS + 64 + cc, tS + kKeys + 64 + cc, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float lo_keys = v[j] + v[16 + j], hi_keys = v[32 + j] + v[48 + j];
          const float got = __shfl_xor_sync(0xffffffffu, half ? lo_keys : hi_keys, 16);
          const float x = half ? hi_keys + got : lo_keys + got;
          pv[c0 + j] = (64 * half + cc + j < nk) ? x : kNegInf;
        }
      }
    } else {   // one key plane: two 16-key steps per load
#pragma unroll
      for (int c0 = 0; c0 < KC; c0 += 32) {
        const int cc = KC * part + c0;
        float v[64];   // [keys cc.., keys 64+cc.., keys cc+16.., keys 64+cc+16..]
        ptx::tmem_ld16x4(tS + cc, tS + 64 + cc, tS + cc + 16, tS + 64 + cc + 16, v);
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float lo_keys = v[32 * u + j], hi_keys = v[32 * u + 16 + j];
            const float got = __shfl_xor_sync(0xffffffffu, half ? lo_keys : hi_keys, 16);
            const float x = half ? hi_keys + got : lo_keys + got;
            pv[c0 + 16 * u + j] = (64 * half + cc + 16 * u + j < nk) ? x : kNegInf;
          }
      }
    }
    float mx = kNegInf;
#pragma unroll
    for (int j = 0; j < KC; ++j) mx = fmaxf(mx, pv[j]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    if constexpr (NP == 2) {   // the row's maximum over both warps of the lane quarter
      if (lane < 16) xch[64 * part + i] = mx;
      sync();
      mx = fmaxf(xch[i], xch[64 + i]);
    }
    float alpha = 1.f;
    if (t == t0) {
      m_used = mx;
    } else if (mx > m_used + kLazy) {
      alpha = exp2f(m_used - mx);
      m_used = mx;
    }
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      pv[j] = exp2f(pv[j] - m_used);
      sum += pv[j];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 16);
    l_sum = l_sum * alpha + sum;   // this warp's keys; the parts are added at the end

    // the previous P V has finished: P may be overwritten, O rescaled
    if (t > t0) ok = ptx::mbar_wait(&bars->odone, par ^ 1u, kBudget, status) && ok;
    ptx::tc_fence_after();
    if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
      for (int d0 = ocols * part; d0 < ocols * (part + 1); d0 += 32) {
        float v[32];
        ptx::tmem_ld32(tO + d0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= alpha;
        ptx::tmem_st32(tO + d0, v);
      }
    }
    {
      uint8_t* pt = sm + C::kOffP + half * kTile16;
      const int rh = a_row(i, 0), rl = a_row(i, 1);
#pragma unroll
      for (int cl = 0; cl < KC / 8; ++cl) {
        const int ch = KC / 8 * part + cl;
        uint4 hi, lo;
        split8(pv + 8 * cl, hi, lo);
        *reinterpret_cast<uint4*>(pt + sw(rh, ch)) = hi;
        *reinterpret_cast<uint4*>(pt + sw(rl, ch)) = lo;
      }
    }
    ptx::fence_proxy_async_shared();
    ptx::tc_fence_before();
    if (stamps && tid == 0 && t == t0) stamps[5] = ptx::globaltimer();
    sync();

    // ---- O += P V (thread 0)
    if (tid == 0 && ok) {
      ptx::tc_fence_after();
      ok = ptx::mbar_wait(&bars->vfull, par, kBudget, status);
      if (stamps && t == t0) stamps[4] = ptx::globaltimer();
      if (ok) {
        // both planes in one N = 2 hd product, or the hi plane alone; the
        // block tile of a one-plane cache adds its lo plane to the O lo columns
        const bool split_lo = np == 2 && p.kvp == 1;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = ptx::smem_desc_sw128(sm + C::kOffP + h * kTile16) + 2 * k;
            const uint64_t bd = ptx::smem_desc_sw128(sm + C::kOffV + h * 2 * C::kVHalf) + 2 * k;
            const uint32_t acc = (t > t0 || h | k) ? 1u : 0u;
            if (np == 2 && !split_lo) {
              ptx::mma_bf16(tmem + 2 * kKeys, ad, bd, idO2, acc);
            } else {
              ptx::mma_bf16(tmem + 2 * kKeys, ad, bd, idO1, acc);
              if (split_lo) {
                const uint64_t bl = ptx::smem_desc_sw128(sm + C::kOffV + (h * 2 + 1) * C::kVHalf) + 2 * k;
                ptx::mma_bf16(tmem + 2 * kKeys + HD, ad, bl, idO1, (h | k) ? 1u : 0u);
              }
            }
          }
        ptx::mma_commit(&bars->odone);
      }
    }
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) ok = false;
  }
  if (t1 > t0) {
    ok = ptx::mbar_wait(&bars->odone, static_cast<uint32_t>(uses + (t1 - 1 - t0)) & 1u, kBudget, status) && ok;
    ptx::tc_fence_after();
    if (stamps && tid == 0) stamps[2] = ptx::globaltimer();
    const int r = 64 * pass + i;
    // the O lo columns hold something when the cache has two planes or the
    // block tile (always the last) was among this item's tiles
    const bool lo_cols = p.kvp == 2 || t1 > nct;
#pragma unroll 1
    for (int d0 = DC * part; d0 < DC * (part + 1); d0 += 32) {
      float v[64];   // O columns d0.. of the Vhi and the Vlo products
      if (lo_cols) {
        ptx::tmem_ld32x2(tO + d0, tO + HD + d0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += v[32 + j];
      } else {
        ptx::tmem_ld32(tO + d0, v);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], 16);
      if (lane < 16 && r < rows) out(r, d0, v);
    }
    if constexpr (NP == 2) {   // the row's sum over both warps of the lane quarter
      if (lane < 16) xch[128 + 64 * part + i] = l_sum;
      sync();
      l_sum = xch[128 + i] + xch[192 + i];
    }
    if (lane < 16 && part == 0 && r < rows) done(r, m_used, l_sum);
    ptx::tc_fence_before();
    if (stamps && tid == 0) stamps[3] = ptx::globaltimer();
  }
  uses += t1 - t0;
  sync();
  return ok;
}

}  // namespace attn_tc
}  // namespace dflash
