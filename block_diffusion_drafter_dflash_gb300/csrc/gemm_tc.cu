// Tensor-core projection GEMM for sm_100-family GPUs (tcgen05 + TMA + TMEM).
//
// Swap-AB form: the weight tile is the MMA's M side and the token rows are
// its N side,
//     D[128 features x PL*BN] += W[128 x 64] . [X_hi ; X_lo][PL*BN x 64]^T   per stage,
// so one kernel covers batch 1 (BN = 16: weight streaming, HBM-bound) and
// batch 32 (BN = 128: dense, tensor-bound).  Activations carried as a hi/lo
// bf16 pair (PL = 2) occupy two row blocks of the N side; the epilogue adds
// the two accumulator columns of each token.  One thread issues TMA loads of
// both operands (128-B swizzle, K-major) into a ring of shared-memory stages;
// one thread issues tcgen05.mma into a tensor-memory accumulator and frees
// each stage with tcgen05.commit; all four warps then read the accumulator
// back (tcgen05.ld) and run the fused epilogue.  Split-K writes fp32 partial
// tiles; the last CTA of a tile (atomic ticket, no waiting) sums them in split
// order and runs the epilogue, so results do not depend on scheduling.
// Every mbarrier wait is bounded: on expiry the kernel sets
// DFLASH_ERR_TIMEOUT in the status word, skips its output and still frees
// its tensor memory.
#include <cuda.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>

#include "gemm.cuh"
#include "ptx.cuh"

namespace dflash {

namespace {

constexpr int kMaxStages = 12;
constexpr int kBarBytes = 8 * (2 * kMaxStages + 1) + 16;
constexpr size_t kSmemPerSM = 228 * 1024;     // shared memory of one SM
constexpr size_t kSmemReservedPerCta = 1024;
constexpr size_t kSmemMaxPerCta = 227 * 1024;  // opt-in limit of one CTA

template <int BN, int PL>
struct TcCfg {
  static constexpr int kN = BN * PL;                  // MMA N
  static constexpr int kABytes = kTileN * 128;        // 128 rows x 64 bf16
  static constexpr int kBBytes = kN * 128;            // PL*BN rows x 64 bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = kN <= 32 ? 32 : kN;
  static constexpr int kChunk = BN < 32 ? BN : 32;    // token columns per epilogue pass
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-B alignment");
  static_assert(kN <= 256 && kN % 16 == 0, "MMA N must be a multiple of 16 up to 256");
  static_assert(kTileN * (kChunk + 1) * 4 <= kStageBytes, "epilogue tile must fit one stage");
  static size_t smem(int stages) { return 1024 + (size_t)stages * kStageBytes + kBarBytes; }
};

size_t stage_bytes(int bm, int planes) { return kTileN * 128 + (size_t)bm * planes * 128; }

// Accumulator columns c0..c0+CH-1 of this warp's lanes; with a hi/lo operand
// pair the lo block (columns BN..2BN-1) is added.
template <int BN, int PL, int CH>
__device__ __forceinline__ void load_acc(uint32_t trow, int c0, float* v) {
#pragma unroll
  for (int h = 0; h < CH; h += 16) ptx::tmem_ld16(trow + c0 + h, v + h);
  if constexpr (PL == 2) {
    float w[CH];
#pragma unroll
    for (int h = 0; h < CH; h += 16) ptx::tmem_ld16(trow + BN + c0 + h, w + h);
#pragma unroll
    for (int j = 0; j < CH; ++j) v[j] += w[j];
  }
}

constexpr long long kWaitBudget = 200000000LL;   // SM cycles (~0.1 s): far beyond any legal wait

template <int BN, int PL, class Epi>
__global__ void __launch_bounds__(128, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap xmap,
                                                         const __grid_constant__ GemmProblem p,
                                                         const __grid_constant__ Epi epi, int32_t* status) {
  using C = TcCfg<BN, PL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * C::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);   // [0] abort, [1] last split, [2] loads issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gtile = blockIdx.x, split = blockIdx.y, mt = blockIdx.z;
  const int m0 = mt * BN, mc = min(BN, p.M - m0);
  const int si = find_seg(p, gtile);
  const GemmSeg& sg = p.seg[si];
  const int tis = gtile - sg.tile_begin;
  const int kb0 = split * p.kblocks_per_split;
  const int nk = min(p.K / 64, kb0 + p.kblocks_per_split) - kb0;
  const CUtensorMap* wmaps = static_cast<const CUtensorMap*>(p.wmaps);
  const CUtensorMap* map0 = wmaps + sg.map0;
  const CUtensorMap* map1 = wmaps + (sg.paired ? sg.map1 : sg.map0);
  // optional timestamps: [0] start, [1] set up, [2] first stage landed,
  // [3] last stage landed, [4] accumulator ready, [5] done, [6] SM, [7] reduced
  unsigned long long* tr = p.trace ? p.trace + 8 * ((size_t)(blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x)
                                   : nullptr;
  if (tr && threadIdx.x == 0) {
    tr[0] = ptx::globaltimer();
    tr[6] = ptx::smid();
    tr[7] = 0;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full + s, 1);
      ptx::mbar_init(empty + s, 1);
    }
    ptx::mbar_init(accf, 1);
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&xmap);
    ptx::prefetch_tmap(map0);
    ptx::prefetch_tmap(map1);
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, C::kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_trigger();
  if (tr && threadIdx.x == 0) tr[1] = ptx::globaltimer();

  if (warp == 0 && lane == 0) {
    // ---- TMA producer.  The weight tiles of the first stages do not depend
    // on earlier kernels and are requested before griddep_wait(), so they
    // stream in while the previous kernel drains.
    const uint64_t pol_w = ptx::policy_evict_first(), pol_x = ptx::policy_evict_last();
    const int r0 = half_first_row(sg, tis, 0), r1 = half_first_row(sg, tis, 1);
    const int prow = static_cast<int>(p.plane_stride / p.ldx);
    auto load_w = [&](int i) {
      uint8_t* a = smem + (i % S) * C::kStageBytes;
      const int kx = (kb0 + i) * 64;
      ptx::tma_load_2d(a, map0, full + i % S, kx, r0, pol_w);
      ptx::tma_load_2d(a + kHalfN * 128, map1, full + i % S, kx, r1, pol_w);
    };
    auto load_x = [&](int i) {
      uint8_t* b = smem + (i % S) * C::kStageBytes + C::kABytes;
      const int kx = (kb0 + i) * 64;
#pragma unroll
      for (int pl = 0; pl < PL; ++pl)
        ptx::tma_load_2d(b + pl * BN * 128, &xmap, full + i % S, kx, pl * prow + m0, pol_x);
    };
    const int pre = min(nk, S);
    for (int i = 0; i < pre; ++i) {
      ptx::mbar_arrive_expect_tx(full + i, C::kStageBytes);
      load_w(i);
    }
    griddep_wait();
    for (int i = 0; i < pre; ++i) load_x(i);
    int issued = pre;
    for (int i = pre; i < nk; ++i) {
      const int s = i % S;
      if (!ptx::mbar_wait(empty + s, ((i / S) & 1) ^ 1, kWaitBudget, status)) {
        flags[0] = 1;
        break;
      }
      ptx::mbar_arrive_expect_tx(full + s, C::kStageBytes);
      load_w(i);
      load_x(i);
      ++issued;
    }
    flags[2] = issued;
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(kTileN, C::kN);
    for (int i = 0; i < nk; ++i) {
      const int s = i % S;
      if (!ptx::mbar_wait(full + s, (i / S) & 1, kWaitBudget, status)) {
        flags[0] = 1;
        break;
      }
      if (tr && (i == 0 || i == nk - 1)) tr[i == 0 ? 2 : 3] = ptx::globaltimer();
      ptx::tc_fence_after();
      const uint64_t ad = ptx::smem_desc_sw128(smem + s * C::kStageBytes);
      const uint64_t bd = ptx::smem_desc_sw128(smem + s * C::kStageBytes + C::kABytes);
#pragma unroll
      for (int k = 0; k < 4; ++k)   // 4 x K=16 per 64-column stage; +32 B per step inside the swizzle row
        ptx::mma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (i | k) != 0 ? 1u : 0u);
      ptx::mma_commit(empty + s);
    }
    ptx::mma_commit(accf);
  }
  __syncwarp();

  // ---- epilogue (all 4 warps; warp w owns accumulator lanes 32w..32w+31)
  griddep_wait();
  const bool ok = ptx::mbar_wait(accf, 0, kWaitBudget, status);
  ptx::tc_fence_after();
  __syncthreads();
  const bool abort = !ok || flags[0] != 0;
  if (tr && threadIdx.x == 0) tr[4] = ptx::globaltimer();
  float* st = reinterpret_cast<float*>(smem);   // [128][kChunk+1], reuses the drained stages
  constexpr int ld = C::kChunk + 1;
  const int n = warp * 32 + lane;
  const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);

  if (!abort) {
    if (p.splits == 1) {
      for (int c0 = 0; c0 < mc; c0 += C::kChunk) {
        float v[C::kChunk];
        load_acc<BN, PL, C::kChunk>(trow, c0, v);
#pragma unroll
        for (int j = 0; j < C::kChunk; ++j) st[n * ld + j] = v[j];
        __syncthreads();
        epi(st, ld, m0 + c0, min(C::kChunk, mc - c0), gtile, sg, tis, threadIdx.x, blockDim.x);
        __syncthreads();
      }
    } else {
      const size_t ntot = static_cast<size_t>(p.total_tiles) * kTileN;
      for (int c0 = 0; c0 < mc; c0 += C::kChunk) {
        float v[C::kChunk];
        load_acc<BN, PL, C::kChunk>(trow, c0, v);
#pragma unroll
        for (int j = 0; j < C::kChunk; ++j)
          if (c0 + j < mc)
            p.partial[(static_cast<size_t>(split) * p.M + m0 + c0 + j) * ntot + static_cast<size_t>(gtile) * kTileN + n] =
                v[j];
      }
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) {
        int* c = p.counters + mt * p.total_tiles + gtile;
        const int old = atomicAdd(c, 1);
        flags[1] = old == p.splits - 1;
        if (flags[1]) *c = 0;   // ready for the next launch
      }
      __syncthreads();
      if (flags[1]) {
        __threadfence();
        // thread t sums features 4(t%32)..+3 of rows t/32, t/32+4, ... over
        // all splits with 16-byte loads, 4 splits' loads in flight at a time
        const size_t sstride = static_cast<size_t>(p.M) * ntot;
        const int fq = (threadIdx.x & 31) * 4, r0 = threadIdx.x >> 5;
        constexpr int kRows = C::kChunk / 4;
        for (int c0 = 0; c0 < mc; c0 += C::kChunk) {
          const int cc = min(C::kChunk, mc - c0);
          const float* base =
              p.partial + static_cast<size_t>(m0 + c0) * ntot + static_cast<size_t>(gtile) * kTileN + fq;
          float4 acc[kRows];
#pragma unroll
          for (int i = 0; i < kRows; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          int sp = 0;
          for (; sp + 4 <= p.splits; sp += 4) {
            float4 v[4][kRows];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int i = 0; i < kRows; ++i) {
                const int r = r0 + 4 * i;
                v[u][i] = r < cc ? __ldcg(reinterpret_cast<const float4*>(base + (sp + u) * sstride +
                                                                          static_cast<size_t>(r) * ntot))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int i = 0; i < kRows; ++i) {
                acc[i].x += v[u][i].x;
                acc[i].y += v[u][i].y;
                acc[i].z += v[u][i].z;
                acc[i].w += v[u][i].w;
              }
          }
          for (; sp < p.splits; ++sp)
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
              const int r = r0 + 4 * i;
              if (r < cc) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(base + sp * sstride + static_cast<size_t>(r) * ntot));
                acc[i].x += v.x;
                acc[i].y += v.y;
                acc[i].z += v.z;
                acc[i].w += v.w;
              }
            }
#pragma unroll
          for (int i = 0; i < kRows; ++i) {
            const int r = r0 + 4 * i;
            st[(fq + 0) * ld + r] = acc[i].x;
            st[(fq + 1) * ld + r] = acc[i].y;
            st[(fq + 2) * ld + r] = acc[i].z;
            st[(fq + 3) * ld + r] = acc[i].w;
          }
          __syncthreads();
          epi(st, ld, m0 + c0, cc, gtile, sg, tis, threadIdx.x, blockDim.x);
          __syncthreads();
        }
      }
    }
  } else if (threadIdx.x == 0) {
    // a wait ran out: let every load this CTA issued land before the CTA exits
    const int issued = flags[2];
    for (int i = max(0, issued - S); i < issued; ++i)
      ptx::mbar_wait(full + (i % S), (i / S) & 1, kWaitBudget, status);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (tr && threadIdx.x == 0) {
    tr[5] = ptx::globaltimer();
    tr[7] = flags[1];
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- dense persistent kernel
// Many token rows (tensor-bound): one CTA per SM walks the output tiles
// (128 features x BN tokens) round-robin, tile = CTA + k * grid, the token
// tiles of one weight tile adjacent so that CTAs running at the same time
// read that weight tile from L2.  Roles (192 threads):
//   warp 4 lane 0   TMA producer: weight halves and activation planes of every
//                   K block into an S-stage ring
//   warp 5          TMEM allocation (two 256-column accumulators); lane 0
//                   issues tcgen05.mma, frees ring stages and signals each
//                   finished accumulator with tcgen05.commit
//   warps 0..3      epilogue of the previous tile (TMEM lanes 32w..32w+31)
//                   while the MMAs of the next tile run
// No split-K: every tile runs its whole K, so results match the one-tile
// kernel's order of summation within a tile (fp32 accumulation in TMEM).
constexpr int kDenseThreads = 192;

template <int BN, int PL>
struct DenseCfg {
  using C = TcCfg<BN, PL>;
  static constexpr int kLd = C::kChunk + 1;
  static constexpr int kStBytes = kTileN * kLd * 4;   // epilogue staging tile
  static constexpr size_t smem(int stages) {
    return 1024 + (size_t)stages * C::kStageBytes + kStBytes + 8 * (2 * kMaxStages + 5) + 16;
  }
};

template <int BN, int PL, class Epi>
__global__ void __launch_bounds__(kDenseThreads, 1) gemm_dense_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                      const __grid_constant__ GemmProblem p,
                                                                      const __grid_constant__ Epi epi,
                                                                      int token_tiles, int32_t* status) {
  using C = TcCfg<BN, PL>;
  using D = DenseCfg<BN, PL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  float* st = reinterpret_cast<float*>(smem + (size_t)S * C::kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * C::kStageBytes + D::kStBytes);
  uint64_t* empty = full + kMaxStages;
  uint64_t* accf = empty + kMaxStages;     // [2]
  uint64_t* accfree = accf + 2;            // [2]
  uint64_t* mdone = accfree + 2;           // every MMA of this CTA has finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, ntiles = p.total_tiles * token_tiles, nk = p.K / 64;
  const CUtensorMap* wmaps = static_cast<const CUtensorMap*>(p.wmaps);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(full + i, 1);
      ptx::mbar_init(empty + i, 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(accf + b, 1);
      ptx::mbar_init(accfree + b, 1);
    }
    ptx::mbar_init(mdone, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&xmap);
  }
  if (warp == 5) ptx::tmem_alloc(tmem_slot, 2 * C::kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_trigger();

  if (warp == 4) {
    if (lane == 0) {
      // ---- TMA producer
      const uint64_t pol_w = ptx::policy_evict_first(), pol_x = ptx::policy_evict_last();
      const int prow = static_cast<int>(p.plane_stride / p.ldx);
      int it = 0;
      bool waited = false;   // griddep_wait() done (activations of earlier kernels visible)
      for (int tile = blockIdx.x; tile < ntiles && !*reinterpret_cast<volatile int*>(abort_flag); tile += G) {
        const int gtile = tile / token_tiles, m0 = (tile - gtile * token_tiles) * BN;
        const GemmSeg& sg = p.seg[find_seg(p, gtile)];
        const int tis = gtile - sg.tile_begin;
        const CUtensorMap* map0 = wmaps + sg.map0;
        const CUtensorMap* map1 = wmaps + (sg.paired ? sg.map1 : sg.map0);
        const int r0 = half_first_row(sg, tis, 0), r1 = half_first_row(sg, tis, 1);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % S;
          if (it >= S && !ptx::mbar_wait(empty + s, ((it / S) & 1) ^ 1, kWaitBudget, status)) {
            *abort_flag = 1;
            break;
          }
          uint8_t* a = smem + (size_t)s * C::kStageBytes;
          ptx::mbar_arrive_expect_tx(full + s, C::kStageBytes);
          // weights first: they do not depend on earlier kernels
          ptx::tma_load_2d(a, map0, full + s, kb * 64, r0, pol_w);
          ptx::tma_load_2d(a + kHalfN * 128, map1, full + s, kb * 64, r1, pol_w);
          if (!waited) {
            griddep_wait();
            waited = true;
          }
#pragma unroll
          for (int pl = 0; pl < PL; ++pl)
            ptx::tma_load_2d(a + C::kABytes + pl * BN * 128, &xmap, full + s, kb * 64, pl * prow + m0, pol_x);
        }
      }
      // every load issued lands before the CTA can exit
      for (int j = max(0, it - S); j < it; ++j) ptx::mbar_wait(full + (j % S), (j / S) & 1, kWaitBudget, status);
      if (!waited) griddep_wait();
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ---- MMA issuer
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kTileN, C::kN);
      int it = 0, seq = 0;
      bool any = false;
      for (int tile = blockIdx.x; tile < ntiles; tile += G, ++seq) {
        const int buf = seq & 1, use = seq >> 1;
        if (use >= 1 && !ptx::mbar_wait(accfree + buf, (use - 1) & 1, kWaitBudget, status)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + buf * C::kTmemCols;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % S;
          if (!ptx::mbar_wait(full + s, (it / S) & 1, kWaitBudget, status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t ad = ptx::smem_desc_sw128(smem + (size_t)s * C::kStageBytes);
          const uint64_t bd = ptx::smem_desc_sw128(smem + (size_t)s * C::kStageBytes + C::kABytes);
#pragma unroll
          for (int k = 0; k < 4; ++k) ptx::mma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
          ptx::mma_commit(empty + s);
          any = true;
        }
        if (!ok) break;
        ptx::mma_commit(accf + buf);
      }
      if (any) {   // every MMA issued has finished before the tensor memory is freed
        ptx::mma_commit(mdone);
        ptx::mbar_wait(mdone, 0, kWaitBudget, status);
      }
    }
  } else {
    // ---- epilogue warps 0..3
    const int tid = threadIdx.x, n = warp * 32 + lane;
    constexpr int ld = D::kLd;
    griddep_wait();   // outputs may be read by the kernel before this one
    int seq = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += G, ++seq) {
      const int buf = seq & 1, use = seq >> 1;
      if (!ptx::mbar_wait(accf + buf, use & 1, kWaitBudget, status)) break;
      ptx::tc_fence_after();
      const int gtile = tile / token_tiles, m0 = (tile - gtile * token_tiles) * BN, mc = min(BN, p.M - m0);
      const GemmSeg& sg = p.seg[find_seg(p, gtile)];
      const int tis = gtile - sg.tile_begin;
      const uint32_t trow = tmem + buf * C::kTmemCols + (static_cast<uint32_t>(warp * 32) << 16);
      for (int c0 = 0; c0 < mc; c0 += C::kChunk) {
        float v[C::kChunk];
        load_acc<BN, PL, C::kChunk>(trow, c0, v);
#pragma unroll
        for (int j = 0; j < C::kChunk; ++j) st[n * ld + j] = v[j];
        if (c0 + C::kChunk >= mc) {   // the accumulator is read: the MMAs of tile + 2G may start
          ptx::tc_fence_before();
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (c0 + C::kChunk >= mc && tid == 0) ptx::mbar_arrive(accfree + buf);
        epi(st, ld, m0 + c0, min(C::kChunk, mc - c0), gtile, sg, tis, tid, 128);
        asm volatile("bar.sync 1, 128;" ::: "memory");
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 2 * C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

template <int BN, int PL, class Epi>
cudaError_t launch_bn(const GemmProblem& p, const GemmPlan& plan, const Epi& epi, cudaStream_t s) {
  using C = TcCfg<BN, PL>;
  static bool attr_set = false;   // per instantiation; the attribute is per device function
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, PL, Epi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)std::min(C::smem(kMaxStages), kSmemMaxPerCta));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (p.stages < 1 || p.stages > kMaxStages || C::smem(p.stages) != plan.smem) return cudaErrorInvalidValue;
  if (p.planes != PL || p.plane_stride % p.ldx) return cudaErrorInvalidValue;
  // one map over both planes: plane 1 starts plane_stride/ldx rows after plane 0
  const int rows = PL == 1 ? p.M : static_cast<int>(p.plane_stride / p.ldx) + p.M;
  CUtensorMap xmap;
  if (!encode_activation_map(&xmap, p.x, p.K, rows, p.ldx, BN)) return cudaErrorInvalidValue;
  dim3 grid(p.total_tiles, plan.splits, plan.token_tiles);
  static const bool log = debug_env("DFLASH_GEMM_LOG") != nullptr;   // plan of every launch, to stderr
  if (log)
    std::fprintf(stderr, "gemm_tc M=%d K=%d tiles=%d BN=%d PL=%d splits=%d kb/split=%d stages=%d grid=%dx%dx%d%s\n",
                 p.M, p.K, p.total_tiles, BN, PL, plan.splits, plan.kblocks_per_split, p.stages, grid.x, grid.y,
                 grid.z, p.trace ? " [traced]" : "");
  return launch_pdl(gemm_tc_kernel<BN, PL, Epi>, grid, dim3(128), C::smem(p.stages), s, xmap, p, epi, p.status);
}

template <int BN, int PL, class Epi>
cudaError_t launch_dense_cfg(const GemmProblem& p, const GemmPlan& plan, const Epi& epi, cudaStream_t s) {
  using D = DenseCfg<BN, PL>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_dense_kernel<BN, PL, Epi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)D::smem(4));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (p.stages != 4 || plan.smem != D::smem(4) || p.planes != PL || plan.bm != BN || (PL == 2 && p.plane_stride % p.ldx) ||
      p.K % 64)
    return cudaErrorInvalidValue;
  const int rows = PL == 1 ? p.M : static_cast<int>(p.plane_stride / p.ldx) + p.M;
  CUtensorMap xmap;
  if (!encode_activation_map(&xmap, p.x, p.K, rows, p.ldx, BN)) return cudaErrorInvalidValue;
  static const bool log = debug_env("DFLASH_GEMM_LOG") != nullptr;
  if (log)
    std::fprintf(stderr, "gemm_dense M=%d K=%d tiles=%d BN=%d PL=%d token_tiles=%d grid=%d\n", p.M, p.K,
                 p.total_tiles, BN, PL, plan.token_tiles, plan.grid);
  return launch_pdl(gemm_dense_kernel<BN, PL, Epi>, dim3(plan.grid), dim3(kDenseThreads), D::smem(4), s, xmap, p,
                    epi, plan.token_tiles, p.status);
}

template <class Epi>
cudaError_t launch_dense(const GemmProblem& p, const GemmPlan& plan, const Epi& epi, cudaStream_t s) {
  static_assert(DenseCfg<128, 2>::smem(4) == DenseCfg<256, 1>::smem(4), "one plan size for both shapes");
  return p.planes == 2 ? launch_dense_cfg<128, 2, Epi>(p, plan, epi, s) : launch_dense_cfg<256, 1, Epi>(p, plan, epi, s);
}

}  // namespace

size_t dense_smem(int stages) { return DenseCfg<128, 2>::smem(stages); }

bool encode_weight_map(void* map, const void* base, int inner, int rows, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_activation_map(void* map, const void* base, int inner, int rows, int row_stride, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_stride * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t tensor_map_bytes() { return sizeof(CUtensorMap); }

// Plan of one launch from a small streaming model.  For every pipeline depth
// S (which fixes the CTAs that fit on an SM) and split-K factor, the launch
// runs in waves of resident CTAs; a CTA streams its weight tiles at
// min(HBM bandwidth / resident CTAs, bytes in flight / latency), and pays a
// fixed start cost per wave plus a reduction tail when K is split.  The
// cheapest plan wins.  With DFLASH_DEBUG=1, DFLASH_TC_STAGES forces S,
// DFLASH_TC_KMIN is the fewest 64-column K blocks per split and
// DFLASH_TC_SPLITS forces the split factor (environment, read once).
int env_int(const char* name, int dflt, bool debug_only = true) {
  const char* v = debug_only ? debug_env(name) : getenv(name);
  return v ? atoi(v) : dflt;
}

GemmPlan plan_gemm_tc(int M, int K, int tiles, int sms, int planes) {
  static const int env_stages = env_int("DFLASH_TC_STAGES", 0);
  static const int env_kmin = env_int("DFLASH_TC_KMIN", 4);
  static const int env_splits = env_int("DFLASH_TC_SPLITS", 0);   // force a split factor (experiments)
  constexpr double kBw = 6.5e12, kLat = 3.2e-6, kStart = 2.0e-6, kReduce = 3.0e-6;
  GemmPlan g{};
  g.tc = 1;
  g.planes = planes;
  const int bm_max = planes == 2 ? 128 : 256;   // MMA N = planes * bm <= 256
  g.bm = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
  g.bm = std::min(g.bm, bm_max);
  g.token_tiles = (M + g.bm - 1) / g.bm;
  static const int env_dense = env_int("DFLASH_DENSE", 1, false);   // 0: never the persistent many-row kernel
  const long dense_tiles = (long)tiles * g.token_tiles;
  // (both shapes have MMA N = 256: 128 rows of a hi/lo pair, or 256 one-plane rows)
  if (env_dense && ((planes == 2 && g.bm == 128) || (planes == 1 && g.bm == 256)) && g.token_tiles >= 2 &&
      4 * dense_tiles >= 3L * sms) {
    // tensor-bound: a persistent kernel with every tile's whole K (no split-K
    // reduction) and the epilogue overlapped with the next tile's MMAs
    g.dense = 1;
    g.grid = (int)std::min<long>(sms, dense_tiles);
    g.stages = 4;
    g.smem = dense_smem(g.stages);
    g.splits = 1;
    g.kblocks_per_split = K / 64;
    g.partial_floats = 0;
    g.counters = 0;
    return g;
  }
  const size_t sb = stage_bytes(g.bm, planes);
  const int s_max = std::min<int>(kMaxStages, (int)((kSmemMaxPerCta - 1024 - kBarBytes) / sb));
  const int kblocks = K / 64;
  const int kmax = std::max(1, kblocks / std::max(1, env_kmin));
  const long base = (long)tiles * g.token_tiles;
  double best = 1e30;
  for (int S : {3, 4, 5, 6, 7, 8, 10}) {
    if (env_stages > 0 && S != std::min(env_stages, s_max)) continue;
    if (S > s_max) continue;
    const size_t smem = 1024 + (size_t)S * sb + kBarBytes;
    const long slots = (long)sms * std::max<long>(1, (long)(kSmemPerSM / (smem + kSmemReservedPerCta)));
    for (int sp = 1; sp <= kmax; ++sp) {
      if (env_splits > 0 && sp != std::min(env_splits, kmax)) continue;
      const int kbps = (kblocks + sp - 1) / sp;
      const int splits = (kblocks + kbps - 1) / kbps;
      if (splits != sp && env_splits <= 0) continue;
      const long ctas = base * splits;
      // One-plane 256-row tiles (exact target features): a stage's activation
      // tile is twice its weight tile, and a split that runs in more than one
      // wave costs more than this model says (512 rows x 20,480 x 4,096 on 152
      // SMs: 7 splits in three waves 174 us, 2 splits in one wave 105 us), so
      // split-K stays within one wave there.
      if (planes == 1 && g.bm == 256 && splits > 1 && ctas > slots && env_splits <= 0) continue;
      // HBM side: the weight tile of each stage (activation tiles come from L2)
      const double wtile = kTileN * 128.0;
      const double bytes = kbps * wtile, inflight = std::min(S, kbps) * wtile;
      double t = splits > 1 ? kReduce : 0.0;
      for (long left = ctas; left > 0; left -= slots) {
        const long n = std::min(left, slots);
        t += bytes / std::min(kBw / n, inflight / kLat) + kStart;
      }
      if (t < best * 0.999) {
        best = t;
        g.stages = S;
        g.smem = smem;
        g.kblocks_per_split = kbps;
        g.splits = splits;
      }
    }
  }
  g.partial_floats = g.splits > 1 ? (size_t)g.splits * M * tiles * kTileN : 0;
  g.counters = g.splits > 1 ? g.token_tiles * tiles : 0;
  return g;
}

template <class Epi>
cudaError_t gemm_tc_launch(const GemmProblem& p, const GemmPlan& plan, const Epi& epi, cudaStream_t s) {
  if (plan.dense) return launch_dense<Epi>(p, plan, epi, s);
  if (plan.planes == 1) {   // operands that are exact in bf16 (target features)
    switch (plan.bm) {
      case 16: return launch_bn<16, 1, Epi>(p, plan, epi, s);
      case 32: return launch_bn<32, 1, Epi>(p, plan, epi, s);
      case 64: return launch_bn<64, 1, Epi>(p, plan, epi, s);
      case 128: return launch_bn<128, 1, Epi>(p, plan, epi, s);
      case 256: return launch_bn<256, 1, Epi>(p, plan, epi, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (plan.bm) {
    case 16: return launch_bn<16, 2, Epi>(p, plan, epi, s);
    case 32: return launch_bn<32, 2, Epi>(p, plan, epi, s);
    case 64: return launch_bn<64, 2, Epi>(p, plan, epi, s);
    case 128: return launch_bn<128, 2, Epi>(p, plan, epi, s);
    default: return cudaErrorInvalidValue;
  }
}

template cudaError_t gemm_tc_launch<EpiStoreF32>(const GemmProblem&, const GemmPlan&, const EpiStoreF32&, cudaStream_t);
template cudaError_t gemm_tc_launch<EpiResidual>(const GemmProblem&, const GemmPlan&, const EpiResidual&, cudaStream_t);
template cudaError_t gemm_tc_launch<EpiSwiGLU<__nv_bfloat16>>(const GemmProblem&, const GemmPlan&,
                                                              const EpiSwiGLU<__nv_bfloat16>&, cudaStream_t);
template cudaError_t gemm_tc_launch<EpiQKV<__nv_bfloat16>>(const GemmProblem&, const GemmPlan&,
                                                           const EpiQKV<__nv_bfloat16>&, cudaStream_t);
template cudaError_t gemm_tc_launch<EpiInject<__nv_bfloat16>>(const GemmProblem&, const GemmPlan&,
                                                              const EpiInject<__nv_bfloat16>&, cudaStream_t);
template cudaError_t gemm_tc_launch<EpiArgmax>(const GemmProblem&, const GemmPlan&, const EpiArgmax&, cudaStream_t);
template cudaError_t gemm_tc_launch<EpiRowsRope>(const GemmProblem&, const GemmPlan&, const EpiRowsRope&, cudaStream_t);

}  // namespace dflash
