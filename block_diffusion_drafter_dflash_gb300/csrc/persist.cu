// Persistent draft-cycle kernel for bf16 drafters at small batch (at most 16
// token rows per call): every projection of one API call — for the drafter
// pass Q/K/V, W_O, gate/up and W_D of every layer and the shared LM head, for
// an injection the fusion W_c and all layers' W_K/W_V — together with the
// block attention between them, run as the phases of ONE launch with one CTA
// per SM, separated by grid-wide barriers.
//
// Why: at a few token rows each projection streams its weights once from HBM
// and does almost no arithmetic.  Launched as one kernel per projection, the
// weight stream drains and refills at every kernel boundary.  Here the TMA
// producers of each CTA stream the weight tiles of all phases back to back
// through a shared-memory ring and run ahead across the barriers (weights do
// not depend on activations), so HBM keeps working while a phase's inputs are
// still being produced.
//
// MMA orientation.  tcgen05.mma costs about the same time per instruction
// whatever its N (measured on this part: ~133 SM cycles for M=128 and any N
// up to 256), so the bigger projections (gate/up, the LM head) put weights on
// the N side, 256 features per instruction (8 KB of weights per K=16 step),
// and the token rows on the M side: A rows 0..15 are the activations' hi
// plane, rows 16..31 the lo plane; rows 32..127 of A are never read back
// (their accumulator rows are discarded), so that A tile overlaps the
// stage's own weight tile.  Only TMEM lanes 0..31 (warp 4) then hold results.
// The small projections (Q/K/V, W_O, W_D, fusion, injection) keep weights on
// the M side (128 features x 32 token columns an instruction): their tiles
// are split over fewer CTAs and all four compute warps read the accumulator
// back, which keeps the phase tail short where it matters more than the
// tensor-pipe rate.  A stage is [8 KB activations][32 KB weights] either way:
// 64 K columns of 256 features for the wide phases, 128 K columns of 128
// features (two 64-column boxes of each operand) for the narrow ones, so
// every phase keeps the same bytes in flight.
//
// Roles (256 threads):
//   warps 0, 3      lane 0: weight producers (even / odd ring slots), TMA of the
//                   <=256 x 64 weight tile of each stage (128-row boxes)
//   warp 1          TMEM allocation (512 columns); lane 0 issues tcgen05.mma
//   warp 2 lane 0   activation producer: TMA of the 16-row hi/lo activation
//                   tiles of each stage, once every earlier phase is complete
//   warps 4..7      accumulator read-back, epilogues, stream-K reductions,
//                   attention and its merge, grid barriers
// The accumulator of an output tile (<= 256 TMEM columns) is double-buffered
// so that the MMAs of one tile overlap the epilogue of the previous one.
//
// Work split (stream-K): the (tile, 64-column K block) iterations of a
// projection are divided evenly over the CTAs.  A tile cut between CTAs
// leaves fp32 partial tiles.  Its reducer is the CTA holding its first K
// blocks: that piece ends the reducer's span, so it finishes last anyway.
// The other CTAs publish their pieces and announce each with one atomic add;
// the reducer keeps its own piece in shared memory, waits (bounded) for the
// count, adds the others in CTA order and runs the epilogue — the sum does
// not depend on timing, and the reducer's chain has no publish, fence or
// ticket round trip of its own.
//
// RMSNorm folds into its neighbours: whoever produces a normed input (the
// residual-stream epilogues, the fusion epilogue, the draft prologue) writes
// it multiplied by the norm's gain as hi/lo bf16 planes, plus per (128-feature
// tile, row) sums of squares; the consuming projection multiplies row m of its
// accumulator by 1/rms(row m) = (sum_t ssq[t][m] / D + eps)^(-1/2).
//
// Data one CTA writes and another reads within the launch (sums of squares,
// partial tiles, Q, attention partials, the residual stream) is read with
// L2-only loads (L1 is not coherent across SMs); activations read by TMA are
// published with a generic-to-async proxy fence on both sides of the barrier.
//
// Every wait is bounded (mbarriers, grid barrier): on expiry the kernel sets
// DFLASH_ERR_TIMEOUT in the status word, waits for its own copies in flight,
// frees its tensor memory and returns.
#include <cuda.h>

#include <algorithm>
#include <atomic>

#include "attn_tc.cuh"
#include "gemm.cuh"
#include "persist.cuh"
#include "ptx.cuh"

namespace dflash {

namespace {

constexpr int kThreads = 256;
constexpr int kXHalf = 2 * kPRows * 128;          // activations of 64 K columns: two 16-row planes (A rows 0..31)
constexpr int kXBytes = 2 * kXHalf;               // a stage holds up to 128 K columns of activations
constexpr int kTwMax = 256;                       // features per tile (MMA N)
constexpr int kWBox = 128 * 128;                  // one 128-row weight box
constexpr int kStage = kXBytes + 2 * kWBox;       // 40 KB
constexpr int kLd = kPRows + 1;                   // staging tile pitch (floats)
constexpr int kTmemCols = 2 * kTwMax;             // double-buffered 256-column accumulator
constexpr long long kBudget = 200000000LL;        // SM cycles (~0.1 s): far beyond any legal wait
constexpr size_t kSmemMax = 227 * 1024;

template <int HD>
struct PCfg {
  static constexpr int kRegion = kTwMax * kLd * 4;   // epilogue staging tile st[256][kLd]
};

struct PBook {
  uint64_t fullW[kPMaxStages], fullX[kPMaxStages], empty[kPMaxStages];
  uint64_t accf[2], accfree[2], mma_done;
  uint32_t tmem;
  int flag_acc, flag_tk, flag_bar;
  uint64_t ring_free;   // attention is done with the ring (one phase per attention phase)
  attn_tc::Bars abars;  // the attention's TMA and MMA barriers
  int ctx_len[kPRows];  // context length of every request (constant during the launch)
  float rs[kPRows];
};

static_assert(kStage % 1024 == 0 && kXBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");

size_t region_bytes(int hd) { return hd == 64 ? PCfg<64>::kRegion : PCfg<128>::kRegion; }

// ---------------------------------------------------------------- stream-K bookkeeping
struct Span {
  int i0, i1;
};

// 32-bit arithmetic (a 64-bit division is a long software sequence, and the
// reducer of a tile runs several before its first load): persist_launch
// refuses a program whose tiles * kb * grid reaches 2^31.
__device__ __forceinline__ int phase_iters(const PPhase& ph) { return ph.tiles * ph.kb; }
__device__ __forceinline__ int phase_ctas(const PPhase& ph, int G) { return min(G, phase_iters(ph)); }
// iterations [i0, i1) of CTA c (CTAs >= phase_ctas get none)
__device__ __forceinline__ Span cta_span(const PPhase& ph, int G, int c) {
  const int W = phase_iters(ph);
  const int g = phase_ctas(ph, G);
  if (c >= g) return {0, 0};
  return {c * W / g, (c + 1) * W / g};
}
// the CTA whose span holds iteration i
__device__ __forceinline__ int cta_of(const PPhase& ph, int G, int i) {
  const int W = phase_iters(ph);
  const int g = phase_ctas(ph, G);
  return ((i + 1) * g - 1) / W;
}
__device__ __forceinline__ int seg_of(const PParams& p, const PPhase& ph, int t) {
  int s = ph.seg0;
  while (s + 1 < ph.seg0 + ph.nseg && t >= p.seg[s + 1].tile_begin) ++s;
  return s;
}

// ---------------------------------------------------------------- grid barrier
__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait until `target` arrivals have been counted (bounded).
__device__ bool grid_wait(const unsigned int* bar, unsigned int target, int32_t* status) {
  if (ld_acquire(bar) >= target) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(32);
    if (ld_acquire(bar) >= target) return true;
    if ((it & 63) == 0) {
      if (*reinterpret_cast<volatile int32_t*>(status) == DFLASH_ERR_TIMEOUT) return false;
      if (clock64() - t0 > kBudget) {
        report_status(status, DFLASH_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Optional timestamps (globaltimer ns), per (CTA, phase): [0] compute warps
// start the phase, [1] they are done with it, [2] / [3] first / last weight
// load issued, [4] activation loads released, [5] first MMA issued, [6] last
// MMA of the phase committed, [7] SM id (phase 0 only).
// [8..11]: SM cycles the MMA issuer waited for weights / activations, and the
// weight producer (even stages) / activation producer waited for free slots.
// [12..15]: for the CTA's last piece of the phase: accumulator ready, tile
// staged, epilogue done or partial published, reduction + epilogue done; in
// an attention phase: Q staged, first scores ready, last P V done, written.
enum { kTrStart = 0, kTrDone, kTrW0, kTrW1, kTrX0, kTrM0, kTrM1, kTrSm, kTrWaitW, kTrWaitX, kTrWaitWEmpty,
       kTrWaitXEmpty, kTrAcc, kTrStaged, kTrPub, kTrRed, kTrReadBack, kTrCombined, kTrSlots };
__device__ __forceinline__ void trace_val(const PParams& p, int cta, int pi, int slot, unsigned long long v) {
  if (p.trace) p.trace[((size_t)cta * kPMaxPhases + pi) * kTrSlots + slot] = v;
}
__device__ __forceinline__ void trace_at(const PParams& p, int cta, int pi, int slot) {
  if (p.trace) trace_val(p, cta, pi, slot, ptx::globaltimer());
}
// mbar_wait that adds the cycles spent to `acc` (for the trace); `sleep`:
// back off between polls (producers, which run ahead of everything else)
__device__ __forceinline__ bool wait_timed(uint64_t* bar, uint32_t parity, int32_t* status, long long& acc,
                                           bool sleep = false) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  const bool ok = sleep ? ptx::mbar_wait_sleep(bar, parity, kBudget, status) : ptx::mbar_wait(bar, parity, kBudget, status);
  acc += clock64() - t0;
  return ok;
}

struct ComputeSync {
  __device__ __forceinline__ void operator()() const { csync(); }
};

// Wait for the loads of the last use of every ring slot that this producer
// filled (slots of parity `par`, or all when par < 0); bounded, and they were
// issued, so they complete.
__device__ void drain_slots(uint64_t* full, int issued, int S, int par, int32_t* status) {
  for (int j = max(0, issued - S); j < issued; ++j)
    if (par < 0 || ((j % S) & 1) == par) ptx::mbar_wait(full + (j % S), (j / S) & 1, kBudget, status);
}

// ---------------------------------------------------------------- producers and MMA
// Weight rows of box h (128 rows) of tile `tis` of a segment: unpaired tiles
// are tw consecutive rows of w0; a paired tile is 128 rows of w0 (SwiGLU gate)
// then the same 128 rows of w1 (up).
__device__ __forceinline__ int box_row(const GemmSeg& sg, int tis, int h) {
  return sg.paired ? 128 * tis : sg.tw * tis + 128 * h;
}

// Attention work item of CTA `cta`: (request b, kv head, chunk of key tiles
// [t0, t1)) of nct context tiles and one block tile; false if it has none.
struct AttnItem {
  int b, kvh, t0, t1, nct, c;
};
__device__ __forceinline__ bool attn_item(const AttnParams& ap, const int* ctx_len, int cta, AttnItem& it) {
  const int nch = ap.splits;
  if (cta >= ap.B * ap.nkv * nch) return false;
  const int r = cta % (ap.nkv * nch), ch = r % nch;
  it.b = cta / (ap.nkv * nch);
  it.kvh = r / nch;
  it.c = ctx_len[it.b];
  it.nct = (it.c + attn_tc::kKeys - 1) / attn_tc::kKeys;
  const int T = it.nct + 1;
  it.t0 = ch * T / nch;
  it.t1 = (ch + 1) * T / nch;
  return true;
}

// Two weight producers (warps 0 and 3) own the even and the odd ring slots:
// one issuing thread sustains only ~5 TB/s of TMA traffic across the device
// (its wait-and-issue loop, not bytes in flight, is the limit), two reach the
// HBM copy rate.
__device__ void weight_producer(const PParams& p, PBook* bk, uint8_t* ring, int G, int cta, int par) {
  const int S = p.stages;
  const uint64_t pol = ptx::policy_evict_first();
  int it = 0, attn_seen = 0;
  for (int pi = 0; pi < p.nphase; ++pi) {
    const PPhase& ph = p.ph[pi];
    if (ph.kind == kPhAttn) {
      // the attention phase borrows the ring's shared memory: load nothing
      // more until this CTA's attention is done
      if (!ptx::mbar_wait_sleep(&bk->ring_free, attn_seen & 1, kBudget, p.status)) goto done;
      ++attn_seen;
      continue;
    }
    if (ph.kind != kPhGemm) continue;
    const Span sp = cta_span(ph, G, cta);
    long long we = 0;
    for (int i = sp.i0; i < sp.i1; ++i, ++it) {
      const int s = it % S;
      if ((s & 1) != par) continue;
      if (it >= S && !wait_timed(&bk->empty[s], ((it / S) & 1) ^ 1, p.status, we, true)) goto done;
      if (i - sp.i0 < 2) trace_at(p, cta, pi, kTrW0);
      if (i + 2 >= sp.i1) trace_at(p, cta, pi, kTrW1);
      {
        const int t = i / ph.kb, kx = (i - t * ph.kb) * ph.kw;
        const GemmSeg& sg = p.seg[seg_of(p, ph, t)];
        const int tis = t - sg.tile_begin;
        uint8_t* w = ring + (size_t)s * kStage + kXBytes;
        ptx::mbar_arrive_expect_tx(&bk->fullW[s], 2 * kWBox);
        if (ph.kw == 128) {   // 128 features x 128 K columns: one box per 64-column half of K
          for (int h = 0; h < 2; ++h)
            ptx::tma_load_2d(w + h * kWBox, p.wmaps + sg.map0, &bk->fullW[s], kx + 64 * h, box_row(sg, tis, 0), pol);
        } else {              // 256 features x 64 K columns: two 128-row boxes
          for (int h = 0; h < 2; ++h)
            ptx::tma_load_2d(w + h * kWBox, p.wmaps + ((sg.paired && h) ? sg.map1 : sg.map0), &bk->fullW[s], kx,
                             box_row(sg, tis, h), pol);
        }
      }
    }
    if (par == 0) trace_val(p, cta, pi, kTrWaitWEmpty, we);
  }
done:
  drain_slots(bk->fullW, it, S, par, p.status);
}

// The activation producer (lane 0 of warp 2): the hi and lo 16-row tiles of
// each stage's 64-column K block, A rows 0..15 and 16..31.
__device__ void activation_producer(const PParams& p, PBook* bk, uint8_t* ring, int G, int cta) {
  const int S = p.stages;
  const uint64_t pol = ptx::policy_evict_last();
  int it = 0;
  long long wx = 0;
  for (int pi = 0; pi < p.nphase; ++pi) {
    const PPhase& ph = p.ph[pi];
    if (ph.kind != kPhGemm) continue;
    const Span sp = cta_span(ph, G, cta);
    if (sp.i0 == sp.i1) continue;
    // the phase's activations exist once every earlier phase is complete
    if (pi > 0 && !grid_wait(p.bar, (unsigned)pi * (unsigned)G, p.status)) goto done;
    ptx::fence_proxy_async_global();
    trace_at(p, cta, pi, kTrX0);
    wx = 0;
    for (int i = sp.i0; i < sp.i1; ++i, ++it) {
      const int s = it % S;
      if (it >= S && !wait_timed(&bk->empty[s], ((it / S) & 1) ^ 1, p.status, wx, true)) goto done;
      const int kx = (i % ph.kb) * ph.kw, halves = ph.kw / 64;
      uint8_t* x = ring + (size_t)s * kStage;
      ptx::mbar_arrive_expect_tx(&bk->fullX[s], halves * ph.planes * kPRows * 128);
      for (int hh = 0; hh < halves; ++hh)
        for (int pl = 0; pl < ph.planes; ++pl)
          ptx::tma_load_2d(x + hh * kXHalf + pl * kPRows * 128, &p.xmap[ph.xmap], &bk->fullX[s], kx + 64 * hh,
                           pl * ph.prow, pol);
    }
    trace_val(p, cta, pi, kTrWaitXEmpty, wx);
  }
done:
  drain_slots(bk->fullX, it, S, -1, p.status);
}

__device__ void mma_issuer(const PParams& p, PBook* bk, uint8_t* ring, uint32_t tmem, int G, int cta) {
  const int S = p.stages;
  int it = 0, seq = 0;
  bool any = false;
  for (int pi = 0; pi < p.nphase; ++pi) {
    const PPhase& ph = p.ph[pi];
    if (ph.kind != kPhGemm) continue;
    const Span sp = cta_span(ph, G, cta);
    long long ww = 0, wxx = 0;
    for (int i = sp.i0; i < sp.i1;) {
      const int t = i / ph.kb, k0 = i - t * ph.kb, k1 = min(sp.i1 - t * ph.kb, ph.kb);
      const bool wide = p.seg[seg_of(p, ph, t)].tw == kTwMax;   // weights on N
      const uint32_t idesc = wide ? ptx::idesc_bf16_f32(128, kTwMax) : ptx::idesc_bf16_f32(128, kPRows * ph.planes);
      const int buf = seq & 1, use = seq >> 1;
      if (use >= 1 && !ptx::mbar_wait(&bk->accfree[buf], (use - 1) & 1, kBudget, p.status)) goto done;
      ptx::tc_fence_after();
      const uint32_t d = tmem + buf * kTwMax;
      for (int kk = k0; kk < k1; ++kk, ++it) {
        const int s = it % S;
        if (!wait_timed(&bk->fullW[s], (it / S) & 1, p.status, ww) ||
            !wait_timed(&bk->fullX[s], (it / S) & 1, p.status, wxx))
          goto done;
        ptx::tc_fence_after();
        if (i == sp.i0 && kk == k0) trace_at(p, cta, pi, kTrM0);
        uint8_t* st = ring + (size_t)s * kStage;
        for (int hh = 0; hh < ph.kw / 64; ++hh) {   // 64 K columns at a time
          const uint64_t xd = ptx::smem_desc_sw128(st + hh * kXHalf);             // activations (token rows 0..31)
          const uint64_t wd = ptx::smem_desc_sw128(st + kXBytes + hh * kWBox);    // weights (tw rows)
          const uint64_t ad = wide ? xd : wd, bd = wide ? wd : xd;
#pragma unroll
          for (int k = 0; k < 4; ++k)   // 4 x K=16 per 64 columns; +32 B per step inside the swizzle row
            ptx::mma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kk > k0 || hh > 0 || k > 0) ? 1u : 0u);
        }
        ptx::mma_commit(&bk->empty[s]);
        any = true;
      }
      ptx::mma_commit(&bk->accf[buf]);
      ++seq;
      i = t * ph.kb + k1;
      if (i == sp.i1) trace_at(p, cta, pi, kTrM1);
    }
    trace_val(p, cta, pi, kTrWaitW, ww);
    trace_val(p, cta, pi, kTrWaitX, wxx);
  }
done:
  if (any) {   // every MMA issued has finished before the tensor memory is freed
    ptx::mma_commit(&bk->mma_done);
    ptx::mbar_wait(&bk->mma_done, 0, kBudget, p.status);
  }
}

// ---------------------------------------------------------------- epilogues
// The staged tile: st[n * kLd + m] for features n < tw of the tile, rows m < M.

// 128 features starting at feature f0 of the output (rows of x / u):
// out = acc (+ x): x keeps out, planes u keep out * gain, ssq[f0/128][m] = sum
// of out^2 over the 128 features.  Thread ct owns feature f0 + ct.
// Residual-stream values x[m][f0 + ct] of the rows (zero for the fusion, which
// has no residual input).
__device__ __forceinline__ void load_resid(const PParams& p, const PPhase& ph, int f0, int ct, float* v) {
  const bool resid = ph.epi == kEpResid;
#pragma unroll
  for (int m = 0; m < kPRows; ++m) v[m] = (m < ph.mrows && resid) ? __ldcg(p.x + (size_t)m * p.D + f0 + ct) : 0.f;
}

// `xr`: kPRows residual values of load_resid followed by the gain of feature
// f0 + ct, or nullptr to load them here.
__device__ void epi_norm_out(const PParams& p, const PPhase& ph, int f0, float* st, int ct, const float* xr) {
  const int f = f0 + ct;
  const float g = xr ? xr[kPRows] : __bfloat162float(ph.gain[f]);
  const bool resid = ph.epi == kEpResid;
  float v[kPRows];
  if (xr) {
#pragma unroll
    for (int m = 0; m < kPRows; ++m) v[m] = xr[m];
  } else {
    load_resid(p, ph, f0, ct, v);
  }
#pragma unroll
  for (int m = 0; m < kPRows; ++m) {
    if (m >= ph.mrows) break;
    const float o = v[m] + st[ct * kLd + m];
    if (resid) p.x[(size_t)m * p.D + f] = o;
    put_act(ph.u_out, p.u_plane, (size_t)m * p.D + f, o * g);
    st[ct * kLd + m] = o * o;
  }
  csync();
  // row m = ct / 8 sums features ct%8, ct%8 + 8, ... then across the 8 lanes
  const int m = ct >> 3, part = ct & 7;
  float a = 0.f;
  if (m < ph.mrows)
    for (int n = part; n < 128; n += 8) a += st[n * kLd + m];
  a += __shfl_xor_sync(0xffffffffu, a, 1);
  a += __shfl_xor_sync(0xffffffffu, a, 2);
  a += __shfl_xor_sync(0xffffffffu, a, 4);
  if (part == 0 && m < ph.mrows) ph.ssq_out[(f0 / 128) * kPRows + m] = a;
  csync();
}

// silu(gate) * up for a paired tile (features 0..127 gate, 128..255 up) into
// the W_D GEMM's activation planes.
__device__ void epi_swiglu(const PParams& p, const PPhase& ph, int tis, const float* st, int ct) {
  const EpiSwiGLU<__nv_bfloat16>& e = p.swiglu;
  for (int idx = ct; idx < ph.mrows * 128; idx += 128) {
    const int m = idx >> 7, c = idx & 127;
    const float g = st[c * kLd + m], u = st[(128 + c) * kLd + m];
    put_act(e.a, e.plane, (size_t)m * e.lda + (size_t)tis * 128 + c, g / (1.0f + __expf(-g)) * u);
  }
}

// Argmax of the tile's logits (features f0 .. f0+tw-1 below the vocabulary)
// for every mask row (block position >= 1) into slots[row]; optional logits.
__device__ void epi_lm(const PParams& p, const PPhase& ph, int f0, int tw, const float* st, int ct) {
  const int lane = ct & 31, w = ct >> 5;
  const int nv = min(tw, p.vocab - f0);
  for (int m = w; m < ph.mrows; m += 4) {
    if (m % p.block == 0) continue;
    unsigned long long best = 0ull;
    for (int n = lane; n < nv; n += 32) {
      const unsigned long long k = pack_argmax(st[n * kLd + m], f0 + n);
      best = k > best ? k : best;
    }
    for (int o = 16; o; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    if (lane == 0) atomicMax(p.slots + m, best);
  }
  if (p.logits) {
    for (int idx = ct; idx < ph.mrows * tw; idx += 128) {
      const int m = idx / tw, n = idx - m * tw;
      const int b = m / p.block, k = m - b * p.block;
      if (k == 0 || n >= nv) continue;
      p.logits[(size_t)(b * (p.block - 1) + k - 1) * p.vocab + (size_t)f0 + n] = st[n * kLd + m];
    }
  }
}

// Partial tiles [16 rows][tw features] in global memory (row pitch kTwMax).
// Thread ct moves feature quad 4(ct % (TW/4)) of rows ct / (TW/4) + k * 512/TW:
// all 128 threads take part at either width.
template <int TW>
struct PieceMap {
  static constexpr int kQ = TW / 4;              // feature quads of a row
  static constexpr int kStep = 128 / kQ;         // rows between a thread's rows
  static constexpr int kR = kPRows / kStep;      // rows of a thread
  static constexpr int kU = 24 / kR;             // pieces loaded at once (24 float4 in flight per thread)
};

template <int TW>
__device__ __forceinline__ void publish_tw(int rows, const float* st, float* dst, int ct) {
  using PM = PieceMap<TW>;
  const int fq = 4 * (ct % PM::kQ), r0 = ct / PM::kQ;
  for (int m = r0; m < rows; m += PM::kStep)
    *reinterpret_cast<float4*>(dst + m * kTwMax + fq) =
        make_float4(st[fq * kLd + m], st[(fq + 1) * kLd + m], st[(fq + 2) * kLd + m], st[(fq + 3) * kLd + m]);
}
__device__ __forceinline__ void publish_piece(int rows, int tw, const float* st, float* dst, int ct) {
  if (tw == kTwMax)
    publish_tw<kTwMax>(rows, st, dst, ct);
  else
    publish_tw<128>(rows, st, dst, ct);
}

// Add the pieces of tile t from CTAs cf+1..cl (in CTA order) to the reducer's
// own piece, staged in st: the sum runs in CTA order cf, cf+1, .., cl, so the
// result does not depend on timing.
template <int TW>
__device__ void add_pieces(const PParams& p, const PPhase& ph, int G, int t, int cf, int cl, float* st, int ct) {
  using PM = PieceMap<TW>;
  const int fq = 4 * (ct % PM::kQ), r0 = ct / PM::kQ;
  const int W = phase_iters(ph);
  const int g = phase_ctas(ph, G);
  const int rows = ph.mrows;
  float4 acc[PM::kR];
#pragma unroll
  for (int j = 0; j < PM::kR; ++j) {
    const int m = r0 + PM::kStep * j;
    acc[j] = m < rows ? make_float4(st[fq * kLd + m], st[(fq + 1) * kLd + m], st[(fq + 2) * kLd + m],
                                   st[(fq + 3) * kLd + m])
                     : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int c = cf + 1; c <= cl; c += PM::kU) {
    float4 a[PM::kU][PM::kR];
#pragma unroll
    for (int u = 0; u < PM::kU; ++u) {
      const int cu = min(c + u, cl);
      const float* src =
          p.partial + (size_t)(cu * 2 + ((cu * W / g) / ph.kb == t ? 0 : 1)) * (kPRows * kTwMax) + fq;
#pragma unroll
      for (int j = 0; j < PM::kR; ++j) {
        const int m = r0 + PM::kStep * j;
        a[u][j] = (c + u <= cl && m < rows) ? __ldcg(reinterpret_cast<const float4*>(src + m * kTwMax))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < PM::kU; ++u)
#pragma unroll
      for (int j = 0; j < PM::kR; ++j) {
        acc[j].x += a[u][j].x;
        acc[j].y += a[u][j].y;
        acc[j].z += a[u][j].z;
        acc[j].w += a[u][j].w;
      }
  }
#pragma unroll
  for (int j = 0; j < PM::kR; ++j) {
    const int m = r0 + PM::kStep * j;
    if (m < rows) {
      st[fq * kLd + m] = acc[j].x;
      st[(fq + 1) * kLd + m] = acc[j].y;
      st[(fq + 2) * kLd + m] = acc[j].z;
      st[(fq + 3) * kLd + m] = acc[j].w;
    }
  }
}

// Wait (bounded) until `n` pieces of a tile have been announced.
__device__ bool wait_pieces(const int* counter, int n, int32_t* status) {
  if ((int)ld_acquire(reinterpret_cast<const unsigned int*>(counter)) >= n) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if ((int)ld_acquire(reinterpret_cast<const unsigned int*>(counter)) >= n) return true;
    if ((it & 63) == 0) {
      if (*reinterpret_cast<volatile int32_t*>(status) == DFLASH_ERR_TIMEOUT) return false;
      if (clock64() - t0 > kBudget) {
        report_status(status, DFLASH_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Epilogue of output tile t (all 128 compute threads; the tile is staged).
// `xr`: this thread's residual values and gain for the tile's first 128
// features (see epi_norm_out), or nullptr.
__device__ void run_epilogue(const PParams& p, const PPhase& ph, int t, float* st, int ct, const float* xr = nullptr) {
  const GemmSeg& sg = p.seg[seg_of(p, ph, t)];
  const int tis = t - sg.tile_begin, halves = sg.tw / 128;
  switch (ph.epi) {
    case kEpFuse:
    case kEpResid:   // one segment starting at feature 0
      for (int h = 0; h < halves; ++h)
        epi_norm_out(p, ph, tis * sg.tw + h * 128, st + h * 128 * kLd, ct, h == 0 ? xr : nullptr);
      break;
    case kEpQKV:
      for (int h = 0; h < halves; ++h) p.qkv(st + h * 128 * kLd, kLd, 0, ph.mrows, 0, sg, tis * halves + h, ct, 128);
      break;
    case kEpInject:
      for (int h = 0; h < halves; ++h) p.inject(st + h * 128 * kLd, kLd, 0, ph.mrows, 0, sg, tis * halves + h, ct, 128);
      break;
    case kEpSwiGLU: epi_swiglu(p, ph, tis, st, ct); break;
    default: epi_lm(p, ph, tis * sg.tw, sg.tw, st, ct); break;
  }
}

// One projection phase, compute-warp side.  Returns false on a timeout.
__device__ bool gemm_phase(const PParams& p, const PPhase& ph, int pi, PBook* bk, float* st, uint32_t tmem, int G,
                           int cta, int ct, int& seq) {
  if (ph.scaled) {
    const int m = ct >> 3, part = ct & 7, nt = p.D / 128;
    float a = 0.f;
    if (m < ph.mrows)
      for (int t = part; t < nt; t += 8) a += __ldcg(ph.ssq_in + t * kPRows + m);
    for (int o = 1; o < 8; o <<= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (part == 0) bk->rs[m] = m < ph.mrows ? rsqrtf(a / (float)p.D + p.eps) : 0.f;
  }
  csync();
  const Span sp = cta_span(ph, G, cta);
  const int first_tile = sp.i0 / max(ph.kb, 1);
  for (int i = sp.i0; i < sp.i1;) {
    const int t = i / ph.kb, k0 = i - t * ph.kb, k1 = min(sp.i1 - t * ph.kb, ph.kb);
    i = t * ph.kb + k1;
    const int tw = p.seg[seg_of(p, ph, t)].tw;
    const int buf = seq & 1, use = seq >> 1;
    ++seq;
    const bool last = i == sp.i1;
    if (ct == 0) bk->flag_acc = ptx::mbar_wait(&bk->accf[buf], use & 1, kBudget, p.status);
    if (ct == 0 && last) trace_at(p, cta, pi, kTrAcc);
    csync();
    if (!bk->flag_acc) return false;
    const uint32_t tb = tmem + buf * kTwMax;
    if (tw == kTwMax) {
      // weights on N: token rows in TMEM lanes 0..15 (hi) and 16..31 (lo), warp 4
      if (ct < 32) {
        ptx::tc_fence_after();
        const float sc = (ct < ph.mrows && ph.scaled) ? bk->rs[ct] : 1.f;
        for (int c0 = 0; c0 < kTwMax; c0 += 64) {
          float v[64];
          ptx::tmem_ld32x2(tb + c0, tb + c0 + 32, v);
          if (ph.planes == 2) {
#pragma unroll
            for (int j = 0; j < 64; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], 16);
          }
          if (ct < ph.mrows) {
#pragma unroll
            for (int j = 0; j < 64; ++j) st[(c0 + j) * kLd + ct] = v[j] * sc;
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (ct == 0) ptx::mbar_arrive(&bk->accfree[buf]);
        if (ct == 0 && last) trace_at(p, cta, pi, kTrReadBack);
      }
    } else {
      // weights on M: feature ct in TMEM lane ct (warp q owns lanes 32q..),
      // token columns 0..15 (hi) and 16..31 (lo)
      ptx::tc_fence_after();
      float v[kPRows];
      const uint32_t ta = tb + (static_cast<uint32_t>((ct >> 5) * 32) << 16);
      ptx::tmem_ld16(ta, v);
      if (ph.planes == 2) {
        float w[kPRows];
        ptx::tmem_ld16(ta + kPRows, w);
#pragma unroll
        for (int m = 0; m < kPRows; ++m) v[m] += w[m];
      }
      ptx::tc_fence_before();
#pragma unroll
      for (int m = 0; m < kPRows; ++m) st[ct * kLd + m] = ph.scaled ? v[m] * bk->rs[m] : v[m];
    }
    csync();
    if (tw != kTwMax) {   // every compute thread has read its lane
      if (ct == 0) ptx::mbar_arrive(&bk->accfree[buf]);
    }
    if (ct == 0 && last) trace_at(p, cta, pi, kTrStaged);

    if (k0 == 0 && k1 == ph.kb) {   // the whole tile is here
      run_epilogue(p, ph, t, st, ct);
      csync();
      if (ct == 0 && last) trace_at(p, cta, pi, kTrPub);
      continue;
    }
    const int cf = cta_of(ph, G, t * ph.kb), cl = cta_of(ph, G, (t + 1) * ph.kb - 1);
    if (cta != cf) {
      // a piece for the tile's reducer: publish it and announce it (release);
      // nothing here waits for the reduction
      publish_piece(ph.mrows, tw, st, p.partial + (size_t)(cta * 2 + (t == first_tile ? 0 : 1)) * (kPRows * kTwMax),
                    ct);
      __threadfence();
      csync();
      if (ct == 0) {
        atomicAdd(p.tickets + t, 1);
        if (last) trace_at(p, cta, pi, kTrPub);
      }
      continue;
    }
    // The designated reducer of tile t: the CTA holding its first K blocks.
    // That piece ends this CTA's span (the tile continues into the next CTA),
    // so it is this CTA's last one and is reduced at once, from shared memory.
    // The residual input and the gain of a norm epilogue do not depend on the
    // pieces: their loads go out first, parked in the staging tile's upper half
    // (unused at 128 features; a row of kLd = kPRows + 1 floats holds both).
    const GemmSeg& sg = p.seg[seg_of(p, ph, t)];
    const bool norm = (ph.epi == kEpResid || ph.epi == kEpFuse) && sg.tw == 128;
    float* xr = norm ? st + 128 * kLd + ct * kLd : nullptr;
    if (xr) {
      const int f0 = (t - sg.tile_begin) * sg.tw;
      float v[kPRows];
      load_resid(p, ph, f0, ct, v);
      const float g = __bfloat162float(ph.gain[f0 + ct]);
#pragma unroll
      for (int m = 0; m < kPRows; ++m) xr[m] = v[m];
      xr[kPRows] = g;
    }
    if (ct == 0) {
      if (last) trace_at(p, cta, pi, kTrPub);
      bk->flag_tk = wait_pieces(p.tickets + t, cl - cf, p.status);
    }
    csync();
    if (!bk->flag_tk) return false;
    if (sg.tw == kTwMax)
      add_pieces<kTwMax>(p, ph, G, t, cf, cl, st, ct);
    else
      add_pieces<128>(p, ph, G, t, cf, cl, st, ct);
    csync();
    run_epilogue(p, ph, t, st, ct, xr);
    csync();
    if (ct == 0) {
      p.tickets[t] = 0;   // every piece has arrived: ready for the next phase
      trace_at(p, cta, pi, kTrRed);
    }
  }
  return true;
}

// Attention of item = this CTA: (request, kv head, chunk of key tiles) on the
// tensor cores (attn_tc.cuh), using the ring's shared memory and all 512 TMEM
// columns (idle between projections); partial (unnormalised output, max, sum)
// rows to global memory, maxima in log2 units.  Returns false on a timeout.
template <int HD>
__device__ bool attn_phase(const PParams& p, const PPhase& ph, int pi, PBook* bk, uint8_t* sm, uint32_t tmem, int cta,
                           int ct, int& uses) {
  const AttnParams& ap = p.attn;
  AttnItem item;
  if (!attn_item(ap, bk->ctx_len, cta, item)) return true;
  const int b = item.b, kvh = item.kvh, t0 = item.t0, t1 = item.t1, nct = item.nct;
  const int rows = (ap.nq / ap.nkv) * ap.block;
  float* op = ap.opart + (size_t)cta * kPAttnRows * HD;
  float2* ml = ap.ml + (size_t)cta * kPAttnRows;
  if (t0 >= t1) {   // no tiles: an empty partial (weight 0 in the merge)
    for (int i = ct; i < rows; i += 128) ml[i] = make_float2(attn_tc::kNegInf, 0.f);
    if (ct == 0) trace_at(p, cta, pi, kTrM1);
    return true;
  }
  AttnParams a = ap;
  a.layer = ph.layer;
  auto out = [&](int row, int d0, const float* v) {
    float* dst = op + (size_t)row * HD + d0;
#pragma unroll
    for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
  };
  auto done = [&](int row, float m_log2, float l) { ml[row] = make_float2(m_log2, l); };
  // trace slots kTrAcc..kTrRed of an attention phase: the core's stamps
  unsigned long long* stamps = p.trace ? p.trace + ((size_t)cta * kPMaxPhases + pi) * kTrSlots + kTrAcc : nullptr;
  const bool ok = attn_tc::run<HD, 128>(a, p.amaps, b, kvh, 0, t0, t1, nct, item.c, sm, tmem, &bk->abars, uses, ct,
                                        ComputeSync{}, p.status, out, done, nullptr, stamps);
  if (ct == 0) trace_at(p, cta, pi, kTrM1);
  return ok;
}

// Merge of the key chunks of one output row (request b, q head qh, block row
// k) into the W_O GEMM's activation planes, by one warp.  Lane ch holds chunk
// ch's (max, sum) and weight; lane l owns output elements [HD/32 * l, +HD/32).
template <int HD>
__device__ void merge_row(const PParams& p, int b, int qh, int k, int lane) {
  constexpr int E = HD / 32;   // elements per lane: 4 (float4) or 2 (float2)
  const AttnParams& ap = p.attn;
  const int nch = ap.splits, Gq = ap.nq / ap.nkv;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(ap.out);
  const int kvh = qh / Gq, r = (qh - kvh * Gq) * ap.block + k;
  const size_t item0 = ((size_t)b * ap.nkv + kvh) * nch;
  float L = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  // 32 chunks at a time: their (max, sum) once, the running maximum (a batch
  // beyond the first rescales what was accumulated), then their partial rows,
  // 16 chunks' vector loads in flight at once.  The first 16 partial rows are
  // loaded together with the (max, sum) pairs, before their weights are known;
  // a chunk of weight 0 (no keys) is then dropped by a select, so whatever its
  // unwritten row holds never enters the sum.
  float M = attn_tc::kNegInf;
  auto load16 = [&](float (&v)[16][E], int c0, int u0, int n) {
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float* src = ap.opart + ((item0 + c0 + u0 + u) * kPAttnRows + r) * HD + E * lane;
      if constexpr (E == 4) {
        const float4 x = u0 + u < n ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
      } else {
        const float2 x = u0 + u < n ? __ldcg(reinterpret_cast<const float2*>(src)) : make_float2(0.f, 0.f);
        v[u][0] = x.x; v[u][1] = x.y;
      }
    }
  };
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const int ch = c0 + lane, n = min(32, nch - c0);
    const float2 ml = ch < nch ? __ldcg(ap.ml + (item0 + ch) * kPAttnRows + r) : make_float2(attn_tc::kNegInf, 0.f);
    float v[16][E];
    load16(v, c0, 0, n);
    float mb = ml.y > 0.f ? ml.x : attn_tc::kNegInf;
    for (int o = 16; o; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    const float Mn = fmaxf(M, mb);
    if (c0 > 0 && Mn > M) {
      const float sc = exp2f(M - Mn);
      L *= sc;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= sc;
    }
    M = Mn;
    const float wgt = ml.y > 0.f ? exp2f(ml.x - M) : 0.f;
    L += wgt * ml.y;
    for (int u0 = 0; u0 < n; u0 += 16) {
      if (u0 > 0) load16(v, c0, u0, n);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float wu = __shfl_sync(0xffffffffu, wgt, (u0 + u) & 31);
        const bool have = u0 + u < n && wu != 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += have ? wu * v[u][e] : 0.f;
      }
    }
  }
  for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = 1.f / L;
  const size_t obase = ((size_t)b * ap.block + k) * ap.nq * HD + (size_t)qh * HD + E * lane;
#pragma unroll
  for (int e = 0; e < E; ++e) put_act(out, ap.out_plane, obase + e, acc[e] * inv);
}

// After this CTA's attention chunk: announce it on its (request, kv head)
// group's counter (release), wait (bounded) for the group's other chunks,
// then merge this chunk's share of the group's output rows (rows
// [ch R / nch, (ch + 1) R / nch) of R = q heads per kv head x block), one warp
// per row.  No grid barrier and no phase of its own: the W_O phase follows.
// Returns false on a timeout.
template <int HD>
__device__ bool attn_merge(const PParams& p, const PPhase& ph, PBook* bk, int cta, int ct) {
  const AttnParams& ap = p.attn;
  AttnItem item;
  if (!attn_item(ap, bk->ctx_len, cta, item)) return true;
  const int nch = ap.splits, Gq = ap.nq / ap.nkv, R = Gq * ap.block;
  const int ch = cta % nch;
  int* cnt = p.gcnt + (size_t)ph.layer * ap.B * ap.nkv + item.b * ap.nkv + item.kvh;
  __threadfence();   // this chunk's partial rows are visible before the count says so
  csync();
  if (ct == 0) {
    atomicAdd(cnt, 1);
    bk->flag_tk = wait_pieces(cnt, nch, p.status);
  }
  csync();
  if (!bk->flag_tk) return false;
  const int r1 = (ch + 1) * R / nch;
  for (int r = ch * R / nch + (ct >> 5); r < r1; r += 4) {
    const int gh = r / ap.block, k = r - gh * ap.block;
    merge_row<HD>(p, item.b, item.kvh * Gq + gh, k, ct & 31);
  }
  return true;
}

__device__ void compute_warps(const PParams& p, PBook* bk, uint8_t* ring, uint8_t* region, uint32_t tmem, int G,
                              int cta) {
  const int ct = threadIdx.x - 128;
  float* st = reinterpret_cast<float*>(region);
  int seq = 0, attn_uses = 0;
  // the requests' context lengths, read once (nothing in the launch changes them)
  if (p.attn.ctx_len)
    for (int i = ct; i < p.attn.B && i < kPRows; i += 128) bk->ctx_len[i] = p.attn.ctx_len[i];
  csync();
  for (int pi = 0; pi < p.nphase; ++pi) {
    const PPhase& ph = p.ph[pi];
    if (ct == 0) trace_at(p, cta, pi, kTrStart);
    // the next phase's attention: its tensor maps into the descriptor cache now
    if (ct == 0 && pi + 1 < p.nphase && p.ph[pi + 1].kind == kPhAttn) attn_tc::prefetch_maps(p.amaps);
    if (ph.kind == kPhGemm) {
      if (!gemm_phase(p, ph, pi, bk, st, tmem, G, cta, ct, seq)) return;
    } else {
      // attention; the weight producers hold off until it releases the ring,
      // which happens before its chunks are merged
      const bool ok = p.attn.hd == 64 ? attn_phase<64>(p, ph, pi, bk, ring, tmem, cta, ct, attn_uses)
                                      : attn_phase<128>(p, ph, pi, bk, ring, tmem, cta, ct, attn_uses);
      csync();
      if (ct == 0) ptx::mbar_arrive(&bk->ring_free);
      if (!ok) return;
      if (!(p.attn.hd == 64 ? attn_merge<64>(p, ph, bk, cta, ct) : attn_merge<128>(p, ph, bk, cta, ct))) return;
    }
    // ---- grid barrier: this CTA's writes of the phase are published
    ptx::fence_proxy_async_global();
    __threadfence();
    csync();
    if (ct == 0) trace_at(p, cta, pi, kTrDone);
    if (pi + 1 < p.nphase) {
      if (ct == 0) {
        atomicAdd(p.bar, 1u);
        bk->flag_bar = grid_wait(p.bar, (unsigned)(pi + 1) * (unsigned)G, p.status);
      }
      csync();
      if (!bk->flag_bar) return;
    } else {
      // the last CTA to finish reads the argmax slots out
      if (ct == 0) bk->flag_bar = atomicAdd(p.bar, 1u) == (unsigned)p.nphase * (unsigned)G - 1u;
      csync();
      if (bk->flag_bar && p.drafts) {
        __threadfence();
        for (int m = ct; m < p.M; m += 128) {
          const int b = m / p.block, k = m - b * p.block;
          if (k > 0) p.drafts[b * (p.block - 1) + k - 1] = unpack_argmax_index(__ldcg(p.slots + m));
        }
      }
    }
  }
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1) persist_kernel(const __grid_constant__ PParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  uint8_t* ring = smem;
  uint8_t* region = smem + (size_t)S * kStage;
  PBook* bk = reinterpret_cast<PBook*>(region + PCfg<HD>::kRegion);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&bk->fullW[s], 1);
      ptx::mbar_init(&bk->fullX[s], 1);
      ptx::mbar_init(&bk->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&bk->accf[b], 1);
      ptx::mbar_init(&bk->accfree[b], 1);
    }
    ptx::mbar_init(&bk->mma_done, 1);
    ptx::mbar_init(&bk->ring_free, 1);
    attn_tc::init_bars(&bk->abars);
    ptx::fence_mbar_init();
    for (int i = 0; i < kPXMaps; ++i) ptx::prefetch_tmap(&p.xmap[i]);
  }
  if (warp == 1) ptx::tmem_alloc(&bk->tmem, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bk->tmem;
  griddep_trigger();
  if (threadIdx.x == 0) trace_val(p, cta, 0, kTrSm, ptx::smid());

  if (warp == 0 || warp == 3) {
    // weights are constant: streaming starts before the previous kernel has finished
    if (lane == 0) weight_producer(p, bk, ring, G, cta, warp == 0 ? 0 : 1);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) mma_issuer(p, bk, ring, tmem, G, cta);
    __syncwarp();
  } else if (warp == 2) {
    griddep_wait();
    if (lane == 0) activation_producer(p, bk, ring, G, cta);
    __syncwarp();
  } else if (warp >= 4) {
    griddep_wait();
    compute_warps(p, bk, ring, region, tmem, G, cta);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- draft prologue
__global__ void __launch_bounds__(256) persist_draft_prep_kernel(
    const __nv_bfloat16* embed, const int32_t* anchor, int mask_id, int vocab, int block, int D,
    const __nv_bfloat16* g, float* x, __nv_bfloat16* u, size_t u_plane, float* ssq, unsigned long long* slots,
    int* zero, int nzero, int32_t* status, const int32_t* ctx_len, const double* inv_freq, int hd, float2* rope) {
  griddep_wait();
  griddep_trigger();
  const int row = blockIdx.x, b = row / block, k = row - b * block;
  if (row == 0)
    for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
  if (threadIdx.x == 0) slots[row] = 0ull;
  const int pos = ctx_len[b] + k;
  for (int i = threadIdx.x; i < (hd >> 1); i += blockDim.x) {
    float sn, cs;
    rope_sincos(pos, inv_freq, i, &sn, &cs);
    rope[(size_t)row * (hd >> 1) + i] = make_float2(cs, sn);
  }
  int tok = k == 0 ? anchor[b] : mask_id;
  if (tok < 0 || tok >= vocab) {   // an anchor outside the vocabulary: flag it, read row 0
    if (threadIdx.x == 0) report_status(status, DFLASH_ERR_INVALID_ARG);
    tok = 0;
  }
  const __nv_bfloat16* e = embed + (size_t)tok * D;
  // warp w covers features [128w + 1024j, +128): one tile of the sums of squares
  for (int f = threadIdx.x * 4; f < D; f += blockDim.x * 4) {
    const float4 v = load4(e + f), gg = load4(g + f);
    *reinterpret_cast<float4*>(x + (size_t)row * D + f) = v;
    put_act4(u, u_plane, (size_t)row * D + f, make_float4(v.x * gg.x, v.y * gg.y, v.z * gg.z, v.w * gg.w));
    float sq = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if ((threadIdx.x & 31) == 0) ssq[(f / kTileN) * kPRows + row] = sq;
  }
}

template <int HD>
cudaError_t launch_hd(const PParams& p, int grid, cudaStream_t s) {
  const size_t smem = persist_smem(p.stages, HD);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // programmatic launch on top of the cooperative one where the runtime takes
  // both; once refused, never asked again (any host thread may launch)
  static std::atomic<int> pdl_ok{1};
  cfg.numAttrs = (pdl_enabled() && pdl_ok.load(std::memory_order_relaxed)) ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, persist_kernel<HD>, p);
  if (e != cudaSuccess && cfg.numAttrs == 2) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone) {
      (void)cudaGetLastError();
      pdl_ok.store(0, std::memory_order_relaxed);
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, persist_kernel<HD>, p);
    }
  }
  return e;
}

}  // namespace

int persist_stages(int hd) {
  const size_t fixed = 1024 + region_bytes(hd) + sizeof(PBook);
  return std::min<int>(kPMaxStages, (int)((kSmemMax - fixed) / kStage));
}

size_t persist_smem(int stages, int hd) { return 1024 + (size_t)stages * kStage + region_bytes(hd) + sizeof(PBook); }

cudaError_t persist_prepare(int hd) {
  const int S = persist_stages(hd);
  if (hd == 64)
    return cudaFuncSetAttribute(persist_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)persist_smem(S, 64));
  return cudaFuncSetAttribute(persist_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)persist_smem(S, 128));
}

cudaError_t persist_launch(const PParams& p, int grid, int hd, cudaStream_t s) {
  // attention borrows the ring and the staging region for its key tiles
  const size_t attn_bytes = hd == 64 ? attn_tc::Cfg<64>::kBytes : attn_tc::Cfg<128>::kBytes;
  if (attn_bytes > (size_t)p.stages * kStage + region_bytes(hd)) return cudaErrorInvalidValue;
  if (p.stages < 2 || p.stages > kPMaxStages || p.M < 1 || p.M > kPRows || p.nphase < 1 || p.nphase > kPMaxPhases)
    return cudaErrorInvalidValue;
  for (int i = 0; i < p.nphase; ++i)   // the stream-K index arithmetic is 32-bit
    if ((long long)p.ph[i].tiles * p.ph[i].kb * grid >= (1LL << 31)) return cudaErrorInvalidValue;
  return hd == 64 ? launch_hd<64>(p, grid, s) : launch_hd<128>(p, grid, s);
}

cudaError_t persist_draft_prep_launch(const __nv_bfloat16* embed, const int32_t* anchor, int mask_id, int vocab,
                                      int B, int block, int D, const __nv_bfloat16* g, float* x, __nv_bfloat16* u,
                                      size_t u_plane, float* ssq, unsigned long long* slots, int* zero, int nzero,
                                      int32_t* status, const int32_t* ctx_len, const double* inv_freq, int hd,
                                      float2* rope, cudaStream_t s) {
  return launch_pdl(persist_draft_prep_kernel, dim3(B * block), dim3(256), 0, s, embed, anchor, mask_id, vocab, block,
                    D, g, x, u, u_plane, ssq, slots, zero, nzero, status, ctx_len, inv_freq, hd, rope);
}

}  // namespace dflash
