// Stochastic lossless verification and inverse-CDF sampling over the
// vocabulary (explainer page "DFlash: Block Diffusion for Flash Speculative
// Decoding", section "The Target Verifier Remains the Correctness Anchor":
// a draft x drawn from p_d is kept with probability min(1, p_t(x) / p_d(x)),
// verification stops at the first rejection, the target then draws a
// correction from the residual distribution, and a bonus token when the whole
// block survives; paper §5.1 reports the temperature-1 results).
//
// Every distribution is softmax(logits / T) of an fp32 logits row (V up to a
// few hundred thousand).  The work is HBM-bound: the logits are read once to
// get each row's (max, sum of exponentials), then only the one or two rows a
// request draws from are read again.  Four launches:
//
//   row_stats   grid (chunks, rows): per 8192-logit chunk of a row, the max m
//               of z = l * log2(e) / T and s = sum exp2(z - m) (online form);
//   accept      one CTA per request: the (max, sum) of its rows from their
//               chunks (all warps, loads first), then one warp: lane k takes
//               draft position k's two rows and reads its token's two logits
//               (all positions at once), takes the acceptance test, and a ballot
//               finds the first rejection; the distribution to draw from is
//               the residual there, or the target's row after the block;
//               writes tau and the accepted tokens;
//   draw_sums   grid (chunks, draws): per chunk, the unnormalised mass of
//               the chosen distribution (max(0, p_t - p_d), or p_t);
//   draw_pick   one CTA per draw: the chunk where the running mass first
//               exceeds u * total, then the token inside it (block scan).
//
// Inverse CDF: the drawn token is the smallest id whose cumulative mass
// (ids in increasing order) exceeds u times the total; when rounding leaves
// u * total at or beyond the total, the last id with non-zero mass is taken.
// Sampling a drafter row (dflash_sample_tokens) is the same draw with p_d
// alone.
#include <cstdint>

#include "common.cuh"
#include "sampling.cuh"

namespace dflash {
namespace {

constexpr int kChunk = 8192;       // logits per chunk (32 KB of fp32)
constexpr int kMaxChunks = (1 << 24) / kChunk;   // the vocabulary is at most 2^24 ids
constexpr int kThreads = 256;      // kChunk / kThreads = 32 logits a thread
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float2 merge_ms(float2 a, float2 b) {
  // (max, sum exp2(z - max)) of the union of two sets
  if (a.y == 0.f) return b;
  if (b.y == 0.f) return a;
  const float m = fmaxf(a.x, b.x);
  return make_float2(m, a.y * exp2f(a.x - m) + b.y * exp2f(b.x - m));
}

__device__ __forceinline__ float2 warp_merge(float2 v) {
  for (int o = 16; o; o >>= 1) {
    float2 w = make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o));
    v = merge_ms(v, w);
  }
  return v;
}

// Row r < nd is drafter row r, otherwise target row r - nd.
__device__ __forceinline__ const float* row_ptr(const float* draft, const float* target, int nd, int r, int V) {
  return r < nd ? draft + (size_t)r * V : target + (size_t)(r - nd) * V;
}

// At most 40 registers a thread, so that 6 CTAs share an SM: 192 KB of loads
// in flight per SM instead of 160 KB at 5 (112 -> 106 us for 603 MB).
__global__ void __launch_bounds__(kThreads, 6) row_stats_kernel(const float* draft, const float* target, int nd, int V,
                                                             float zscale, float2* part, int nchunk) {
  griddep_wait();
  griddep_trigger();
  const int c = blockIdx.x, r = blockIdx.y;
  const float* x = row_ptr(draft, target, nd, r, V);
  const int v0 = c * kChunk, v1 = min(V, v0 + kChunk);
  // 8 float4 per thread, all loads issued before the arithmetic
  float4 a[kChunk / kThreads / 4];
#pragma unroll
  for (int j = 0; j < kChunk / kThreads / 4; ++j) {
    const int v = v0 + 4 * (threadIdx.x + j * kThreads);
    a[j] = v < v1 ? __ldcs(reinterpret_cast<const float4*>(x + v)) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < kChunk / kThreads / 4; ++j) m = fmaxf(m, fmaxf(fmaxf(a[j].x, a[j].y), fmaxf(a[j].z, a[j].w)));
  m *= zscale;
  float s = 0.f;
  if (m > -INFINITY) {
#pragma unroll
    for (int j = 0; j < kChunk / kThreads / 4; ++j) {
      const int v = v0 + 4 * (threadIdx.x + j * kThreads);
      if (v < v1)
        s += exp2f(a[j].x * zscale - m) + exp2f(a[j].y * zscale - m) + exp2f(a[j].z * zscale - m) +
             exp2f(a[j].w * zscale - m);
    }
  }
  float2 t = warp_merge(make_float2(m, s));
  __shared__ float2 ws[kThreads / 32];
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = t;
  __syncthreads();
  if (threadIdx.x < 32) {
    t = threadIdx.x < kThreads / 32 ? ws[threadIdx.x] : make_float2(-INFINITY, 0.f);
    t = warp_merge(t);
    if (threadIdx.x == 0) part[(size_t)r * nchunk + c] = t;
  }
}

// (max, sum) of row r from its chunk partials, by one warp.
__device__ __forceinline__ float2 row_total(const float2* part, int r, int nchunk) {
  float2 t = make_float2(-INFINITY, 0.f);
  for (int c = threadIdx.x & 31; c < nchunk; c += 32) t = merge_ms(t, part[(size_t)r * nchunk + c]);
  return warp_merge(t);
}

// p(x) of one logit given its row's (max, sum).
__device__ __forceinline__ float prob(float logit, float zscale, float2 ms) { return exp2f(logit * zscale - ms.x) / ms.y; }

// One CTA per request.  First the (max, sum) of its 2g-1 rows from their
// chunk partials, by all warps (every warp issues the loads of its rows, one
// row a round, before merging any; lane c takes chunk c, then a warp merge):
// tot[k] draft position k (k < g-1), tot[32 + k] the target's row k (k < g).
// Then warp 0 walks the block.  g <= 32.
__global__ void __launch_bounds__(kThreads) accept_kernel(const float* draft, const float* target,
                                                          const int32_t* tokens, const float* u_accept,
                                                          const float2* part, int nchunk, int B, int g, int V,
                                                          float zscale, DrawSel* sel, int32_t* accept_len,
                                                          int32_t* out_tokens) {
  griddep_wait();
  griddep_trigger();
  const int b = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nd = B * (g - 1), nrow = 2 * g - 1;
  __shared__ float2 tot[64];
  {
    constexpr int kW = kThreads / 32, kRounds = (63 + kW - 1) / kW;
    float2 first[kRounds];
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
      const int j = warp + kW * u;   // draft rows first, then the target's
      const int r = j < g - 1 ? b * (g - 1) + j : nd + b * g + (j - (g - 1));
      first[u] = j < nrow && lane < nchunk ? part[(size_t)r * nchunk + lane] : make_float2(-INFINITY, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
      const int j = warp + kW * u;
      if (j >= nrow) break;
      const int r = j < g - 1 ? b * (g - 1) + j : nd + b * g + (j - (g - 1));
      float2 t = first[u];
      for (int c = lane + 32; c < nchunk; c += 32) t = merge_ms(t, part[(size_t)r * nchunk + c]);
      t = warp_merge(t);
      if (lane == 0) tot[j < g - 1 ? j : 32 + (j - (g - 1))] = t;
    }
  }
  __syncthreads();
  if (warp > 0) return;
  // every input of the walk first, in parallel: lane k < g-1 takes draft
  // position k (its two rows' (max, sum) and the two logits of its token),
  // lane g-1 the target row after the block
  float2 md = make_float2(0.f, 1.f), mt = make_float2(0.f, 1.f);
  float ld = 0.f, lt = 0.f, ua = 0.f;
  int d = -1;
  if (lane < g) {
    mt = tot[32 + lane];
    if (lane < g - 1) {
      const int rd = b * (g - 1) + lane;
      md = tot[lane];
      d = tokens[rd];
      ua = u_accept[rd];
      if (d >= 0 && d < V) {
        ld = draft[(size_t)rd * V + d];
        lt = target[(size_t)(b * g + lane) * V + d];
      }
    }
  }
  // lane k keeps its draft iff u < min(1, p_t / p_d); the first lane that does
  // not is the first rejection (an id outside the vocabulary is rejected)
  bool keep = false;
  if (lane < g - 1 && d >= 0 && d < V) {
    const float pd = prob(ld, zscale, md), pt = prob(lt, zscale, mt);
    const float a = pd <= 0.f ? 1.f : fminf(1.f, pt / pd);
    keep = ua < a;
  }
  const unsigned rejected = __ballot_sync(0xffffffffu, lane < g - 1 && !keep);
  const int kstar = rejected ? __ffs(rejected) - 1 : g - 1;   // g - 1: none rejected, the bonus
  const float2 mst = make_float2(__shfl_sync(0xffffffffu, mt.x, kstar), __shfl_sync(0xffffffffu, mt.y, kstar));
  const float2 msd = make_float2(__shfl_sync(0xffffffffu, md.x, kstar), __shfl_sync(0xffffffffu, md.y, kstar));
  if (lane == 0) {
    DrawSel s;
    s.pt = target + (size_t)(b * g + kstar) * V;
    s.pd = kstar < g - 1 ? draft + (size_t)(b * (g - 1) + kstar) * V : nullptr;
    s.mst = mst;
    s.msd = kstar < g - 1 ? msd : make_float2(0.f, 1.f);
    s.out = out_tokens + (size_t)b * g + kstar;
    sel[b] = s;
    accept_len[b] = kstar + 1;
  }
  for (int k = lane; k < g; k += 32)
    if (k != kstar) out_tokens[(size_t)b * g + k] = k < kstar ? tokens[b * (g - 1) + k] : -1;
}

// Sampling rows on their own: draw i comes from softmax(row i).
__global__ void __launch_bounds__(32) sample_sel_kernel(const float* logits, const float2* part, int nchunk, int V,
                                                        DrawSel* sel, int32_t* tokens) {
  griddep_wait();
  griddep_trigger();
  const int r = blockIdx.x;
  const float2 ms = row_total(part, r, nchunk);
  if (threadIdx.x == 0) {
    DrawSel s;
    s.pt = logits + (size_t)r * V;
    s.pd = nullptr;
    s.mst = ms;
    s.msd = make_float2(0.f, 1.f);
    s.out = tokens + r;
    sel[r] = s;
  }
}

// Unnormalised mass of draw i's distribution at the four logit indices of a
// float4 (lt: the target's or sampled row's logits there, ld: the drafter's).
__device__ __forceinline__ float mass1(const DrawSel& s, float lt, float ld, float zscale) {
  const float pt = prob(lt, zscale, s.mst);
  return s.pd ? fmaxf(0.f, pt - prob(ld, zscale, s.msd)) : pt;
}
__device__ __forceinline__ float4 mass4(const DrawSel& s, float4 lt, float4 ld, float zscale) {
  return make_float4(mass1(s, lt.x, ld.x, zscale), mass1(s, lt.y, ld.y, zscale), mass1(s, lt.z, ld.z, zscale),
                     mass1(s, lt.w, ld.w, zscale));
}
// The logits of draw i's rows at v (a multiple of 4; vocab % 4 == 0 and the
// rows are 16-byte aligned, so a float4 never crosses the row's end).
__device__ __forceinline__ void load4(const DrawSel& s, int v, float4& lt, float4& ld) {
  lt = __ldg(reinterpret_cast<const float4*>(s.pt + v));
  ld = s.pd ? __ldg(reinterpret_cast<const float4*>(s.pd + v)) : make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(kThreads) draw_sums_kernel(const DrawSel* sel, int V, float zscale, float* csum,
                                                             int nchunk) {
  griddep_wait();
  griddep_trigger();
  const int c = blockIdx.x, i = blockIdx.y;
  const DrawSel s = sel[i];
  const int v0 = c * kChunk, v1 = min(V, v0 + kChunk);
  // 8 float4 of each row per thread, all loads issued before the arithmetic
  constexpr int kV4 = kChunk / kThreads / 4;
  float4 lt[kV4], ld[kV4];
#pragma unroll
  for (int j = 0; j < kV4; ++j) {
    const int v = v0 + 4 * (threadIdx.x + j * kThreads);
    if (v < v1) load4(s, v, lt[j], ld[j]);
  }
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < kV4; ++j) {
    const int v = v0 + 4 * (threadIdx.x + j * kThreads);
    if (v < v1) {
      const float4 m = mass4(s, lt[j], ld[j], zscale);
      acc += (m.x + m.y) + (m.z + m.w);
    }
  }
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ float ws[kThreads / 32];
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) t += ws[w];
    csum[(size_t)i * nchunk + c] = t;
  }
}

__global__ void __launch_bounds__(kThreads) draw_pick_kernel(const DrawSel* sel, int V, float zscale,
                                                             const float* csum, int nchunk, const float* u,
                                                             int32_t* next_anchor) {
  griddep_wait();
  griddep_trigger();
  const int i = blockIdx.x;
  const DrawSel s = sel[i];
  __shared__ int s_chunk;
  __shared__ float s_rem;
  __shared__ float s_tsum[kThreads / 32];
  __shared__ int s_tok;
  __shared__ float s_cs[kMaxChunks];
  for (int c = threadIdx.x; c < nchunk; c += kThreads) s_cs[c] = csum[(size_t)i * nchunk + c];   // all loads at once
  __syncthreads();
  if (threadIdx.x == 0) {
    // running mass over the chunks in id order (double: the chunk sums are few)
    double total = 0.0;
    for (int c = 0; c < nchunk; ++c) total += s_cs[c];
    const double target = (double)__ldg(u + i) * total;
    double run = 0.0;
    int pick = -1, last_nz = 0;
    double before = 0.0;
    for (int c = 0; c < nchunk; ++c) {
      const double m = s_cs[c];
      if (m > 0.0) last_nz = c;
      if (pick < 0 && run + m > target && m > 0.0) {
        pick = c;
        before = run;
      }
      run += m;
    }
    if (pick < 0) {   // u * total at or past the total: the last chunk with mass
      pick = last_nz;
      s_rem = INFINITY;
    } else {
      s_rem = (float)(target - before);
    }
    s_chunk = pick;
    s_tok = INT32_MAX;
  }
  __syncthreads();
  const int v0 = s_chunk * kChunk, v1 = min(V, v0 + kChunk);
  constexpr int kPer = kChunk / kThreads;
  // thread t owns ids [v0 + kPer t, v0 + kPer (t+1)): its mass, then a block scan
  float mv[kPer];
  float own = 0.f;
  {
    float4 lt[kPer / 4], ld[kPer / 4];   // all loads first (float4: kPer and the chunk end are multiples of 4)
#pragma unroll
    for (int j = 0; j < kPer / 4; ++j) {
      const int v = v0 + kPer * threadIdx.x + 4 * j;
      if (v < v1) load4(s, v, lt[j], ld[j]);
    }
#pragma unroll
    for (int j = 0; j < kPer / 4; ++j) {
      const int v = v0 + kPer * threadIdx.x + 4 * j;
      const float4 m = v < v1 ? mass4(s, lt[j], ld[j], zscale) : make_float4(0.f, 0.f, 0.f, 0.f);
      mv[4 * j] = m.x;
      mv[4 * j + 1] = m.y;
      mv[4 * j + 2] = m.z;
      mv[4 * j + 3] = m.w;
      own += (m.x + m.y) + (m.z + m.w);
    }
  }
  // exclusive scan of the 256 partial sums in id order: within each warp by
  // shuffles, then across the 8 warp totals
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  float inc = own;
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) s_tsum[wid] = inc;
  __syncthreads();
  float wbase = 0.f;
  for (int w = 0; w < wid; ++w) wbase += s_tsum[w];
  const float rem = s_rem;
  const float before = wbase + inc - own;
  if (rem != INFINITY && before <= rem && rem < before + own) {
    // this thread's ids hold the remainder: the first whose running mass
    // exceeds it (or, if rounding says none does, the last with mass)
    float run = before;
    int tok = -1, last = -1;
    for (int j = 0; j < kPer; ++j) {
      if (mv[j] > 0.f) last = v0 + kPer * threadIdx.x + j;
      run += mv[j];
      if (mv[j] > 0.f && run > rem) {
        tok = v0 + kPer * threadIdx.x + j;
        break;
      }
    }
    if (tok < 0) tok = last;
    if (tok >= 0) atomicMin(&s_tok, tok);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int tok = s_tok;
    if (tok == INT32_MAX) {
      // the remainder lies beyond the chunk's mass (rounding, or u * total at
      // or past the total): the chunk's last id with mass
      tok = v0;
      for (int v = v1 - 1; v >= v0; --v)
        if (mass1(s, __ldg(s.pt + v), s.pd ? __ldg(s.pd + v) : 0.f, zscale) > 0.f) {
          tok = v;
          break;
        }
    }
    *s.out = tok;
    if (next_anchor) next_anchor[i] = tok;
  }
}

}  // namespace

int sampling_chunks(int vocab) { return (vocab + kChunk - 1) / kChunk; }

size_t sampling_workspace_bytes(int rows, int draws, int vocab) {
  const size_t nc = (size_t)sampling_chunks(vocab);
  auto a = [](size_t v) { return (v + 255) & ~(size_t)255; };
  return a(sizeof(float2) * (size_t)rows * nc) + a(sizeof(DrawSel) * (size_t)draws) + a(sizeof(float) * (size_t)draws * nc);
}

namespace {
struct SamplingWs {
  float2* part;
  DrawSel* sel;
  float* csum;
};
SamplingWs carve(void* ws, int rows, int draws, int vocab) {
  const size_t nc = (size_t)sampling_chunks(vocab);
  auto a = [](size_t v) { return (v + 255) & ~(size_t)255; };
  char* p = static_cast<char*>(ws);
  SamplingWs w;
  w.part = reinterpret_cast<float2*>(p);
  p += a(sizeof(float2) * (size_t)rows * nc);
  w.sel = reinterpret_cast<DrawSel*>(p);
  p += a(sizeof(DrawSel) * (size_t)draws);
  w.csum = reinterpret_cast<float*>(p);
  return w;
}
}  // namespace

cudaError_t verify_sampled_launch(const float* draft_logits, const float* target_logits, const int32_t* drafts,
                                  const float* u_accept, const float* u_sample, int B, int g, int V,
                                  float temperature, int32_t* accept_len, int32_t* out_tokens,
                                  int32_t* next_anchor, void* ws, int* launches, cudaStream_t s) {
  const int nchunk = sampling_chunks(V);
  const int nd = B * (g - 1), rows = nd + B * g;
  const float zscale = kLog2e / temperature;
  SamplingWs w = carve(ws, rows, B, V);
  *launches = 0;
  cudaError_t e = launch_pdl(row_stats_kernel, dim3(nchunk, rows), dim3(kThreads), 0, s, draft_logits, target_logits,
                             nd, V, zscale, w.part, nchunk);
  if (e != cudaSuccess) return e;
  ++*launches;
  e = launch_pdl(accept_kernel, dim3(B), dim3(kThreads), 0, s, draft_logits, target_logits, drafts, u_accept,
                 static_cast<const float2*>(w.part), nchunk, B, g, V, zscale, w.sel, accept_len, out_tokens);
  if (e != cudaSuccess) return e;
  ++*launches;
  e = launch_pdl(draw_sums_kernel, dim3(nchunk, B), dim3(kThreads), 0, s, static_cast<const DrawSel*>(w.sel), V, zscale,
                 w.csum, nchunk);
  if (e != cudaSuccess) return e;
  ++*launches;
  e = launch_pdl(draw_pick_kernel, dim3(B), dim3(kThreads), 0, s, static_cast<const DrawSel*>(w.sel), V, zscale,
                 static_cast<const float*>(w.csum), nchunk, u_sample, next_anchor);
  if (e != cudaSuccess) return e;
  ++*launches;
  return cudaSuccess;
}

cudaError_t sample_tokens_launch(const float* logits, int rows, int V, float temperature, const float* u,
                                 int32_t* tokens, void* ws, int* launches, cudaStream_t s) {
  const int nchunk = sampling_chunks(V);
  const float zscale = kLog2e / temperature;
  SamplingWs w = carve(ws, rows, rows, V);
  *launches = 0;
  cudaError_t e = launch_pdl(row_stats_kernel, dim3(nchunk, rows), dim3(kThreads), 0, s, logits,
                             static_cast<const float*>(nullptr), rows, V, zscale, w.part, nchunk);
  if (e != cudaSuccess) return e;
  ++*launches;
  e = launch_pdl(sample_sel_kernel, dim3(rows), dim3(32), 0, s, logits, static_cast<const float2*>(w.part), nchunk, V,
                 w.sel, tokens);
  if (e != cudaSuccess) return e;
  ++*launches;
  e = launch_pdl(draw_sums_kernel, dim3(nchunk, rows), dim3(kThreads), 0, s, static_cast<const DrawSel*>(w.sel), V,
                 zscale, w.csum, nchunk);
  if (e != cudaSuccess) return e;
  ++*launches;
  e = launch_pdl(draw_pick_kernel, dim3(rows), dim3(kThreads), 0, s, static_cast<const DrawSel*>(w.sel), V, zscale,
                 static_cast<const float*>(w.csum), nchunk, u, static_cast<int32_t*>(nullptr));
  if (e != cudaSuccess) return e;
  ++*launches;
  return cudaSuccess;
}

}  // namespace dflash
