// C ABI of the DFlash draft-cycle library: argument checks, memory plans and
// the launch sequence of each stage.  Every step of the cycle runs in the
// kernels of this library; this file only validates and orders launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "gemm.cuh"
#include "kernels.cuh"
#include "attn_tc.cuh"
#include "persist.cuh"
#include "sampling.cuh"
#include "packed_attention.cuh"

using namespace dflash;

namespace {
// CUDA event pairs around each launch while profiling is on.
struct Profiler {
  bool on = false;
  int used = 0;                    // events used so far (2 per launch)
  std::vector<cudaEvent_t> ev;
  std::vector<int> stage;          // stage of each recorded launch
};
std::atomic<uint64_t> g_launch_count{0};
}  // namespace

struct dflash_model {
  dflash_config cfg;
  const void* embed;
  const void* lm_head;
  const void* w_c;
  const void* g_c;
  const void* g_final;
  std::vector<dflash_layer_weights> layers;
  int device;
  int sms;
  int32_t* status_dev;     // device status word (first device-detected error)
  double* inv_freq_dev;    // RoPE frequencies theta^(-2i/hd), i < hd/2
  void* tmaps_dev;         // tensor maps of every weight matrix (bf16 models), 64-row boxes
  void* tmaps128_dev;      // the same maps with 128-row boxes (persistent kernel)
  int use_tc;              // bf16 projections on the tcgen05 kernel
  int persist;             // calls of at most 16 token rows run as one persistent launch
  int persist_stages;      // its shared-memory ring depth
  unsigned long long* trace_dev;  // GEMM timestamps (DFLASH_TRACE_GEMM=<launch index>)
  long trace_target;
  int trace_persist;       // DFLASH_TRACE_PERSIST: the persistent drafter records phase timestamps
  long gemm_launches;
  Profiler prof;
};

// Index of a weight matrix's tensor map: 0 lm_head, 1 w_c, then 7 per layer.
enum { kMapLm = 0, kMapWc = 1, kMapLayer0 = 2 };
enum { kMapQ = 0, kMapK, kMapV, kMapO, kMapG, kMapU, kMapD, kMapsPerLayer };
inline int layer_map(int l, int which) { return kMapLayer0 + kMapsPerLayer * l + which; }

struct dflash_cache {
  const dflash_model* model;
  char* base;
  size_t bytes;
  int batch;
  int cap;
  size_t k_off, v_off, len_off;
  std::vector<int32_t> len_host;  // host mirror of ctx_len, exact while len_known
  bool len_known;
};

namespace {

thread_local std::string g_last_error;

int32_t fail(int32_t code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

}  // namespace

namespace dflash {
int32_t set_error(int32_t code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace dflash

namespace {

int32_t cuda_fail(cudaError_t e, const char* what) {
  return fail(DFLASH_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define DF_CUDA(call, what)                              \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return cuda_fail(e_, what);   \
  } while (0)

// Launch `call` (which makes `kernels` kernel launches) for profiler stage
// `stage`, with an event pair around it while profiling is on.
#define DF_LAUNCH(stg, kernels, call, what)                                         \
  do {                                                                                \
    Profiler& pr_ = const_cast<dflash_model*>(m)->prof;                               \
    const bool rec_ = pr_.on && pr_.used + 2 <= (int)pr_.ev.size();                   \
    if (rec_) DF_CUDA(cudaEventRecord(pr_.ev[pr_.used], s), "profiler event");        \
    DF_CUDA((call), what);                                                            \
    g_launch_count += (kernels);                                                      \
    if (rec_) {                                                                       \
      DF_CUDA(cudaEventRecord(pr_.ev[pr_.used + 1], s), "profiler event");            \
      pr_.stage.push_back(stg);                                                       \
      pr_.used += 2;                                                                  \
    }                                                                                 \
  } while (0)

constexpr size_t kTraceEntries = 8u << 16;   // 8 timestamps for up to 65536 CTAs

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
// row pitch of hd-major V (bf16 models): positions rounded up to 8 (16-byte rows for TMA)
int pad8(int n) { return (n + 7) & ~7; }
// bf16 planes of every cached context K/V value: hi and lo, or one rounded value
int kv_planes(const dflash_config& c) { return c.kv_bf16 ? 1 : 2; }
// operand planes the LM head reads: 1 with head_bf16 (the hi plane of the pair
// the final norm writes is the value rounded to nearest bf16)
int head_planes(const dflash_config& c) { return c.dtype == DFLASH_DTYPE_F32 ? 1 : (c.head_bf16 ? 1 : 2); }
// planes of the cache of a T model (an fp32 cache is one fp32 plane)
template <typename T> int cache_planes(const dflash_config& c) { return ActPlanes<T>::n == 2 ? kv_planes(c) : 1; }

int32_t check_config(const dflash_config* c) {
  if (!c) return fail(DFLASH_ERR_INVALID_ARG, "config is NULL");
  if (c->dtype != DFLASH_DTYPE_F32 && c->dtype != DFLASH_DTYPE_BF16)
    return fail(DFLASH_ERR_INVALID_ARG, "dtype %d is not DFLASH_DTYPE_F32 or DFLASH_DTYPE_BF16", c->dtype);
  if (c->hidden <= 0 || c->hidden % kTileN || c->hidden > 8192)
    return fail(DFLASH_ERR_SHAPE, "hidden %d must be a positive multiple of 128, at most 8192", c->hidden);
  if (c->layers <= 0 || c->layers > kMaxSeg / 2) return fail(DFLASH_ERR_SHAPE, "layers %d must be in [1, %d]", c->layers, kMaxSeg / 2);
  if (c->head_dim != 64 && c->head_dim != 128) return fail(DFLASH_ERR_SHAPE, "head_dim %d must be 64 or 128", c->head_dim);
  if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->n_q_heads % c->n_kv_heads)
    return fail(DFLASH_ERR_SHAPE, "n_q_heads %d must be a positive multiple of n_kv_heads %d", c->n_q_heads, c->n_kv_heads);
  if ((c->n_q_heads * c->head_dim) % kTileN || (c->n_kv_heads * c->head_dim) % kTileN)
    return fail(DFLASH_ERR_SHAPE, "n_q_heads*head_dim and n_kv_heads*head_dim must be multiples of 128");
  if (c->ffn <= 0 || c->ffn % kHalfN) return fail(DFLASH_ERR_SHAPE, "ffn %d must be a positive multiple of 64", c->ffn);
  if (c->vocab <= 0 || c->vocab % kTileN) return fail(DFLASH_ERR_SHAPE, "vocab %d must be a positive multiple of 128", c->vocab);
  if (c->n_target_feats < 1 || c->n_target_feats > 8) return fail(DFLASH_ERR_SHAPE, "n_target_feats %d must be in [1, 8]", c->n_target_feats);
  if (c->max_block < 1 || c->max_block > kMaxBlock) return fail(DFLASH_ERR_SHAPE, "max_block %d must be in [1, %d]", c->max_block, kMaxBlock);
  if ((c->n_q_heads / c->n_kv_heads) * c->max_block > attention_max_rows())
    return fail(DFLASH_ERR_SHAPE, "(n_q_heads/n_kv_heads)*max_block must be <= %d", attention_max_rows());
  if (c->mask_token_id < 0 || c->mask_token_id >= c->vocab) return fail(DFLASH_ERR_INVALID_ARG, "mask_token_id %d out of [0, vocab)", c->mask_token_id);
  if (!(c->rope_theta > 1.0f) || !(c->rms_eps >= 0.0f)) return fail(DFLASH_ERR_INVALID_ARG, "rope_theta must be > 1 and rms_eps >= 0");
  if (c->qk_norm != 0 && c->qk_norm != 1) return fail(DFLASH_ERR_INVALID_ARG, "qk_norm %d must be 0 or 1", c->qk_norm);
  if (c->input_fusion != 0 && c->input_fusion != 1)
    return fail(DFLASH_ERR_INVALID_ARG, "input_fusion %d must be 0 or 1", c->input_fusion);
  if (c->input_fusion && c->qk_norm) return fail(DFLASH_ERR_UNSUPPORTED, "input_fusion with qk_norm is not built");
  if (c->kv_bf16 != 0 && c->kv_bf16 != 1) return fail(DFLASH_ERR_INVALID_ARG, "kv_bf16 %d must be 0 or 1", c->kv_bf16);
  if (c->kv_bf16 && c->dtype != DFLASH_DTYPE_BF16) return fail(DFLASH_ERR_INVALID_ARG, "kv_bf16 needs a bf16 model");
  if (c->kv_bf16 && c->qk_norm) return fail(DFLASH_ERR_UNSUPPORTED, "kv_bf16 with qk_norm is not built");
  if (c->head_bf16 != 0 && c->head_bf16 != 1)
    return fail(DFLASH_ERR_INVALID_ARG, "head_bf16 %d must be 0 or 1", c->head_bf16);
  if (c->head_bf16 && c->dtype != DFLASH_DTYPE_BF16) return fail(DFLASH_ERR_INVALID_ARG, "head_bf16 needs a bf16 model");
  return DFLASH_OK;
}

int32_t check_device(const dflash_model* m) {
  int dev = -1;
  DF_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev != m->device) return fail(DFLASH_ERR_INVALID_ARG, "current device %d is not the model's device %d", dev, m->device);
  return DFLASH_OK;
}

// ---------------------------------------------------------------- workspace plan
struct WsPlan {
  size_t total;
  size_t rowinfo, yf, ht, rope_c;                              // injection
  size_t x, u, q, kb, vb, opart, ml, o, a, hm, slots, rope_q;  // drafter
  size_t partial, counters;                                    // split-K scratch
  int counters_n;
  int attn_splits, attn_chunk;
  GemmPlan g_fuse, g_inject, g_qkv, g_o, g_gu, g_down, g_lm;
  // input-fusion injection: context rows through the layers
  GemmPlan gf_q, gf_kv, gf_o, gf_gu, gf_down;
  size_t xc, uc, qc, oc, ac;
  // persistent path: sums of squares, attention chunk partials, tickets + barrier
  int persist;
  int fused;   // one persistent launch runs the injection and the drafter pass
  size_t ssq, ssq2, aml, tickets;
  int ntickets, nch;
  int ngcnt;   // persistent drafter: per (layer, request, kv head) attention chunk counters after the barrier
};

// The persistent path serves bf16 calls of at most 16 token rows whose
// attention groups fit 64 query rows.
bool persist_draft_ok(const dflash_model* m, int B, int block) {
  const dflash_config& c = m->cfg;
  return m->persist && !c.qk_norm && !c.head_bf16 && B * block <= kPRows && (c.n_q_heads / c.n_kv_heads) * block <= kPAttnRows &&
         5 * c.layers + 1 <= kPMaxPhases && c.ffn % kTileN == 0;
}
// A whole cycle in one launch: fusion and injection phases before the drafter's
// (5 phases a layer + 3; segments: 6 a layer, 2 a layer for the injection, the
// fusion and the LM head).
bool persist_cycle_ok(const dflash_model* m) {
  return 5 * m->cfg.layers + 3 <= kPMaxPhases && 8 * m->cfg.layers + 2 <= kPMaxSeg;
}
bool persist_inject_ok(const dflash_model* m, int max_rows) {
  return m->persist && !m->cfg.qk_norm && !m->cfg.input_fusion && max_rows <= kPRows && 1 + 2 * m->cfg.layers <= kPMaxSeg;
}

// One call's scratch: the injection part when max_rows > 0, the drafter part
// when block > 0.  Each call lays out only its own regions from offset 0, so a
// single workspace of max(inject, draft) bytes serves both on one stream.
WsPlan plan_ws(const dflash_model* m, int B, int cap, int block, int max_rows) {
  const dflash_config& c = m->cfg;
  const size_t es = c.dtype == DFLASH_DTYPE_F32 ? 4 : 2;
  const int pl = c.dtype == DFLASH_DTYPE_F32 ? 1 : 2;   // activation planes
  const size_t ea = es * pl;                             // bytes per activation element
  const int D = c.hidden, hq = c.n_q_heads * c.head_dim, hk = c.n_kv_heads * c.head_dim, F = c.ffn;
  const int R = B * block, Rm = B * std::max(block - 1, 0);
  WsPlan p{};
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off += align256(std::max<size_t>(bytes, 1)); return o; };
  const bool inj_p = max_rows > 0 && persist_inject_ok(m, max_rows);
  const bool drf_p = block > 0 && persist_draft_ok(m, B, block);
  if ((max_rows > 0 && block > 0) ? (inj_p && drf_p && persist_cycle_ok(m)) : (inj_p || drf_p)) {
    // one persistent launch: activation planes padded to 16 rows, stream-K scratch per CTA;
    // with both an injection and a block, one launch runs the whole cycle
    const int half = c.head_dim / 2;
    p.persist = 1;
    p.fused = max_rows > 0 && block > 0;
    if (max_rows > 0) {
      p.ntickets = std::max(D / kTileN, c.layers * 2 * (hk / kTileN));
      p.rowinfo = take(sizeof(int2) * (size_t)max_rows);
      p.ht = take(2 * 2 * (size_t)kPRows * D);
      p.rope_c = take(sizeof(float2) * (size_t)kPRows * half);
      if (p.fused) p.ssq2 = take(sizeof(float) * (size_t)(D / kTileN) * kPRows);
    }
    if (block > 0) {
      p.ntickets = std::max({p.ntickets, (hq + 2 * hk) / kTileN, D / kTileN, F / kTileN, (c.vocab + 255) / 256});
      const int groups = B * c.n_kv_heads;
      p.nch = std::max(1, std::min(m->sms / groups, (cap + block + 31) / 32));
      p.x = take(sizeof(float) * (size_t)kPRows * D);
      p.u = take(2 * 2 * (size_t)kPRows * D);
      p.q = take(sizeof(float) * (size_t)R * hq);
      p.kb = take(2 * 2 * (size_t)R * hk);
      p.vb = take(2 * 2 * (size_t)B * hk * pad8(block));   // hd-major, rows padded to 8
      p.o = take(2 * 2 * (size_t)kPRows * hq);
      p.a = take(2 * 2 * (size_t)kPRows * F);
      p.slots = take(sizeof(unsigned long long) * kPRows);
      p.rope_q = take(sizeof(float2) * (size_t)kPRows * half);
      p.opart = take(sizeof(float) * (size_t)groups * p.nch * kPAttnRows * c.head_dim);
      p.aml = take(sizeof(float2) * (size_t)groups * p.nch * kPAttnRows);
    }
    p.ssq = take(sizeof(float) * (size_t)(D / kTileN) * kPRows);
    p.partial = take(sizeof(float) * (size_t)m->sms * 2 * kPRows * 256);
    p.ngcnt = block > 0 ? c.layers * B * c.n_kv_heads : 0;
    // tickets, then the barrier counter, then the attention chunk counters
    p.tickets = take(sizeof(int) * (size_t)(p.ntickets + 1 + p.ngcnt));
    p.total = off;
    return p;
  }
  std::vector<const GemmPlan*> used;
  if (max_rows > 0) {
    p.g_fuse = plan_gemm(c.dtype, max_rows, c.n_target_feats * D, D / kTileN, m->sms, m->use_tc, 1);
    p.g_inject = plan_gemm(c.dtype, max_rows, D, c.layers * 2 * (hk / kTileN), m->sms, m->use_tc, pl);
    used = {&p.g_fuse, &p.g_inject};
    if (c.input_fusion) {
      p.gf_q = plan_gemm(c.dtype, max_rows, D, hq / kTileN, m->sms, m->use_tc, pl);
      p.gf_kv = plan_gemm(c.dtype, max_rows, D, 2 * (hk / kTileN), m->sms, m->use_tc, pl);
      p.gf_o = plan_gemm(c.dtype, max_rows, hq, D / kTileN, m->sms, m->use_tc, pl);
      p.gf_gu = plan_gemm(c.dtype, max_rows, D, F / kHalfN, m->sms, m->use_tc, pl);
      p.gf_down = plan_gemm(c.dtype, max_rows, F, D / kTileN, m->sms, m->use_tc, pl);
      used.insert(used.end(), {&p.gf_q, &p.gf_kv, &p.gf_o, &p.gf_gu, &p.gf_down});
    }
  }
  if (block > 0) {
    p.g_qkv = plan_gemm(c.dtype, R, D, (hq + 2 * hk) / kTileN, m->sms, m->use_tc, pl);
    p.g_o = plan_gemm(c.dtype, R, hq, D / kTileN, m->sms, m->use_tc, pl);
    p.g_gu = plan_gemm(c.dtype, R, D, F / kHalfN, m->sms, m->use_tc, pl);
    p.g_down = plan_gemm(c.dtype, R, F, D / kTileN, m->sms, m->use_tc, pl);
    p.g_lm = plan_gemm(c.dtype, std::max(Rm, 1), D, c.vocab / kTileN, m->sms, m->use_tc, head_planes(c));
    used.insert(used.end(), {&p.g_qkv, &p.g_o, &p.g_gu, &p.g_down, &p.g_lm});
  }
  size_t partial = 0;
  int counters = 0;
  for (const GemmPlan* g : used) {
    partial = std::max(partial, g->partial_floats);
    counters = std::max(counters, g->counters);
  }
  if (max_rows > 0) {
    p.rowinfo = take(sizeof(int2) * (size_t)max_rows);
    p.yf = take(sizeof(float) * (size_t)max_rows * D);
    p.ht = take(ea * (size_t)max_rows * D);
    p.rope_c = take(sizeof(float2) * (size_t)max_rows * (c.head_dim / 2));
    if (c.input_fusion) {   // the context rows' residual stream and operands
      p.xc = take(sizeof(float) * (size_t)max_rows * D);
      p.uc = take(ea * (size_t)max_rows * D);
      p.qc = take(sizeof(float) * (size_t)max_rows * hq);
      p.oc = take(ea * (size_t)max_rows * hq);
      p.ac = take(ea * (size_t)max_rows * F);
    }
  }
  if (block > 0) {
    // attention splits: enough CTAs to cover the device twice over
    const int keys = cap + block;
    const int groups = std::max(1, B * c.n_kv_heads);
    const int want = std::max(1, (2 * m->sms + groups - 1) / groups);
    int chunk = (keys + want - 1) / want;
    chunk = std::max(64, (chunk + 31) / 32 * 32);
    p.attn_chunk = chunk;
    p.attn_splits = (keys + chunk - 1) / chunk;
    if (c.dtype == DFLASH_DTYPE_BF16) {
      // tensor-core attention: 128-key tiles (context tiles + the block tile)
      // cut into splits so that there are ~4 CTAs per SM over all groups
      const int tiles = (cap + 127) / 128 + 1;
      p.attn_splits = std::max(1, std::min(tiles, (4 * m->sms + groups - 1) / groups));
    }
    p.x = take(sizeof(float) * (size_t)R * D);
    p.u = take(ea * (size_t)R * D);
    p.q = take(sizeof(float) * (size_t)R * hq);
    p.kb = take(sizeof(float) * (size_t)R * hk);
    p.vb = take(sizeof(float) * (size_t)B * hk * pad8(block));   // bf16: hd-major, rows padded to 8
    // split partials of the split-KV attention, merged by a second kernel
    const size_t nsplit = (size_t)p.attn_splits;
    p.opart = take(sizeof(float) * (size_t)B * c.n_q_heads * block * nsplit * c.head_dim);
    p.ml = take(sizeof(float2) * (size_t)B * c.n_q_heads * block * nsplit);
    p.o = take(ea * (size_t)R * hq);
    p.a = take(ea * (size_t)R * F);
    p.hm = take(ea * (size_t)std::max(Rm, 1) * D);
    p.slots = take(sizeof(unsigned long long) * (size_t)std::max(Rm, 1));
    p.rope_q = take(sizeof(float2) * (size_t)R * (c.head_dim / 2));
  }
  p.partial = take(sizeof(float) * partial);
  p.counters = take(sizeof(int) * (size_t)counters);
  p.counters_n = counters;
  p.total = off;
  return p;
}

// X is `planes` planes of [M][ldx], plane_stride elements apart.
GemmProblem make_problem(const dflash_model* m, const void* x, int ldx, int M, int K, int planes = 1,
                         size_t plane_stride = 0) {
  GemmProblem p{};
  p.x = x;
  p.ldx = ldx;
  p.planes = planes;
  p.plane_stride = plane_stride;
  p.M = M;
  p.K = K;
  p.wmaps = m->tmaps_dev;
  p.status = m->status_dev;
  if (m->trace_dev) {   // timestamps of one chosen GEMM launch
    dflash_model* mm = const_cast<dflash_model*>(m);
    p.trace = mm->gemm_launches++ == mm->trace_target ? mm->trace_dev : nullptr;
  }
  return p;
}

void add_seg(GemmProblem& p, const void* w0, int map0, const void* w1, int map1, int tiles, int paired, int tag) {
  GemmSeg& s = p.seg[p.nseg++];
  s.w0 = w0;
  s.w1 = w1;
  s.map0 = map0;
  s.map1 = map1;
  s.tiles = tiles;
  s.tile_begin = p.total_tiles;
  s.paired = paired;
  s.tag = tag;
  p.total_tiles += tiles;
}

// Input-fusion ablation: the injected rows' hidden states start at H_t (x_c,
// fp32) and go through the draft layers like sequence positions; layer l's
// K/V projection of its context rows is appended to the cache (RoPE on K at
// each row's position), then the rows attend causally to the cache (keys up
// to their own position) and take the layer's W_O, norm and SwiGLU FFN.  The
// last layer needs only its K/V: its outputs feed nothing.
template <typename T>
int32_t run_context_layers(const dflash_model* m, dflash_cache* cache, int max_rows, char* ws, const WsPlan& P,
                           cudaStream_t s) {
  const dflash_config& c = m->cfg;
  const int D = c.hidden, F = c.ffn, hq = c.n_q_heads * c.head_dim, hk = c.n_kv_heads * c.head_dim;
  const int pl = ActPlanes<T>::n;
  const size_t R = (size_t)max_rows;
  int2* rowinfo = reinterpret_cast<int2*>(ws + P.rowinfo);
  const float2* rope_c = reinterpret_cast<const float2*>(ws + P.rope_c);
  float* xc = reinterpret_cast<float*>(ws + P.xc);
  T* uc = reinterpret_cast<T*>(ws + P.uc);
  float* qc = reinterpret_cast<float*>(ws + P.qc);
  T* oc = reinterpret_cast<T*>(ws + P.oc);
  T* ac = reinterpret_cast<T*>(ws + P.ac);
  float* partial = reinterpret_cast<float*>(ws + P.partial);
  int* counters = reinterpret_cast<int*>(ws + P.counters);
  T* kc = reinterpret_cast<T*>(cache->base + cache->k_off);
  T* vc = reinterpret_cast<T*>(cache->base + cache->v_off);
  for (int l = 0; l < c.layers; ++l) {
    const dflash_layer_weights& L = m->layers[l];
    DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
              rmsnorm_launch<T>(xc, static_cast<const T*>(L.g_in), c.rms_eps, max_rows, D, uc, R * D, s),
              "context input norm");
    GemmProblem pkv = make_problem(m, uc, D, max_rows, D, pl, R * D);
    add_seg(pkv, L.w_k, layer_map(l, kMapK), L.w_k, layer_map(l, kMapK), hk / kTileN, 0, 2 * l);
    add_seg(pkv, L.w_v, layer_map(l, kMapV), L.w_v, layer_map(l, kMapV), hk / kTileN, 0, 2 * l + 1);
    apply_plan(pkv, P.gf_kv, partial, counters);
    EpiInject<T> ei{kc, vc, rowinfo, rope_c, c.layers, c.n_kv_heads, c.head_dim, cache->cap, pad8(cache->cap),
                    cache_planes<T>(c)};
    DF_LAUNCH(DFLASH_STAGE_INJECT, 1, (gemm_launch<T, EpiInject<T>>(pkv, P.gf_kv, ei, s)), "context K/V GEMM");
    if (l + 1 == c.layers) break;
    GemmProblem pq = make_problem(m, uc, D, max_rows, D, pl, R * D);
    add_seg(pq, L.w_q, layer_map(l, kMapQ), L.w_q, layer_map(l, kMapQ), hq / kTileN, 0, 0);
    apply_plan(pq, P.gf_q, partial, counters);
    DF_LAUNCH(DFLASH_STAGE_INJECT, 1,
              (gemm_launch<T, EpiRowsRope>(pq, P.gf_q, EpiRowsRope{qc, hq, rope_c, c.head_dim}, s)),
              "context Q GEMM");
    DF_LAUNCH(DFLASH_STAGE_ATTN, 1,
              ctx_attention_launch<T>(qc, kc, vc, rowinfo, max_rows, l, c.layers, c.n_q_heads, c.n_kv_heads,
                                      c.head_dim, cache->cap, pad8(cache->cap), cache_planes<T>(c),
                                      1.0f / sqrtf((float)c.head_dim), oc, R * hq, s),
              "context attention");
    GemmProblem po = make_problem(m, oc, hq, max_rows, hq, pl, R * hq);
    add_seg(po, L.w_o, layer_map(l, kMapO), L.w_o, layer_map(l, kMapO), D / kTileN, 0, 0);
    apply_plan(po, P.gf_o, partial, counters);
    DF_LAUNCH(DFLASH_STAGE_INJECT, 1, (gemm_launch<T, EpiResidual>(po, P.gf_o, EpiResidual{xc, D}, s)), "context O GEMM");
    DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
              rmsnorm_launch<T>(xc, static_cast<const T*>(L.g_post), c.rms_eps, max_rows, D, uc, R * D, s),
              "context post-attention norm");
    GemmProblem pg = make_problem(m, uc, D, max_rows, D, pl, R * D);
    add_seg(pg, L.w_g, layer_map(l, kMapG), L.w_u, layer_map(l, kMapU), F / kHalfN, 1, 0);
    apply_plan(pg, P.gf_gu, partial, counters);
    DF_LAUNCH(DFLASH_STAGE_INJECT, 1,
              (gemm_launch<T, EpiSwiGLU<T>>(pg, P.gf_gu, EpiSwiGLU<T>{ac, F, R * F}, s)), "context gate/up GEMM");
    GemmProblem pd = make_problem(m, ac, F, max_rows, F, pl, R * F);
    add_seg(pd, L.w_d, layer_map(l, kMapD), L.w_d, layer_map(l, kMapD), D / kTileN, 0, 0);
    apply_plan(pd, P.gf_down, partial, counters);
    DF_LAUNCH(DFLASH_STAGE_INJECT, 1, (gemm_launch<T, EpiResidual>(pd, P.gf_down, EpiResidual{xc, D}, s)),
              "context down GEMM");
  }
  return DFLASH_OK;
}

template <typename T>
int32_t run_inject(const dflash_model* m, dflash_cache* cache, const void* feats, const int32_t* n_new, int max_rows,
                   char* ws, const WsPlan& P, cudaStream_t s) {
  const dflash_config& c = m->cfg;
  const int D = c.hidden, hk = c.n_kv_heads * c.head_dim;
  const int pl = ActPlanes<T>::n;
  int2* rowinfo = reinterpret_cast<int2*>(ws + P.rowinfo);
  float* yf = reinterpret_cast<float*>(ws + P.yf);
  T* ht = reinterpret_cast<T*>(ws + P.ht);
  float* partial = reinterpret_cast<float*>(ws + P.partial);
  int* counters = reinterpret_cast<int*>(ws + P.counters);
  int32_t* ctx_len = reinterpret_cast<int32_t*>(cache->base + cache->len_off);

  DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
            inject_prep_launch(n_new, ctx_len, cache->batch, max_rows, cache->cap, rowinfo, counters, P.counters_n,
                               m->status_dev, s), "inject_prep");
  GemmProblem pf = make_problem(m, feats, c.n_target_feats * D, max_rows, c.n_target_feats * D);
  add_seg(pf, m->w_c, kMapWc, m->w_c, kMapWc, D / kTileN, 0, 0);
  apply_plan(pf, P.g_fuse, partial, counters);
  DF_LAUNCH(DFLASH_STAGE_FUSE, 1, (gemm_launch<T, EpiStoreF32>(pf, P.g_fuse, EpiStoreF32{yf, D}, s)), "fusion GEMM");
  DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
            fuse_norm_launch<T>(yf, static_cast<const T*>(m->g_c), c.rms_eps, rowinfo, max_rows, D, ht,
                                (size_t)max_rows * D, m->inv_freq_dev, c.head_dim,
                                reinterpret_cast<float2*>(ws + P.rope_c), s,
                                c.input_fusion ? reinterpret_cast<float*>(ws + P.xc) : nullptr),
            "fusion norm");
  if (c.input_fusion) return run_context_layers<T>(m, cache, max_rows, ws, P, s);

  GemmProblem pi = make_problem(m, ht, D, max_rows, D, pl, (size_t)max_rows * D);
  for (int l = 0; l < c.layers; ++l) {
    add_seg(pi, m->layers[l].w_k, layer_map(l, kMapK), m->layers[l].w_k, layer_map(l, kMapK), hk / kTileN, 0, 2 * l);
    add_seg(pi, m->layers[l].w_v, layer_map(l, kMapV), m->layers[l].w_v, layer_map(l, kMapV), hk / kTileN, 0, 2 * l + 1);
  }
  apply_plan(pi, P.g_inject, partial, counters);
  const float2* rope_c = reinterpret_cast<const float2*>(ws + P.rope_c);
  T* kc = reinterpret_cast<T*>(cache->base + cache->k_off);
  EpiInject<T> ei{kc, reinterpret_cast<T*>(cache->base + cache->v_off), rowinfo, c.qk_norm ? nullptr : rope_c,
                  c.layers, c.n_kv_heads, c.head_dim, cache->cap, pad8(cache->cap), cache_planes<T>(c)};
  DF_LAUNCH(DFLASH_STAGE_INJECT, 1, (gemm_launch<T, EpiInject<T>>(pi, P.g_inject, ei, s)), "injection GEMM");
  if (c.qk_norm)   // per-head key norm, then RoPE, of the injected keys
    for (int l = 0; l < c.layers; ++l)
      DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
                qknorm_cache_launch<T>(kc, rowinfo, max_rows, l, c.layers, c.n_kv_heads, c.head_dim, cache->cap,
                                       cache_planes<T>(c), static_cast<const T*>(m->layers[l].g_k), c.rms_eps,
                                       rope_c, s),
                "injected key norm");
  return DFLASH_OK;
}

template <typename T>
int32_t run_draft(const dflash_model* m, const dflash_cache* cache, const int32_t* anchor, int block, int32_t* drafts,
                  float* logits, char* ws, const WsPlan& P, cudaStream_t s) {
  const dflash_config& c = m->cfg;
  const int B = cache->batch, D = c.hidden, F = c.ffn;
  const int hq = c.n_q_heads * c.head_dim, hk = c.n_kv_heads * c.head_dim;
  const int R = B * block, Rm = B * (block - 1);
  const int pl = ActPlanes<T>::n;
  float* x = reinterpret_cast<float*>(ws + P.x);
  T* u = reinterpret_cast<T*>(ws + P.u);
  float* q = reinterpret_cast<float*>(ws + P.q);
  T* kb = reinterpret_cast<T*>(ws + P.kb);
  T* vb = reinterpret_cast<T*>(ws + P.vb);
  T* o = reinterpret_cast<T*>(ws + P.o);
  T* a = reinterpret_cast<T*>(ws + P.a);
  T* hm = reinterpret_cast<T*>(ws + P.hm);
  unsigned long long* slots = reinterpret_cast<unsigned long long*>(ws + P.slots);
  float* partial = reinterpret_cast<float*>(ws + P.partial);
  int* counters = reinterpret_cast<int*>(ws + P.counters);
  const int32_t* ctx_len = reinterpret_cast<const int32_t*>(cache->base + cache->len_off);

  DF_LAUNCH(DFLASH_STAGE_OTHER, 1, embed_norm_launch<T>(static_cast<const T*>(m->embed), anchor, c.mask_token_id, c.vocab, B, block, D,
                               static_cast<const T*>(m->layers[0].g_in), c.rms_eps, x, u, (size_t)R * D, counters,
                               P.counters_n, m->status_dev, ctx_len, m->inv_freq_dev, c.head_dim,
                               reinterpret_cast<float2*>(ws + P.rope_q), s),
          "embedding");
  attn_tc::Maps amaps;   // bf16 models: tensor maps of the K/V cache and of the block K/V
  if constexpr (ActPlanes<T>::n == 2) {
    if (!encode_attention_maps(&amaps, cache->base + cache->k_off, cache->base + cache->v_off, kb, vb, B, c.layers,
                               c.n_kv_heads, c.head_dim, cache->cap, pad8(cache->cap), kv_planes(c), block,
                               pad8(block)))
      return fail(DFLASH_ERR_CUDA, "could not encode attention tensor maps");
  }
  for (int l = 0; l < c.layers; ++l) {
    const dflash_layer_weights& L = m->layers[l];
    GemmProblem pq = make_problem(m, u, D, R, D, pl, (size_t)R * D);
    add_seg(pq, L.w_q, layer_map(l, kMapQ), L.w_q, layer_map(l, kMapQ), hq / kTileN, 0, 0);
    add_seg(pq, L.w_k, layer_map(l, kMapK), L.w_k, layer_map(l, kMapK), hk / kTileN, 0, 1);
    add_seg(pq, L.w_v, layer_map(l, kMapV), L.w_v, layer_map(l, kMapV), hk / kTileN, 0, 2);
    apply_plan(pq, P.g_qkv, partial, counters);
    const float2* rope_q = reinterpret_cast<const float2*>(ws + P.rope_q);
    EpiQKV<T> eq{q, kb, vb, c.qk_norm ? nullptr : rope_q, block, c.n_q_heads, c.n_kv_heads, c.head_dim, pad8(block)};
    DF_LAUNCH(DFLASH_STAGE_QKV, 1, (gemm_launch<T, EpiQKV<T>>(pq, P.g_qkv, eq, s)), "QKV GEMM");
    if (c.qk_norm)   // per-head query / key norm, then RoPE
      DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
                qknorm_block_launch<T>(q, kb, static_cast<const T*>(L.g_q), static_cast<const T*>(L.g_k), B, block,
                                       c.n_q_heads, c.n_kv_heads, c.head_dim, c.rms_eps, rope_q, s),
                "query/key norm");

    AttnParams ap{};
    ap.q = q; ap.kb = kb; ap.vb = vb;
    ap.kc = cache->base + cache->k_off;
    ap.vc = cache->base + cache->v_off;
    ap.ctx_len = ctx_len;
    ap.layer = l; ap.layers = c.layers; ap.cap = cache->cap; ap.kvp = cache_planes<T>(c);
    ap.B = B; ap.nq = c.n_q_heads; ap.nkv = c.n_kv_heads; ap.hd = c.head_dim; ap.block = block;
    ap.chunk = P.attn_chunk; ap.splits = P.attn_splits;
    ap.opart = reinterpret_cast<float*>(ws + P.opart);
    ap.ml = reinterpret_cast<float2*>(ws + P.ml);
    ap.out = o;
    ap.out_plane = (size_t)R * hq;
    ap.scale = 1.0f / sqrtf((float)c.head_dim);
    if constexpr (ActPlanes<T>::n == 2)
      DF_LAUNCH(DFLASH_STAGE_ATTN, 2, attention_bf16_launch(ap, amaps, m->status_dev, s), "attention");
    else
      DF_LAUNCH(DFLASH_STAGE_ATTN, 2, attention_launch<T>(ap, s), "attention");

    GemmProblem po = make_problem(m, o, hq, R, hq, pl, (size_t)R * hq);
    add_seg(po, L.w_o, layer_map(l, kMapO), L.w_o, layer_map(l, kMapO), D / kTileN, 0, 0);
    apply_plan(po, P.g_o, partial, counters);
    DF_LAUNCH(DFLASH_STAGE_O, 1, (gemm_launch<T, EpiResidual>(po, P.g_o, EpiResidual{x, D}, s)), "O GEMM");
    DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
              rmsnorm_launch<T>(x, static_cast<const T*>(L.g_post), c.rms_eps, R, D, u, (size_t)R * D, s),
              "post-attention norm");

    GemmProblem pg = make_problem(m, u, D, R, D, pl, (size_t)R * D);
    add_seg(pg, L.w_g, layer_map(l, kMapG), L.w_u, layer_map(l, kMapU), F / kHalfN, 1, 0);
    apply_plan(pg, P.g_gu, partial, counters);
    DF_LAUNCH(DFLASH_STAGE_GATEUP, 1, (gemm_launch<T, EpiSwiGLU<T>>(pg, P.g_gu, EpiSwiGLU<T>{a, F, (size_t)R * F}, s)),
              "gate/up GEMM");

    GemmProblem pd = make_problem(m, a, F, R, F, pl, (size_t)R * F);
    add_seg(pd, L.w_d, layer_map(l, kMapD), L.w_d, layer_map(l, kMapD), D / kTileN, 0, 0);
    apply_plan(pd, P.g_down, partial, counters);
    DF_LAUNCH(DFLASH_STAGE_DOWN, 1, (gemm_launch<T, EpiResidual>(pd, P.g_down, EpiResidual{x, D}, s)), "down GEMM");
    if (l + 1 < c.layers)
      DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
                rmsnorm_launch<T>(x, static_cast<const T*>(m->layers[l + 1].g_in), c.rms_eps, R, D, u, (size_t)R * D, s),
                "input norm");
  }
  if (Rm == 0) return DFLASH_OK;
  DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
            final_norm_launch<T>(x, static_cast<const T*>(m->g_final), c.rms_eps, B, block, D, hm, (size_t)Rm * D, slots,
                                 s),
            "final norm");
  GemmProblem plm = make_problem(m, hm, D, Rm, D, head_planes(c), (size_t)Rm * D);
  add_seg(plm, m->lm_head, kMapLm, m->lm_head, kMapLm, c.vocab / kTileN, 0, 0);
  apply_plan(plm, P.g_lm, partial, counters);
  DF_LAUNCH(DFLASH_STAGE_LMHEAD, 1, (gemm_launch<T, EpiArgmax>(plm, P.g_lm, EpiArgmax{slots, logits, c.vocab}, s)),
            "LM head GEMM");
  DF_LAUNCH(DFLASH_STAGE_OTHER, 1, argmax_finalize_launch(slots, Rm, drafts, s), "argmax");
  return DFLASH_OK;
}

// ---------------------------------------------------------------- persistent path
struct PhaseBuilder {
  PParams& p;
  int add_gemm(int epi, int K, int xmap, int planes, int prow, int scaled, const void* gain) {
    PPhase& ph = p.ph[p.nphase++];
    ph = PPhase{};
    ph.kind = kPhGemm;
    ph.epi = epi;
    ph.kw = 64;
    ph.kb = K / 64;
    ph.xmap = xmap;
    ph.planes = planes;
    ph.prow = prow;
    ph.scaled = scaled;
    ph.layer = -1;
    ph.gain = static_cast<const __nv_bfloat16*>(gain);
    ph.seg0 = nseg_total();
    ph.mrows = p.M;
    ph.ssq_in = p.ssq;
    ph.u_out = p.u;
    ph.ssq_out = p.ssq;
    return p.nphase - 1;
  }
  void add_other(int kind, int layer) {
    PPhase& ph = p.ph[p.nphase++];
    ph = PPhase{};
    ph.kind = kind;
    ph.layer = layer;
  }
  // segment of `features` output features (per matrix when paired) of the
  // last projection phase; tile_begin relative to the phase.  Wide segments
  // (gate/up, the LM head) use 256-feature tiles with the weights on the MMA's
  // N side; a paired tile is 128 gate + 128 up rows; `ragged` lets the last
  // tile run past the matrix (its missing rows read as zeros).  The others
  // use 128-feature tiles with the weights on the M side.
  bool all_wide = false;   // DFLASH_DEBUG=1 DFLASH_PERSIST_WIDE=1: every segment that allows it (experiments)
  void seg(int map0, int map1, int features, int paired, int tag, bool wide = false, bool ragged = false) {
    PPhase& ph = p.ph[p.nphase - 1];
    GemmSeg& g = p.seg[ph.seg0 + ph.nseg++];
    g = GemmSeg{};
    g.map0 = map0;
    g.map1 = map1;
    g.tw = (paired || ragged || ((wide || all_wide) && features % 256 == 0)) ? 256 : 128;
    g.tiles = paired ? features / 128 : (features + g.tw - 1) / g.tw;
    g.tile_begin = ph.tiles;
    g.paired = paired;
    g.tag = tag;
    ph.tiles += g.tiles;
    ++segs;
  }
  int segs = 0;
  int nseg_total() const { return segs; }
  // Phases whose tiles are all 128 features wide (weights on the MMA's M side)
  // take 128 K columns a stage, so that their stages carry as many weight
  // bytes as the wide phases' (more in flight across the phase boundaries).
  void finish() {
    for (int i = 0; i < p.nphase; ++i) {
      PPhase& ph = p.ph[i];
      if (ph.kind != kPhGemm || ph.kb % 2) continue;
      bool narrow = true;
      for (int j = ph.seg0; j < ph.seg0 + ph.nseg; ++j) narrow = narrow && p.seg[j].tw == 128;
      if (narrow) {
        ph.kw = 128;
        ph.kb /= 2;
      }
    }
  }
};

int32_t run_inject_persist(const dflash_model* m, dflash_cache* cache, const void* feats, const int32_t* n_new,
                           int max_rows, char* ws, const WsPlan& P, cudaStream_t s) {
  const dflash_config& c = m->cfg;
  const int D = c.hidden, hk = c.n_kv_heads * c.head_dim, F5 = c.n_target_feats * D;
  int2* rowinfo = reinterpret_cast<int2*>(ws + P.rowinfo);
  float2* rope = reinterpret_cast<float2*>(ws + P.rope_c);
  int* tickets = reinterpret_cast<int*>(ws + P.tickets);
  int32_t* ctx_len = reinterpret_cast<int32_t*>(cache->base + cache->len_off);
  __nv_bfloat16* ht = reinterpret_cast<__nv_bfloat16*>(ws + P.ht);
  DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
            inject_prep_launch(n_new, ctx_len, cache->batch, max_rows, cache->cap, rowinfo, tickets, P.ntickets + 1,
                               m->status_dev, s, m->inv_freq_dev, c.head_dim, rope),
            "inject_prep");
  PParams pp{};
  if (!encode_activation_map(&pp.xmap[0], feats, F5, max_rows, F5, kPRows) ||
      !encode_activation_map(&pp.xmap[1], ht, D, 2 * kPRows, D, kPRows))
    return fail(DFLASH_ERR_INVALID_ARG, "could not encode activation tensor maps (16-B aligned features needed)");
  pp.wmaps = static_cast<const CUtensorMap*>(m->tmaps128_dev);
  pp.M = max_rows;
  pp.D = D;
  pp.eps = c.rms_eps;
  pp.stages = m->persist_stages;
  pp.u = ht;
  pp.u_plane = (size_t)kPRows * D;
  pp.ssq = reinterpret_cast<float*>(ws + P.ssq);
  pp.partial = reinterpret_cast<float*>(ws + P.partial);
  pp.tickets = tickets;
  pp.bar = reinterpret_cast<unsigned int*>(tickets + P.ntickets);
  pp.status = m->status_dev;
  pp.inject = EpiInject<__nv_bfloat16>{reinterpret_cast<__nv_bfloat16*>(cache->base + cache->k_off),
                                       reinterpret_cast<__nv_bfloat16*>(cache->base + cache->v_off), rowinfo, rope,
                                       c.layers, c.n_kv_heads, c.head_dim, cache->cap, pad8(cache->cap),
                                       kv_planes(c)};
  pp.block = 1;
  pp.attn.hd = c.head_dim;
  PhaseBuilder pb{pp};
  pb.add_gemm(kEpFuse, F5, 0, 1, 0, 0, m->g_c);
  pb.seg(kMapWc, kMapWc, D, 0, 0);
  pb.add_gemm(kEpInject, D, 1, 2, kPRows, 1, nullptr);
  for (int l = 0; l < c.layers; ++l) {
    pb.seg(layer_map(l, kMapK), layer_map(l, kMapK), hk, 0, 2 * l);
    pb.seg(layer_map(l, kMapV), layer_map(l, kMapV), hk, 0, 2 * l + 1);
  }
  pb.finish();
  DF_LAUNCH(DFLASH_STAGE_INJECT_PERSIST, 1, persist_launch(pp, m->sms, c.head_dim, s), "persistent injection");
  return DFLASH_OK;
}

// The drafter pass as one persistent launch.  With inj_rows > 0 (a plan with
// P.fused) the same launch first runs the injection of those rows: a fusion
// phase (W_c) writes H_t's planes and sums of squares, an injection phase
// projects every layer's context K/V into the cache, then the drafter's
// phases follow.
int32_t run_draft_persist(const dflash_model* m, const dflash_cache* cache, const int32_t* anchor, int block,
                          int32_t* drafts, float* logits, char* ws, const WsPlan& P, cudaStream_t s,
                          const void* feats = nullptr, const int32_t* n_new = nullptr, int inj_rows = 0) {
  const dflash_config& c = m->cfg;
  const int B = cache->batch, D = c.hidden, F = c.ffn;
  const int hq = c.n_q_heads * c.head_dim, hk = c.n_kv_heads * c.head_dim;
  const int R = B * block;
  const bool fused = inj_rows > 0;
  const int F5 = c.n_target_feats * D;
  if (fused) {   // the injection's row map, ctx_len update and RoPE table come first
    DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
              inject_prep_launch(n_new, reinterpret_cast<int32_t*>(cache->base + cache->len_off), B, inj_rows,
                                 cache->cap, reinterpret_cast<int2*>(ws + P.rowinfo),
                                 reinterpret_cast<int*>(ws + P.tickets), P.ntickets + 1 + P.ngcnt, m->status_dev, s,
                                 m->inv_freq_dev, c.head_dim, reinterpret_cast<float2*>(ws + P.rope_c)),
              "inject_prep");
  }
  float* x = reinterpret_cast<float*>(ws + P.x);
  __nv_bfloat16* u = reinterpret_cast<__nv_bfloat16*>(ws + P.u);
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(ws + P.o);
  __nv_bfloat16* a = reinterpret_cast<__nv_bfloat16*>(ws + P.a);
  float* ssq = reinterpret_cast<float*>(ws + P.ssq);
  int* tickets = reinterpret_cast<int*>(ws + P.tickets);
  unsigned long long* slots = reinterpret_cast<unsigned long long*>(ws + P.slots);
  float2* rope = reinterpret_cast<float2*>(ws + P.rope_q);
  const int32_t* ctx_len = reinterpret_cast<const int32_t*>(cache->base + cache->len_off);

  DF_LAUNCH(DFLASH_STAGE_OTHER, 1,
            persist_draft_prep_launch(static_cast<const __nv_bfloat16*>(m->embed), anchor, c.mask_token_id, c.vocab,
                                      B, block, D, static_cast<const __nv_bfloat16*>(m->layers[0].g_in), x, u,
                                      (size_t)kPRows * D, ssq, slots, tickets, P.ntickets + 1 + P.ngcnt, m->status_dev,
                                      ctx_len,
                                      m->inv_freq_dev, c.head_dim, rope, s),
            "embedding");
  PParams pp{};
  if (!encode_activation_map(&pp.xmap[0], u, D, 2 * kPRows, D, kPRows) ||
      !encode_activation_map(&pp.xmap[1], o, hq, 2 * kPRows, hq, kPRows) ||
      !encode_activation_map(&pp.xmap[2], a, F, 2 * kPRows, F, kPRows))
    return fail(DFLASH_ERR_CUDA, "could not encode activation tensor maps");
  __nv_bfloat16* ht = fused ? reinterpret_cast<__nv_bfloat16*>(ws + P.ht) : nullptr;
  if (fused && (!encode_activation_map(&pp.xmap[3], feats, F5, inj_rows, F5, kPRows) ||
                !encode_activation_map(&pp.xmap[4], ht, D, 2 * kPRows, D, kPRows)))
    return fail(DFLASH_ERR_INVALID_ARG, "could not encode activation tensor maps (16-B aligned features needed)");
  pp.wmaps = static_cast<const CUtensorMap*>(m->tmaps128_dev);
  pp.M = R;
  pp.D = D;
  pp.eps = c.rms_eps;
  pp.stages = m->persist_stages;
  pp.x = x;
  pp.u = u;
  pp.u_plane = (size_t)kPRows * D;
  pp.ssq = ssq;
  pp.partial = reinterpret_cast<float*>(ws + P.partial);
  pp.tickets = tickets;
  pp.bar = reinterpret_cast<unsigned int*>(tickets + P.ntickets);
  pp.gcnt = tickets + P.ntickets + 1;
  pp.status = m->status_dev;
  float* q = reinterpret_cast<float*>(ws + P.q);
  __nv_bfloat16* kb = reinterpret_cast<__nv_bfloat16*>(ws + P.kb);
  __nv_bfloat16* vb = reinterpret_cast<__nv_bfloat16*>(ws + P.vb);
  pp.qkv = EpiQKV<__nv_bfloat16>{q, kb, vb, rope, block, c.n_q_heads, c.n_kv_heads, c.head_dim, pad8(block)};
  pp.swiglu = EpiSwiGLU<__nv_bfloat16>{a, F, (size_t)kPRows * F};
  pp.slots = slots;
  pp.logits = logits;
  pp.drafts = block > 1 ? drafts : nullptr;
  pp.vocab = c.vocab;
  pp.block = block;
  AttnParams& ap = pp.attn;
  ap.q = q;
  ap.kb = kb;
  ap.vb = vb;
  ap.kc = cache->base + cache->k_off;
  ap.vc = cache->base + cache->v_off;
  ap.ctx_len = ctx_len;
  ap.layers = c.layers;
  ap.cap = cache->cap;
  ap.kvp = kv_planes(c);
  ap.B = B;
  ap.nq = c.n_q_heads;
  ap.nkv = c.n_kv_heads;
  ap.hd = c.head_dim;
  ap.block = block;
  ap.splits = P.nch;
  ap.opart = reinterpret_cast<float*>(ws + P.opart);
  ap.ml = reinterpret_cast<float2*>(ws + P.aml);
  ap.out = o;
  ap.out_plane = (size_t)kPRows * hq;
  ap.scale = 1.0f / sqrtf((float)c.head_dim);
  if (!encode_attention_maps(&pp.amaps, ap.kc, ap.vc, kb, vb, B, c.layers, c.n_kv_heads, c.head_dim, cache->cap,
                             pad8(cache->cap), ap.kvp, block, pad8(block)))
    return fail(DFLASH_ERR_CUDA, "could not encode attention tensor maps");

  float* ssq_ht = fused ? reinterpret_cast<float*>(ws + P.ssq2) : nullptr;
  if (fused) {
    pp.inject = EpiInject<__nv_bfloat16>{reinterpret_cast<__nv_bfloat16*>(cache->base + cache->k_off),
                                         reinterpret_cast<__nv_bfloat16*>(cache->base + cache->v_off),
                                         reinterpret_cast<const int2*>(ws + P.rowinfo),
                                         reinterpret_cast<const float2*>(ws + P.rope_c), c.layers, c.n_kv_heads,
                                         c.head_dim, cache->cap, pad8(cache->cap), kv_planes(c)};
  }

  PhaseBuilder pb{pp};
  if (const char* w = debug_env("DFLASH_PERSIST_WIDE")) pb.all_wide = std::strcmp(w, "1") == 0;
  if (fused) {   // context fusion: H_t planes * g_c and their sums of squares
    const int ph = pb.add_gemm(kEpFuse, F5, 3, 1, 0, 0, m->g_c);
    pp.ph[ph].mrows = inj_rows;
    pp.ph[ph].u_out = ht;
    pp.ph[ph].ssq_out = ssq_ht;
    pb.seg(kMapWc, kMapWc, D, 0, 0);
    // every layer's context K/V of the injected rows
    const int ip = pb.add_gemm(kEpInject, D, 4, 2, kPRows, 1, nullptr);
    pp.ph[ip].mrows = inj_rows;
    pp.ph[ip].ssq_in = ssq_ht;
    for (int l = 0; l < c.layers; ++l) {
      pb.seg(layer_map(l, kMapK), layer_map(l, kMapK), hk, 0, 2 * l);
      pb.seg(layer_map(l, kMapV), layer_map(l, kMapV), hk, 0, 2 * l + 1);
    }
  }
  for (int l = 0; l < c.layers; ++l) {
    const dflash_layer_weights& L = m->layers[l];
    pb.add_gemm(kEpQKV, D, 0, 2, kPRows, 1, nullptr);
    pb.seg(layer_map(l, kMapQ), layer_map(l, kMapQ), hq, 0, 0);
    pb.seg(layer_map(l, kMapK), layer_map(l, kMapK), hk, 0, 1);
    pb.seg(layer_map(l, kMapV), layer_map(l, kMapV), hk, 0, 2);
    pb.add_other(kPhAttn, l);
    pb.add_gemm(kEpResid, hq, 1, 2, kPRows, 0, L.g_post);
    pb.seg(layer_map(l, kMapO), layer_map(l, kMapO), D, 0, 0);
    pb.add_gemm(kEpSwiGLU, D, 0, 2, kPRows, 1, nullptr);
    pb.seg(layer_map(l, kMapG), layer_map(l, kMapU), F, 1, 0, true);
    pb.add_gemm(kEpResid, F, 2, 2, kPRows, 0, l + 1 < c.layers ? m->layers[l + 1].g_in : m->g_final);
    pb.seg(layer_map(l, kMapD), layer_map(l, kMapD), D, 0, 0);
  }
  if (block > 1) {
    pb.add_gemm(kEpLM, D, 0, 2, kPRows, 1, nullptr);
    pb.seg(kMapLm, kMapLm, c.vocab, 0, 0, true, true);
  }
  pb.finish();
  pp.trace = m->trace_persist ? m->trace_dev : nullptr;
  if (fused)
    DF_LAUNCH(DFLASH_STAGE_CYCLE_PERSIST, 1, persist_launch(pp, m->sms, c.head_dim, s), "persistent cycle");
  else
    DF_LAUNCH(DFLASH_STAGE_DRAFT_PERSIST, 1, persist_launch(pp, m->sms, c.head_dim, s), "persistent drafter");
  return DFLASH_OK;
}

// Tensor maps of every weight matrix, copied once to device memory.
int32_t build_weight_maps(dflash_model* m) {
  const dflash_config& c = m->cfg;
  const int D = c.hidden, hq = c.n_q_heads * c.head_dim, hk = c.n_kv_heads * c.head_dim, F = c.ffn;
  const size_t mb = tensor_map_bytes();
  const int n = kMapLayer0 + kMapsPerLayer * c.layers;
  std::vector<unsigned char> host(mb * n), host128(mb * n);
  auto enc = [&](int idx, const void* w, int inner, int rows) {
    if (reinterpret_cast<uintptr_t>(w) % 16) return false;
    return encode_weight_map(host.data() + mb * idx, w, inner, rows) &&
           encode_weight_map(host128.data() + mb * idx, w, inner, rows, 128);
  };
  bool ok = enc(kMapLm, m->lm_head, D, c.vocab) && enc(kMapWc, m->w_c, c.n_target_feats * D, D);
  for (int l = 0; ok && l < c.layers; ++l) {
    const dflash_layer_weights& L = m->layers[l];
    ok = enc(layer_map(l, kMapQ), L.w_q, D, hq) && enc(layer_map(l, kMapK), L.w_k, D, hk) &&
         enc(layer_map(l, kMapV), L.w_v, D, hk) && enc(layer_map(l, kMapO), L.w_o, hq, D) &&
         enc(layer_map(l, kMapG), L.w_g, D, F) && enc(layer_map(l, kMapU), L.w_u, D, F) &&
         enc(layer_map(l, kMapD), L.w_d, F, D);
  }
  if (!ok) return fail(DFLASH_ERR_UNSUPPORTED, "could not encode weight tensor maps (16-B aligned weights needed)");
  DF_CUDA(cudaMalloc(&m->tmaps_dev, host.size()), "tensor maps");
  DF_CUDA(cudaMemcpy(m->tmaps_dev, host.data(), host.size(), cudaMemcpyHostToDevice), "tensor maps");
  DF_CUDA(cudaMalloc(&m->tmaps128_dev, host128.size()), "tensor maps");
  DF_CUDA(cudaMemcpy(m->tmaps128_dev, host128.data(), host128.size(), cudaMemcpyHostToDevice), "tensor maps");
  return DFLASH_OK;
}

// K [b][layer][kvh][cap][hd] fp32, or kv_planes bf16 planes [..][P][cap][hd];
// V the same for fp32 models and hd-major [..][P][hd][pad8(cap)] for bf16 models.
size_t cache_k_bytes(const dflash_config* cfg, int batch, int capacity) {
  const size_t elem = cfg->dtype == DFLASH_DTYPE_BF16 ? 2 * (size_t)kv_planes(*cfg) : sizeof(float);
  return elem * (size_t)batch * cfg->layers * cfg->n_kv_heads * (size_t)capacity * cfg->head_dim;
}
size_t cache_v_bytes(const dflash_config* cfg, int batch, int capacity) {
  return cache_k_bytes(cfg, batch, cfg->dtype == DFLASH_DTYPE_BF16 ? pad8(capacity) : capacity);
}

}  // namespace

extern "C" {

int32_t dflash_version(void) { return 10100; }

const char* dflash_last_error(void) { return g_last_error.c_str(); }

int32_t dflash_model_create(const dflash_config* cfg, const dflash_weights* w, dflash_model** out) {
  if (!out) return fail(DFLASH_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int32_t rc = check_config(cfg);
  if (rc) return rc;
  if (!w || !w->embed || !w->lm_head || !w->w_c || !w->g_c || !w->g_final || !w->layers)
    return fail(DFLASH_ERR_INVALID_ARG, "a top-level weight pointer is NULL");
  for (int l = 0; l < cfg->layers; ++l) {
    const dflash_layer_weights& L = w->layers[l];
    if (!L.g_in || !L.w_q || !L.w_k || !L.w_v || !L.w_o || !L.g_post || !L.w_g || !L.w_u || !L.w_d)
      return fail(DFLASH_ERR_INVALID_ARG, "a weight pointer of layer %d is NULL", l);
    if (cfg->qk_norm && (!L.g_q || !L.g_k)) return fail(DFLASH_ERR_INVALID_ARG, "qk_norm: g_q or g_k of layer %d is NULL", l);
  }
  dflash_model* m = new dflash_model();
  m->cfg = *cfg;
  m->embed = w->embed;
  m->lm_head = w->lm_head;
  m->w_c = w->w_c;
  m->g_c = w->g_c;
  m->g_final = w->g_final;
  m->layers.assign(w->layers, w->layers + cfg->layers);
  cudaError_t e = cudaGetDevice(&m->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m->sms, cudaDevAttrMultiProcessorCount, m->device);
  if (e == cudaSuccess) e = cudaMalloc(&m->status_dev, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(m->status_dev, 0, sizeof(int32_t));
  const int half = cfg->head_dim / 2;
  std::vector<double> inv(half);
  for (int i = 0; i < half; ++i) inv[i] = std::pow((double)cfg->rope_theta, -2.0 * i / cfg->head_dim);
  if (e == cudaSuccess) e = cudaMalloc(&m->inv_freq_dev, sizeof(double) * half);
  if (e == cudaSuccess) e = cudaMemcpy(m->inv_freq_dev, inv.data(), sizeof(double) * half, cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cfg->dtype == DFLASH_DTYPE_F32
            ? attention_prepare<float>((cfg->n_q_heads / cfg->n_kv_heads) * cfg->max_block, cfg->head_dim)
            : attention_prepare<__nv_bfloat16>((cfg->n_q_heads / cfg->n_kv_heads) * cfg->max_block, cfg->head_dim);
  if (e != cudaSuccess) {
    dflash_model_destroy(m);
    return cuda_fail(e, "model state");
  }
  const char* tr = std::getenv("DFLASH_TRACE_GEMM");
  const char* tp = std::getenv("DFLASH_TRACE_PERSIST");
  m->trace_persist = tp && std::strcmp(tp, "0") != 0;
  if (tr || m->trace_persist) {
    m->trace_target = tr ? std::atol(tr) : -1;
    if (cudaMalloc(&m->trace_dev, kTraceEntries * sizeof(unsigned long long)) != cudaSuccess ||
        cudaMemset(m->trace_dev, 0, kTraceEntries * sizeof(unsigned long long)) != cudaSuccess) {
      dflash_model_destroy(m);
      return fail(DFLASH_ERR_CUDA, "trace buffer");
    }
  }
  const char* gemm_env = std::getenv("DFLASH_GEMM");
  m->use_tc = cfg->dtype == DFLASH_DTYPE_BF16 && !(gemm_env && std::strcmp(gemm_env, "simt") == 0);
  if (m->use_tc) {
    rc = build_weight_maps(m);
    if (rc) {
      dflash_model_destroy(m);
      return rc;
    }
    const char* pe = std::getenv("DFLASH_PERSIST");
    if (!(pe && std::strcmp(pe, "0") == 0) && (cfg->head_dim == 64 || cfg->head_dim == 128) &&
        cfg->vocab % kTileN == 0) {
      m->persist_stages = persist_stages(cfg->head_dim);
      e = persist_prepare(cfg->head_dim);
      if (e != cudaSuccess) {
        dflash_model_destroy(m);
        return cuda_fail(e, "persistent kernel set-up");
      }
      m->persist = 1;
    }
  }
  *out = m;
  return DFLASH_OK;
}

int32_t dflash_model_destroy(dflash_model* m) {
  if (!m) return DFLASH_OK;
  if (m->status_dev) cudaFree(m->status_dev);
  if (m->inv_freq_dev) cudaFree(m->inv_freq_dev);
  if (m->tmaps_dev) cudaFree(m->tmaps_dev);
  if (m->tmaps128_dev) cudaFree(m->tmaps128_dev);
  if (m->trace_dev) cudaFree(m->trace_dev);
  for (cudaEvent_t e : m->prof.ev) cudaEventDestroy(e);
  delete m;
  return DFLASH_OK;
}

int32_t dflash_get_status(const dflash_model* m, dflash_stream_t stream, int32_t* status_host) {
  if (!m || !status_host) return fail(DFLASH_ERR_INVALID_ARG, "model or status_host is NULL");
  DF_CUDA(cudaMemcpyAsync(status_host, m->status_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream),
          "status read");
  DF_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "status sync");
  return DFLASH_OK;
}

int32_t dflash_clear_status(const dflash_model* m, dflash_stream_t stream) {
  if (!m) return fail(DFLASH_ERR_INVALID_ARG, "model is NULL");
  DF_CUDA(cudaMemsetAsync(m->status_dev, 0, sizeof(int32_t), (cudaStream_t)stream), "status clear");
  return DFLASH_OK;
}

int32_t dflash_selftest_wait_timeout(const dflash_model* m, int64_t budget_cycles, dflash_stream_t stream) {
  if (!m) return fail(DFLASH_ERR_INVALID_ARG, "model is NULL");
  if (budget_cycles <= 0 || budget_cycles > (int64_t)4000000000LL)
    return fail(DFLASH_ERR_INVALID_ARG, "budget_cycles %lld outside (0, 4e9]", (long long)budget_cycles);
  int32_t rc = check_device(m);
  if (rc) return rc;
  DF_CUDA(wait_selftest_launch(budget_cycles, m->status_dev, (cudaStream_t)stream), "wait self-test");
  g_launch_count += 1;
  return DFLASH_OK;
}

size_t dflash_cache_bytes(const dflash_config* cfg, int32_t batch, int32_t capacity) {
  if (check_config(cfg) != DFLASH_OK || batch < 0 || capacity < 0) return 0;
  return align256(cache_k_bytes(cfg, batch, capacity)) + align256(cache_v_bytes(cfg, batch, capacity)) +
         align256(sizeof(int32_t) * std::max(batch, 1));
}

int32_t dflash_cache_init(const dflash_model* m, void* dev_mem, size_t bytes, int32_t batch, int32_t capacity,
                          dflash_stream_t stream, dflash_cache** out) {
  if (!out) return fail(DFLASH_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!m || !dev_mem) return fail(DFLASH_ERR_INVALID_ARG, "model or dev_mem is NULL");
  if (batch <= 0 || capacity <= 0) return fail(DFLASH_ERR_INVALID_ARG, "batch %d and capacity %d must be positive", batch, capacity);
  if (batch > 4096) return fail(DFLASH_ERR_SHAPE, "batch %d > 4096", batch);
  if (reinterpret_cast<uintptr_t>(dev_mem) % 256) return fail(DFLASH_ERR_INVALID_ARG, "dev_mem must be 256-byte aligned");
  const size_t need = dflash_cache_bytes(&m->cfg, batch, capacity);
  if (bytes < need) return fail(DFLASH_ERR_CAPACITY, "cache memory %zu bytes < %zu needed", bytes, need);
  int32_t rc = check_device(m);
  if (rc) return rc;
  const size_t kb = align256(cache_k_bytes(&m->cfg, batch, capacity));
  const size_t vb = align256(cache_v_bytes(&m->cfg, batch, capacity));
  dflash_cache* c = new dflash_cache();
  c->model = m;
  c->base = static_cast<char*>(dev_mem);
  c->bytes = bytes;
  c->batch = batch;
  c->cap = capacity;
  c->k_off = 0;
  c->v_off = kb;
  c->len_off = kb + vb;
  c->len_host.assign(batch, 0);
  c->len_known = true;
  // zeroed once: positions past a request's context are then always finite
  // (the attention reads whole tiles and gives those keys probability 0)
  cudaError_t e = cudaMemsetAsync(c->base, 0, c->len_off + sizeof(int32_t) * batch, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "cache init");
  }
  *out = c;
  return DFLASH_OK;
}

int32_t dflash_cache_destroy(dflash_cache* c) {
  delete c;
  return DFLASH_OK;
}

int32_t dflash_cache_layout(const dflash_cache* c, size_t* k_off, size_t* v_off, size_t* len_off) {
  if (!c || !k_off || !v_off || !len_off) return fail(DFLASH_ERR_INVALID_ARG, "NULL argument");
  *k_off = c->k_off;
  *v_off = c->v_off;
  *len_off = c->len_off;
  return DFLASH_OK;
}

int32_t dflash_cache_set_lengths(dflash_cache* c, const int32_t* len_host, dflash_stream_t stream) {
  if (!c || !len_host) return fail(DFLASH_ERR_INVALID_ARG, "cache or ctx_len_host is NULL");
  for (int b = 0; b < c->batch; ++b)
    if (len_host[b] < 0 || len_host[b] > c->cap)
      return fail(DFLASH_ERR_CAPACITY, "ctx_len[%d] = %d outside [0, %d]", b, len_host[b], c->cap);
  DF_CUDA(cudaMemcpyAsync(c->base + c->len_off, len_host, sizeof(int32_t) * c->batch, cudaMemcpyHostToDevice,
                          (cudaStream_t)stream), "set lengths");
  c->len_host.assign(len_host, len_host + c->batch);
  c->len_known = true;
  return DFLASH_OK;
}

size_t dflash_workspace_bytes(const dflash_model* m, int32_t batch, int32_t capacity, int32_t block_size,
                              int32_t max_inject_rows) {
  if (!m || batch <= 0 || capacity < 0 || block_size < 1 || block_size > m->cfg.max_block || max_inject_rows < 0) return 0;
  // smaller calls may take the persistent path, whose scratch differs: cover
  // every block size up to block_size and injections of up to 16 rows too
  size_t need = plan_ws(m, batch, capacity, 0, max_inject_rows).total;
  if (max_inject_rows > 0)
    need = std::max(need, plan_ws(m, batch, capacity, 0, std::min(max_inject_rows, kPRows)).total);
  for (int b = 1; b <= block_size; ++b) {
    need = std::max(need, plan_ws(m, batch, capacity, b, 0).total);
    // dflash_draft_cycle: injection and drafter pass in one launch
    if (max_inject_rows > 0) need = std::max(need, plan_ws(m, batch, capacity, b, std::min(max_inject_rows, kPRows)).total);
  }
  return need;
}

int32_t dflash_inject_context(const dflash_model* m, dflash_cache* cache, const void* feats, const int32_t* n_new_dev,
                              const int32_t* n_new_host, int32_t max_rows, void* workspace, size_t ws_bytes,
                              dflash_stream_t stream) {
  if (!m || !cache) return fail(DFLASH_ERR_INVALID_ARG, "model or cache is NULL");
  if (cache->model != m) return fail(DFLASH_ERR_INVALID_ARG, "cache was made for another model");
  if (max_rows < 0) return fail(DFLASH_ERR_INVALID_ARG, "max_rows %d < 0", max_rows);
  if (!n_new_dev) return fail(DFLASH_ERR_INVALID_ARG, "n_new_dev is NULL");
  if (max_rows > 0 && (!feats || !workspace)) return fail(DFLASH_ERR_INVALID_ARG, "feats or workspace is NULL");
  int32_t rc = check_device(m);
  if (rc) return rc;
  if (n_new_host) {
    long total = 0;
    for (int b = 0; b < cache->batch; ++b) {
      if (n_new_host[b] < 0) return fail(DFLASH_ERR_INVALID_ARG, "n_new[%d] = %d < 0", b, n_new_host[b]);
      total += n_new_host[b];
      if (cache->len_known && cache->len_host[b] + (long)n_new_host[b] > cache->cap)
        return fail(DFLASH_ERR_CAPACITY, "request %d: %d + %d tokens exceed capacity %d", b, cache->len_host[b],
                    n_new_host[b], cache->cap);
    }
    if (total > max_rows) return fail(DFLASH_ERR_SHAPE, "sum of n_new (%ld) > max_rows (%d)", total, max_rows);
  }
  if (max_rows == 0) return DFLASH_OK;
  const WsPlan P = plan_ws(m, cache->batch, cache->cap, 0, max_rows);
  if (ws_bytes < P.total) return fail(DFLASH_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, P.total);
  cudaStream_t s = (cudaStream_t)stream;
  rc = P.persist ? run_inject_persist(m, cache, feats, n_new_dev, max_rows, static_cast<char*>(workspace), P, s)
       : m->cfg.dtype == DFLASH_DTYPE_F32
           ? run_inject<float>(m, cache, feats, n_new_dev, max_rows, static_cast<char*>(workspace), P, s)
           : run_inject<__nv_bfloat16>(m, cache, feats, n_new_dev, max_rows, static_cast<char*>(workspace), P, s);
  if (rc) return rc;
  if (n_new_host) {
    if (cache->len_known)
      for (int b = 0; b < cache->batch; ++b) cache->len_host[b] += n_new_host[b];
  } else {
    cache->len_known = false;
  }
  return DFLASH_OK;
}

int32_t dflash_draft_block(const dflash_model* m, const dflash_cache* cache, const int32_t* anchor_dev,
                           int32_t block_size, int32_t* draft_dev, float* logits_dev, void* workspace,
                           size_t ws_bytes, dflash_stream_t stream) {
  if (!m || !cache) return fail(DFLASH_ERR_INVALID_ARG, "model or cache is NULL");
  if (cache->model != m) return fail(DFLASH_ERR_INVALID_ARG, "cache was made for another model");
  if (block_size < 1 || block_size > m->cfg.max_block)
    return fail(DFLASH_ERR_SHAPE, "block_size %d outside [1, %d]", block_size, m->cfg.max_block);
  if (!anchor_dev || !workspace) return fail(DFLASH_ERR_INVALID_ARG, "anchor_dev or workspace is NULL");
  if (block_size > 1 && !draft_dev) return fail(DFLASH_ERR_INVALID_ARG, "draft_dev is NULL");
  int32_t rc = check_device(m);
  if (rc) return rc;
  const WsPlan P = plan_ws(m, cache->batch, cache->cap, block_size, 0);
  if (ws_bytes < P.total) return fail(DFLASH_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, P.total);
  cudaStream_t s = (cudaStream_t)stream;
  if (P.persist)
    return run_draft_persist(m, cache, anchor_dev, block_size, draft_dev, logits_dev, static_cast<char*>(workspace), P, s);
  return m->cfg.dtype == DFLASH_DTYPE_F32
             ? run_draft<float>(m, cache, anchor_dev, block_size, draft_dev, logits_dev, static_cast<char*>(workspace), P, s)
             : run_draft<__nv_bfloat16>(m, cache, anchor_dev, block_size, draft_dev, logits_dev,
                                        static_cast<char*>(workspace), P, s);
}

int32_t dflash_draft_cycle(const dflash_model* m, dflash_cache* cache, const void* feats, const int32_t* n_new_dev,
                           const int32_t* n_new_host, int32_t max_rows, const int32_t* anchor_dev, int32_t block_size,
                           int32_t* draft_dev, float* logits_dev, void* workspace, size_t ws_bytes,
                           dflash_stream_t stream) {
  if (!m || !cache) return fail(DFLASH_ERR_INVALID_ARG, "model or cache is NULL");
  if (cache->model != m) return fail(DFLASH_ERR_INVALID_ARG, "cache was made for another model");
  if (max_rows < 0) return fail(DFLASH_ERR_INVALID_ARG, "max_rows %d < 0", max_rows);
  if (!n_new_dev) return fail(DFLASH_ERR_INVALID_ARG, "n_new_dev is NULL");
  if (block_size < 1 || block_size > m->cfg.max_block)
    return fail(DFLASH_ERR_SHAPE, "block_size %d outside [1, %d]", block_size, m->cfg.max_block);
  if (!anchor_dev || !workspace || (max_rows > 0 && !feats))
    return fail(DFLASH_ERR_INVALID_ARG, "anchor_dev, feats or workspace is NULL");
  if (block_size > 1 && !draft_dev) return fail(DFLASH_ERR_INVALID_ARG, "draft_dev is NULL");
  int32_t rc = check_device(m);
  if (rc) return rc;
  const WsPlan P = plan_ws(m, cache->batch, cache->cap, block_size, max_rows);
  if (max_rows == 0 || !P.fused) {   // the two calls one after the other
    rc = dflash_inject_context(m, cache, feats, n_new_dev, n_new_host, max_rows, workspace, ws_bytes, stream);
    if (rc) return rc;
    return dflash_draft_block(m, cache, anchor_dev, block_size, draft_dev, logits_dev, workspace, ws_bytes, stream);
  }
  if (n_new_host) {
    long total = 0;
    for (int b = 0; b < cache->batch; ++b) {
      if (n_new_host[b] < 0) return fail(DFLASH_ERR_INVALID_ARG, "n_new[%d] = %d < 0", b, n_new_host[b]);
      total += n_new_host[b];
      if (cache->len_known && cache->len_host[b] + (long)n_new_host[b] > cache->cap)
        return fail(DFLASH_ERR_CAPACITY, "request %d: %d + %d tokens exceed capacity %d", b, cache->len_host[b],
                    n_new_host[b], cache->cap);
    }
    if (total > max_rows) return fail(DFLASH_ERR_SHAPE, "sum of n_new (%ld) > max_rows (%d)", total, max_rows);
  }
  if (ws_bytes < P.total) return fail(DFLASH_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, P.total);
  rc = run_draft_persist(m, cache, anchor_dev, block_size, draft_dev, logits_dev, static_cast<char*>(workspace), P,
                         (cudaStream_t)stream, feats, n_new_dev, max_rows);
  if (rc) return rc;
  if (n_new_host) {
    if (cache->len_known)
      for (int b = 0; b < cache->batch; ++b) cache->len_host[b] += n_new_host[b];
  } else {
    cache->len_known = false;
  }
  return DFLASH_OK;
}

int32_t dflash_verify_greedy(const int32_t* draft_dev, const int32_t* target_argmax_dev, int32_t batch,
                             int32_t block_size, int32_t* accept_len_dev, int32_t* out_tokens_dev,
                             int32_t* next_anchor_dev, dflash_stream_t stream) {
  if (batch < 0) return fail(DFLASH_ERR_INVALID_ARG, "batch %d < 0", batch);
  if (block_size < 1 || block_size > kMaxBlock) return fail(DFLASH_ERR_SHAPE, "block_size %d outside [1, %d]", block_size, kMaxBlock);
  if (batch == 0) return DFLASH_OK;
  if ((block_size > 1 && !draft_dev) || !target_argmax_dev || !accept_len_dev || !out_tokens_dev || !next_anchor_dev)
    return fail(DFLASH_ERR_INVALID_ARG, "a device pointer is NULL");
  DF_CUDA(verify_launch(draft_dev, target_argmax_dev, batch, block_size, accept_len_dev, out_tokens_dev,
                        next_anchor_dev, (cudaStream_t)stream), "verify");
  g_launch_count += 1;
  return DFLASH_OK;
}

size_t dflash_sampling_workspace_bytes(int32_t rows, int32_t draws, int32_t vocab) {
  if (rows < 0 || draws < 0 || vocab <= 0) return 0;
  return sampling_workspace_bytes(std::max(rows, 1), std::max(draws, 1), vocab);
}

namespace {
int32_t check_sampling(const void* p_logits, int rows, int vocab, float temperature, const void* ws, size_t ws_bytes,
                       int draws) {
  if (vocab <= 0 || vocab % 4 || vocab > (1 << 24))
    return fail(DFLASH_ERR_SHAPE, "vocab %d must be a positive multiple of 4, at most 2^24", vocab);
  if (rows > 65535) return fail(DFLASH_ERR_SHAPE, "%d logits rows > 65535", rows);
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(DFLASH_ERR_INVALID_ARG, "temperature must be positive and finite");
  if (reinterpret_cast<uintptr_t>(p_logits) % 16) return fail(DFLASH_ERR_INVALID_ARG, "logits must be 16-byte aligned");
  if (!ws) return fail(DFLASH_ERR_INVALID_ARG, "workspace is NULL");
  const size_t need = sampling_workspace_bytes(rows, draws, vocab);
  if (ws_bytes < need) return fail(DFLASH_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
  return DFLASH_OK;
}
}  // namespace

int32_t dflash_verify_sampled(const float* draft_logits, const float* target_logits, const int32_t* drafts,
                              const float* u_accept, const float* u_sample, int32_t batch, int32_t block_size,
                              int32_t vocab, float temperature, int32_t* accept_len, int32_t* out_tokens,
                              int32_t* next_anchor, void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  if (batch < 0) return fail(DFLASH_ERR_INVALID_ARG, "batch %d < 0", batch);
  if (block_size < 1 || block_size > kMaxBlock)
    return fail(DFLASH_ERR_SHAPE, "block_size %d outside [1, %d]", block_size, kMaxBlock);
  if (batch == 0) return DFLASH_OK;
  if ((block_size > 1 && (!draft_logits || !drafts || !u_accept)) || !target_logits || !u_sample || !accept_len ||
      !out_tokens || !next_anchor)
    return fail(DFLASH_ERR_INVALID_ARG, "a device pointer is NULL");
  if (block_size > 1 && reinterpret_cast<uintptr_t>(draft_logits) % 16)
    return fail(DFLASH_ERR_INVALID_ARG, "logits must be 16-byte aligned");
  const int rows = batch * (2 * block_size - 1);
  int32_t rc = check_sampling(target_logits, rows, vocab, temperature, workspace, ws_bytes, batch);
  if (rc) return rc;
  int launches = 0;
  DF_CUDA(verify_sampled_launch(draft_logits, target_logits, drafts, u_accept, u_sample, batch, block_size, vocab,
                                temperature, accept_len, out_tokens, next_anchor, workspace, &launches,
                                (cudaStream_t)stream),
          "sampled verification");
  g_launch_count += launches;
  return DFLASH_OK;
}

int32_t dflash_sample_tokens(const float* logits, int32_t rows, int32_t vocab, float temperature, const float* u,
                             int32_t* tokens, void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  if (rows < 0) return fail(DFLASH_ERR_INVALID_ARG, "rows %d < 0", rows);
  if (rows == 0) return DFLASH_OK;
  if (!logits || !u || !tokens) return fail(DFLASH_ERR_INVALID_ARG, "a device pointer is NULL");
  int32_t rc = check_sampling(logits, rows, vocab, temperature, workspace, ws_bytes, rows);
  if (rc) return rc;
  int launches = 0;
  DF_CUDA(sample_tokens_launch(logits, rows, vocab, temperature, u, tokens, workspace, &launches,
                               (cudaStream_t)stream),
          "token sampling");
  g_launch_count += launches;
  return DFLASH_OK;
}

namespace {
int32_t packed_shape(int32_t n_blocks, int32_t block, int32_t seq_len, int32_t nq, int32_t nkv, int32_t hd) {
  if (n_blocks < 0 || block < 1 || block > kMaxBlock || seq_len < 0)
    return fail(DFLASH_ERR_SHAPE, "n_blocks %d >= 0, block %d in [1, %d], seq_len %d >= 0 needed", n_blocks, block,
                kMaxBlock, seq_len);
  if (hd != 64 && hd != 128) return fail(DFLASH_ERR_SHAPE, "head_dim %d must be 64 or 128", hd);
  if (nq <= 0 || nkv <= 0 || nq % nkv) return fail(DFLASH_ERR_SHAPE, "n_q_heads must be a positive multiple of n_kv_heads");
  if ((long long)n_blocks * nkv > 65535) return fail(DFLASH_ERR_SHAPE, "n_blocks * n_kv_heads > 65535");
  if ((long long)nkv * 2 * (seq_len + 1) * hd >= (1LL << 31) || (long long)n_blocks * nkv * 2 * hd * 64 >= (1LL << 31))
    return fail(DFLASH_ERR_SHAPE, "packed attention operands exceed 2^31 rows");
  return DFLASH_OK;
}
int current_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}
}  // namespace

size_t dflash_packed_attention_workspace_bytes(int32_t n_blocks, int32_t block, int32_t seq_len, int32_t nq,
                                               int32_t nkv, int32_t hd) {
  if (packed_shape(n_blocks, block, seq_len, nq, nkv, hd) != DFLASH_OK) return 0;
  const int sms = current_sms();
  if (sms <= 0) return 0;
  return packed_workspace_bytes(std::max(n_blocks, 1), block, seq_len, nq, nkv, hd, sms);
}

int32_t dflash_packed_block_attention(const void* q, const void* k_ctx, const void* v_ctx, const void* k_blk,
                                      const void* v_blk, const int32_t* anchors_dev, const int32_t* anchors_host,
                                      int32_t n_blocks, int32_t block, int32_t seq_len, int32_t nq, int32_t nkv,
                                      int32_t hd, int32_t dtype, float* out, void* workspace, size_t ws_bytes,
                                      dflash_stream_t stream) {
  int32_t rc = packed_shape(n_blocks, block, seq_len, nq, nkv, hd);
  if (rc) return rc;
  if (dtype != DFLASH_DTYPE_F32 && dtype != DFLASH_DTYPE_BF16) return fail(DFLASH_ERR_INVALID_ARG, "bad dtype %d", dtype);
  if (n_blocks == 0) return DFLASH_OK;
  if (!q || !k_blk || !v_blk || !anchors_dev || !out || !workspace || (seq_len > 0 && (!k_ctx || !v_ctx)))
    return fail(DFLASH_ERR_INVALID_ARG, "a device pointer is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(DFLASH_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (anchors_host)
    for (int n = 0; n < n_blocks; ++n)
      if (anchors_host[n] < 0 || anchors_host[n] > seq_len)
        return fail(DFLASH_ERR_INVALID_ARG, "anchor[%d] = %d outside [0, %d]", n, anchors_host[n], seq_len);
  const int sms = current_sms();
  if (sms <= 0) return fail(DFLASH_ERR_CUDA, "no current device");
  const size_t need = packed_workspace_bytes(n_blocks, block, seq_len, nq, nkv, hd, sms);
  if (ws_bytes < need) return fail(DFLASH_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
  // shared-memory opt-in of the split kernel, once per device and head size
  static std::atomic<unsigned> prepared[64];
  int dev = 0;
  DF_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  const unsigned bit = hd == 64 ? 1u : 2u;
  if (dev < 0 || dev >= 64 || !(prepared[dev].load() & bit)) {
    DF_CUDA(attention_tc_prepare(hd), "packed attention set-up");
    if (dev >= 0 && dev < 64) prepared[dev].fetch_or(bit);
  }
  // (with no context no block has a context tile: the one-row slabs are never read)
  const PackedPlan pl = packed_plan(workspace, n_blocks, block, seq_len, nq, nkv, hd, sms);
  int launches = 0;
  DF_CUDA(packed_attention_run(pl, dtype == DFLASH_DTYPE_F32, q, seq_len ? k_ctx : nullptr, seq_len ? v_ctx : nullptr,
                               k_blk, v_blk, anchors_dev, out, sms, &launches, (cudaStream_t)stream),
          "packed block attention");
  g_launch_count += launches;
  return DFLASH_OK;
}

int32_t dflash_packed_attention_status(const void* workspace, dflash_stream_t stream, int32_t* status_host) {
  if (!workspace || !status_host) return fail(DFLASH_ERR_INVALID_ARG, "workspace or status_host is NULL");
  DF_CUDA(cudaMemcpyAsync(status_host, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream),
          "status read");
  DF_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "status sync");
  return DFLASH_OK;
}

uint64_t dflash_launch_count(void) { return g_launch_count.load(); }

int32_t dflash_synthetic_target(const int32_t* draft_dev, const uint8_t* match_dev, const int32_t* off_dev,
                                const int32_t* bonus_dev, int32_t n_patterns, int64_t* pattern_idx_dev,
                                const int32_t* tau_dev, int64_t* tau_sum_dev, int32_t batch, int32_t block_size,
                                int32_t vocab, int32_t* target_dev, dflash_stream_t stream) {
  if (batch < 0 || n_patterns <= 0 || vocab <= 0) return fail(DFLASH_ERR_INVALID_ARG, "bad synthetic target sizes");
  if (block_size < 1 || block_size > kMaxBlock) return fail(DFLASH_ERR_SHAPE, "block_size %d outside [1, %d]", block_size, kMaxBlock);
  if (batch == 0) return DFLASH_OK;
  if ((block_size > 1 && (!draft_dev || !match_dev || !off_dev)) || !bonus_dev || !pattern_idx_dev || !target_dev)
    return fail(DFLASH_ERR_INVALID_ARG, "a device pointer is NULL");
  DF_CUDA(synthetic_target_launch(draft_dev, match_dev, off_dev, bonus_dev, n_patterns,
                                  reinterpret_cast<long long*>(pattern_idx_dev), tau_dev,
                                  reinterpret_cast<long long*>(tau_sum_dev), batch, block_size, vocab, target_dev,
                                  (cudaStream_t)stream),
          "synthetic target");
  g_launch_count += 1;
  return DFLASH_OK;
}

int32_t dflash_trace_read(const dflash_model* m, uint64_t* host, size_t n) {
  if (!m || !host) return fail(DFLASH_ERR_INVALID_ARG, "NULL argument");
  if (!m->trace_dev) return fail(DFLASH_ERR_UNSUPPORTED, "GEMM tracing is off (set DFLASH_TRACE_GEMM)");
  n = std::min(n, kTraceEntries);
  DF_CUDA(cudaMemcpy(host, m->trace_dev, n * sizeof(uint64_t), cudaMemcpyDeviceToHost), "trace read");
  return DFLASH_OK;
}

int32_t dflash_profile_start(dflash_model* m, int32_t max_launches) {
  if (!m || max_launches <= 0) return fail(DFLASH_ERR_INVALID_ARG, "model is NULL or max_launches <= 0");
  int32_t rc = check_device(m);
  if (rc) return rc;
  Profiler& p = m->prof;
  while ((int)p.ev.size() < 2 * max_launches) {
    cudaEvent_t e;
    DF_CUDA(cudaEventCreate(&e), "cudaEventCreate");
    p.ev.push_back(e);
  }
  p.used = 0;
  p.stage.clear();
  p.on = true;
  return DFLASH_OK;
}

int32_t dflash_profile_stop(dflash_model* m, dflash_stream_t stream, float* ms_by_stage, int32_t* launches_by_stage,
                            int32_t n_stages) {
  if (!m || !ms_by_stage || !launches_by_stage || n_stages <= 0 || n_stages > DFLASH_NUM_STAGES)
    return fail(DFLASH_ERR_INVALID_ARG, "bad profile_stop arguments");
  Profiler& p = m->prof;
  p.on = false;
  DF_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "profile sync");
  for (int i = 0; i < n_stages; ++i) {
    ms_by_stage[i] = 0.f;
    launches_by_stage[i] = 0;
  }
  for (size_t i = 0; i < p.stage.size(); ++i) {
    float ms = 0.f;
    DF_CUDA(cudaEventElapsedTime(&ms, p.ev[2 * i], p.ev[2 * i + 1]), "cudaEventElapsedTime");
    if (p.stage[i] < n_stages) {
      ms_by_stage[p.stage[i]] += ms;
      launches_by_stage[p.stage[i]] += 1;
    }
  }
  p.used = 0;
  p.stage.clear();
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of dflash_inject_context (scratch in a static array).
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

// Scratch of dflash_inject_context_noalloc.  A file-scope device array: every
// GPU that loads this library holds it until the process exits.  In host code
// the name is only a stand-in for the symbol, never a device address.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};
void* g_noalloc_ctx[kMaxDevices] = {};   // the context the address was looked up in

// The current driver context (CUcontext), through the runtime's driver entry
// point; nullptr if it cannot be had.
void* current_context() {
  using Fn = int (*)(void**);
  static Fn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<Fn>(f);
  }();
  void* ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

// Device address of the scratch array on the current device, looked up once
// per device and context (with that device current) and then reused; a
// context created anew (after cudaDeviceReset, which unloads the module that
// holds the array) gets a fresh look-up.
int32_t noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(DFLASH_ERR_UNSUPPORTED, "device %d out of range", dev);
  void* ctx = current_context();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev] || ctx == nullptr || ctx != g_noalloc_ctx[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(noalloc scratch)");
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = ctx;
  }
  *out = g_noalloc_ptr[dev];
  return DFLASH_OK;
}

}  // namespace

extern "C" {

size_t dflash_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int32_t dflash_inject_context_noalloc(const dflash_model* m, dflash_cache* cache, const void* feats,
                                      const int32_t* n_new_dev, const int32_t* n_new_host, int32_t max_rows,
                                      dflash_stream_t stream) {
  if (!m || !cache) return fail(DFLASH_ERR_INVALID_ARG, "model or cache is NULL");
  if (cache->model != m) return fail(DFLASH_ERR_INVALID_ARG, "cache was made for another model");
  if (max_rows < 0) return fail(DFLASH_ERR_INVALID_ARG, "max_rows %d < 0", max_rows);
  if (!n_new_dev) return fail(DFLASH_ERR_INVALID_ARG, "n_new_dev is NULL");
  if (max_rows > 0 && !feats) return fail(DFLASH_ERR_INVALID_ARG, "feats is NULL");
  int32_t rc = check_device(m);
  if (rc) return rc;
  if (n_new_host) {
    long total = 0;
    for (int b = 0; b < cache->batch; ++b) {
      if (n_new_host[b] < 0) return fail(DFLASH_ERR_INVALID_ARG, "n_new[%d] = %d < 0", b, n_new_host[b]);
      total += n_new_host[b];
      if (cache->len_known && cache->len_host[b] + (long)n_new_host[b] > cache->cap)
        return fail(DFLASH_ERR_CAPACITY, "request %d: %d + %d tokens exceed capacity %d", b, cache->len_host[b],
                    n_new_host[b], cache->cap);
    }
    if (total > max_rows) return fail(DFLASH_ERR_SHAPE, "sum of n_new (%ld) > max_rows (%d)", total, max_rows);
  }
  if (max_rows == 0) return DFLASH_OK;
  const WsPlan P = plan_ws(m, cache->batch, cache->cap, 0, max_rows);
  if (P.total > kNoAllocScratchBytes)
    return fail(DFLASH_ERR_CAPACITY,
                "dflash_inject_context_noalloc: %d rows need %zu bytes of scratch, more than the fixed %zu; "
                "inject fewer rows per call or use dflash_inject_context with a workspace",
                max_rows, P.total, kNoAllocScratchBytes);
  void* scratch = nullptr;
  rc = noalloc_scratch(m->device, &scratch);
  if (rc) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  rc = P.persist ? run_inject_persist(m, cache, feats, n_new_dev, max_rows, static_cast<char*>(scratch), P, s)
       : m->cfg.dtype == DFLASH_DTYPE_F32
           ? run_inject<float>(m, cache, feats, n_new_dev, max_rows, static_cast<char*>(scratch), P, s)
           : run_inject<__nv_bfloat16>(m, cache, feats, n_new_dev, max_rows, static_cast<char*>(scratch), P, s);
  if (rc) return rc;
  if (n_new_host) {
    if (cache->len_known)
      for (int b = 0; b < cache->batch; ++b) cache->len_host[b] += n_new_host[b];
  } else {
    cache->len_known = false;
  }
  return DFLASH_OK;
}

}  // extern "C"
