// Block-size scheduling for the draft cycle (paper "DFlash: Block Diffusion
// for Flash Speculative Decoding", §5.5.4: a drafter trained at a large block
// size serves smaller inference-time block sizes nearly as well, which makes
// choosing the block size per cycle possible; large blocks raise the
// verification cost when the target is compute-bound, e.g. at large batch).
//
// Host-side policy over the existing kernels: per draft position j it keeps
// decayed counts of how often position j was attempted (every earlier draft
// of its block kept, j < block) and kept (j <= tau - 1), from the accepted
// lengths tau that verification returns each cycle.  Its estimate of the
// conditional acceptance probability is alpha_j = (kept_j + prior * weight) /
// (attempted_j + weight).  For a candidate block size g the expected accepted
// length per request is E[tau | g] = 1 + sum_{i<g} prod_{j<=i} alpha_j (the
// closed form of the blog page "Inside DFlash & Block Diffusion Speculative
// Decoding", section 1), and the cycle cost is the linear model
// cost_fixed + cost_per_row * batch * g + cost_per_request * batch (drafting
// and verifying batch * g token rows).  The choice maximises
// batch * E[tau | g] / cost, ties to the smaller block.  All arithmetic is in
// double precision.
#include <algorithm>
#include <cmath>
#include <new>

#include "dflash.h"

namespace dflash {
int32_t set_error(int32_t code, const char* msg);   // api.cu: thread-local message for dflash_last_error
}
using dflash::set_error;

struct dflash_block_policy {
  dflash_block_policy_config cfg;
  int max_pos;            // largest candidate - 1: draft positions tracked
  double kept[DFLASH_POLICY_MAX_BLOCK];
  double tried[DFLASH_POLICY_MAX_BLOCK];
};

namespace {

double alpha_at(const dflash_block_policy* p, int j) {   // j: 0-based draft position
  return (p->kept[j] + (double)p->cfg.prior_accept * p->cfg.prior_weight) / (p->tried[j] + p->cfg.prior_weight);
}

double expected_tau(const dflash_block_policy* p, int g) {
  double total = 1.0, prod = 1.0;
  for (int j = 0; j < g - 1; ++j) {
    prod *= alpha_at(p, j);
    total += prod;
  }
  return total;
}

}  // namespace

extern "C" {

int32_t dflash_block_policy_create(const dflash_block_policy_config* cfg, dflash_block_policy** out) {
  if (!out) return set_error(DFLASH_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!cfg) return set_error(DFLASH_ERR_INVALID_ARG, "config is NULL");
  const int n = cfg->n_candidates;
  if (n < 1 || n > DFLASH_POLICY_MAX_CANDIDATES)
    return set_error(DFLASH_ERR_INVALID_ARG, "n_candidates must be in [1, DFLASH_POLICY_MAX_CANDIDATES]");
  for (int i = 0; i < n; ++i) {
    const int g = cfg->candidates[i];
    if (g < 1 || g > DFLASH_POLICY_MAX_BLOCK)
      return set_error(DFLASH_ERR_SHAPE, "candidate block sizes must be in [1, DFLASH_POLICY_MAX_BLOCK]");
    if (i > 0 && g <= cfg->candidates[i - 1])
      return set_error(DFLASH_ERR_INVALID_ARG, "candidate block sizes must be strictly ascending");
  }
  if (!(cfg->decay > 0.f && cfg->decay <= 1.f) || !(cfg->prior_accept >= 0.f && cfg->prior_accept <= 1.f) ||
      !(cfg->prior_weight > 0.f))
    return set_error(DFLASH_ERR_INVALID_ARG, "need 0 < decay <= 1, 0 <= prior_accept <= 1, prior_weight > 0");
  if (!(cfg->cost_fixed_ms >= 0.f) || !(cfg->cost_per_row_ms >= 0.f) || !(cfg->cost_per_request_ms >= 0.f) ||
      !(cfg->cost_fixed_ms + cfg->cost_per_row_ms + cfg->cost_per_request_ms > 0.f))
    return set_error(DFLASH_ERR_INVALID_ARG, "costs must be non-negative with a positive sum");
  dflash_block_policy* p = new (std::nothrow) dflash_block_policy();
  if (!p) return set_error(DFLASH_ERR_INVALID_ARG, "out of host memory");
  p->cfg = *cfg;
  p->max_pos = cfg->candidates[n - 1] - 1;
  *out = p;
  return DFLASH_OK;
}

int32_t dflash_block_policy_destroy(dflash_block_policy* p) {
  delete p;
  return DFLASH_OK;
}

int32_t dflash_block_policy_observe(dflash_block_policy* p, int32_t block_size, const int32_t* accept_len_host,
                                    int32_t batch) {
  if (!p || batch < 0 || (batch > 0 && !accept_len_host))
    return set_error(DFLASH_ERR_INVALID_ARG, "policy or accept_len_host is NULL, or batch < 0");
  if (block_size < 1 || block_size > p->max_pos + 1)
    return set_error(DFLASH_ERR_SHAPE, "block_size outside [1, largest candidate]");
  for (int b = 0; b < batch; ++b)
    if (accept_len_host[b] < 1 || accept_len_host[b] > block_size)
      return set_error(DFLASH_ERR_INVALID_ARG, "an accepted length lies outside [1, block_size]");
  const double d = p->cfg.decay;
  for (int j = 0; j < p->max_pos; ++j) {
    p->kept[j] *= d;
    p->tried[j] *= d;
  }
  for (int b = 0; b < batch; ++b) {
    const int n = accept_len_host[b] - 1;   // drafts kept
    // positions 1 .. min(n + 1, block - 1) were attempted, 1 .. n kept
    const int attempted = std::min(n + 1, block_size - 1);
    for (int j = 0; j < attempted; ++j) p->tried[j] += 1.0;
    for (int j = 0; j < n; ++j) p->kept[j] += 1.0;
  }
  return DFLASH_OK;
}

int32_t dflash_block_policy_choose(const dflash_block_policy* p, int32_t batch, int32_t* block_size_out,
                                   double* expected_tau_out) {
  if (!p || !block_size_out || batch < 1)
    return set_error(DFLASH_ERR_INVALID_ARG, "policy or block_size_out is NULL, or batch < 1");
  const dflash_block_policy_config& c = p->cfg;
  double best = -1.0, best_e = 1.0;
  int best_g = c.candidates[0];
  for (int i = 0; i < c.n_candidates; ++i) {
    const int g = c.candidates[i];
    const double e = expected_tau(p, g);
    const double cost = (double)c.cost_fixed_ms + (double)c.cost_per_row_ms * batch * g +
                        (double)c.cost_per_request_ms * batch;
    const double score = batch * e / cost;
    if (score > best) {
      best = score;
      best_g = g;
      best_e = e;
    }
  }
  *block_size_out = best_g;
  if (expected_tau_out) *expected_tau_out = best_e;
  return DFLASH_OK;
}

int32_t dflash_block_policy_acceptance(const dflash_block_policy* p, double* alpha_out, int32_t n) {
  if (!p || !alpha_out || n < 0) return set_error(DFLASH_ERR_INVALID_ARG, "policy or alpha_out is NULL, or n < 0");
  for (int j = 0; j < n; ++j) alpha_out[j] = j < p->max_pos ? alpha_at(p, j) : 0.0;
  return DFLASH_OK;
}

}  // extern "C"
