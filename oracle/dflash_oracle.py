"""CPU oracle for one DFlash draft cycle — TEST INFRASTRUCTURE, not a product path.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may import this module.  It is a plain, slow, float64 numpy restatement of what
the DFlash drafter computes, written from the method's description so that a
reader can check each function against it by eye:

* "DFlash: Block Diffusion for Flash Speculative Decoding" (paper), §3.1 (accepted
  length tau in [1, gamma+1]), §4.1 (persistent context K/V in the draft KV cache),
  §4.2 (anchor + masked block, block_size - 1 predictions, shared frozen
  embedding and LM head), §7.3 (fusion equation for H_t and the K/V injection
  equations for layer i).
* The companion explainer page "DFlash: Block Diffusion for Flash Speculative
  Decoding" (zhongzhoutan-coder.github.io), sections "The Target Verifier Remains
  the Correctness Anchor" (lossless acceptance rule, stop at first rejection,
  worked example), "Target Hidden States Supply the Missing Context" (fusion
  equation) and "Putting It Together" (one cycle, steps 1-5).
* The blog page "Inside DFlash & Block Diffusion Speculative Decoding"
  (abrarakhunji.com), section "2. Non-Causal Block Diffusion Denoising
  Objective" (case definition of the non-causal mask and its 4+4 printed
  matrix) and section "1. Arithmetic Intensity & Speculative Speedup" (E[L]).

Where those pages leave a step open (RoPE pairing, norm epsilon, final norm,
which rows get drafts, argmax ties) the reading taken is stated in the
function's docstring.  Every floating-point step is float64; matrices are
[out_features, in_features] and are converted to float64 in row chunks so that
8B-shaped weights fit in host memory — each output element is still one
complete dot product, unchanged by the chunking.

Pins (tests/test_oracle_pins.py) tie each function to something other than
itself: the printed mask matrix, the worked verification example, exhaustive
brute force, the E[L] closed form by Monte Carlo, complex-number RoPE, library
scaled-dot-product attention, invariants and special cases; the stochastic
verification (verify_sampled) to the losslessness of speculative sampling
(the first emitted token follows the target's distribution), the acceptance
overlap sum_x min(p_t, p_d), its greedy limit and its special cases.  The end-to-end
drafter logits have no printed values on the pages: beyond the component pins
and the special cases in the tests, that composition is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

F64 = np.float64
_CHUNK_ELEMS = 1 << 25


def _f64(a) -> np.ndarray:
    """float64 copy of a numpy array or a host torch tensor (conversion only)."""
    if hasattr(a, "detach"):
        return a.detach().to("cpu").float().numpy().astype(F64)
    return np.asarray(a, dtype=F64)


# Tensor classes the storage study can round one at a time (see `store`).
STORE_CLASSES = ("ht", "kv", "u", "qkv", "attn_out", "ffn_act", "h")


def store(x: np.ndarray, mode="f64", cls: str = "") -> np.ndarray:
    """Round values to the storage type a drafter keeps its activations in.

    "f64": no rounding (the exact definition).  "fp32": round to float32.
    "bf16": round to float32, then to bfloat16 (round to nearest, ties to
    even, on the upper 16 bits) — a bf16 drafter keeps every tensor handed
    from one step to the next in bf16 while accumulating in float32.  The
    result is returned as float64.  `mode` may also map tensor classes
    (STORE_CLASSES: the fused context H_t, the cached context K/V, the normed
    projection inputs, block Q/K/V, the attention output, the SwiGLU product,
    the final h) to modes, the rest staying exact: the per-tensor study.
    """
    if isinstance(mode, dict):
        mode = mode.get(cls, "f64")
    if mode == "f64":
        return x
    f = np.asarray(x, dtype=np.float32)
    if mode == "fp32":
        return f.astype(F64)
    if mode != "bf16":
        raise ValueError(mode)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(F64)


# ---------------------------------------------------------------------------
# Small building blocks
# ---------------------------------------------------------------------------

def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x W^T in float64 for W stored [out, in] (any float dtype).

    W is upcast in chunks of output rows; each output column is the full dot
    product of x with one row of W.
    """
    x = np.asarray(x, dtype=F64)
    out = np.empty(x.shape[:-1] + (w.shape[0],), dtype=F64)
    step = max(1, _CHUNK_ELEMS // max(1, w.shape[1]))
    for r0 in range(0, w.shape[0], step):
        r1 = min(r0 + step, w.shape[0])
        out[..., r0:r1] = x @ _f64(w[r0:r1]).T
    return out


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: g * x / sqrt(mean(x^2) + eps).

    The paper applies RMSNorm to the fused context (§7.3, H_t equation); the
    Qwen3-style drafter layers use the same norm before attention and before
    the FFN, and once more before the LM head (reading: a final norm is taken,
    as in the Qwen3 decoder the drafter is shaped after).
    """
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(g)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def rope(x: np.ndarray, positions: Sequence[int], theta: float) -> np.ndarray:
    """Rotary position embedding, rotate-half pairing.

    x: [n, heads, hd]; positions: [n].  Element i of the first half pairs with
    element i + hd/2; the pair turns by angle pos * theta^(-2i/hd).  (The pages
    call the drafter Qwen3-style but do not spell RoPE out; this is the pairing
    Qwen3 uses.)
    """
    x = np.asarray(x, dtype=F64)
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = np.power(F64(theta), -2.0 * np.arange(half, dtype=F64) / hd)
    ang = np.asarray(positions, dtype=F64)[:, None] * inv_freq[None, :]      # [n, half]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


# ---------------------------------------------------------------------------
# Stage 1: context fusion  (paper §7.3; explainer "Target Hidden States ...")
# ---------------------------------------------------------------------------

def fuse_context(feats: np.ndarray, w_c: np.ndarray, g_c: np.ndarray, eps: float, mode: str = "f64") -> np.ndarray:
    """H_t = RMSNorm(W_c [H^(l1); ...; H^(lm)]) for every new context token.

    feats: [n, m, D], the hidden state of token j at each of the m selected
    target layers; the m vectors are concatenated along features in layer order
    to a length-mD vector, projected by W_c [D, mD] and normalised.
    """
    feats = _f64(feats)
    n = feats.shape[0]
    x = feats.reshape(n, -1)                     # [n, m*D]: [H^(l1)_j ; ... ; H^(lm)_j]
    return store(rms_norm(linear(x, w_c), g_c, eps), mode, "ht")


# ---------------------------------------------------------------------------
# Stage 2: K/V injection into every draft layer  (paper §7.3, §4.1)
# ---------------------------------------------------------------------------

def inject_kv(h_t: np.ndarray, w_k: np.ndarray, w_v: np.ndarray, positions: Sequence[int],
              n_kv_heads: int, head_dim: int, theta: float, mode: str = "f64", g_k=None, eps: float = 1e-6):
    """Context keys and values of one draft layer: W^K H_t and W^V H_t.

    Only keys get the rotary embedding; a context token j injected for a
    request holding c tokens sits at absolute position c + j (reading: context
    positions count from 0 and the block continues after them).  No per-layer
    norm is applied to H_t — the equation feeds H_t straight into W^K, W^V.
    With a QK-norm gain g_k (a Qwen3 option the pages do not mention; reading:
    it belongs to the layer's key path, so context keys get it like block
    keys) each key head is RMS-normalised over head_dim and scaled by g_k
    before RoPE.  Returns K, V as [n, n_kv_heads, head_dim].
    """
    n = h_t.shape[0]
    k = linear(h_t, w_k).reshape(n, n_kv_heads, head_dim)
    if g_k is not None:
        k = rms_norm(k, g_k, eps)
    v = linear(h_t, w_v).reshape(n, n_kv_heads, head_dim)
    return store(rope(k, positions, theta), mode, "kv"), store(v, mode, "kv")


class RequestCache:
    """Persistent context K/V of one request for every draft layer (§4.1:
    "stored in the draft model's KV cache and reused across drafting
    iterations").  Only context entries live here; block K/V never does."""

    def __init__(self, layers: int, n_kv_heads: int, head_dim: int):
        self.k: List[np.ndarray] = [np.zeros((0, n_kv_heads, head_dim)) for _ in range(layers)]
        self.v: List[np.ndarray] = [np.zeros((0, n_kv_heads, head_dim)) for _ in range(layers)]

    @property
    def length(self) -> int:
        return self.k[0].shape[0]


def inject_context(weights: Dict, cfg, cache: RequestCache, feats: np.ndarray, mode: str = "f64") -> np.ndarray:
    """Stages 1+2 for one request: fuse the new tokens' target features and
    append their K/V to every layer of the cache.  Returns H_t.  `mode` is the
    storage rounding of H_t and of the cached K/V (see `store`).  With
    cfg.input_fusion the ablation path inject_context_input_fusion runs."""
    if getattr(cfg, "input_fusion", False):
        return inject_context_input_fusion(weights, cfg, cache, feats, mode)
    h_t = fuse_context(feats, weights["w_c"], weights["g_c"], cfg.rms_eps, mode)
    c = cache.length
    pos = np.arange(c, c + h_t.shape[0])
    qk = getattr(cfg, "qk_norm", False)
    for i, lw in enumerate(weights["layers"]):
        k, v = inject_kv(h_t, lw["w_k"], lw["w_v"], pos, cfg.n_kv_heads, cfg.head_dim, cfg.rope_theta, mode,
                         g_k=lw["g_k"] if qk else None, eps=cfg.rms_eps)
        cache.k[i] = np.concatenate([cache.k[i], k], axis=0)
        cache.v[i] = np.concatenate([cache.v[i], v], axis=0)
    return h_t


def inject_context_input_fusion(weights: Dict, cfg, cache: RequestCache, feats: np.ndarray,
                                mode="f64") -> np.ndarray:
    """The input-fusion ablation (paper §5.5.5, against KV injection; explainer
    "Per-Layer K/V Injection Prevents Context Dilution": with input fusion the
    target context enters only at the first layer).  Reading: the new context
    tokens' layer-0 hidden states are H_t itself (no extra weights), and every
    draft layer processes them like sequence positions, causally among the
    context (the DFlash mask's context rows, j <= i); layer i's context keys
    and values are that layer's own projections of its context hidden states.
    Earlier context rows never see later ones, so the per-layer K/V of the
    context can be cached and extended: this function appends the new rows'
    K/V of every layer to the cache.  Drafting is unchanged (draft_forward).
    draft_forward_full_sequence is the same computation without a cache.
    `mode` rounds the cached K/V (storage class "kv", see `store`) before the
    context rows' own attention reads them, as the cache holds them."""
    h_t = fuse_context(feats, weights["w_c"], weights["g_c"], cfg.rms_eps)
    D, nq, nkv, hd = cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    c, n = cache.length, h_t.shape[0]
    pos = np.arange(c, c + n)
    rows = dflash_mask(c + n, 0)[c:, :]                          # causal context rows over keys 0..c+n-1
    x = h_t.copy()
    for i, lw in enumerate(weights["layers"]):
        u = rms_norm(x, lw["g_in"], cfg.rms_eps)
        q = linear(u, lw["w_q"]).reshape(n, nq, hd)
        k = linear(u, lw["w_k"]).reshape(n, nkv, hd)
        if getattr(cfg, "qk_norm", False):
            q = rms_norm(q, lw["g_q"], cfg.rms_eps)
            k = rms_norm(k, lw["g_k"], cfg.rms_eps)
        q, k = rope(q, pos, cfg.rope_theta), rope(k, pos, cfg.rope_theta)
        v = linear(u, lw["w_v"]).reshape(n, nkv, hd)
        cache.k[i] = np.concatenate([cache.k[i], store(k, mode, "kv")], axis=0)
        cache.v[i] = np.concatenate([cache.v[i], store(v, mode, "kv")], axis=0)
        o = attention_masked(q, cache.k[i], cache.v[i], rows)
        x = x + linear(o.reshape(n, nq * hd), lw["w_o"])
        u = rms_norm(x, lw["g_post"], cfg.rms_eps)
        x = x + linear(silu(linear(u, lw["w_g"])) * linear(u, lw["w_u"]), lw["w_d"])
    return h_t


# ---------------------------------------------------------------------------
# The non-causal DFlash mask  (blog, "2. Non-Causal Block Diffusion ...")
# ---------------------------------------------------------------------------

def dflash_mask(t: int, K: int) -> np.ndarray:
    """M[i, j] over the sequence [c_1..c_t ; m_1..m_K], 1-indexed as printed.

    Block rows (t < i <= t+K) see every context position (j <= t) and every
    block position (t < j <= t+K).  Context rows carry the "causal context"
    case: j <= i.  (The case list writes "j <= t" for the context case without
    a condition on i; the printed 4+4 matrix and the case's own label make the
    context rows causal.  Context rows are never drafter queries — target
    features bypass the Q projection — so only block rows reach the drafter.)
    """
    n = t + K
    M = np.zeros((n, n), dtype=np.int64)
    for i in range(1, n + 1):
        for j in range(1, n + 1):
            if i <= t:
                M[i - 1, j - 1] = 1 if j <= i else 0
            elif j <= t:
                M[i - 1, j - 1] = 1
            elif t < j <= t + K:
                M[i - 1, j - 1] = 1
    return M


# ---------------------------------------------------------------------------
# Stage 3: drafter forward over [anchor, mask x (block-1)]
# ---------------------------------------------------------------------------

def attention_masked(q: np.ndarray, k_all: np.ndarray, v_all: np.ndarray, mask_rows: np.ndarray) -> np.ndarray:
    """Softmax attention of the block queries through an explicit mask.

    q: [g, nq, hd] (block rows); k_all, v_all: [t+g, nkv, hd] = [context ; block];
    mask_rows: [g, t+g], the block rows of the DFlash mask.  Scale 1/sqrt(hd),
    no bias; query head h reads kv head h // (nq / nkv) (grouped-query).
    """
    g, nq, hd = q.shape
    nkv = k_all.shape[1]
    group = nq // nkv
    out = np.zeros((g, nq, hd), dtype=F64)
    scale = 1.0 / math.sqrt(hd)
    allowed = mask_rows.astype(bool)
    for h in range(nq):
        kh = k_all[:, h // group, :]
        vh = v_all[:, h // group, :]
        s = (q[:, h, :] @ kh.T) * scale                      # [g, t+g]
        s = np.where(allowed, s, -np.inf)
        s = s - np.max(s, axis=1, keepdims=True)
        p = np.exp(s)
        p = p / np.sum(p, axis=1, keepdims=True)
        out[:, h, :] = p @ vh
    return out


def attention_block(q: np.ndarray, k_ctx: np.ndarray, v_ctx: np.ndarray,
                    k_blk: np.ndarray, v_blk: np.ndarray) -> np.ndarray:
    """Block queries against every context key and every block key, no mask:
    the form the DFlash mask reduces to for block rows."""
    k_all = np.concatenate([k_ctx, k_blk], axis=0)
    v_all = np.concatenate([v_ctx, v_blk], axis=0)
    return attention_masked(q, k_all, v_all, np.ones((q.shape[0], k_all.shape[0]), dtype=np.int64))


def draft_forward(weights: Dict, cfg, cache: RequestCache, anchor: int, block: int,
                  use_mask: bool = True, mode: str = "f64") -> Dict[str, np.ndarray]:
    """One non-causal drafter pass over [anchor, mask, ..., mask] (block rows).

    Per layer i (Qwen3-style): u = RMSNorm(x); Q = W^Q u, K = W^K u, V = W^V u
    with RoPE on Q and K at positions c..c+block-1; the block keys/values are
    appended after the layer's injected context K/V (paper §7.3: K_i =
    [W^K H_t ; W^K H_d], V_i likewise); attention through the DFlash mask;
    x += W^O o; u = RMSNorm(x); x += W^D (silu(W^G u) * W^U u).  After the
    last layer h = RMSNorm_final(x).  The block's own K/V is not kept.
    `mode` rounds every tensor handed from one step to the next (normed
    inputs, Q/K/V, attention output, SwiGLU product, h) to a storage type; the
    residual stream x stays exact.  With cfg.qk_norm, every query and key head
    is RMS-normalised over head_dim and scaled by the layer's g_q / g_k before
    RoPE (Qwen3's q_norm / k_norm).
    """
    D, nq, nkv, hd = cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    c = cache.length
    tokens = [int(anchor)] + [cfg.mask_id] * (block - 1)
    x = _f64(weights["embed"][tokens])                             # shared embedding rows
    pos = np.arange(c, c + block)
    mask_rows = dflash_mask(c, block)[c:, :]                       # block rows only
    for i, lw in enumerate(weights["layers"]):
        u = store(rms_norm(x, lw["g_in"], cfg.rms_eps), mode, "u")
        q = linear(u, lw["w_q"]).reshape(block, nq, hd)
        k = linear(u, lw["w_k"]).reshape(block, nkv, hd)
        if getattr(cfg, "qk_norm", False):
            q = rms_norm(q, lw["g_q"], cfg.rms_eps)
            k = rms_norm(k, lw["g_k"], cfg.rms_eps)
        q = store(rope(q, pos, cfg.rope_theta), mode, "qkv")
        k = store(rope(k, pos, cfg.rope_theta), mode, "qkv")
        v = store(linear(u, lw["w_v"]).reshape(block, nkv, hd), mode, "qkv")
        if use_mask:
            o = attention_masked(q, np.concatenate([cache.k[i], k]), np.concatenate([cache.v[i], v]), mask_rows)
        else:
            o = attention_block(q, cache.k[i], cache.v[i], k, v)
        x = x + linear(store(o, mode, "attn_out").reshape(block, nq * hd), lw["w_o"])
        u = store(rms_norm(x, lw["g_post"], cfg.rms_eps), mode, "u")
        x = x + linear(store(silu(linear(u, lw["w_g"])) * linear(u, lw["w_u"]), mode, "ffn_act"), lw["w_d"])
    h = store(rms_norm(x, weights["g_final"], cfg.rms_eps), mode, "h")
    return {"h": h}


def draft_forward_full_sequence(weights: Dict, cfg, ctx_feats: np.ndarray, anchor: int, block: int) -> Dict:
    """The input-fusion drafter written out over the whole sequence, with no
    cache: x = [H_t of every context token ; E[anchor, mask, ..]]; every layer
    processes every position under the full DFlash mask (context rows causal,
    block rows see all context and the whole block); h = RMSNorm_final of the
    block rows.  Equal to inject_context_input_fusion + draft_forward."""
    D, nq, nkv, hd = cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    h_t = fuse_context(ctx_feats, weights["w_c"], weights["g_c"], cfg.rms_eps)
    c = h_t.shape[0]
    tokens = [int(anchor)] + [cfg.mask_id] * (block - 1)
    x = np.concatenate([h_t, _f64(weights["embed"][tokens])], axis=0)
    n = c + block
    pos = np.arange(n)
    M = dflash_mask(c, block)
    for lw in weights["layers"]:
        u = rms_norm(x, lw["g_in"], cfg.rms_eps)
        q = linear(u, lw["w_q"]).reshape(n, nq, hd)
        k = linear(u, lw["w_k"]).reshape(n, nkv, hd)
        if getattr(cfg, "qk_norm", False):
            q = rms_norm(q, lw["g_q"], cfg.rms_eps)
            k = rms_norm(k, lw["g_k"], cfg.rms_eps)
        q, k = rope(q, pos, cfg.rope_theta), rope(k, pos, cfg.rope_theta)
        v = linear(u, lw["w_v"]).reshape(n, nkv, hd)
        o = attention_masked(q, k, v, M)
        x = x + linear(o.reshape(n, nq * hd), lw["w_o"])
        u = rms_norm(x, lw["g_post"], cfg.rms_eps)
        x = x + linear(silu(linear(u, lw["w_g"])) * linear(u, lw["w_u"]), lw["w_d"])
    return {"h": rms_norm(x[c:], weights["g_final"], cfg.rms_eps)}


# ---------------------------------------------------------------------------
# Stage 4: shared LM head + argmax  (paper §4.2 shared head; explainer step 3)
# ---------------------------------------------------------------------------

def lm_head_argmax(h_rows: np.ndarray, lm_head: np.ndarray):
    """logits = h W_lm^T for the mask rows; draft = argmax, lowest index on ties.

    Reading: the anchor row's output is not a draft; rows 1..block-1 give the
    block_size - 1 predictions (paper §4.2)."""
    logits = linear(h_rows, lm_head)
    drafts = np.argmax(logits, axis=-1).astype(np.int64)   # first occurrence of the maximum
    return logits, drafts


# ---------------------------------------------------------------------------
# Stage 5: greedy verification  (explainer, "The Target Verifier ...")
# ---------------------------------------------------------------------------

def verify_greedy(drafts: Sequence[int], target: Sequence[int]):
    """Greedy lossless verification of one block.

    drafts d_1..d_{g-1}; target y_0..y_{g-1} where y_k is the target's greedy
    token after block position k (y_0 judges d_1).  Walk left to right and stop
    at the first rejection; n = number of accepted drafts, tau = n + 1, the
    emitted tokens are d_1..d_n followed by y_n (the correction, or the bonus
    when every draft survives).  Returns (tau, out[g] padded with -1,
    next_anchor = y_n).
    """
    g = len(target)
    n = 0
    while n < len(drafts) and int(drafts[n]) == int(target[n]):
        n += 1
    out = [int(d) for d in drafts[:n]] + [int(target[n])]
    out = out + [-1] * (g - len(out))
    return n + 1, out, int(target[n])


def softmax(logits: np.ndarray, temperature: float = 1.0) -> np.ndarray:
    """The distribution a row of logits stands for at a sampling temperature:
    p_v = exp(l_v / T) / sum_w exp(l_w / T), in float64, over the last axis.
    (The pages sample at temperature 1; T scales the logits before the
    normalisation, the usual reading.)  The largest logit is subtracted first,
    which changes nothing mathematically and keeps exp finite."""
    z = np.asarray(logits, dtype=F64) / F64(temperature)
    z = z - np.max(z, axis=-1, keepdims=True)
    e = np.exp(z)
    return e / np.sum(e, axis=-1, keepdims=True)


def sample_inverse_cdf(p: np.ndarray, u: float) -> int:
    """The token a single uniform u in [0, 1) draws from distribution p: the
    smallest id whose cumulative probability (ids in increasing order) exceeds
    u; rounding that leaves u beyond the total falls back to the last id with
    non-zero probability."""
    p = np.asarray(p, dtype=F64)
    c = np.cumsum(p)
    idx = int(np.searchsorted(c, u, side="right"))   # c[idx] > u >= c[idx-1]: p[idx] > 0
    if idx >= len(p):
        idx = int(np.nonzero(p > 0.0)[0][-1])
    return idx


def verify_sampled(drafts: Sequence[int], p_draft: np.ndarray, p_target: np.ndarray,
                   u_accept: Sequence[float], u_sample: float):
    """Stochastic lossless verification of one block (explainer, "The Target
    Verifier Remains the Correctness Anchor").

    drafts d_1..d_n (n = block_size - 1), d_k drawn from the drafter's
    distribution p_draft[k-1] ([n, V]); p_target [n+1, V], row k the target's
    distribution for the token after block position k (row 0 judges d_1, as in
    verify_greedy; row n gives the bonus).  Left to right, d_k is accepted iff
    u_accept[k-1] < min(1, p_t(d_k) / p_d(d_k)); at the first rejection the
    target draws a correction from its residual distribution and the rest of
    the block is dropped; if every draft survives the target draws a bonus
    token from p_target[n].  Reading of "residual distribution": the standard
    one of lossless speculative sampling, max(0, p_t - p_d) normalised.  The
    draw uses one uniform u_sample (sample_inverse_cdf).  The uniforms are
    inputs.  Returns (tau, out[n+1] padded with -1, next_anchor) like
    verify_greedy.
    """
    n = len(drafts)
    p_draft, p_target = np.asarray(p_draft, dtype=F64), np.asarray(p_target, dtype=F64)
    for k in range(n):
        d = int(drafts[k])
        pt, pd = p_target[k, d], p_draft[k, d]
        accept = 1.0 if pd <= 0.0 else min(1.0, pt / pd)
        if u_accept[k] < accept:
            continue
        resid = np.maximum(p_target[k] - p_draft[k], 0.0)
        tok = sample_inverse_cdf(resid / resid.sum(), u_sample)
        out = [int(x) for x in drafts[:k]] + [tok]
        return k + 1, out + [-1] * (n + 1 - len(out)), tok
    tok = sample_inverse_cdf(p_target[n], u_sample)
    return n + 1, [int(x) for x in drafts] + [tok], tok


def expected_accept_len(alpha: Sequence[float]) -> float:
    """E[L] = 1 + sum_i prod_{j<=i} alpha_j (blog, section 1), alpha_j the
    probability that draft j is accepted given the ones before it were."""
    total, prod = 1.0, 1.0
    for a in alpha:
        prod *= a
        total += prod
    return total


# ---------------------------------------------------------------------------
# Training-time packed block attention  (paper §4.2 "all blocks are
# concatenated into a single sequence and processed jointly using a sparse
# attention mask"; explainer "Training Rehearses the Same Masked Blocks Used
# at Runtime" and its Figure 4)
# ---------------------------------------------------------------------------

def packed_block_mask(seq_len: int, anchors: Sequence[int], block: int) -> np.ndarray:
    """M[r, j] over keys [context positions 0..seq_len-1 ; block rows of every
    block], for the query rows r of every block (block n's rows are n*block ..
    n*block + block - 1).  A row of block n sees context position j iff
    j < a_n (the clean target features before its anchor: the anchor itself is
    the block's first row, as at inference, where the block starts right after
    the injected context), every row of its own block (bidirectional), and no
    row of another block.  Built element by element from those cases."""
    N = len(anchors)
    M = np.zeros((N * block, seq_len + N * block), dtype=np.int64)
    for n, a in enumerate(anchors):
        for i in range(block):
            r = n * block + i
            for j in range(seq_len):
                if j < a:
                    M[r, j] = 1
            for m in range(N):
                for l in range(block):
                    if m == n:
                        M[r, seq_len + m * block + l] = 1
    return M


def attention_packed(q: np.ndarray, k_ctx: np.ndarray, v_ctx: np.ndarray, k_blk: np.ndarray, v_blk: np.ndarray,
                     anchors: Sequence[int]) -> np.ndarray:
    """Forward attention of the packed training sequence: q [N*block, nq, hd]
    (every block's rows, RoPE applied), k_ctx / v_ctx [S, nkv, hd] (the
    sequence's injected context keys / values), k_blk / v_blk [N*block, nkv,
    hd] (the blocks' own keys / values), through packed_block_mask; scale
    1/sqrt(hd), grouped-query heads as in attention_masked."""
    N, S = len(anchors), k_ctx.shape[0]
    block = q.shape[0] // N
    mask = packed_block_mask(S, anchors, block)
    return attention_masked(np.asarray(q, dtype=F64), np.concatenate([k_ctx, k_blk]).astype(F64),
                            np.concatenate([v_ctx, v_blk]).astype(F64), mask)


# ---------------------------------------------------------------------------
# Block-size scheduling  (paper §5.5.4: a drafter trained at a large block
# size serves smaller ones about as well, which allows choosing the block size
# per cycle; large blocks cost more verification when compute-bound)
# ---------------------------------------------------------------------------

def acceptance_update(accepts: np.ndarray, attempts: np.ndarray, block: int, taus: Sequence[int],
                      decay: float):
    """Per-position acceptance counts after one cycle of blocks of size
    `block` with accepted lengths `taus` (one per request).  Draft position j
    (1-based) of a block is attempted when every draft before it was kept and
    j <= block - 1, and kept when j <= tau - 1.  Older counts are first
    multiplied by `decay` (forgetting factor per cycle).  Returns new arrays."""
    accepts = np.asarray(accepts, dtype=F64) * decay
    attempts = np.asarray(attempts, dtype=F64) * decay
    for tau in taus:
        n = int(tau) - 1                      # drafts kept
        for j in range(1, block):
            if j <= n + 1:
                attempts[j - 1] += 1.0
            if j <= n:
                accepts[j - 1] += 1.0
    return accepts, attempts


def acceptance_estimate(accepts: np.ndarray, attempts: np.ndarray, prior: float, weight: float) -> np.ndarray:
    """alpha_j = P(draft j kept | drafts before it kept), estimated from the
    counts with `weight` pseudo-observations of the prior probability."""
    return (np.asarray(accepts, dtype=F64) + prior * weight) / (np.asarray(attempts, dtype=F64) + weight)


def choose_block(candidates: Sequence[int], alpha: Sequence[float], batch: int, cost_fixed: float,
                 cost_per_row: float, cost_per_request: float):
    """The block size that maximises expected accepted tokens per unit of
    cycle cost: E[tau | g] = expected_accept_len(alpha_1 .. alpha_{g-1}) per
    request, cycle cost = cost_fixed + cost_per_row * batch * g +
    cost_per_request * batch (a linear model of drafting plus verifying
    batch * g token rows).  Ties go to the smaller block.  Returns (g, E[tau])."""
    best = None
    for g in sorted(candidates):
        e = expected_accept_len(list(alpha[:g - 1]))
        score = batch * e / (cost_fixed + cost_per_row * batch * g + cost_per_request * batch)
        if best is None or score > best[0]:
            best = (score, g, e)
    return best[1], best[2]


# ---------------------------------------------------------------------------
# One whole cycle for one request
# ---------------------------------------------------------------------------

def draft_cycle(weights: Dict, cfg, cache: RequestCache, new_feats: Optional[np.ndarray], anchor: int,
                block: int, use_mask: bool = True, mode: str = "f64") -> Dict[str, np.ndarray]:
    """inject(new tokens) -> draft forward -> LM head + argmax for one request."""
    if new_feats is not None and new_feats.shape[0] > 0:
        inject_context(weights, cfg, cache, new_feats, mode)
    fw = draft_forward(weights, cfg, cache, anchor, block, use_mask=use_mask, mode=mode)
    logits, drafts = lm_head_argmax(fw["h"][1:], weights["lm_head"])
    return {"h": fw["h"], "logits": logits, "drafts": drafts}


def weights_to_host(w: Dict) -> Dict:
    """Host copies of a weight dict of torch tensors, dtype kept (bf16 stays
    bf16; every oracle step upcasts what it reads to float64)."""
    def conv(t):
        return t.detach().to("cpu")
    out = {k: conv(v) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: conv(v) for k, v in lw.items()} for lw in w["layers"]]
    return out


def weights_to_numpy(w: Dict) -> Dict:
    """Host float32 copies of a weight dict whose leaves are torch tensors
    (bf16 values are exact in float32).  Conversion only."""
    def conv(t):
        return t.detach().to("cpu").float().numpy()
    out = {k: conv(v) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: conv(v) for k, v in lw.items()} for lw in w["layers"]]
    return out
