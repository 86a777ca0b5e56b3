"""GB300 (sm_103a) DFlash draft cycle: thin Python binding over the C ABI.

The functions below carry the C ABI's names and only marshal arguments (torch
tensors -> device pointers, the current torch stream -> cudaStream_t); every
step of the cycle — context fusion, K/V injection, the non-causal drafter
pass, the LM head argmax and greedy verification — runs in the CUDA library
``libdflash_gb300.so`` built from ``csrc/``.  There is no CPU fallback: if the
library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _abi
from ._abi import DFlashError, check, lib

__all__ = ["DFlashError", "Model", "Cache", "lib", "dflash_model_create", "dflash_cache_init",
           "dflash_workspace_bytes", "dflash_workspace", "dflash_inject_context", "dflash_draft_block",
           "dflash_verify_greedy", "dflash_draft_cycle", "dflash_get_status", "dflash_clear_status", "dflash_version",
           "dflash_launch_count", "dflash_profile_start", "dflash_profile_stop", "dflash_inject_context_noalloc",
           "dflash_selftest_wait_timeout", "dflash_sampling_workspace", "dflash_verify_sampled", "dflash_sample_tokens",
           "BlockPolicy", "dflash_packed_attention_workspace", "dflash_packed_block_attention",
           "dflash_packed_attention_status"]


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _config_struct(cfg) -> _abi.Config:
    mask = cfg.mask_id if hasattr(cfg, "mask_id") else cfg.mask_token_id
    return _abi.Config(hidden=cfg.hidden, layers=cfg.layers, n_q_heads=cfg.n_q_heads, n_kv_heads=cfg.n_kv_heads,
                       head_dim=cfg.head_dim, ffn=cfg.ffn, vocab=cfg.vocab, n_target_feats=cfg.n_target_feats,
                       max_block=cfg.max_block, rope_theta=float(cfg.rope_theta), rms_eps=float(cfg.rms_eps),
                       mask_token_id=int(mask), dtype=_abi.DTYPE_F32 if cfg.dtype == "fp32" else _abi.DTYPE_BF16,
                       qk_norm=1 if getattr(cfg, "qk_norm", False) else 0,
                       input_fusion=1 if getattr(cfg, "input_fusion", False) else 0,
                       kv_bf16=1 if getattr(cfg, "kv_bf16", False) else 0,
                       head_bf16=1 if getattr(cfg, "head_bf16", False) else 0)


def dflash_version() -> int:
    return lib().dflash_version()


class Model:
    """A created dflash_model; keeps the borrowed weight tensors alive."""

    def __init__(self, cfg, weights: dict):
        self.cfg = cfg
        self.weights = weights
        self.dtype = torch.float32 if cfg.dtype == "fp32" else torch.bfloat16
        tensors = [weights[k] for k in ("embed", "lm_head", "w_c", "g_c", "g_final")]
        for lw in weights["layers"]:
            tensors += list(lw.values())
        for t in tensors:
            if t.dtype != self.dtype or not t.is_cuda or not t.is_contiguous():
                raise ValueError("weights must be contiguous CUDA tensors of the model dtype")
        self._layers = (_abi.LayerWeights * cfg.layers)(*[
            _abi.LayerWeights(**{k: (lw[k].data_ptr() if k in lw else None)
                                 for k in ("g_in", "w_q", "w_k", "w_v", "w_o", "g_post", "w_g", "w_u", "w_d", "g_q",
                                           "g_k")})
            for lw in weights["layers"]])
        w = _abi.Weights(embed=weights["embed"].data_ptr(), lm_head=weights["lm_head"].data_ptr(),
                         w_c=weights["w_c"].data_ptr(), g_c=weights["g_c"].data_ptr(),
                         g_final=weights["g_final"].data_ptr(), layers=self._layers)
        self._cfg = _config_struct(cfg)
        h = ctypes.c_void_p()
        check(lib().dflash_model_create(ctypes.byref(self._cfg), ctypes.byref(w), ctypes.byref(h)),
              "dflash_model_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            lib().dflash_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Cache:
    """A dflash_cache carved out of a torch-owned device buffer."""

    def __init__(self, model: Model, batch: int, capacity: int, stream=None):
        self.model, self.batch, self.capacity = model, batch, capacity
        nbytes = lib().dflash_cache_bytes(ctypes.byref(model._cfg), batch, capacity)
        if nbytes == 0:
            raise ValueError("invalid cache shape")
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        h = ctypes.c_void_p()
        check(lib().dflash_cache_init(model.handle, self.buffer.data_ptr(), nbytes, batch, capacity,
                                      _stream_ptr(stream), ctypes.byref(h)), "dflash_cache_init")
        self.handle = h
        k, v, ln = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
        check(lib().dflash_cache_layout(h, ctypes.byref(k), ctypes.byref(v), ctypes.byref(ln)), "dflash_cache_layout")
        self.k_off, self.v_off, self.len_off = k.value, v.value, ln.value

    def _kv_view(self, off: int, hd_major: bool = False) -> torch.Tensor:
        c = self.model.cfg
        B, L, H, cap, hd = self.batch, c.layers, c.n_kv_heads, self.capacity, c.head_dim
        if self.model.dtype == torch.float32:
            raw = self.buffer[off:off + B * L * H * cap * hd * 4]
            return raw.view(torch.float32).view(B, L, H, cap, hd)
        P = 1 if getattr(c, "kv_bf16", False) else 2   # bf16 planes of each value
        if hd_major:   # bf16 V: [B][L][H][P][hd][pitch], pitch = capacity rounded up to 8
            pitch = (cap + 7) // 8 * 8
            raw = self.buffer[off:off + B * L * H * P * hd * pitch * 2]
            planes = raw.view(torch.bfloat16).view(B, L, H, P, hd, pitch)[..., :cap].transpose(-1, -2)
        else:
            raw = self.buffer[off:off + B * L * H * P * cap * hd * 2]
            planes = raw.view(torch.bfloat16).view(B, L, H, P, cap, hd)
        return planes.float().sum(dim=3)

    def k(self) -> torch.Tensor:
        """Context keys as fp32 [batch][layers][n_kv_heads][capacity][head_dim]
        (a view for fp32 models; the sum of the bf16 planes otherwise)."""
        return self._kv_view(self.k_off)

    def v(self) -> torch.Tensor:
        """Context values as fp32 [batch][layers][n_kv_heads][capacity][head_dim]
        (bf16 models store them head-dim-major; this returns them position-major)."""
        return self._kv_view(self.v_off, hd_major=True)

    def ctx_len(self) -> torch.Tensor:
        return self.buffer[self.len_off:self.len_off + 4 * self.batch].view(torch.int32)

    def set_lengths(self, lengths, stream=None):
        arr = (ctypes.c_int32 * self.batch)(*[int(v) for v in lengths])
        check(lib().dflash_cache_set_lengths(self.handle, arr, _stream_ptr(stream)), "dflash_cache_set_lengths")

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            lib().dflash_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dflash_model_create(cfg, weights: dict) -> Model:
    return Model(cfg, weights)


def dflash_cache_init(model: Model, batch: int, capacity: int, stream=None) -> Cache:
    return Cache(model, batch, capacity, stream)


def dflash_workspace_bytes(model: Model, batch: int, capacity: int, block_size: int, max_inject_rows: int) -> int:
    return int(lib().dflash_workspace_bytes(model.handle, batch, capacity, block_size, max_inject_rows))


def dflash_workspace(model: Model, batch: int, capacity: int, block_size: int, max_inject_rows: int) -> torch.Tensor:
    n = dflash_workspace_bytes(model, batch, capacity, block_size, max_inject_rows)
    if n == 0:
        raise ValueError("invalid workspace shape")
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def dflash_inject_context(model: Model, cache: Cache, feats: torch.Tensor, n_new_dev: torch.Tensor,
                          n_new_host=None, max_rows: Optional[int] = None, workspace: torch.Tensor = None,
                          stream=None) -> None:
    """feats [max_rows, m, D] (model dtype), n_new_dev int32 [batch] on the device."""
    if n_new_dev.dtype != torch.int32 or feats.dtype != model.dtype:
        raise ValueError("n_new_dev must be int32 and feats of the model dtype")
    rows = feats.shape[0] if max_rows is None else int(max_rows)
    host = None
    if n_new_host is not None:
        host = (ctypes.c_int32 * cache.batch)(*[int(v) for v in n_new_host])
    check(lib().dflash_inject_context(model.handle, cache.handle, _ptr(feats), _ptr(n_new_dev), host, rows,
                                      _ptr(workspace), workspace.numel(), _stream_ptr(stream)),
          "dflash_inject_context")


def dflash_inject_context_noalloc(model: Model, cache: Cache, feats: torch.Tensor, n_new_dev: torch.Tensor,
                                  n_new_host=None, max_rows: Optional[int] = None, stream=None) -> None:
    """dflash_inject_context without a workspace, for callers that cannot
    allocate device memory: the library's fixed static scratch is used."""
    if n_new_dev.dtype != torch.int32 or feats.dtype != model.dtype:
        raise ValueError("n_new_dev must be int32 and feats of the model dtype")
    rows = feats.shape[0] if max_rows is None else int(max_rows)
    host = None
    if n_new_host is not None:
        host = (ctypes.c_int32 * cache.batch)(*[int(v) for v in n_new_host])
    check(lib().dflash_inject_context_noalloc(model.handle, cache.handle, _ptr(feats), _ptr(n_new_dev), host, rows,
                                              _stream_ptr(stream)), "dflash_inject_context_noalloc")


def dflash_draft_block(model: Model, cache: Cache, anchor_dev: torch.Tensor, block_size: int,
                       draft_dev: torch.Tensor, logits_dev: Optional[torch.Tensor] = None,
                       workspace: torch.Tensor = None, stream=None) -> None:
    """anchor_dev int32 [batch]; draft_dev int32 [batch, block-1]; logits_dev fp32 [batch, block-1, V] or None."""
    if anchor_dev.dtype != torch.int32 or draft_dev.dtype != torch.int32:
        raise ValueError("anchor_dev and draft_dev must be int32")
    if logits_dev is not None and logits_dev.dtype != torch.float32:
        raise ValueError("logits_dev must be float32")
    check(lib().dflash_draft_block(model.handle, cache.handle, _ptr(anchor_dev), int(block_size), _ptr(draft_dev),
                                   _ptr(logits_dev), _ptr(workspace), workspace.numel(), _stream_ptr(stream)),
          "dflash_draft_block")


def dflash_draft_cycle(model: Model, cache: Cache, feats: torch.Tensor, n_new_dev: torch.Tensor, anchor_dev: torch.Tensor,
                       block_size: int, draft_dev: torch.Tensor, logits_dev: Optional[torch.Tensor] = None,
                       n_new_host=None, max_rows: Optional[int] = None, workspace: torch.Tensor = None,
                       stream=None) -> None:
    """Injection of feats [max_rows, m, D] (n_new_dev rows per request) then a
    drafter pass of block_size from anchor_dev; one persistent launch when
    both fit it."""
    if n_new_dev.dtype != torch.int32 or anchor_dev.dtype != torch.int32 or draft_dev.dtype != torch.int32:
        raise ValueError("n_new_dev, anchor_dev and draft_dev must be int32")
    if feats.dtype != model.dtype:
        raise ValueError("feats must be of the model dtype")
    rows = feats.shape[0] if max_rows is None else int(max_rows)
    host = None
    if n_new_host is not None:
        host = (ctypes.c_int32 * cache.batch)(*[int(v) for v in n_new_host])
    check(lib().dflash_draft_cycle(model.handle, cache.handle, _ptr(feats), _ptr(n_new_dev), host, rows,
                                   _ptr(anchor_dev), int(block_size), _ptr(draft_dev), _ptr(logits_dev),
                                   _ptr(workspace), workspace.numel(), _stream_ptr(stream)), "dflash_draft_cycle")


def dflash_verify_greedy(draft_dev: torch.Tensor, target_argmax_dev: torch.Tensor, accept_len_dev: torch.Tensor,
                         out_tokens_dev: torch.Tensor, next_anchor_dev: torch.Tensor, stream=None) -> None:
    """draft int32 [B, g-1], target int32 [B, g] -> tau [B], out [B, g], next anchor [B] (all int32)."""
    B, g = target_argmax_dev.shape
    for t in (draft_dev, target_argmax_dev, accept_len_dev, out_tokens_dev, next_anchor_dev):
        if t.dtype != torch.int32:
            raise ValueError("verify tensors must be int32")
    check(lib().dflash_verify_greedy(_ptr(draft_dev), _ptr(target_argmax_dev), B, g, _ptr(accept_len_dev),
                                     _ptr(out_tokens_dev), _ptr(next_anchor_dev), _stream_ptr(stream)),
          "dflash_verify_greedy")


def dflash_sampling_workspace(rows: int, draws: int, vocab: int) -> torch.Tensor:
    """Device scratch for dflash_verify_sampled / dflash_sample_tokens."""
    n = int(lib().dflash_sampling_workspace_bytes(int(rows), int(draws), int(vocab)))
    if n == 0:
        raise ValueError("invalid sampling workspace shape")
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def dflash_verify_sampled(draft_logits: Optional[torch.Tensor], target_logits: torch.Tensor,
                          drafts: Optional[torch.Tensor], u_accept: Optional[torch.Tensor], u_sample: torch.Tensor,
                          temperature: float, accept_len: torch.Tensor, out_tokens: torch.Tensor,
                          next_anchor: torch.Tensor, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Stochastic lossless verification: draft logits fp32 [B, g-1, V], target
    logits fp32 [B, g, V], drafts int32 [B, g-1], uniforms fp32 u_accept
    [B, g-1] and u_sample [B] -> tau [B], out [B, g], next anchor [B]."""
    B, g, V = target_logits.shape
    for t in (draft_logits, target_logits, u_accept, u_sample):
        if t is not None and t.dtype != torch.float32:
            raise ValueError("logits and uniforms must be float32")
    for t in (drafts, accept_len, out_tokens, next_anchor):
        if t is not None and t.dtype != torch.int32:
            raise ValueError("token tensors must be int32")
    if workspace is None:
        workspace = dflash_sampling_workspace(B * (2 * g - 1), B, V)
    check(lib().dflash_verify_sampled(_ptr(draft_logits), _ptr(target_logits), _ptr(drafts), _ptr(u_accept),
                                      _ptr(u_sample), B, g, V, float(temperature), _ptr(accept_len),
                                      _ptr(out_tokens), _ptr(next_anchor), _ptr(workspace), workspace.numel(),
                                      _stream_ptr(stream)), "dflash_verify_sampled")


def dflash_sample_tokens(logits: torch.Tensor, temperature: float, u: torch.Tensor, tokens: torch.Tensor,
                         workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """tokens[r] = inverse-CDF draw with uniform u[r] from softmax(logits[r] / T); logits fp32 [..., V]."""
    V = logits.shape[-1]
    rows = logits.numel() // V
    if logits.dtype != torch.float32 or u.dtype != torch.float32 or tokens.dtype != torch.int32:
        raise ValueError("logits and u must be float32, tokens int32")
    if workspace is None:
        workspace = dflash_sampling_workspace(rows, rows, V)
    check(lib().dflash_sample_tokens(_ptr(logits), rows, V, float(temperature), _ptr(u), _ptr(tokens),
                                     _ptr(workspace), workspace.numel(), _stream_ptr(stream)), "dflash_sample_tokens")


def dflash_packed_attention_workspace(n_blocks: int, block: int, seq_len: int, n_q_heads: int, n_kv_heads: int,
                                      head_dim: int) -> torch.Tensor:
    n = int(lib().dflash_packed_attention_workspace_bytes(n_blocks, block, seq_len, n_q_heads, n_kv_heads, head_dim))
    if n == 0:
        raise ValueError("invalid packed attention shape")
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def dflash_packed_block_attention(q: torch.Tensor, k_ctx: torch.Tensor, v_ctx: torch.Tensor, k_blk: torch.Tensor,
                                  v_blk: torch.Tensor, anchors_dev: torch.Tensor, out: torch.Tensor,
                                  workspace: torch.Tensor, anchors_host=None, stream=None) -> None:
    """Packed training attention: q [N, g, nq, hd], k_ctx / v_ctx [S, nkv, hd],
    k_blk / v_blk [N, g, nkv, hd] (fp32 or bf16), anchors int32 [N] -> out fp32 [N, g, nq, hd]."""
    N, g, nq, hd = q.shape
    S, nkv = k_ctx.shape[0], k_blk.shape[2]
    dt = _abi.DTYPE_F32 if q.dtype == torch.float32 else _abi.DTYPE_BF16
    for t in (k_ctx, v_ctx, k_blk, v_blk):
        if t.dtype != q.dtype:
            raise ValueError("q, k and v must share one dtype")
    if out.dtype != torch.float32 or anchors_dev.dtype != torch.int32:
        raise ValueError("out must be float32 and anchors int32")
    host = None
    if anchors_host is not None:
        host = (ctypes.c_int32 * N)(*[int(a) for a in anchors_host])
    check(lib().dflash_packed_block_attention(_ptr(q), _ptr(k_ctx), _ptr(v_ctx), _ptr(k_blk), _ptr(v_blk),
                                              _ptr(anchors_dev), host, N, g, S, nq, nkv, hd, dt, _ptr(out),
                                              _ptr(workspace), workspace.numel(), _stream_ptr(stream)),
          "dflash_packed_block_attention")


def dflash_packed_attention_status(workspace: torch.Tensor, stream=None) -> int:
    st = ctypes.c_int32(0)
    check(lib().dflash_packed_attention_status(_ptr(workspace), _stream_ptr(stream), ctypes.byref(st)),
          "dflash_packed_attention_status")
    return st.value


class BlockPolicy:
    """Host block-size scheduling policy (dflash_block_policy_*): observe each
    cycle's accepted lengths, choose the next cycle's block size."""

    def __init__(self, candidates, cost_fixed_ms: float, cost_per_row_ms: float, cost_per_request_ms: float = 0.0,
                 decay: float = 0.9, prior_accept: float = 0.8, prior_weight: float = 2.0):
        cfg = _abi.PolicyConfig()
        cand = [int(c) for c in candidates]
        if len(cand) > _abi.POLICY_MAX_CANDIDATES:
            raise ValueError("too many candidates")
        cfg.n_candidates = len(cand)
        for i, c in enumerate(cand):
            cfg.candidates[i] = c
        cfg.cost_fixed_ms, cfg.cost_per_row_ms, cfg.cost_per_request_ms = cost_fixed_ms, cost_per_row_ms, \
            cost_per_request_ms
        cfg.decay, cfg.prior_accept, cfg.prior_weight = decay, prior_accept, prior_weight
        h = ctypes.c_void_p()
        check(lib().dflash_block_policy_create(ctypes.byref(cfg), ctypes.byref(h)), "dflash_block_policy_create")
        self.handle = h
        self.candidates = cand

    def observe(self, block_size: int, taus) -> None:
        arr = (ctypes.c_int32 * len(taus))(*[int(t) for t in taus])
        check(lib().dflash_block_policy_observe(self.handle, int(block_size), arr, len(taus)),
              "dflash_block_policy_observe")

    def choose(self, batch: int):
        g, e = ctypes.c_int32(0), ctypes.c_double(0.0)
        check(lib().dflash_block_policy_choose(self.handle, int(batch), ctypes.byref(g), ctypes.byref(e)),
              "dflash_block_policy_choose")
        return g.value, e.value

    def acceptance(self, n: int):
        out = (ctypes.c_double * n)()
        check(lib().dflash_block_policy_acceptance(self.handle, out, n), "dflash_block_policy_acceptance")
        return list(out)

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            lib().dflash_block_policy_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dflash_synthetic_target(drafts: torch.Tensor, match: torch.Tensor, off: torch.Tensor, bonus: torch.Tensor,
                            pattern_idx: torch.Tensor, target_out: torch.Tensor, vocab: int,
                            tau: Optional[torch.Tensor] = None, tau_sum: Optional[torch.Tensor] = None,
                            stream=None) -> None:
    """Benchmark utility: the synthetic target's answer for stacked agreement
    patterns (match bool/uint8 [P,B,g-1], off int32 [P,B,g-1], bonus int32
    [P,B]) selected by the device counter pattern_idx (int64 [1])."""
    P, B = bonus.shape
    g = target_out.shape[1]
    m = match.view(torch.uint8) if match.dtype == torch.bool else match
    check(lib().dflash_synthetic_target(_ptr(drafts) if g > 1 else None, _ptr(m), _ptr(off), _ptr(bonus), P,
                                        _ptr(pattern_idx), _ptr(tau), _ptr(tau_sum), B, g, int(vocab),
                                        _ptr(target_out), _stream_ptr(stream)), "dflash_synthetic_target")


def dflash_get_status(model: Model, stream=None) -> int:
    st = ctypes.c_int32(0)
    check(lib().dflash_get_status(model.handle, _stream_ptr(stream), ctypes.byref(st)), "dflash_get_status")
    return st.value


def dflash_clear_status(model: Model, stream=None) -> None:
    check(lib().dflash_clear_status(model.handle, _stream_ptr(stream)), "dflash_clear_status")


def dflash_selftest_wait_timeout(model: Model, budget_cycles: int, stream=None) -> None:
    """Run the bounded-wait self-test: a wait that nothing completes gives up
    after budget_cycles SM cycles and sets the status word to DFLASH_ERR_TIMEOUT."""
    check(lib().dflash_selftest_wait_timeout(model.handle, int(budget_cycles), _stream_ptr(stream)),
          "dflash_selftest_wait_timeout")


def dflash_launch_count() -> int:
    """Kernel launches made by the library in this process."""
    return int(lib().dflash_launch_count())


def dflash_profile_start(model: Model, max_launches: int = 4096) -> None:
    check(lib().dflash_profile_start(model.handle, int(max_launches)), "dflash_profile_start")


def dflash_profile_stop(model: Model, stream=None) -> dict:
    """{stage: (milliseconds, launches)} recorded since dflash_profile_start."""
    n = len(_abi.STAGES)
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int32 * n)()
    check(lib().dflash_profile_stop(model.handle, _stream_ptr(stream), ms, cnt, n), "dflash_profile_stop")
    return {name: (float(ms[i]), int(cnt[i])) for i, name in enumerate(_abi.STAGES)}
