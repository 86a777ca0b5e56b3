"""Seeded synthetic inputs for the DFlash draft cycle.

This module holds shapes and random-number recipes only: drafter shapes, the
workloads they are measured on, seeded weights, target hidden features, anchor
tokens and the synthetic target's agreement pattern.  It contains none of the
method's arithmetic, so both the CUDA path (through its binding) and the CPU
oracle can be fed from it without sharing any of the method's code.

Shapes follow the DFlash drafter described in "DFlash: Block Diffusion for
Flash Speculative Decoding" (§5 Implementation: 5 draft layers, block size 16,
5 target feature layers; §7.3: W_c in R^{D x 5D}) with Qwen3-style dimensions.
All draws are seeded: the same (config, seed) gives the same tensors on the
same device type.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional

import torch


@dataclass(frozen=True)
class DraftConfig:
    """Drafter shape.  Field names follow the paper's symbols where it has one."""

    name: str
    hidden: int            # D, draft hidden size (= target hidden size)
    layers: int            # number of draft transformer layers
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int               # SwiGLU intermediate width
    vocab: int             # shared embedding / LM head rows
    n_target_feats: int = 5   # m, target layers whose hidden states are fused
    rope_theta: float = 1e6
    rms_eps: float = 1e-6
    dtype: str = "bf16"    # "fp32" or "bf16": storage type of weights and activations
    max_block: int = 32    # largest block_size the drafter is asked for
    mask_token_id: Optional[int] = None   # defaults to vocab - 1
    qk_norm: bool = False  # per-head RMSNorm of queries and keys before RoPE (Qwen3's q_norm / k_norm)
    input_fusion: bool = False  # ablation: the fused context enters once, at the input, instead of every layer's K/V
    kv_bf16: bool = False  # bf16 models: the context K/V cache holds one bf16 per value (else a hi/lo pair)
    head_bf16: bool = False  # bf16 models: the LM head reads the final normed state as one bf16 (else a hi/lo pair)

    @property
    def mask_id(self) -> int:
        return self.vocab - 1 if self.mask_token_id is None else self.mask_token_id

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "fp32" else 2

    def layer_params(self) -> int:
        D, hq, hk, F = self.hidden, self.n_q_heads * self.head_dim, self.n_kv_heads * self.head_dim, self.ffn
        return D * hq + 2 * D * hk + hq * D + 3 * D * F + 2 * D

    def layer_matrix_params(self) -> int:
        D, hq, hk, F = self.hidden, self.n_q_heads * self.head_dim, self.n_kv_heads * self.head_dim, self.ffn
        return D * hq + 2 * D * hk + hq * D + 3 * D * F


TINY = DraftConfig("tiny-fp32", hidden=256, layers=2, n_q_heads=4, n_kv_heads=2, head_dim=64,
                   ffn=768, vocab=1024, dtype="fp32", max_block=32)
QWEN3_8B = DraftConfig("qwen3-8b-shaped", hidden=4096, layers=5, n_q_heads=32, n_kv_heads=8,
                       head_dim=128, ffn=12288, vocab=151936, dtype="bf16", max_block=32)
QWEN3_4B = DraftConfig("qwen3-4b-shaped", hidden=2560, layers=5, n_q_heads=32, n_kv_heads=8,
                       head_dim=128, ffn=9728, vocab=151936, dtype="bf16", max_block=32)


@dataclass(frozen=True)
class Workload:
    """One measured or parity-tested configuration of the draft cycle."""

    name: str
    cfg: DraftConfig
    batch: int
    block: int                       # block_size = anchor + (block - 1) mask tokens
    ctx: List[int]                   # injected context length per request at setup
    accept_p: List[float]            # per-request probability that the target agrees with a draft
    cycles: int = 1
    seed: int = 0
    first_inject: int = 8            # tau of the (synthetic) previous cycle, injected in cycle 0


def _ragged_ctx(batch: int, lo: int, hi: int, seed: int) -> List[int]:
    g = torch.Generator().manual_seed(seed)
    return [int(v) for v in torch.randint(lo, hi + 1, (batch,), generator=g)]


def _ragged_p(batch: int, lo: float, hi: float, seed: int) -> List[float]:
    g = torch.Generator().manual_seed(seed + 1)
    return [float(lo + (hi - lo) * v) for v in torch.rand(batch, generator=g, dtype=torch.float64)]


def workloads() -> Dict[str, Workload]:
    """The five configurations of the draft-cycle study, by name."""
    w = {
        "tiny": Workload("tiny", TINY, batch=1, block=4, ctx=[64], accept_p=[0.9], cycles=1, seed=0,
                         first_inject=2),
        "8b_bs1": Workload("8b_bs1", QWEN3_8B, batch=1, block=16, ctx=[2048], accept_p=[0.9],
                           cycles=1, seed=1000),
        "8b_bs32": Workload("8b_bs32", QWEN3_8B, batch=32, block=16, ctx=_ragged_ctx(32, 512, 8192, 3),
                            accept_p=_ragged_p(32, 0.6, 0.95, 3), cycles=1, seed=2000),
        "8b_long": Workload("8b_long", QWEN3_8B, batch=4, block=16, ctx=[32768] * 4, accept_p=[0.9] * 4,
                            cycles=16, seed=3000),
    }
    for g in (8, 10, 16):
        for b in (1, 4, 16):
            w[f"4b_g{g}_b{b}"] = Workload(f"4b_g{g}_b{b}", QWEN3_4B, batch=b, block=g, ctx=[4096] * b,
                                          accept_p=[0.9] * b, cycles=64, seed=4000 + 10 * g + b)
    return w


# ---------------------------------------------------------------------------
# Seeded tensors.  Every draw goes through a torch.Generator on `device`.
# ---------------------------------------------------------------------------

def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(int(seed))


def _normal(shape, std, g, device, dtype):
    t = torch.empty(shape, device=device, dtype=torch.float32)
    t.normal_(0.0, std, generator=g)
    return t.to(dtype)


def make_weights(cfg: DraftConfig, seed: int, device="cpu", std: float = 0.02) -> Dict[str, object]:
    """Drafter weights: matrices N(0, std), RMSNorm gains ones.

    Matrices are [out_features, in_features] row-major.  Keys:
    embed [V, D], lm_head [V, D], w_c [D, m*D], g_c [D], g_final [D] and
    layers[i] with g_in, w_q, w_k, w_v, w_o, g_post, w_g, w_u, w_d (and, when
    cfg.qk_norm, g_q and g_k [head_dim] drawn as 1 + N(0, 0.1)).
    """
    g = _gen(seed, device)
    dt = cfg.torch_dtype
    D, V, m = cfg.hidden, cfg.vocab, cfg.n_target_feats
    hq, hk, F = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim, cfg.ffn
    ones = lambda n: torch.ones(n, device=device, dtype=dt)
    w: Dict[str, object] = {
        "embed": _normal((V, D), std, g, device, dt),
        "lm_head": _normal((V, D), std, g, device, dt),
        "w_c": _normal((D, m * D), std, g, device, dt),
        "g_c": ones(D),
        "g_final": ones(D),
    }
    layers = []
    for _ in range(cfg.layers):
        layers.append({
            "g_in": ones(D),
            "w_q": _normal((hq, D), std, g, device, dt),
            "w_k": _normal((hk, D), std, g, device, dt),
            "w_v": _normal((hk, D), std, g, device, dt),
            "w_o": _normal((D, hq), std, g, device, dt),
            "g_post": ones(D),
            "w_g": _normal((F, D), std, g, device, dt),
            "w_u": _normal((F, D), std, g, device, dt),
            "w_d": _normal((D, F), std, g, device, dt),
        })
    w["layers"] = layers
    if cfg.qk_norm:
        # per-head query / key norm gains [head_dim], near one so that a
        # missing gain is visible; a generator of their own keeps every other
        # weight of the configuration unchanged
        gq = _gen(seed + 7777, device)
        for lw in layers:
            lw["g_q"] = (1.0 + _normal((cfg.head_dim,), 0.1, gq, device, torch.float32)).to(dt)
            lw["g_k"] = (1.0 + _normal((cfg.head_dim,), 0.1, gq, device, torch.float32)).to(dt)
    return w


def make_features(cfg: DraftConfig, n_tokens: int, seed: int, device="cpu") -> torch.Tensor:
    """Target hidden states of the m selected target layers, N(0,1): [n, m, D]."""
    g = _gen(seed, device)
    return _normal((n_tokens, cfg.n_target_feats, cfg.hidden), 1.0, g, device, cfg.torch_dtype)


def make_tokens(cfg: DraftConfig, n: int, seed: int, device="cpu") -> torch.Tensor:
    """Uniform token ids in [0, V) as int32 (anchors or a uniform target argmax)."""
    g = _gen(seed, device)
    return torch.randint(0, cfg.vocab, (n,), generator=g, device=device, dtype=torch.int64).to(torch.int32)


@dataclass
class AgreementPattern:
    """How the synthetic target answers a block of drafts.

    match[b, k] is True when the target's argmax after block position k agrees
    with draft k+1; off[b, k] picks the disagreeing token; bonus[b] is the
    target's token after the last block position.
    """

    match: torch.Tensor    # bool  [B, block-1]
    off: torch.Tensor      # int32 [B, block-1], uniform in [0, V-2]
    bonus: torch.Tensor    # int32 [B]


def make_agreement(cfg: DraftConfig, batch: int, block: int, accept_p, seed: int, device="cpu") -> AgreementPattern:
    g = _gen(seed, device)
    p = torch.as_tensor(list(accept_p), dtype=torch.float32, device=device).reshape(batch, 1)
    u = torch.rand((batch, max(block - 1, 0)), generator=g, device=device)
    off = torch.randint(0, max(cfg.vocab - 1, 1), (batch, max(block - 1, 0)), generator=g, device=device)
    bonus = torch.randint(0, cfg.vocab, (batch,), generator=g, device=device)
    return AgreementPattern(match=u < p, off=off.to(torch.int32), bonus=bonus.to(torch.int32))


def synthetic_target_argmax(drafts: torch.Tensor, pat: AgreementPattern, vocab: int) -> torch.Tensor:
    """The synthetic target's greedy tokens y[b, 0..block-1] for a block of drafts.

    y[b, k] (k < block-1) equals drafts[b, k] where the pattern says the target
    agrees, and (drafts[b, k] + 1 + off[b, k]) mod V (never equal) elsewhere;
    y[b, block-1] is the bonus.  Torch ops on whatever device `drafts` is on.
    """
    d = drafts.to(torch.int64)
    other = (d + 1 + pat.off.to(torch.int64)) % vocab
    y = torch.where(pat.match, d, other)
    return torch.cat([y, pat.bonus.to(torch.int64).reshape(-1, 1)], dim=1).to(torch.int32)


def seed_for(workload: Workload, cycle: int, stream: int = 0) -> int:
    """Seed of one draw: workload seed, cycle index and a per-tensor stream id."""
    return workload.seed + 7919 * cycle + 104729 * stream


__all__ = [
    "DraftConfig", "Workload", "AgreementPattern", "TINY", "QWEN3_8B", "QWEN3_4B", "workloads",
    "make_weights", "make_features", "make_tokens", "make_agreement", "synthetic_target_argmax",
    "seed_for", "replace", "field",
]
