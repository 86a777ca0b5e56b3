"""Training-time packed block attention (paper §4.2; explainer "Training
Rehearses the Same Masked Blocks Used at Runtime", Figure 4) on the GPU
against the float64 oracle: oracle.attention_packed (the brute-force mask) on
small sequences, and — at the training shape of paper §7.1 (sequences of 3072
tokens, 512 anchor blocks of 16, Qwen3-8B-shaped heads) — sampled blocks
against oracle.attention_block over the context truncated at the anchor (the
pinned identity between the two).  Bar: per (row, head) max |g - o| /
max |o| <= 1e-4 (the kernel carries every operand at fp32 precision through
the tensor cores), for fp32 and bf16 inputs alike."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

TOL = 1e-4


def _df():
    import block_diffusion_drafter_dflash_gb300 as df
    return df


def _inputs(S, N, g, nq, nkv, hd, dtype, seed):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    r = lambda *shape: torch.randn(shape, generator=gen, device="cuda").to(dtype).contiguous()
    return r(N, g, nq, hd), r(S, nkv, hd), r(S, nkv, hd), r(N, g, nkv, hd), r(N, g, nkv, hd)


def _run(q, kc, vc, kb, vb, anchors, dtype):
    df = _df()
    N, g, nq, hd = q.shape
    S, nkv = kc.shape[0], kc.shape[1]
    out = torch.full((N, g, nq, hd), float("nan"), device="cuda")
    ws = df.dflash_packed_attention_workspace(N, g, S, nq, nkv, hd)
    a_dev = torch.tensor(anchors, dtype=torch.int32, device="cuda")
    df.dflash_packed_block_attention(q, kc, vc, kb, vb, a_dev, out, ws, anchors_host=anchors)
    return out, ws


def _rel(g, o):
    g = np.asarray(g, dtype=np.float64).reshape(-1, g.shape[-1])
    o = np.asarray(o, dtype=np.float64).reshape(-1, o.shape[-1])
    return float(np.max(np.max(np.abs(g - o), axis=1) / np.maximum(np.max(np.abs(o), axis=1), 1e-30)))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("S,anchors,g,nq,nkv,hd", [
    (200, [0, 200, 77, 128, 129, 5], 4, 4, 2, 64),     # an anchor at 0 and one at the sequence end
    (300, [150, 10, 299, 256, 31], 16, 32, 8, 128),    # 8B-shaped heads, block 16, ragged context tiles
    (0, [0, 0, 0], 8, 8, 2, 128),                      # no context: each block sees only itself
])
def test_packed_attention_matches_oracle(dtype, S, anchors, g, nq, nkv, hd):
    N = len(anchors)
    q, kc, vc, kb, vb = _inputs(S, N, g, nq, nkv, hd, dtype, seed=S + N)
    out, ws = _run(q, kc, vc, kb, vb, anchors, dtype)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().numpy()
    ref = oracle.attention_packed(f(q).reshape(N * g, nq, hd), f(kc), f(vc), f(kb).reshape(N * g, nkv, hd),
                                  f(vb).reshape(N * g, nkv, hd), anchors)
    err = _rel(f(out).reshape(N * g, nq, hd), ref)
    print(f"S={S} N={N} g={g} {dtype}: rel err {err:.2e}")
    assert err <= TOL
    assert _df().dflash_packed_attention_status(ws) == 0


def test_packed_attention_training_shape_sampled_blocks():
    """Paper §7.1: up to 3072 tokens a sequence, 512 anchors; 8B-shaped
    attention (32 q / 8 kv heads of 128), block 16, bf16 inputs."""
    S, N, g, nq, nkv, hd = 3072, 512, 16, 32, 8, 128
    rng = np.random.default_rng(7)
    anchors = sorted(int(a) for a in rng.choice(np.arange(1, S - g), size=N, replace=False))
    q, kc, vc, kb, vb = _inputs(S, N, g, nq, nkv, hd, torch.bfloat16, seed=71)
    out, ws = _run(q, kc, vc, kb, vb, anchors, torch.bfloat16)
    torch.cuda.synchronize()
    assert _df().dflash_packed_attention_status(ws) == 0
    f = lambda t: t.float().cpu().numpy()
    kc_h, vc_h = f(kc), f(vc)
    worst = 0.0
    for n in [0, 1, 100, 255, 256, 400, 510, N - 1]:
        ref = oracle.attention_block(f(q[n]), kc_h[:anchors[n]], vc_h[:anchors[n]], f(kb[n]), f(vb[n]))
        worst = max(worst, _rel(f(out[n]), ref))
    print(f"training shape: worst sampled rel err {worst:.2e}")
    assert worst <= TOL
    assert torch.isfinite(out).all()


def test_packed_attention_flags_anchors_outside_the_sequence():
    df = _df()
    S, N, g, nq, nkv, hd = 64, 3, 4, 4, 2, 64
    q, kc, vc, kb, vb = _inputs(S, N, g, nq, nkv, hd, torch.float32, seed=9)
    with pytest.raises(df.DFlashError):            # checked on the host when the host copy is given
        _run(q, kc, vc, kb, vb, [3, 65, 7], torch.float32)
    out = torch.empty((N, g, nq, hd), device="cuda")
    ws = df.dflash_packed_attention_workspace(N, g, S, nq, nkv, hd)
    a_dev = torch.tensor([3, 999, 7], dtype=torch.int32, device="cuda")
    df.dflash_packed_block_attention(q, kc, vc, kb, vb, a_dev, out, ws)   # device copy only: clamped and flagged
    assert df.dflash_packed_attention_status(ws) == -1
    f = lambda t: t.float().cpu().numpy()
    ref = oracle.attention_packed(f(q).reshape(N * g, nq, hd), f(kc), f(vc), f(kb).reshape(N * g, nkv, hd),
                                  f(vb).reshape(N * g, nkv, hd), [3, S, 7])
    assert _rel(f(out).reshape(N * g, nq, hd), ref) <= TOL
