"""Phase timeline of the persistent cycle launch (a diagnostic).

Runs a few draft cycles (dflash_draft_cycle: injection and drafter pass in one
launch) of a bf16 workload whose calls have at most 16 token rows with
DFLASH_TRACE_PERSIST=1, so that every persistent drafter launch records
per-CTA globaltimer stamps, reads the stamps of the last one and prints one
line per phase: when its first CTA started it, the median and the latest
CTA's last MMA issue, and the median and the latest CTA's end.

    python -m block_diffusion_drafter_dflash_gb300.phase_trace [workload] [--raw out.npy]
"""
from __future__ import annotations

import ctypes
import os
import sys
from typing import List

import numpy as np

GRID_MAX, PHASES, SLOTS = 512, 56, 18           # the kernel's trace layout [cta][phase][slot]
START, DONE, MMA_LAST = 0, 1, 6                  # slots used here


def phase_names(layers: int, lm_head: bool = True, fusion: bool = False) -> List[str]:
    """Phases of a persistent drafter launch; `fusion`: the launch of a whole
    cycle (dflash_draft_cycle), which starts with the context fusion and the
    injection of every layer's context K/V."""
    names = ["fusion", "inject"] if fusion else []
    for l in range(layers):
        names += [f"L{l} qkv", f"L{l} attn", f"L{l} o", f"L{l} gateup", f"L{l} down"]   # attn: chunks and their merge
    return names + (["lmhead"] if lm_head else [])


def phase_table(t: np.ndarray, names: List[str]) -> List[dict]:
    """Per phase (microseconds from the first CTA's start of phase 0): first
    start, median / latest last-MMA issue (projection phases), median / latest
    end, and the phase's length up to the next phase's first start.  `t` is
    [ctas][phases][slots] of globaltimer nanoseconds (0 = not stamped)."""
    t = np.asarray(t, dtype=np.float64)
    t0 = t[:, 0, START][t[:, 0, START] > 0].min()
    us = lambda a: (a - t0) / 1e3
    rows = []
    for p, name in enumerate(names):
        st, dn, m1 = t[:, p, START], t[:, p, DONE], t[:, p, MMA_LAST]
        st, dn, m1 = st[st > 0], dn[dn > 0], m1[m1 > 0]
        nxt = t[:, p + 1, START] if p + 1 < len(names) else None
        end = nxt[nxt > 0].min() if nxt is not None and (nxt > 0).any() else dn.max()
        rows.append({"phase": name, "start": us(st.min()),
                     "mma_last_med": us(np.median(m1)) if m1.size else None,
                     "mma_last_max": us(m1.max()) if m1.size else None,
                     "done_med": us(np.median(dn)), "done_max": us(dn.max()),
                     "length": (end - st.min()) / 1e3})
    return rows


def format_table(rows: List[dict]) -> str:
    f = lambda v: "      -" if v is None else f"{v:7.1f}"
    out = ["| phase | start | last MMA (median / latest) | end (median / latest) | length |",
           "|---|---|---|---|---|"]
    for r in rows:
        out.append(f"| {r['phase']} | {r['start']:.1f} | {f(r['mma_last_med'])} / {f(r['mma_last_max'])} | "
                   f"{r['done_med']:.1f} / {r['done_max']:.1f} | {r['length']:.1f} |")
    return "\n".join(out)


def run(workload: str = "8b_bs1", cycles: int = 4):
    os.environ["DFLASH_TRACE_PERSIST"] = "1"     # read when the model is created
    import torch

    import block_diffusion_drafter_dflash_gb300 as df
    from dflash_inputs import make_features, make_tokens, make_weights, workloads

    wl = workloads()[workload]
    cfg, B, block = wl.cfg, wl.batch, wl.block
    if cfg.dtype != "bf16" or B * block > 16:
        raise ValueError(f"{workload}: the persistent path serves bf16 calls of at most 16 token rows")
    torch.cuda.set_device(0)
    w = make_weights(cfg, wl.seed, device="cuda")
    model = df.Model(cfg, w)
    cap = max(wl.ctx) + block * (cycles + 2)
    cache = df.Cache(model, B, cap)
    ws = df.dflash_workspace(model, B, cap, block, max(sum(wl.ctx), B * block))
    feats = torch.cat([make_features(cfg, c, seed=wl.seed + 17 * b, device="cuda") for b, c in enumerate(wl.ctx)])
    df.dflash_inject_context(model, cache, feats, torch.tensor(wl.ctx, dtype=torch.int32, device="cuda"), wl.ctx,
                             sum(wl.ctx), ws)
    new = make_features(cfg, B * block, seed=wl.seed + 999, device="cuda")
    tau = torch.full((B,), wl.first_inject, dtype=torch.int32, device="cuda")
    anchor = make_tokens(cfg, B, seed=wl.seed + 3, device="cuda")
    drafts = torch.empty((B, block - 1), dtype=torch.int32, device="cuda")
    for _ in range(cycles):   # the benchmark's cycle: injection and drafter pass in one launch
        df.dflash_draft_cycle(model, cache, new, tau, anchor, block, drafts, None, max_rows=B * block, workspace=ws)
    torch.cuda.synchronize()
    n = GRID_MAX * PHASES * SLOTS
    buf = (ctypes.c_uint64 * n)()
    df.check(df.lib().dflash_trace_read(model.handle, buf, n), "dflash_trace_read")
    t = np.frombuffer(buf, dtype=np.uint64).reshape(GRID_MAX, PHASES, SLOTS)
    t = t[: torch.cuda.get_device_properties(0).multi_processor_count]
    return t, phase_names(cfg.layers, fusion=True)


def main(argv: List[str]) -> None:
    args = [a for a in argv if not a.startswith("--")]
    t, names = run(args[0] if args else "8b_bs1")
    if "--raw" in argv:
        np.save(argv[argv.index("--raw") + 1], t)
    print(format_table(phase_table(t, names)))


if __name__ == "__main__":
    main(sys.argv[1:])
