"""Storage-precision study of the bf16 drafter — test infrastructure, run by hand.

Rounds one tensor class at a time (oracle.STORE_CLASSES) to bf16 in the
float64 oracle and reports, against the exact definition, the largest per-row
logit error (max_v |l - l_exact| / max_v |l_exact|) and how many drafts flip
among the rows whose exact top-1 minus top-2 logit exceeds 1e-2 — the two
parity bars of the draft cycle.  It tells which tensors the GPU path could
keep in one bf16 plane without leaving those bars.  Uses only the oracle and
the seeded input generators:

    python -m oracle.precision_study [--ctx 2048] [--anchors 3] [--drafter 8b]
"""
from __future__ import annotations

import argparse
import time

import numpy as np
import torch

from dflash_inputs import QWEN3_4B, QWEN3_8B, make_features, make_tokens, make_weights

from . import dflash_oracle as o


def row_err(a, b):
    return float(np.max(np.max(np.abs(a - b), axis=1) / np.max(np.abs(b), axis=1)))


def flips(logits, exact, margin=1e-2):
    top2 = np.sort(exact, axis=1)[:, -2:]
    ok = (top2[:, 1] - top2[:, 0]) > margin
    return int(np.sum((np.argmax(logits, 1) != np.argmax(exact, 1)) & ok)), int(np.sum(ok))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--ctx", type=int, default=2048)
    ap.add_argument("--anchors", type=int, default=3)
    ap.add_argument("--drafter", default="8b", choices=["8b", "4b"])
    ap.add_argument("--block", type=int, default=16)
    ap.add_argument("--classes", default=",".join(o.STORE_CLASSES) + ",all",
                    help="comma-separated classes to study (all: every class at once; a+b: "
                         "classes a and b at once)")
    args = ap.parse_args()
    cfg = QWEN3_8B if args.drafter == "8b" else QWEN3_4B
    torch.set_num_threads(max(1, torch.get_num_threads()))
    t0 = time.time()
    w = o.weights_to_host(make_weights(cfg, 1000))
    feats = make_features(cfg, args.ctx, seed=1001)
    wanted = args.classes.split(",")
    modes = [("exact", "f64")] + [(c, {c: "bf16"}) for c in o.STORE_CLASSES if c in wanted]
    for combo in (c for c in wanted if "+" in c):
        parts = combo.split("+")
        if any(p not in o.STORE_CLASSES for p in parts):
            raise SystemExit(f"unknown class in {combo}")
        modes.append((combo, {p: "bf16" for p in parts}))
    if "all" in wanted:
        modes.append(("all", "bf16"))
    rows = {name: [] for name, _ in modes}
    caches = {}   # the injected cache depends on the rounding mode only, not on the anchor
    for a in range(args.anchors):
        anchor = int(make_tokens(cfg, 1, seed=1002 + a).item())
        ref = None
        for name, mode in modes:
            own = mode == "bf16" or (isinstance(mode, dict) and ("kv" in mode or "ht" in mode))
            key = name if own else "exact"
            if key not in caches:
                cache = o.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
                for s in range(0, args.ctx, 1024):
                    o.inject_context(w, cfg, cache, feats[s:s + 1024], mode if own else "f64")
                caches[key] = cache
            cache = caches[key]
            fw = o.draft_forward(w, cfg, cache, anchor, args.block, mode=mode)
            logits, _ = o.lm_head_argmax(fw["h"][1:], w["lm_head"])
            if name == "exact":
                ref = logits
            f, n = flips(logits, ref)
            rows[name].append((row_err(logits, ref), f, n))
        print(f"anchor {a} done ({time.time() - t0:.0f} s)", flush=True)
    print(f"\n{cfg.name}, context {args.ctx}, block {args.block}, {args.anchors} anchors")
    print("| tensor class in bf16 | max row logit error | argmax flips / rows with margin > 1e-2 |")
    print("|---|---|---|")
    for name, _ in modes[1:]:
        err = max(r[0] for r in rows[name])
        f = sum(r[1] for r in rows[name])
        n = sum(r[2] for r in rows[name])
        print(f"| {name} | {err:.2e} | {f} / {n} |")


if __name__ == "__main__":
    main()
