"""The phase-timeline diagnostic's table on a hand-made trace: first start,
median and latest last-MMA issue and end, and the length up to the next
phase's first start."""
import numpy as np

from block_diffusion_drafter_dflash_gb300.phase_trace import DONE, MMA_LAST, START, format_table, phase_names, \
    phase_table


def test_phase_names_follow_the_drafter_program():
    assert phase_names(1) == ["L0 qkv", "L0 attn", "L0 o", "L0 gateup", "L0 down", "lmhead"]
    assert len(phase_names(5)) == 26
    assert phase_names(5, fusion=True)[:3] == ["fusion", "inject", "L0 qkv"] and len(phase_names(5, fusion=True)) == 28


def test_phase_table_on_a_hand_made_trace():
    t = np.zeros((3, 4, 18), dtype=np.uint64)
    base = 1_000_000_000
    # phase 0: CTAs start at 0, 1, 2 us; last MMAs at 5, 6, 7 us; end at 8, 9, 12 us
    for c in range(3):
        t[c, 0, START] = base + 1000 * c
        t[c, 0, MMA_LAST] = base + 1000 * (5 + c)
        t[c, 0, DONE] = base + [8000, 9000, 12000][c]
    # phase 1 starts at 13 us (first CTA), no MMA stamps, ends at 20 us
    t[:, 1, START] = base + 13000
    t[1, 1, START] = base + 13500
    t[:, 1, DONE] = base + 20000
    rows = phase_table(t, ["a", "b"])
    a, b = rows
    assert a["start"] == 0.0 and a["mma_last_med"] == 6.0 and a["mma_last_max"] == 7.0
    assert a["done_med"] == 9.0 and a["done_max"] == 12.0 and a["length"] == 13.0
    assert b["start"] == 13.0 and b["mma_last_med"] is None and b["length"] == 7.0
    text = format_table(rows)
    assert text.count("\n") == 3 and "| a | 0.0 |" in text
