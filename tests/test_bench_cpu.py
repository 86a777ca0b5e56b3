"""The benchmark's own arithmetic, on the CPU: the algorithmic bytes and flops
behind every roofline fraction, checked against independent counts from the
weight tensors' shapes and against the documented per-cycle figures; the rule
that uses a committed DRAM-traffic profile only for the workload and the
kernel sources it was taken on; and the whole-job throughput."""
import importlib.util
import os

import pytest

from dflash_inputs import QWEN3_8B, TINY, make_weights, replace, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _streamed_matrices(w):
    """Every matrix a cycle streams from HBM (the embedding is only gathered
    for the block's rows; the gains are vectors)."""
    mats = [w["w_c"], w["lm_head"]]
    for lw in w["layers"]:
        mats += [lw[k] for k in ("w_q", "w_k", "w_v", "w_o", "w_g", "w_u", "w_d")]
    return mats


@pytest.mark.parametrize("cfg", [TINY, replace(TINY, name="tiny-bf16", dtype="bf16")], ids=["fp32", "bf16"])
def test_gemm_bytes_with_no_rows_are_every_weight_byte_of_each_launch(bench, cfg):
    """Each matrix once per launch that uses it: W_K and W_V twice a cycle (the
    injection's context K/V, then the drafter's block K/V)."""
    w = make_weights(cfg, 0)
    nbytes = lambda t: t.numel() * t.element_size()
    expect = sum(nbytes(t) for t in _streamed_matrices(w))
    expect += sum(nbytes(lw["w_k"]) + nbytes(lw["w_v"]) for lw in w["layers"])
    got = bench.gemm_bytes_per_cycle(cfg, B=0, block=1, inject_rows=0)
    assert sum(got.values()) == expect
    assert got["inject"] == sum(nbytes(lw["w_k"]) + nbytes(lw["w_v"]) for lw in w["layers"])


@pytest.mark.parametrize("B,block,rows", [(1, 4, 3), (3, 5, 7)])
def test_gemm_flops_are_two_per_multiply_add_of_each_matrix(bench, B, block, rows):
    cfg = TINY
    w = make_weights(cfg, 0)
    R, Rm = B * block, B * (block - 1)
    expect = 2 * rows * w["w_c"].numel() + 2 * Rm * w["lm_head"].numel()
    for lw in w["layers"]:
        expect += 2 * rows * (lw["w_k"].numel() + lw["w_v"].numel())      # context injection
        expect += 2 * R * sum(lw[k].numel() for k in ("w_q", "w_k", "w_v", "w_o", "w_g", "w_u", "w_d"))
    assert sum(bench.gemm_flops_per_cycle(cfg, B, block, rows).values()) == expect


def test_8b_weight_bytes_match_the_documented_breakdown(bench):
    # layers 5 x 192.94 M parameters (1.929 GB), LM head 151936 x 4096 (1.245 GB),
    # W_c 4096 x 20480 (0.168 GB): 3.342 GB; plus the injection's W_K/W_V (84 MB)
    layer = 4096 * 4096 * 2 + 1024 * 4096 * 2 + 3 * 12288 * 4096
    drafter_and_fusion = 2 * (5 * layer + 151936 * 4096 + 4096 * 20480)
    assert abs(drafter_and_fusion / 1e9 - 3.342) < 5e-4
    got = bench.gemm_bytes_per_cycle(QWEN3_8B, B=0, block=1, inject_rows=0)
    assert got["inject"] == 2 * 5 * 2 * 1024 * 4096
    assert sum(got.values()) == drafter_and_fusion + got["inject"]


def test_context_kv_bytes_method_and_stored(bench):
    wl = workloads()["8b_bs1"]
    # the method's cache: K and V, 5 layers, 8 kv heads of 128, bf16 (20,480 B a token), 2048 tokens
    mb = bench.method_bytes(wl, inject_rows=8)
    assert mb["kv"] == 2 * 5 * 8 * 128 * 2 * 2048 == 41_943_040
    # as stored: hi and lo bf16 planes, 4 bytes a value
    assert bench.kv_storage_bytes(wl) == 2 * 5 * 8 * 128 * 4 * 2048 == 83_886_080
    # drafter launch: layer weights 1.929 GB + LM head 1.245 GB + K/V 41.9 MB = 3.216 GB
    assert abs(mb["drafter"] / 1e9 - 3.216) < 1e-3
    # whole cycle adds W_c and the 8 new tokens' 5 x 4096 bf16 features: 3.384 GB
    assert mb["cycle"] == mb["drafter"] + 2 * 4096 * 20480 + 8 * 5 * 4096 * 2
    assert abs(mb["cycle"] / 1e9 - 3.384) < 1e-3
    assert bench.kv_weight_bytes(QWEN3_8B) == 2 * 5 * 2 * 1024 * 4096


def test_traffic_profile_is_used_only_for_its_workload_and_sources(bench, monkeypatch, tmp_path):
    prof = tmp_path / "traffic.md"
    prof.write_text("# summary\n\nworkload: 8b_bs1\nsource_sha1: " + "a" * 40 + "\n"
                    "traffic_bytes_per_cycle: 3323915712\n")
    monkeypatch.setitem(bench.TRAFFIC_PROFILES, "persist", (str(prof), ["persist.cu"]))
    monkeypatch.setattr(bench, "source_sha1", lambda names: "a" * 40)
    assert bench.measured_traffic("persist", "8b_bs1") == 3323915712
    assert bench.measured_traffic("persist", "8b_bs32") is None
    monkeypatch.setattr(bench, "source_sha1", lambda names: "0" * 40)
    assert bench.measured_traffic("persist", "8b_bs1") is None


def test_job_throughput_counts_every_rank(bench):
    assert bench.job_throughput(2.0, 15, 1) == pytest.approx(7500.0)
    assert bench.job_throughput(2.0, 15, 4) == pytest.approx(30000.0)
