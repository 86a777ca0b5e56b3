"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/dflash.h declares, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def L():
    from block_diffusion_drafter_dflash_gb300 import _abi
    from block_diffusion_drafter_dflash_gb300.csrc import build as b
    srcs = [os.path.join(os.path.dirname(b.__file__), s) for s in b.SOURCES]
    srcs = [s for s in srcs if os.path.exists(s)] + [HEADER]
    lib = b.lib_path()
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(s) for s in srcs):
        b.build()
    return _abi.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z_]+)\s*\(", text)))


def test_header_declares_the_three_stage_entry_points():
    names = declared_functions()
    for n in ("dflash_inject_context", "dflash_draft_block", "dflash_verify_greedy"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    from block_diffusion_drafter_dflash_gb300 import _abi
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in _abi.SIGNATURES, f"{name} has no ctypes signature"
    assert L.dflash_version() >= 100


def _cfg(**kw):
    from block_diffusion_drafter_dflash_gb300 import _abi
    base = dict(hidden=256, layers=2, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=768, vocab=1024,
                n_target_feats=5, max_block=32, rope_theta=1e6, rms_eps=1e-6, mask_token_id=1023, dtype=0)
    base.update(kw)
    return _abi.Config(**base)


def test_cache_bytes_follow_the_documented_layout(L):
    c = _cfg()
    kv = 4 * 3 * 2 * 2 * 100 * 64
    a = lambda v: (v + 255) // 256 * 256
    assert L.dflash_cache_bytes(ctypes.byref(c), 3, 100) == 2 * a(kv) + a(4 * 3)
    c16 = _cfg(dtype=1)        # fp32-sized for bf16 models too (two bf16 planes); V hd-major, rows padded to 8
    kv8 = 4 * 3 * 2 * 2 * 104 * 64
    assert L.dflash_cache_bytes(ctypes.byref(c16), 3, 100) == a(kv) + a(kv8) + a(4 * 3)
    assert L.dflash_cache_bytes(ctypes.byref(c16), 3, 104) == 2 * a(kv8) + a(4 * 3)
    c1 = _cfg(dtype=1, kv_bf16=1)   # one rounded bf16 per value: half the K/V bytes
    assert L.dflash_cache_bytes(ctypes.byref(c1), 3, 100) == a(kv // 2) + a(kv8 // 2) + a(4 * 3)


@pytest.mark.parametrize("bad", [dict(hidden=200), dict(head_dim=96), dict(n_kv_heads=3), dict(ffn=100),
                                 dict(vocab=1000), dict(max_block=33), dict(max_block=0), dict(dtype=5),
                                 dict(mask_token_id=1024), dict(layers=0), dict(n_target_feats=0),
                                 dict(kv_bf16=1), dict(dtype=1, kv_bf16=2), dict(head_bf16=1),
                                 dict(dtype=1, head_bf16=2)])
def test_bad_configs_are_rejected_on_the_host(L, bad):
    c = _cfg(**bad)
    assert L.dflash_cache_bytes(ctypes.byref(c), 1, 16) == 0
    h = ctypes.c_void_p()
    from block_diffusion_drafter_dflash_gb300 import _abi
    w = _abi.Weights()
    rc = L.dflash_model_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h))
    assert rc in (-1, -2) and not h.value
    assert len(L.dflash_last_error()) > 0


def test_verify_argument_checks_need_no_device(L):
    assert L.dflash_verify_greedy(None, None, 0, 16, None, None, None, None) == 0    # empty batch: no launch
    assert L.dflash_verify_greedy(None, None, 1, 0, None, None, None, None) == -2
    assert L.dflash_verify_greedy(None, None, 1, 33, None, None, None, None) == -2
    assert L.dflash_verify_greedy(None, None, -1, 4, None, None, None, None) == -1
    assert L.dflash_verify_greedy(None, None, 2, 4, None, None, None, None) == -1


def test_null_handles_are_rejected(L):
    assert L.dflash_inject_context(None, None, None, None, None, 0, None, 0, None) == -1
    assert L.dflash_draft_block(None, None, None, 4, None, None, None, 0, None) == -1
    assert L.dflash_model_destroy(None) == 0
    assert L.dflash_workspace_bytes(None, 1, 1, 4, 4) == 0
    assert L.dflash_selftest_wait_timeout(None, 1000, None) == -1


def test_product_path_has_no_oracle_or_cpu_fallback():
    """The package never imports the oracle and fails loudly without its library."""
    pkg = os.path.join(ROOT, "block_diffusion_drafter_dflash_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_one_plane_cache_is_20480_bytes_a_token_at_the_8b_shape(L):
    from block_diffusion_drafter_dflash_gb300 import _config_struct
    from dflash_inputs import QWEN3_8B, replace
    cap = 32768 + 512
    two = L.dflash_cache_bytes(ctypes.byref(_config_struct(QWEN3_8B)), 4, cap)
    one = L.dflash_cache_bytes(ctypes.byref(_config_struct(replace(QWEN3_8B, kv_bf16=True))), 4, cap)
    assert abs(two - 2 * one) < 4096
    # 5 layers x 8 kv heads x 128 x (K and V) x 2 bytes = 20,480 bytes a token
    assert abs(one - 4 * cap * 20480) < 4096
