"""The C-ABI library on the CPU: it loads, exports every function include/tinfer.h declares, and
its host-side logic (configuration checks, packed sizes, status strings, the prefill product's
argument checks) behaves as documented.
No compute call is made here."""
import ctypes
import os
import re

import pytest

import decode_persistent_megakernel_gb300 as T
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    T.build()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tinfer.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tinfer_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 18
    lib = ctypes.CDLL(T.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(T.EXPORTS) == names


@pytest.mark.parametrize("name", list(synth.CONFIGS))
def test_workloads_are_valid_configs(name):
    c = T.make_config(synth.config(name))
    assert T.tinfer_check_config(c) == T.TINFER_OK
    for mode in (T.TINFER_MEGAKERNEL, T.TINFER_GRAPH):
        c.exec_mode = mode
        assert T.tinfer_check_config(c) == T.TINFER_OK


def test_invalid_and_unsupported_configs_are_rejected():
    base = synth.config("tiny")
    cases = [
        (dict(n_kv_heads=3), T.TINFER_ERR_INVALID_ARG),
        (dict(head_dim=63), T.TINFER_ERR_INVALID_ARG),
        (dict(vocab=0), T.TINFER_ERR_INVALID_ARG),
        (dict(n_heads=16, n_kv_heads=1), T.TINFER_ERR_UNSUPPORTED),   # 16 query heads per KV head
        (dict(head_dim=256), T.TINFER_ERR_UNSUPPORTED),
        (dict(hidden=260), T.TINFER_ERR_UNSUPPORTED),                  # rows not 16-byte multiples
        (dict(weight_format="int4", group_size=48), T.TINFER_ERR_UNSUPPORTED),
        (dict(weight_format="int4", group_size=64), T.TINFER_ERR_UNSUPPORTED),  # ffn 688 not /64
        (dict(max_ctx=10 ** 6), T.TINFER_ERR_UNSUPPORTED),
        (dict(n_layers=65), T.TINFER_ERR_UNSUPPORTED),
    ]
    for over, want in cases:
        c = dict(base)
        c.update(over)
        assert T.tinfer_check_config(T.make_config(c)) == want, over
    cfg = T.make_config(base)
    cfg.exec_mode = 7
    assert T.tinfer_check_config(cfg) == T.TINFER_ERR_INVALID_ARG
    assert T.lib().tinfer_check_config(None) == T.TINFER_ERR_INVALID_ARG


def test_packed_row_bytes():
    assert T.tinfer_packed_row_bytes(T.TINFER_BF16, 2048, 0) == 4096
    assert T.tinfer_packed_row_bytes(T.TINFER_BF16, 2044, 0) == 0
    assert T.tinfer_packed_row_bytes(T.TINFER_INT4, 2048, 64) == 1024 + 64
    assert T.tinfer_packed_row_bytes(T.TINFER_INT4, 2560, 128) == 1328  # 1280 + 40, padded to 16
    assert T.tinfer_packed_row_bytes(T.TINFER_INT4, 2048, 48) == 0


def test_packed_layer_bytes_cover_every_part():
    c = synth.config("llama1b")
    n = T.tinfer_packed_layer_bytes(T.make_config(c))
    raw = synth.model_bytes(c)["per_layer"]
    # bf16 gains become fp32 (+2 x 2 x hidden bytes); every part starts on a 256-byte boundary
    assert raw + 4 * c["hidden"] <= n <= raw + 4 * c["hidden"] + 6 * 256
    ci = synth.config("int4_3b")
    ni = T.tinfer_packed_layer_bytes(T.make_config(ci))
    assert ni >= synth.model_bytes(ci)["per_layer"]


def test_status_strings():
    assert T.status_string(T.TINFER_OK) == "ok"
    assert T.status_string(T.TINFER_ERR_TIMEOUT) == "device wait timed out"
    assert T.status_string(99) == "unknown status"


def test_gemm_arguments_are_checked_before_any_device_work():
    # every case below fails the host checks of tinfer_op_gemm_bf16 before its first CUDA call, so
    # the stand-in addresses are never dereferenced and the test is safe with or without a GPU
    a = 1 << 20  # 16-byte aligned stand-in address
    bad = T.TINFER_ERR_INVALID_ARG
    assert T.tinfer_op_gemm_bf16(0, 4, 64, a, a, a) == bad        # empty M
    assert T.tinfer_op_gemm_bf16(4, 0, 64, a, a, a) == bad        # empty N
    assert T.tinfer_op_gemm_bf16(4, 4, 0, a, a, a) == bad         # empty K
    assert T.tinfer_op_gemm_bf16(4, 4, 12, a, a, a) == bad        # K not a multiple of 8 (row stride)
    assert T.tinfer_op_gemm_bf16(4, 4, 64, a + 2, a, a) == bad    # X base not 16-byte aligned
    assert T.tinfer_op_gemm_bf16(4, 4, 64, a, a + 8, a) == bad    # W base not 16-byte aligned
    assert T.tinfer_op_gemm_bf16(4, 4, 64, a, a, a + 2) == bad    # Y not 4-byte aligned
    assert T.tinfer_op_gemm_bf16(4, 4, 64, None, a, a) == bad
    assert T.tinfer_op_gemm_bf16(4, 4, 64, a, None, a) == bad
    assert T.tinfer_op_gemm_bf16(4, 4, 64, a, a, None) == bad
