"""Seeded synthetic workloads for the batch-1 decode step.

This module makes input bytes only: weights, gains, biases, int4 nibbles and scales, a prefilled
KV cache and token ids, all from the counter-based generator documented in ``synth.c``. It contains
none of the decode step's arithmetic. Both sides of every comparison (the oracle and the CUDA
path) receive the same arrays from here; neither side imports the other.

Canonical layout of a model (numpy arrays, little-endian):
  bf16 tensors          uint16 bit patterns
  matrices              row-major [out][in]
  int4 matrices         uint8 [out][in/2], element 2j = low nibble of byte j, value (q - 8) * s
  int4 scales           uint16 bits (fp16 or bf16) [out][in/group]
  KV cache              uint16 bf16 bits [n_layers][n_kv_heads][max_ctx][head_dim]
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None
_lock = threading.Lock()

# The five workloads. Sizes and distributions are the benchmark's configurations; fields the
# configurations leave open take the readings listed in the design notes (rope theta 10000 for the
# TinyLlama- and 3B-shaped models, eps 1e-5 everywhere, int4 scale |N(0, 0.005)| for both int4
# models).
CONFIGS = {
    "tiny": dict(
        name="tiny-llama-2L-h256", n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64,
        ffn=688, vocab=2048, rope_theta=10000.0, rms_eps=1e-5, weight_format="bf16",
        group_size=0, scale_dtype="fp16", tied=False, qkv_bias=False,
        prompt=16, prefill=0, steps=16),
    "llama1b": dict(
        name="llama-3.2-1b-shaped-bf16", n_layers=16, hidden=2048, n_heads=32, n_kv_heads=8,
        head_dim=64, ffn=8192, vocab=128256, rope_theta=500000.0, rms_eps=1e-5,
        weight_format="bf16", group_size=0, scale_dtype="fp16", tied=True, qkv_bias=False,
        prompt=0, prefill=1024, steps=128),
    "tinyllama_int4": dict(
        name="tinyllama-1.1b-shaped-int4-g64", n_layers=22, hidden=2048, n_heads=32, n_kv_heads=4,
        head_dim=64, ffn=5632, vocab=32000, rope_theta=10000.0, rms_eps=1e-5,
        weight_format="int4", group_size=64, scale_dtype="fp16", tied=False, qkv_bias=False,
        prompt=0, prefill=2048, steps=128),
    "qwen1.5b": dict(
        name="qwen2.5-1.5b-shaped-bf16", n_layers=28, hidden=1536, n_heads=12, n_kv_heads=2,
        head_dim=128, ffn=8960, vocab=151936, rope_theta=1000000.0, rms_eps=1e-5,
        weight_format="bf16", group_size=0, scale_dtype="fp16", tied=True, qkv_bias=True,
        prompt=0, prefill=4096, steps=64),
    "int4_3b": dict(
        name="3b-class-int4-g128-long", n_layers=40, hidden=2560, n_heads=40, n_kv_heads=8,
        head_dim=64, ffn=8192, vocab=49152, rope_theta=10000.0, rms_eps=1e-5,
        weight_format="int4", group_size=128, scale_dtype="bf16", tied=True, qkv_bias=False,
        prompt=0, prefill=8192, steps=64),
}
for _c in CONFIGS.values():
    _c["max_ctx"] = _c["prompt"] + _c["prefill"] + _c["steps"]

WEIGHT_STD = 0.02
SCALE_STD = 0.005


def config(name: str, **overrides) -> dict:
    c = dict(CONFIGS[name])
    c.update(overrides)
    if "max_ctx" not in overrides:
        c["max_ctx"] = c["prompt"] + c["prefill"] + c["steps"]
    return c


def build(force: bool = False) -> str:
    """Compile libsynth.so next to this file (gcc, OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, i64, dbl, ptr = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.synth_normal_bf16.argtypes = [u64, u64, i64, dbl, dbl, ptr]
            lib.synth_abs_normal_16.argtypes = [u64, u64, i64, dbl, ctypes.c_int, ptr]
            lib.synth_nibbles.argtypes = [u64, u64, i64, ptr]
            lib.synth_uniform_int.argtypes = [u64, u64, i64, ctypes.c_int32, ptr]
            lib.synth_words.argtypes = [u64, u64, i64, ptr]
            lib.synth_normals.argtypes = [u64, u64, i64, ptr]
            lib.synth_splitmix.argtypes = [u64, i64, ptr]
            lib.synth_base.argtypes = [u64, u64]
            lib.synth_base.restype = u64
            _lib = lib
    return _lib


def stream_id(name: str) -> int:
    """FNV-1a 64-bit hash of a tensor name: the generator's stream id for that tensor."""
    h = 0xCBF29CE484222325
    for b in name.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def normal_bf16(name: str, shape, mean: float = 0.0, std: float = 1.0, seed: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_bf16(seed, stream_id(name), out.size, mean, std, _ptr(out))
    return out


def abs_normal_16(name: str, shape, std: float, fmt: str, seed: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_abs_normal_16(seed, stream_id(name), out.size, std, 1 if fmt == "bf16" else 0,
                                _ptr(out))
    return out


def nibbles(name: str, shape, seed: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint8)
    _load().synth_nibbles(seed, stream_id(name), out.size, _ptr(out))
    return out


def uniform_int(name: str, n: int, hi: int, seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_uniform_int(seed, stream_id(name), n, hi, _ptr(out))
    return out


def words(name: str, n: int, seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_words(seed, stream_id(name), n, _ptr(out))
    return out


def normals(name: str, n: int, seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_normals(seed, stream_id(name), n, _ptr(out))
    return out


def splitmix(state: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_splitmix(state, n, _ptr(out))
    return out


def base_state(name: str, seed: int = 0) -> int:
    return int(_load().synth_base(seed, stream_id(name)))


LINEARS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def linear_shapes(cfg: dict) -> dict:
    """(out, in) of each linear of a layer."""
    H, qd, kvd, F = cfg["hidden"], cfg["n_heads"] * cfg["head_dim"], \
        cfg["n_kv_heads"] * cfg["head_dim"], cfg["ffn"]
    return dict(wq=(qd, H), wk=(kvd, H), wv=(kvd, H), wo=(H, qd), wg=(F, H), wu=(F, H), wd=(H, F))


def make_model(cfg: dict, seed: int = 0) -> dict:
    """All weights of one synthetic model in the canonical layout.

    Returns {"embed", "lm_head", "final_norm", "layers": [ {wq.., sq.., bq.., g1, g2} ]}. For a
    tied model "lm_head" is the same array object as "embed". bf16 weights ~ N(0, 0.02), gains
    1 + N(0, 0.02), biases N(0, 0.02); int4 nibbles uniform in 0..15 and scales |N(0, 0.005)|.
    """
    H, V = cfg["hidden"], cfg["vocab"]
    m = {"embed": normal_bf16("embed", (V, H), 0.0, WEIGHT_STD, seed)}
    m["lm_head"] = m["embed"] if cfg["tied"] else normal_bf16("lm_head", (V, H), 0.0, WEIGHT_STD, seed)
    m["final_norm"] = normal_bf16("final_norm", (H,), 1.0, WEIGHT_STD, seed)
    shapes = linear_shapes(cfg)
    layers = []
    for li in range(cfg["n_layers"]):
        L = {}
        for w in LINEARS:
            rows, cols = shapes[w]
            key = f"L{li}.{w}"
            if cfg["weight_format"] == "int4":
                g = cfg["group_size"]
                L[w] = nibbles(key, (rows, cols // 2), seed)
                L["s" + w[1]] = abs_normal_16(key + ".scale", (rows, cols // g), SCALE_STD,
                                              cfg["scale_dtype"], seed)
            else:
                L[w] = normal_bf16(key, (rows, cols), 0.0, WEIGHT_STD, seed)
        if cfg["qkv_bias"]:
            for b, w in (("bq", "wq"), ("bk", "wk"), ("bv", "wv")):
                L[b] = normal_bf16(f"L{li}.{b}", (shapes[w][0],), 0.0, WEIGHT_STD, seed)
        L["g1"] = normal_bf16(f"L{li}.g1", (H,), 1.0, WEIGHT_STD, seed)
        L["g2"] = normal_bf16(f"L{li}.g2", (H,), 1.0, WEIGHT_STD, seed)
        layers.append(L)
    m["layers"] = layers
    return m


def make_kv(cfg: dict, prefill: int, seed: int = 0):
    """K and V caches [L][nkv][max_ctx][d] bf16 with slots [0, prefill) ~ N(0, 1), the rest 0."""
    shape = (cfg["n_layers"], cfg["n_kv_heads"], cfg["max_ctx"], cfg["head_dim"])
    K = np.zeros(shape, dtype=np.uint16)
    V = np.zeros(shape, dtype=np.uint16)
    if prefill > 0:
        sub = shape[:2] + (prefill, shape[3])
        K[:, :, :prefill, :] = normal_bf16("kv.K", sub, 0.0, 1.0, seed)
        V[:, :, :prefill, :] = normal_bf16("kv.V", sub, 0.0, 1.0, seed)
    return K, V


def make_tokens(cfg: dict, n: int, seed: int = 0) -> np.ndarray:
    """Uniform token ids in [0, vocab): the prompt (tiny model) or the first decode token."""
    return uniform_int("tokens", n, cfg["vocab"], seed)


def model_bytes(cfg: dict) -> dict:
    """Stored bytes of each part of a model in the canonical layout (no packing padding)."""
    H, V = cfg["hidden"], cfg["vocab"]
    per_layer = 0
    for rows, cols in linear_shapes(cfg).values():
        if cfg["weight_format"] == "int4":
            per_layer += rows * cols // 2 + rows * (cols // cfg["group_size"]) * 2
        else:
            per_layer += rows * cols * 2
    per_layer += 2 * H * 2
    if cfg["qkv_bias"]:
        per_layer += (cfg["n_heads"] + 2 * cfg["n_kv_heads"]) * cfg["head_dim"] * 2
    return dict(per_layer=per_layer, layers=per_layer * cfg["n_layers"], embed=V * H * 2,
                lm_head=V * H * 2, final_norm=H * 2)


def make_moe(n_experts: int, top_k: int, hidden: int, ffn_e: int, weight_format: str = "bf16",
             group_size: int = 64, scale_dtype: str = "fp16", seed: int = 0) -> dict:
    """One gathered-expert MLP case: every expert's gate and up [ffn_e][hidden] and down
    [hidden][ffn_e] matrices stacked along the first axis (bf16 ~ N(0, 0.02), or int4 nibbles with
    scales |N(0, 0.005)|), top_k distinct expert ids drawn uniformly from [0, n_experts), positive
    routing weights (|N(0, 1)| normalised to sum 1, held as float32) and an input vector x ~ N(0, 1)
    (float32)."""
    m = {}
    for name, rows, cols in (("g", ffn_e, hidden), ("u", ffn_e, hidden), ("d", hidden, ffn_e)):
        key = f"moe.w{name}"
        if weight_format == "int4":
            m["w" + name] = nibbles(key, (n_experts, rows, cols // 2), seed)
            m["s" + name] = abs_normal_16(key + ".scale", (n_experts, rows, cols // group_size), SCALE_STD,
                                          scale_dtype, seed)
        else:
            m["w" + name] = normal_bf16(key, (n_experts, rows, cols), 0.0, WEIGHT_STD, seed)
            m["s" + name] = None
    # distinct ids: the first top_k of a seeded shuffle (Fisher-Yates on the generator's words)
    order = list(range(n_experts))
    r = words("moe.ids", n_experts, seed)
    for i in range(n_experts - 1, 0, -1):
        j = int(r[i] % np.uint64(i + 1))
        order[i], order[j] = order[j], order[i]
    m["ids"] = np.array(order[:top_k], dtype=np.int32)
    w = np.abs(normals("moe.weights", top_k, seed))
    m["weights"] = (w / w.sum()).astype(np.float32)
    m["x"] = normals("moe.x", hidden, seed).astype(np.float32)
    return m
