"""Python binding of the CPU oracle (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import this
package. It loads liboracle_f64.so (double, the default) or liboracle_f32.so (float), built from
oracle.c by :func:`build`. It imports nothing from the CUDA package and the CUDA package imports
nothing from here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_libs: dict = {}
_lock = threading.Lock()

OK, ERR_NONFINITE, ERR_INVALID = 0, -1, -2


def lib_path(precision: str = "f64") -> str:
    return os.path.join(_HERE, f"liboracle_{precision}.so")


def build(force: bool = False) -> None:
    """Compile both precisions of the oracle with gcc (-O2, OpenMP, no fast-math)."""
    for prec, real in (("f64", "double"), ("f32", "float")):
        out = lib_path(prec)
        newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
        if force or not os.path.exists(out) or os.path.getmtime(out) < newest:
            tmp = out + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                                   f"-DORACLE_REAL={real}", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, out)


class _Layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "wq", "wk", "wv", "wo", "wg", "wu", "wd",
        "sq", "sk", "sv", "so", "sg", "su", "sd",
        "bq", "bk", "bv", "g1", "g2")]


class _Model(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "max_ctx")] + [
        ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_double),
        ("weight_format", ctypes.c_int), ("group_size", ctypes.c_int),
        ("scale_is_bf16", ctypes.c_int), ("qkv_bias", ctypes.c_int),
        ("embed", ctypes.c_void_p), ("lm_head", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
        ("layers", ctypes.POINTER(_Layer))]


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags.c_contiguous, "oracle inputs must be contiguous"
    return a.ctypes.data


class Oracle:
    """The oracle's functions on numpy arrays. precision: 'f64' (default) or 'f32'."""

    def __init__(self, precision: str = "f64"):
        with _lock:
            if precision not in _libs:
                build()
                _libs[precision] = self._declare(ctypes.CDLL(lib_path(precision)))
        self.lib = _libs[precision]
        self.precision = precision
        self.real = np.float64 if precision == "f64" else np.float32
        assert self.lib.orc_real_bytes() == np.dtype(self.real).itemsize

    @staticmethod
    def _declare(lib):
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        sig = {
            "orc_real_bytes": ([], I), "orc_set_threads": ([I], None), "orc_get_threads": ([], I),
            "orc_bf16_value": ([ctypes.c_uint16], D), "orc_fp16_value": ([ctypes.c_uint16], D),
            "orc_round_bf16": ([D], ctypes.c_uint16),
            "orc_rmsnorm": ([P, P, I, D, P], None),
            "orc_gemv_bf16": ([P, I, I, P, P], None),
            "orc_dequant_int4": ([P, P, I, I, I, I, P], None),
            "orc_gemv_int4": ([P, P, I, I, I, I, P, P], None),
            "orc_rope": ([P, I, I, D], None),
            "orc_softmax": ([P, I, P], None),
            "orc_attention": ([P, P, P, I, I, I, I, I, P], None),
            "orc_attention_partials": ([P, P, P, I, I, I, I, I, I, I, P, P, P], None),
            "orc_attention_combine": ([P, P, P, I, I, I, P], None),
            "orc_swiglu": ([P, P, I, P], None),
            "orc_argmax": ([P, I, ctypes.POINTER(I)], I),
            "orc_decode_step": ([ctypes.POINTER(_Model), I, I, P, P, P, ctypes.POINTER(I), P], I),
            "orc_moe_mlp": ([I, I, I, I, I, P, P, P, P, P, P, I, P, P, P, P], None),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes, f.restype = args, res
        return lib

    def _r(self, a):
        return np.ascontiguousarray(a, dtype=self.real)

    def set_threads(self, n: int) -> None:
        self.lib.orc_set_threads(int(n))

    def threads(self) -> int:
        return self.lib.orc_get_threads()

    # scalar formats
    def bf16_value(self, bits: int) -> float:
        return self.lib.orc_bf16_value(int(bits))

    def fp16_value(self, bits: int) -> float:
        return self.lib.orc_fp16_value(int(bits))

    def round_bf16(self, v: float) -> int:
        return int(self.lib.orc_round_bf16(float(v)))

    # building blocks
    def rmsnorm(self, x, gain_bits, eps):
        x = self._r(x)
        y = np.empty_like(x)
        self.lib.orc_rmsnorm(_p(x), _p(np.ascontiguousarray(gain_bits, np.uint16)), x.size, eps, _p(y))
        return y

    def gemv_bf16(self, w_bits, x):
        w = np.ascontiguousarray(w_bits, np.uint16)
        x = self._r(x)
        y = np.empty(w.shape[0], self.real)
        self.lib.orc_gemv_bf16(_p(w), w.shape[0], w.shape[1], _p(x), _p(y))
        return y

    def dequant_int4(self, wq, scales, scale_is_bf16, group):
        wq = np.ascontiguousarray(wq, np.uint8)
        s = np.ascontiguousarray(scales, np.uint16)
        rows, cols = wq.shape[0], wq.shape[1] * 2
        out = np.empty((rows, cols), self.real)
        self.lib.orc_dequant_int4(_p(wq), _p(s), int(scale_is_bf16), rows, cols, group, _p(out))
        return out

    def gemv_int4(self, wq, scales, scale_is_bf16, group, x):
        wq = np.ascontiguousarray(wq, np.uint8)
        s = np.ascontiguousarray(scales, np.uint16)
        x = self._r(x)
        y = np.empty(wq.shape[0], self.real)
        self.lib.orc_gemv_int4(_p(wq), _p(s), int(scale_is_bf16), wq.shape[0], wq.shape[1] * 2,
                               group, _p(x), _p(y))
        return y

    def rope(self, v, pos, theta):
        v = self._r(v).copy()
        self.lib.orc_rope(_p(v), v.size, int(pos), float(theta))
        return v

    def softmax(self, s):
        s = self._r(s)
        p = np.empty_like(s)
        self.lib.orc_softmax(_p(s), s.size, _p(p))
        return p

    def attention(self, q, k_bits, v_bits, n_heads, n_kv_heads, head_dim, n_ctx):
        """k_bits, v_bits: uint16 [n_kv_heads][ctx_stride][head_dim] of one layer."""
        q = self._r(q)
        k = np.ascontiguousarray(k_bits, np.uint16)
        v = np.ascontiguousarray(v_bits, np.uint16)
        out = np.empty(n_heads * head_dim, self.real)
        self.lib.orc_attention(_p(q), _p(k), _p(v), n_heads, n_kv_heads, head_dim, n_ctx,
                               k.shape[1], _p(out))
        return out

    def attention_partials(self, q, k_bits, v_bits, n_heads, n_kv_heads, head_dim, n_ctx,
                           chunk_len, n_chunks):
        q = self._r(q)
        k = np.ascontiguousarray(k_bits, np.uint16)
        v = np.ascontiguousarray(v_bits, np.uint16)
        m = np.empty((n_heads, n_chunks), self.real)
        l = np.empty((n_heads, n_chunks), self.real)
        o = np.empty((n_heads, n_chunks, head_dim), self.real)
        self.lib.orc_attention_partials(_p(q), _p(k), _p(v), n_heads, n_kv_heads, head_dim, n_ctx,
                                        k.shape[1], chunk_len, n_chunks, _p(m), _p(l), _p(o))
        return m, l, o

    def attention_combine(self, m, l, o):
        m, l, o = self._r(m), self._r(l), self._r(o)
        n_heads, n_chunks, head_dim = o.shape
        out = np.empty(n_heads * head_dim, self.real)
        self.lib.orc_attention_combine(_p(m), _p(l), _p(o), n_heads, head_dim, n_chunks, _p(out))
        return out

    def swiglu(self, gate, up):
        g, u = self._r(gate), self._r(up)
        a = np.empty_like(g)
        self.lib.orc_swiglu(_p(g), _p(u), g.size, _p(a))
        return a

    def moe_mlp(self, fmt, group, scale_is_bf16, wg, sg, wu, su, wd, sd, ids, weights, x):
        """Gathered-expert SwiGLU MLP (orc_moe_mlp): expert matrices stacked along the first axis,
        wg, wu [E][ffn_e][...] and wd [E][hidden][...] (bf16 bits or int4 bytes, scales alike)."""
        def c(a, t):
            return None if a is None else np.ascontiguousarray(a, t)
        wt = np.uint8 if fmt == 1 else np.uint16
        wg, wu, wd = c(wg, wt), c(wu, wt), c(wd, wt)
        sg, su, sd = c(sg, np.uint16), c(su, np.uint16), c(sd, np.uint16)
        hidden = wd.shape[1]
        ffn_e = wg.shape[1]
        ids = np.ascontiguousarray(ids, np.int32)
        weights = self._r(weights)
        x = self._r(x)
        y = np.empty(hidden, self.real)
        self.lib.orc_moe_mlp(int(fmt), int(group), int(scale_is_bf16), hidden, ffn_e, _p(wg), _p(sg), _p(wu),
                             _p(su), _p(wd), _p(sd), ids.size, _p(ids), _p(weights), _p(x), _p(y))
        return y

    def argmax(self, logits):
        x = self._r(logits)
        idx = ctypes.c_int(0)
        rc = self.lib.orc_argmax(_p(x), x.size, ctypes.byref(idx))
        return idx.value, rc

    # the whole step
    def model(self, cfg: dict, weights: dict) -> "OracleModel":
        return OracleModel(cfg, weights)

    def decode_step(self, om: "OracleModel", token: int, pos: int, K, V, trace: bool = False):
        """Runs one step in place on the bf16 caches K, V ([L][nkv][max_ctx][d] uint16).
        Returns (logits, argmax, rc[, trace_x])."""
        cfg = om.cfg
        assert K.dtype == np.uint16 and K.flags.c_contiguous and V.flags.c_contiguous
        logits = np.empty(cfg["vocab"], self.real)
        tr = np.empty((cfg["n_layers"], cfg["hidden"]), self.real) if trace else None
        am = ctypes.c_int(0)
        rc = self.lib.orc_decode_step(ctypes.byref(om.struct), int(token), int(pos), _p(K), _p(V),
                                      _p(logits), ctypes.byref(am), _p(tr) if trace else None)
        if trace:
            return logits, am.value, rc, tr
        return logits, am.value, rc


class OracleModel:
    """ctypes view of a canonical weight dict (see synth.make_model); keeps the arrays alive."""

    def __init__(self, cfg: dict, w: dict):
        self.cfg = cfg
        self._keep = []
        int4 = cfg["weight_format"] == "int4"
        layers = (_Layer * cfg["n_layers"])()
        for i, L in enumerate(w["layers"]):
            for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
                setattr(layers[i], name, self._hold(L[name]))
                if int4:
                    setattr(layers[i], "s" + name[1], self._hold(L["s" + name[1]]))
            if cfg["qkv_bias"]:
                for b in ("bq", "bk", "bv"):
                    setattr(layers[i], b, self._hold(L[b]))
            layers[i].g1 = self._hold(L["g1"])
            layers[i].g2 = self._hold(L["g2"])
        self._layers = layers
        s = _Model()
        for f in ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
                  "max_ctx"):
            setattr(s, f, int(cfg[f]))
        s.rope_theta, s.rms_eps = float(cfg["rope_theta"]), float(cfg["rms_eps"])
        s.weight_format = 1 if int4 else 0
        s.group_size = int(cfg.get("group_size") or 0)
        s.scale_is_bf16 = 1 if cfg.get("scale_dtype") == "bf16" else 0
        s.qkv_bias = 1 if cfg["qkv_bias"] else 0
        s.embed = self._hold(w["embed"])
        s.lm_head = self._hold(w["lm_head"])
        s.final_norm = self._hold(w["final_norm"])
        s.layers = ctypes.cast(layers, ctypes.POINTER(_Layer))
        self.struct = s

    def _hold(self, a):
        a = np.ascontiguousarray(a)
        self._keep.append(a)
        return a.ctypes.data
