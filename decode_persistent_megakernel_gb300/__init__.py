"""Python binding of libtinfer.so, the GB300 batch-1 decode engine (include/tinfer.h).

The functions below carry the C names and only marshal arguments: every step of the decode path
runs in the library's CUDA kernels. PyTorch is used for device memory and streams. There is no
fallback: if the library is missing or the GPU is absent, calls raise.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtinfer.so")

TINFER_OK, TINFER_ERR_INVALID_ARG, TINFER_ERR_UNSUPPORTED, TINFER_ERR_CUDA, TINFER_ERR_OOM, \
    TINFER_ERR_NONFINITE, TINFER_ERR_TIMEOUT = range(7)
TINFER_BF16, TINFER_INT4 = 0, 1
TINFER_SCALE_FP16, TINFER_SCALE_BF16 = 0, 1
TINFER_MEGAKERNEL, TINFER_GRAPH = 0, 1
TINFER_Q_GRID, TINFER_Q_SMEM, TINFER_Q_RING_STAGES, TINFER_Q_SLOT_BYTES, TINFER_Q_KERNELS_PER_STEP, \
    TINFER_Q_TRACE_BYTES, TINFER_Q_BLOCK_THREADS = range(7)
TINFER_EPI_STORE, TINFER_EPI_RESIDUAL, TINFER_EPI_SWIGLU, TINFER_EPI_ARGMAX = range(4)
TINFER_S_INFLIGHT, TINFER_S_INFLIGHT_LM, TINFER_S_L2_LOOKAHEAD, TINFER_S_L2_PACE, TINFER_S_SYNC, TINFER_S_ATTN_CHUNKS = range(6)
TINFER_SYNC_STAMPS, TINFER_SYNC_GRID_BARRIER = 0, 1
TINFER_NOALLOC_SCRATCH_BYTES = 1 << 20
TRACE_FIELDS = 10  # stamps per CTA and phase of the timeline (tinfer_set_trace)

EXPORTS = [
    "tinfer_status_string", "tinfer_check_config", "tinfer_packed_layer_bytes", "tinfer_pack_layer",
    "tinfer_unpack_layer", "tinfer_create", "tinfer_decode_step", "tinfer_decode_step_dev",
    "tinfer_generate", "tinfer_generate_dev", "tinfer_get_error", "tinfer_query", "tinfer_set_trace", "tinfer_set_timeout_ns",
    "tinfer_debug_withhold_results", "tinfer_set_schedule", "tinfer_get_schedule", "tinfer_destroy",
    "tinfer_packed_row_bytes", "tinfer_pack_matrix", "tinfer_op_gemv", "tinfer_op_attention",
    "tinfer_op_attention_noalloc", "tinfer_op_gemv_batch", "tinfer_moe_packed_bytes", "tinfer_pack_moe", "tinfer_op_moe",
    "tinfer_op_gemm_bf16",
]


class TinferError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: tinfer status {status} ({status_string(status)})")


class tinfer_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "max_ctx")] + [
        ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_double)] + [
        (n, ctypes.c_int) for n in ("weight_format", "group_size", "scale_dtype", "tied_embeddings",
                                    "qkv_bias", "exec_mode", "ffn_split")]


class tinfer_layer_src(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "wq", "wk", "wv", "wo", "wg", "wu", "wd", "sq", "sk", "sv", "so", "sg", "su", "sd",
        "bq", "bk", "bv", "g1", "g2")]


class tinfer_weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("final_norm", ctypes.c_void_p), ("layer_blobs", ctypes.POINTER(ctypes.c_void_p))]


_lib = None


def build(force: bool = False) -> str:
    from .build import build as _build
    return _build(force=force)


def lib():
    """The loaded library. Raises if it has not been built: there is no other implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run decode_persistent_megakernel_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, D, Z, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_size_t, ctypes.c_longlong
        cfgp = ctypes.POINTER(tinfer_config)
        sig = {
            "tinfer_status_string": ([I], ctypes.c_char_p),
            "tinfer_check_config": ([cfgp], I),
            "tinfer_packed_layer_bytes": ([cfgp], Z),
            "tinfer_pack_layer": ([cfgp, ctypes.POINTER(tinfer_layer_src), P, P], I),
            "tinfer_unpack_layer": ([cfgp, P, ctypes.POINTER(tinfer_layer_src), P], I),
            "tinfer_create": ([cfgp, ctypes.POINTER(tinfer_weights), P, P, ctypes.POINTER(P)], I),
            "tinfer_decode_step": ([P, ctypes.c_int32, ctypes.c_int32, P, P, P], I),
            "tinfer_decode_step_dev": ([P, P, ctypes.c_int32, P, P, P], I),
            "tinfer_generate": ([P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P], I),
            "tinfer_generate_dev": ([P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P, P], I),
            "tinfer_get_error": ([P], I),
            "tinfer_query": ([P, I], LL),
            "tinfer_set_trace": ([P, P], I),
            "tinfer_set_timeout_ns": ([P, LL], I),
            "tinfer_debug_withhold_results": ([P, I, I], I),
            "tinfer_set_schedule": ([P, I, LL], I),
            "tinfer_get_schedule": ([P, I], LL),
            "tinfer_destroy": ([P], None),
            "tinfer_packed_row_bytes": ([I, I, I], Z),
            "tinfer_pack_matrix": ([I, I, I, I, I, P, P, P, P], I),
            "tinfer_op_gemv": ([I, I, I, I, I, P, P, P, D, P, I, P, P, P], I),
            "tinfer_op_attention": ([I, I, I, I, D, I, I, P, P, P, P, P, P, P, P], I),
            "tinfer_op_attention_noalloc": ([I, I, I, I, D, I, I, P, P, P, P, P], I),
            "tinfer_op_gemv_batch": ([I, I, I, I, I, I, P, P, P, I, P, P], I),
            "tinfer_moe_packed_bytes": ([I, I, I, I, I, I], Z),
            "tinfer_pack_moe": ([I, I, I, I, I, I, P, P, P, P, P, P, P, P, P], I),
            "tinfer_op_moe": ([I, I, I, I, I, I, I, P, P, P, P, P, P, P, I, P, P], I),
            "tinfer_op_gemm_bf16": ([I, I, I, P, P, P, P], I),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes, f.restype = args, res
        _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().tinfer_status_string(int(s)).decode()


def _check(rc: int, what: str) -> int:
    if rc != TINFER_OK:
        raise TinferError(rc, what)
    return rc


def _ptr(t) -> int | None:
    """Device address of a torch tensor (or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ------------------------------------------------------------------ C entry points, same names

def tinfer_check_config(cfg: tinfer_config) -> int:
    return lib().tinfer_check_config(ctypes.byref(cfg))


def tinfer_packed_layer_bytes(cfg: tinfer_config) -> int:
    return lib().tinfer_packed_layer_bytes(ctypes.byref(cfg))


def tinfer_pack_layer(cfg, src: tinfer_layer_src, packed, stream=None) -> int:
    return lib().tinfer_pack_layer(ctypes.byref(cfg), ctypes.byref(src), _ptr(packed), _stream(stream))


def tinfer_unpack_layer(cfg, packed, dst: tinfer_layer_src, stream=None) -> int:
    return lib().tinfer_unpack_layer(ctypes.byref(cfg), _ptr(packed), ctypes.byref(dst), _stream(stream))


def tinfer_create(cfg, weights: tinfer_weights, k_cache, v_cache):
    out = ctypes.c_void_p()
    rc = lib().tinfer_create(ctypes.byref(cfg), ctypes.byref(weights), _ptr(k_cache), _ptr(v_cache),
                             ctypes.byref(out))
    return rc, out


def tinfer_decode_step(ctx, token: int, pos: int, stream=None, logits=None, argmax=None) -> int:
    return lib().tinfer_decode_step(ctx, int(token), int(pos), _stream(stream), _ptr(logits), _ptr(argmax))


def tinfer_decode_step_dev(ctx, token_dev, pos: int, stream=None, logits=None, argmax=None) -> int:
    return lib().tinfer_decode_step_dev(ctx, _ptr(token_dev), int(pos), _stream(stream), _ptr(logits),
                                        _ptr(argmax))


def tinfer_generate(ctx, first_token: int, pos0: int, n_steps: int, stream, tokens_host) -> int:
    """tokens_host: a ctypes int32 array or a writable numpy int32 array of length >= n_steps."""
    if hasattr(tokens_host, "ctypes"):
        ptr = tokens_host.ctypes.data
    else:
        ptr = ctypes.addressof(tokens_host)
    return lib().tinfer_generate(ctx, int(first_token), int(pos0), int(n_steps), _stream(stream), ptr)


def tinfer_generate_dev(ctx, first_token: int, pos0: int, n_steps: int, eos_token: int, stream, tokens_dev,
                        count_dev=None) -> int:
    return lib().tinfer_generate_dev(ctx, int(first_token), int(pos0), int(n_steps), int(eos_token),
                                     _stream(stream), _ptr(tokens_dev), _ptr(count_dev))


def tinfer_get_error(ctx) -> int:
    return lib().tinfer_get_error(ctx)


def tinfer_query(ctx, what: int) -> int:
    return lib().tinfer_query(ctx, what)


def tinfer_set_trace(ctx, trace_dev) -> int:
    return lib().tinfer_set_trace(ctx, _ptr(trace_dev))


def tinfer_set_timeout_ns(ctx, ns: int) -> int:
    return lib().tinfer_set_timeout_ns(ctx, int(ns))


def tinfer_debug_withhold_results(ctx, cta: int, phase: int) -> int:
    return lib().tinfer_debug_withhold_results(ctx, int(cta), int(phase))


def tinfer_set_schedule(ctx, knob: int, value: int) -> int:
    return lib().tinfer_set_schedule(ctx, int(knob), int(value))


def tinfer_get_schedule(ctx, knob: int) -> int:
    return lib().tinfer_get_schedule(ctx, int(knob))


def tinfer_destroy(ctx) -> None:
    lib().tinfer_destroy(ctx)


def tinfer_packed_row_bytes(fmt: int, cols: int, group: int) -> int:
    return lib().tinfer_packed_row_bytes(fmt, cols, group)


def tinfer_pack_matrix(fmt, group, scale_dtype, rows, cols, w, scales, packed, stream=None) -> int:
    return lib().tinfer_pack_matrix(fmt, group, scale_dtype, rows, cols, _ptr(w), _ptr(scales),
                                    _ptr(packed), _stream(stream))


def tinfer_op_gemv(fmt, group, scale_dtype, rows, cols, packed, x, gain, eps, bias, epilogue, y,
                   argmax, stream=None) -> int:
    return lib().tinfer_op_gemv(fmt, group, scale_dtype, rows, cols, _ptr(packed), _ptr(x), _ptr(gain),
                                float(eps), _ptr(bias), epilogue, _ptr(y), _ptr(argmax), _stream(stream))


def tinfer_op_attention(nq, nkv, d, max_ctx, theta, pos, n_chunks, qkv, k_layer, v_layer, out,
                        part_m=None, part_l=None, part_o=None, stream=None) -> int:
    return lib().tinfer_op_attention(nq, nkv, d, max_ctx, float(theta), pos, n_chunks, _ptr(qkv),
                                     _ptr(k_layer), _ptr(v_layer), _ptr(out), _ptr(part_m),
                                     _ptr(part_l), _ptr(part_o), _stream(stream))


def tinfer_op_attention_noalloc(nq, nkv, d, max_ctx, theta, pos, n_chunks, qkv, k_layer, v_layer,
                                out, stream=None) -> int:
    return lib().tinfer_op_attention_noalloc(nq, nkv, d, max_ctx, float(theta), pos, n_chunks,
                                             _ptr(qkv), _ptr(k_layer), _ptr(v_layer), _ptr(out),
                                             _stream(stream))


def tinfer_op_gemv_batch(fmt, group, scale_dtype, rows, cols, m, packed, x, bias, epilogue, y, stream=None) -> int:
    return lib().tinfer_op_gemv_batch(fmt, group, scale_dtype, rows, cols, m, _ptr(packed), _ptr(x), _ptr(bias),
                                      epilogue, _ptr(y), _stream(stream))


def tinfer_moe_packed_bytes(fmt, group, n_experts, hidden, ffn_e, which) -> int:
    return lib().tinfer_moe_packed_bytes(fmt, group, n_experts, hidden, ffn_e, which)


def tinfer_pack_moe(fmt, group, scale_dtype, n_experts, hidden, ffn_e, wg, sg, wu, su, wd, sd, gu_packed,
                    down_packed, stream=None) -> int:
    return lib().tinfer_pack_moe(fmt, group, scale_dtype, n_experts, hidden, ffn_e, _ptr(wg), _ptr(sg), _ptr(wu),
                                 _ptr(su), _ptr(wd), _ptr(sd), _ptr(gu_packed), _ptr(down_packed),
                                 _stream(stream))


def tinfer_op_moe(fmt, group, scale_dtype, n_experts, top_k, hidden, ffn_e, gu_packed, down_packed, ids, weights,
                  x, h, y, accumulate=0, status=None, stream=None) -> int:
    return lib().tinfer_op_moe(fmt, group, scale_dtype, n_experts, top_k, hidden, ffn_e, _ptr(gu_packed),
                               _ptr(down_packed), _ptr(ids), _ptr(weights), _ptr(x), _ptr(h), _ptr(y),
                               int(accumulate), _ptr(status), _stream(stream))


# ------------------------------------------------------------------ marshalling helpers

def tinfer_op_gemm_bf16(m, n, k, x, w, y, stream=None) -> int:
    return lib().tinfer_op_gemm_bf16(m, n, k, _ptr(x), _ptr(w), _ptr(y), _stream(stream))


def make_config(c: dict, exec_mode: int = TINFER_MEGAKERNEL) -> tinfer_config:
    """tinfer_config from a workload description (synth.CONFIGS entries or the same keys)."""
    cfg = tinfer_config()
    for f in ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "max_ctx"):
        setattr(cfg, f, int(c[f]))
    cfg.rope_theta = float(c["rope_theta"])
    cfg.rms_eps = float(c["rms_eps"])
    cfg.weight_format = TINFER_INT4 if c["weight_format"] == "int4" else TINFER_BF16
    cfg.group_size = int(c.get("group_size") or 0)
    cfg.scale_dtype = TINFER_SCALE_BF16 if c.get("scale_dtype") == "bf16" else TINFER_SCALE_FP16
    cfg.tied_embeddings = 1 if c.get("tied") else 0
    cfg.qkv_bias = 1 if c.get("qkv_bias") else 0
    cfg.exec_mode = int(exec_mode)
    cfg.ffn_split = 1 if c.get("ffn_split") else 0
    return cfg


class Engine:
    """Owns the device copies of a canonical model (torch tensors), the packed layers, the KV cache
    and one tinfer context. The model dict is synth.make_model's layout (numpy arrays)."""

    def __init__(self, c: dict, weights: dict, exec_mode: int = TINFER_MEGAKERNEL, device: str = "cuda",
                 kv=None):
        import numpy as np
        import torch
        self.c = c
        self.cfg = make_config(c, exec_mode)
        _check(tinfer_check_config(self.cfg), "tinfer_check_config")
        dev = torch.device(device)
        self.device = dev

        def up(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
            return t.to(dev)

        self.embed = up(weights["embed"])
        self.lm_head = self.embed if weights["lm_head"] is weights["embed"] else up(weights["lm_head"])
        self.final_norm = up(weights["final_norm"])
        nbytes = tinfer_packed_layer_bytes(self.cfg)
        if nbytes == 0:
            raise TinferError(TINFER_ERR_UNSUPPORTED, "tinfer_packed_layer_bytes")
        self.blobs = []
        int4 = c["weight_format"] == "int4"
        for L in weights["layers"]:
            src = tinfer_layer_src()
            keep = {}
            for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
                keep[name] = up(L[name])
                setattr(src, name, _ptr(keep[name]))
                if int4:
                    sname = "s" + name[1]
                    keep[sname] = up(L[sname])
                    setattr(src, sname, _ptr(keep[sname]))
            if c.get("qkv_bias"):
                for b in ("bq", "bk", "bv"):
                    keep[b] = up(L[b])
                    setattr(src, b, _ptr(keep[b]))
            for g in ("g1", "g2"):
                keep[g] = up(L[g])
                setattr(src, g, _ptr(keep[g]))
            blob = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            _check(tinfer_pack_layer(self.cfg, src, blob, torch.cuda.current_stream(dev)), "tinfer_pack_layer")
            self.blobs.append(blob)
            torch.cuda.current_stream(dev).synchronize()  # canonical copies can go
        shape = (c["n_layers"], c["n_kv_heads"], c["max_ctx"], c["head_dim"])
        if kv is not None:
            self.k = up(kv[0]).view(shape)
            self.v = up(kv[1]).view(shape)
        else:
            self.k = torch.zeros(shape, dtype=torch.int16, device=dev)
            self.v = torch.zeros(shape, dtype=torch.int16, device=dev)
        arr = (ctypes.c_void_p * len(self.blobs))(*[b.data_ptr() for b in self.blobs])
        self._blob_arr = arr
        w = tinfer_weights()
        w.embed, w.lm_head, w.final_norm = _ptr(self.embed), _ptr(self.lm_head), _ptr(self.final_norm)
        w.layer_blobs = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
        self._w = w
        rc, ctx = tinfer_create(self.cfg, w, self.k, self.v)
        _check(rc, "tinfer_create")
        self.ctx = ctx
        self.logits = torch.empty(c["vocab"], dtype=torch.float32, device=dev)
        self.argmax = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(self, token: int, pos: int, stream=None, logits=True):
        rc = tinfer_decode_step(self.ctx, token, pos, stream, self.logits if logits else None, self.argmax)
        _check(rc, "tinfer_decode_step")

    def step_dev(self, token_dev, pos: int, stream=None, logits=True, argmax=None):
        rc = tinfer_decode_step_dev(self.ctx, token_dev, pos, stream, self.logits if logits else None,
                                    self.argmax if argmax is None else argmax)
        _check(rc, "tinfer_decode_step_dev")

    def trace_step(self, token: int, pos: int):
        """Runs one traced megakernel step; returns int64 stamps [grid][phases][fields] (ns,
        relative to the earliest stamp; 0 stays 0 where nothing was recorded)."""
        import numpy as np
        import torch
        nbytes = self.query(TINFER_Q_TRACE_BYTES)
        buf = torch.zeros(nbytes // 8, dtype=torch.int64, device=self.device)
        _check(tinfer_set_trace(self.ctx, buf), "tinfer_set_trace")
        self.step(token, pos)
        torch.cuda.synchronize()
        _check(tinfer_set_trace(self.ctx, None), "tinfer_set_trace")
        t = buf.cpu().numpy().reshape(self.query(TINFER_Q_GRID), -1, TRACE_FIELDS)
        return np.where(t > 0, t - t[t > 0].min(), 0)

    def error(self) -> int:
        return tinfer_get_error(self.ctx)

    def query(self, what: int) -> int:
        return tinfer_query(self.ctx, what)

    def close(self):
        if getattr(self, "ctx", None):
            tinfer_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
