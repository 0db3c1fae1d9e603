"""ctypes front end of the CPU oracle (oracle/dl_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and
bench.py's cpu_baseline leg (and `bench.py --impl reference`) may import this
package.  The product path (pdl_persistent_megakernel_gb300) never imports or
links it, and it never imports the product's CUDA library: the two share only
the seeded input generator pdl_persistent_megakernel_gb300.synth.

Arrays cross the boundary as numpy arrays: bf16 as uint16 bit patterns, FP8
as uint8 codes, fp32 scales as float32.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dl_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, OpenMP over output rows)."""
    os.makedirs(_BUILD, exist_ok=True)
    hdr = os.path.join(_HERE, "dl_oracle.h")
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= max(os.path.getmtime(_SRC),
                                             os.path.getmtime(hdr))):
        return _SO
    tmp = _SO + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


class Config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("inter", C.c_int),
                ("n_q_heads", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("n_layers", C.c_int),
                ("vocab", C.c_int), ("eps", C.c_double),
                ("rope_theta", C.c_double), ("fp8", C.c_int),
                ("num_requests", C.c_int), ("tokens_per_request", C.c_int),
                ("page_size", C.c_int), ("num_pages", C.c_int),
                ("max_pages_per_request", C.c_int)]


class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "ln1_w", "w_qkv", "w_qkv_scale", "q_norm_w", "k_norm_w", "w_o",
        "w_o_scale", "ln2_w", "w_gate_up", "w_gate_up_scale", "w_down",
        "w_down_scale")]


TRACE_FIELDS = ("r1", "h1", "h1_codes", "h1_scales", "q_rot", "k_rot", "v",
                "attn", "attn_codes", "attn_scales", "o2", "r2", "h2",
                "h2_codes", "h2_scales", "act", "act_codes", "act_scales", "y")


class LayerTrace(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in TRACE_FIELDS]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            L.or_bf16_to_double.argtypes = [C.c_uint16]
            L.or_bf16_to_double.restype = C.c_double
            L.or_bf16_from_double.argtypes = [C.c_double]
            L.or_bf16_from_double.restype = C.c_uint16
            L.or_e4m3_decode.argtypes = [C.c_uint8]
            L.or_e4m3_decode.restype = C.c_double
            L.or_e4m3_encode.argtypes = [C.c_double]
            L.or_e4m3_encode.restype = C.c_uint8
            L.or_silu.argtypes = [C.c_double]
            L.or_silu.restype = C.c_double
            L.or_add_rmsnorm.argtypes = [C.c_int, C.c_int, u16p, u16p, u16p,
                                         C.c_double, C.c_void_p, C.c_void_p,
                                         C.c_void_p]
            L.or_quant_group128.argtypes = [C.c_int, C.c_int, f32p, u8p, f32p]
            L.or_gemm_bf16.argtypes = [C.c_int, C.c_int, C.c_int, f64p, u16p,
                                       f64p]
            L.or_gemm_fp8.argtypes = [C.c_int, C.c_int, C.c_int, u8p, f32p,
                                      u8p, f32p, f64p]
            L.or_head_rmsnorm.argtypes = [C.c_int, f64p, u16p, C.c_double,
                                          f64p]
            L.or_rope.argtypes = [C.c_int, f64p, C.c_int, C.c_double, f64p]
            L.or_kv_offset.argtypes = [C.c_int] * 10
            L.or_kv_offset.restype = C.c_size_t
            L.or_kv_page.argtypes = [i32p] + [C.c_int] * 5
            L.or_kv_page.restype = C.c_int
            L.or_kv_gather.argtypes = [u16p, i32p] + [C.c_int] * 10 + [u16p]
            L.or_kv_gather.restype = C.c_int
            L.or_attention_partial.argtypes = [C.c_int, f64p, u16p, u16p,
                                               C.c_int, C.c_int, C.c_int,
                                               f64p, C.POINTER(C.c_double)]
            L.or_lse_combine.argtypes = [C.c_int, C.c_int, f64p, f64p, f64p,
                                         C.POINTER(C.c_double)]
            L.or_argmax.argtypes = [C.c_int, f32p]
            L.or_argmax.restype = C.c_int32
            L.or_decode_layer.argtypes = [
                C.POINTER(Config), C.c_int, C.POINTER(LayerWeights), u16p,
                u16p, u16p, i32p, i32p, u16p, u16p, C.c_void_p]
            L.or_decode_layer.restype = C.c_int
            L.or_decode_step.argtypes = [
                C.POINTER(Config), C.POINTER(LayerWeights), C.c_void_p,
                C.c_void_p, u16p, u16p, u16p, i32p, i32p, C.c_void_p,
                C.c_void_p, C.c_void_p, C.c_void_p]
            L.or_decode_step.restype = C.c_int
            L.or_num_threads.restype = C.c_int
            L.or_set_num_threads.argtypes = [C.c_int]
            _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


# ----------------------------------------------------------------- scalars

def bf16_from_double(v) -> np.ndarray:
    L = lib()
    v = np.asarray(v, dtype=np.float64)
    return np.array([L.or_bf16_from_double(float(x)) for x in v.ravel()],
                    dtype=np.uint16).reshape(v.shape)


def bf16_to_double(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_decode(codes) -> np.ndarray:
    L = lib()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([L.or_e4m3_decode(int(x)) for x in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def e4m3_encode(v) -> np.ndarray:
    L = lib()
    v = np.asarray(v, dtype=np.float64)
    return np.array([L.or_e4m3_encode(float(x)) for x in v.ravel()],
                    dtype=np.uint8).reshape(v.shape)


def silu(z) -> np.ndarray:
    L = lib()
    z = np.asarray(z, dtype=np.float64)
    return np.array([L.or_silu(float(x)) for x in z.ravel()]).reshape(z.shape)


# --------------------------------------------------------------------- ops

def add_rmsnorm(x, res, w, eps):
    x = np.ascontiguousarray(x, np.uint16)
    res = np.ascontiguousarray(res, np.uint16)
    w = np.ascontiguousarray(w, np.uint16)
    M, H = x.shape
    r = np.empty((M, H), np.uint16)
    hb = np.empty((M, H), np.uint16)
    hf = np.empty((M, H), np.float32)
    lib().or_add_rmsnorm(M, H, x, res, w, eps, _ptr(r), _ptr(hb), _ptr(hf))
    return r, hb, hf


def quant_group128(v):
    v = np.ascontiguousarray(v, np.float32)
    M, K = v.shape
    codes = np.empty((M, K), np.uint8)
    scales = np.empty((M, K // 128), np.float32)
    lib().or_quant_group128(M, K, v, codes, scales)
    return codes, scales


def gemm_bf16(a, w):
    a = np.ascontiguousarray(a, np.float64)
    w = np.ascontiguousarray(w, np.uint16)
    M, K = a.shape
    N = w.shape[0]
    out = np.empty((M, N), np.float64)
    lib().or_gemm_bf16(M, N, K, a, w, out)
    return out


def gemm_fp8(a_codes, a_scales, w_codes, w_scales):
    a_codes = np.ascontiguousarray(a_codes, np.uint8)
    w_codes = np.ascontiguousarray(w_codes, np.uint8)
    a_scales = np.ascontiguousarray(a_scales, np.float32)
    w_scales = np.ascontiguousarray(w_scales, np.float32)
    M, K = a_codes.shape
    N = w_codes.shape[0]
    out = np.empty((M, N), np.float64)
    lib().or_gemm_fp8(M, N, K, a_codes, a_scales, w_codes, w_scales, out)
    return out


def head_rmsnorm(v, w, eps):
    v = np.ascontiguousarray(v, np.float64)
    out = np.empty_like(v)
    lib().or_head_rmsnorm(v.shape[0], v, np.ascontiguousarray(w, np.uint16),
                          eps, out)
    return out


def rope(v, pos, theta):
    v = np.ascontiguousarray(v, np.float64)
    out = np.empty_like(v)
    lib().or_rope(v.shape[0], v, int(pos), float(theta), out)
    return out


def kv_offset(num_pages, n_kv_heads, page_size, head_dim, layer, page, kv,
              head, slot, dim) -> int:
    return int(lib().or_kv_offset(num_pages, n_kv_heads, page_size, head_dim,
                                  layer, page, kv, head, slot, dim))


def kv_gather(kv_pages, block_table, n_kv_heads, page_size, head_dim, layer,
              r, h, kv, n_keys):
    kvp = np.ascontiguousarray(kv_pages, np.uint16).reshape(-1)
    bt = np.ascontiguousarray(block_table, np.int32)
    num_pages = kv_pages.shape[1] if kv_pages.ndim == 6 else None
    assert num_pages is not None
    out = np.empty((n_keys, head_dim), np.uint16)
    rc = lib().or_kv_gather(kvp, bt, bt.shape[1], num_pages, n_kv_heads,
                            page_size, head_dim, layer, r, h, kv, n_keys, out)
    if rc != 0:
        raise ValueError("kv_gather: page out of range")
    return out


def attention_partial(q, K, V, k0, k1, last):
    q = np.ascontiguousarray(q, np.float64)
    K = np.ascontiguousarray(K, np.uint16)
    V = np.ascontiguousarray(V, np.uint16)
    o = np.empty(q.shape[0], np.float64)
    lse = C.c_double()
    lib().or_attention_partial(q.shape[0], q, K, V, k0, k1, last, o,
                               C.byref(lse))
    return o, lse.value


def lse_combine(o_parts, lse_parts):
    o_parts = np.ascontiguousarray(o_parts, np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, np.float64)
    n, d = o_parts.shape
    o = np.empty(d, np.float64)
    lse = C.c_double()
    lib().or_lse_combine(d, n, o_parts, lse_parts, o, C.byref(lse))
    return o, lse.value


def argmax(logits) -> int:
    logits = np.ascontiguousarray(logits, np.float32)
    return int(lib().or_argmax(logits.shape[0], logits))


def num_threads() -> int:
    return int(lib().or_num_threads())


def set_num_threads(n: int) -> None:
    lib().or_set_num_threads(int(n))


# ------------------------------------------------------------- composition

def _np(t):
    """torch tensor or numpy array -> contiguous numpy (bf16 -> uint16)."""
    if t is None:
        return None
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy()
    except ImportError:
        pass
    return np.ascontiguousarray(t)


def make_config(cfg) -> Config:
    return Config(cfg.hidden, cfg.inter, cfg.n_q_heads, cfg.n_kv_heads,
                  cfg.head_dim, cfg.n_layers, cfg.vocab, cfg.eps,
                  cfg.rope_theta, int(cfg.fp8), cfg.num_requests,
                  cfg.tokens_per_request, cfg.page_size, cfg.num_pages,
                  cfg.pages_per_request)


def _layer_struct(lw: dict, keep: list) -> LayerWeights:
    s = LayerWeights()
    for name, _ in LayerWeights._fields_:
        a = _np(lw.get(name))
        if a is not None:
            keep.append(a)
            setattr(s, name, a.ctypes.data)
    return s


def _alloc_trace(cfg):
    M, H, I = cfg.M, cfg.hidden, cfg.inter
    qd, kvd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    shapes = {"r1": (M, H), "q_rot": (M, qd), "k_rot": (M, kvd),
              "v": (M, kvd), "o2": (M, H), "r2": (M, H), "y": (M, H)}
    if cfg.fp8:
        shapes.update({"h1_codes": (M, H), "h1_scales": (M, H // 128),
                       "attn_codes": (M, qd), "attn_scales": (M, qd // 128),
                       "h2_codes": (M, H), "h2_scales": (M, H // 128),
                       "act_codes": (M, I), "act_scales": (M, I // 128)})
    else:
        shapes.update({"h1": (M, H), "attn": (M, qd), "h2": (M, H),
                       "act": (M, I)})
    arrs = {}
    for k, shp in shapes.items():
        dt = (np.uint8 if k.endswith("codes") else
              np.float32 if k.endswith("scales") else np.uint16)
        arrs[k] = np.zeros(shp, dt)
    tr = LayerTrace()
    for k, a in arrs.items():
        setattr(tr, k, a.ctypes.data)
    return tr, arrs


def decode_step(cfg, weights: dict, inputs: dict, trace: bool = False,
                threads: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Run the whole step on the CPU.  `inputs["kv_pages"]` is copied; the
    updated cache is returned under "kv_pages".  Returns out [2, M, H] (layer
    plans) or logits [M, V] + ids [M] (full plans), plus the last layer's
    intermediates when trace=True."""
    L = lib()
    if threads is not None:
        L.or_set_num_threads(int(threads))
    keep: list = []
    c = make_config(cfg)
    arr = (LayerWeights * cfg.n_layers)()
    for l, lw in enumerate(weights["layers"]):
        arr[l] = _layer_struct(lw, keep)
    x = _np(inputs["x"])
    res = _np(inputs["residual"])
    kv = _np(inputs["kv_pages"]).copy()
    bt = np.ascontiguousarray(_np(inputs["block_table"]), np.int32)
    pos = np.ascontiguousarray(_np(inputs["positions"]), np.int32)
    fn = _np(weights.get("final_norm_w"))
    lm = _np(weights.get("lm_head_w"))
    M, H = cfg.M, cfg.hidden
    out = np.zeros((2, M, H), np.uint16) if cfg.vocab == 0 else None
    logits = np.zeros((M, cfg.vocab), np.float32) if cfg.vocab else None
    ids = np.zeros((M,), np.int32) if cfg.vocab else None
    tr, tarrs = _alloc_trace(cfg) if trace else (None, {})
    rc = L.or_decode_step(C.byref(c), arr, _ptr(fn), _ptr(lm), x, res,
                          kv.reshape(-1), bt, pos, _ptr(out), _ptr(logits),
                          _ptr(ids), C.byref(tr) if tr is not None else None)
    if rc != 0:
        raise ValueError("oracle decode_step rejected its arguments")
    res_d = {"kv_pages": kv}
    if out is not None:
        res_d["out"] = out
    if logits is not None:
        res_d["logits"] = logits
        res_d["ids"] = ids
    res_d.update(tarrs)
    return res_d
