"""GB300 (sm_103a) small-batch decode step, three schedules, behind a C ABI.

The compute path is the CUDA library libdl.so (include/dl.h): every step of
the decode step runs in its kernels.  This module only marshals arguments
through ctypes; PyTorch supplies device memory and streams.  There is no CPU
fallback: if the library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(_ROOT, "include")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libdl.so")
_SOURCES = ["dl_kernels.cu", "dl_host.cu", "dl_noalloc.cu", "dl_bench.cu"]
_HEADERS = ["dl_internal.h", "dl_device.cuh", "dl_ops.cuh", "dl_kernels.h"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

MODE_SERIAL, MODE_PDL_GRAPH, MODE_MEGAKERNEL = 0, 1, 2
MODE_GRAPH_LINEAR, MODE_GRAPH_LINEAR_PDL, MODE_GRAPH_DAG = 3, 4, 5
MODE_NAMES = {0: "serial", 1: "pdl_graph", 2: "megakernel", 3: "graph_linear",
              4: "graph_linear_pdl", 5: "graph_dag"}
ALL_MODES = (1 << 6) - 1

DEBUG_BUFFERS = {"r1": 0, "h1": 1, "h1_scales": 2, "q_rot": 3, "attn": 4,
                 "attn_scales": 5, "o2": 6, "r2": 7, "h2": 8, "h2_scales": 9,
                 "act": 10, "act_scales": 11, "y": 12, "h_final": 16}


def _nvcc() -> str:
    for cand in ("/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand == "nvcc" or os.path.exists(cand):
            return cand
    return "nvcc"


def _cuda_lib_dir() -> str:
    nv = _nvcc()
    base = os.path.dirname(os.path.dirname(os.path.realpath(nv))) if os.path.sep in nv else "/usr/local/cuda"
    return os.path.join(base, "lib64")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libdl.so for sm_103a in-tree (two translation units in
    parallel, then one link)."""
    os.makedirs(_BUILD, exist_ok=True)
    deps = [os.path.join(_CSRC, f) for f in _SOURCES + _HEADERS]
    deps.append(os.path.join(_INCLUDE, "dl.h"))
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= max(os.path.getmtime(d) for d in deps)):
        return _SO
    nv = _nvcc()
    flags = [ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
             "-I" + _INCLUDE, "-I" + _CSRC]
    objs = []

    def compile_one(src):
        obj = os.path.join(_BUILD, src.replace(".cu", f".{os.getpid()}.o"))
        cmd = [nv] + flags + ["-c", os.path.join(_CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout, r.stderr)
        return obj

    with ThreadPoolExecutor(len(_SOURCES)) as ex:
        objs = list(ex.map(compile_one, _SOURCES))
    tmp = _SO + f".{os.getpid()}.tmp"
    cmd = [nv, ARCH, "-shared", "-cudart", "shared", "-o", tmp] + objs + [
        "-Xlinker", "-rpath," + _cuda_lib_dir()]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, _SO)
    for o in objs:
        try:
            os.remove(o)
        except OSError:
            pass
    return _SO


# ------------------------------------------------------------------ C types
class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "ln1_w", "w_qkv", "w_qkv_scale", "q_norm_w", "k_norm_w", "w_o",
        "w_o_scale", "ln2_w", "w_gate_up", "w_gate_up_scale", "w_down",
        "w_down_scale")]


class Config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("inter", C.c_int), ("n_q_heads", C.c_int),
                ("n_kv_heads", C.c_int), ("head_dim", C.c_int),
                ("n_layers", C.c_int), ("vocab", C.c_int), ("eps", C.c_float),
                ("rope_theta", C.c_float), ("weight_dtype", C.c_int),
                ("num_requests", C.c_int), ("tokens_per_request", C.c_int),
                ("page_size", C.c_int), ("num_pages", C.c_int),
                ("max_pages_per_request", C.c_int), ("max_context", C.c_int),
                ("num_sms", C.c_int), ("modes_mask", C.c_uint),
                ("layers", C.POINTER(LayerWeights)),
                ("final_norm_w", C.c_void_p), ("lm_head_w", C.c_void_p)]


_lock = threading.Lock()
_lib = None

EXPORTS = ("dl_plan_create", "dl_last_error", "dl_decode_step",
           "dl_decode_step_host", "dl_plan_status", "dl_plan_logits",
           "dl_plan_debug_buffer", "dl_plan_kernel_count", "dl_plan_mega_info",
           "dl_plan_debug_perturb_wait", "dl_plan_destroy", "dl_test_kv_write",
           "dl_test_kv_gather", "dl_plan_op_count", "dl_plan_op_info",
           "dl_plan_launch_op", "dl_plan_launch_ops", "dl_attention_noalloc", "dl_plan_trace",
           "dl_test_validate_mega_queues", "dl_bench_mma", "dl_bench_poll_latency",
           "dl_plan_bench_empty_megakernel")


def lib(path: Optional[str] = None):
    """Load libdl.so (building it if missing).  Raises if it cannot load."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        so = path or build()
        L = C.CDLL(so)
        vp, i32, u32 = C.c_void_p, C.c_int, C.c_uint
        L.dl_plan_create.argtypes = [C.POINTER(Config)]
        L.dl_plan_create.restype = vp
        L.dl_last_error.restype = C.c_char_p
        L.dl_decode_step.argtypes = [vp] * 7 + [i32, vp]
        L.dl_decode_step.restype = i32
        L.dl_decode_step_host.argtypes = [vp] * 7 + [i32, vp]
        L.dl_decode_step_host.restype = i32
        L.dl_plan_status.argtypes = [vp]
        L.dl_plan_status.restype = i32
        L.dl_plan_logits.argtypes = [vp]
        L.dl_plan_logits.restype = vp
        L.dl_plan_debug_buffer.argtypes = [vp, i32, C.POINTER(vp), C.POINTER(C.c_size_t)]
        L.dl_plan_debug_buffer.restype = i32
        L.dl_plan_kernel_count.argtypes = [vp, i32]
        L.dl_plan_kernel_count.restype = i32
        L.dl_plan_mega_info.argtypes = [vp, C.POINTER(i32), C.POINTER(i32), C.POINTER(i32)]
        L.dl_plan_mega_info.restype = i32
        L.dl_plan_debug_perturb_wait.argtypes = [vp, u32, C.c_ulonglong, i32]
        L.dl_plan_debug_perturb_wait.restype = i32
        L.dl_plan_destroy.argtypes = [vp]
        L.dl_plan_op_count.argtypes = [vp]
        L.dl_plan_op_count.restype = i32
        L.dl_plan_op_info.argtypes = [vp, i32, C.c_char_p, C.c_size_t, C.POINTER(i32),
                                      C.POINTER(i32)]
        L.dl_plan_op_info.restype = i32
        L.dl_plan_launch_op.argtypes = [vp, i32, vp]
        L.dl_plan_launch_op.restype = i32
        L.dl_plan_launch_ops.argtypes = [vp, i32, i32, i32, i32, vp]
        L.dl_plan_launch_ops.restype = i32
        L.dl_plan_trace.argtypes = [vp, vp, C.c_size_t, C.POINTER(i32), C.POINTER(i32)]
        L.dl_plan_trace.restype = i32
        L.dl_attention_noalloc.argtypes = [C.POINTER(Config), i32] + [vp] * 6 + [i32, vp]
        L.dl_attention_noalloc.restype = i32
        L.dl_test_kv_write.argtypes = [vp] * 4 + [i32] * 8 + [vp]
        L.dl_test_kv_write.restype = i32
        L.dl_test_kv_gather.argtypes = [vp] * 3 + [i32] * 8 + [vp]
        L.dl_test_kv_gather.restype = i32
        L.dl_test_validate_mega_queues.argtypes = [vp, i32, i32, i32]
        L.dl_test_validate_mega_queues.restype = i32
        L.dl_bench_mma.argtypes = [i32, i32, i32, i32, i32, i32, C.POINTER(C.c_double)]
        L.dl_bench_mma.restype = i32
        L.dl_bench_poll_latency.argtypes = [i32, C.POINTER(C.c_double)]
        L.dl_bench_poll_latency.restype = i32
        L.dl_plan_bench_empty_megakernel.argtypes = [vp, i32, C.POINTER(C.c_double), vp]
        L.dl_plan_bench_empty_megakernel.restype = i32
        if path is None:
            _lib = L
        return L


class DLError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"dl status {status}: {msg}")
        self.status = status


def _check(rc: int):
    if rc != 0:
        raise DLError(rc, lib().dl_last_error().decode())


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def attention_noalloc(cfg, layer: int, q, kv_pages, block_table, positions, out,
                      out_scale=None, max_context: Optional[int] = None, num_sms: int = 0,
                      check: bool = True, stream=None):
    """Split-KV attention of one layer that allocates no device memory (its
    scratch is a static device array; dl_attention_noalloc in include/dl.h).
    Meant for callers that may not allocate at the call, such as code whose
    framework owns the device allocator.  Calls on one device must not
    overlap in time: they share the scratch."""
    c = Config()
    c.n_q_heads, c.n_kv_heads, c.head_dim = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    c.n_layers = cfg.n_layers
    c.weight_dtype = 1 if cfg.fp8 else 0
    c.num_requests, c.tokens_per_request = cfg.num_requests, cfg.tokens_per_request
    c.page_size, c.num_pages = cfg.page_size, cfg.num_pages
    c.max_pages_per_request = cfg.pages_per_request
    c.max_context = max_context or cfg.context
    c.num_sms = num_sms
    _check(lib().dl_attention_noalloc(C.byref(c), layer, _ptr(q), _ptr(kv_pages),
                                      _ptr(block_table), _ptr(positions), _ptr(out),
                                      _ptr(out_scale), int(check), _stream_handle(stream)))


def bench_mma(fp8: bool, n: int, n_mma: int, n_accumulators: int = 1,
              n_issuers: int = 1, lean: bool = False) -> float:
    """ns per tcgen05.mma (M = 128, N = n; bf16 K = 16 or e4m3 K = 32) over
    n_mma instructions into n_accumulators TMEM accumulators from n_issuers
    threads; lean: descriptors precomputed (dl_bench_mma)."""
    v = C.c_double()
    _check(lib().dl_bench_mma(int(bool(fp8)), n, n_mma, n_accumulators, n_issuers,
                              int(bool(lean)), C.byref(v)))
    return v.value


def bench_poll_latency(iters: int = 10000) -> float:
    """ns per release-add / acquire-poll round trip between two CTAs
    (dl_bench_poll_latency)."""
    v = C.c_double()
    _check(lib().dl_bench_poll_latency(iters, C.byref(v)))
    return v.value


class Plan:
    """A prepared decode step for one configuration (device-resident weights
    supplied as torch CUDA tensors, kept alive by the plan)."""

    def __init__(self, cfg, weights: Dict, modes_mask: int = ALL_MODES,
                 max_context: Optional[int] = None, num_sms: int = 0):
        L = lib()
        self.cfg = cfg
        self._keep: List = [weights]
        n = cfg.n_layers
        arr = (LayerWeights * n)()
        for l, lw in enumerate(weights["layers"]):
            s = arr[l]
            for name, _ in LayerWeights._fields_:
                setattr(s, name, _ptr(lw.get(name)))
        self._layers = arr
        c = Config()
        c.hidden, c.inter = cfg.hidden, cfg.inter
        c.n_q_heads, c.n_kv_heads, c.head_dim = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
        c.n_layers, c.vocab = n, cfg.vocab
        c.eps, c.rope_theta = cfg.eps, cfg.rope_theta
        c.weight_dtype = 1 if cfg.fp8 else 0
        c.num_requests, c.tokens_per_request = cfg.num_requests, cfg.tokens_per_request
        c.page_size, c.num_pages = cfg.page_size, cfg.num_pages
        c.max_pages_per_request = cfg.pages_per_request
        c.max_context = max_context or cfg.context
        c.num_sms = num_sms
        c.modes_mask = modes_mask
        c.layers = arr
        c.final_norm_w = _ptr(weights.get("final_norm_w"))
        c.lm_head_w = _ptr(weights.get("lm_head_w"))
        self._c = c
        h = L.dl_plan_create(C.byref(c))
        if not h:
            raise DLError(-1, L.dl_last_error().decode())
        self._h = h

    def step(self, x, residual, kv_pages, block_table, positions, out,
             mode: int = MODE_SERIAL, stream=None):
        _check(lib().dl_decode_step(self._h, _ptr(x), _ptr(residual), _ptr(kv_pages),
                                    _ptr(block_table), _ptr(positions), _ptr(out),
                                    mode, _stream_handle(stream)))

    def step_host(self, x, residual, kv_pages, block_table, positions, out,
                  mode: int = MODE_SERIAL, stream=None):
        """x, residual, block_table, positions, out: (pinned) CPU tensors."""
        _check(lib().dl_decode_step_host(self._h, _ptr(x), _ptr(residual), _ptr(kv_pages),
                                         _ptr(block_table), _ptr(positions), _ptr(out),
                                         mode, _stream_handle(stream)))

    def status(self):
        _check(lib().dl_plan_status(self._h))

    def debug_buffer(self, name: str):
        p, n = C.c_void_p(), C.c_size_t()
        _check(lib().dl_plan_debug_buffer(self._h, DEBUG_BUFFERS[name], C.byref(p), C.byref(n)))
        return p.value, n.value

    def trace(self):
        """Trace table uint64 [ops, ctas, 8] (plan created with DL_TRACE=1);
        reading it clears it."""
        import numpy as np
        n_ops, n_ctas = C.c_int(), C.c_int()
        _check(lib().dl_plan_trace(self._h, None, 0, C.byref(n_ops), C.byref(n_ctas)))
        buf = np.zeros((n_ops.value, n_ctas.value, 8), dtype=np.uint64)
        _check(lib().dl_plan_trace(self._h, buf.ctypes.data, buf.nbytes, None, None))
        return buf

    def logits_ptr(self) -> Optional[int]:
        return lib().dl_plan_logits(self._h)

    def kernel_count(self, mode: int) -> int:
        return lib().dl_plan_kernel_count(self._h, mode)

    def mega_info(self):
        w, q, e = C.c_int(), C.c_int(), C.c_int()
        _check(lib().dl_plan_mega_info(self._h, C.byref(w), C.byref(q), C.byref(e)))
        return w.value, q.value, e.value

    def ops(self):
        """[(name, grid, smem_bytes)] of the serial schedule's operations."""
        L = lib()
        res = []
        for i in range(L.dl_plan_op_count(self._h)):
            buf = C.create_string_buffer(64)
            g, s = C.c_int(), C.c_int()
            _check(L.dl_plan_op_info(self._h, i, buf, 64, C.byref(g), C.byref(s)))
            res.append((buf.value.decode(), g.value, s.value))
        return res

    def launch_op(self, i: int, stream=None):
        _check(lib().dl_plan_launch_op(self._h, i, _stream_handle(stream)))

    def launch_ops(self, first: int, count: int, pdl: bool, gdc_mode: int = 0, stream=None):
        """Ops [first, first + count) of the serial list, with or without
        programmatic dependent launch, projections waiting on their producer
        per gdc_mode (0 after their first weight stages, 1 after their
        prologue, 2 at entry): the per-edge ablation hook."""
        _check(lib().dl_plan_launch_ops(self._h, first, count, int(bool(pdl)), gdc_mode,
                                        _stream_handle(stream)))

    def bench_empty_megakernel(self, iters: int = 50, stream=None) -> float:
        """µs per launch of the megakernel with all-NoOp queues."""
        v = C.c_double()
        _check(lib().dl_plan_bench_empty_megakernel(self._h, iters, C.byref(v),
                                                     _stream_handle(stream)))
        return v.value

    def perturb_wait(self, delta: int, budget_ns: int, validate: bool):
        return lib().dl_plan_debug_perturb_wait(self._h, delta, budget_ns, int(validate))

    def close(self):
        if getattr(self, "_h", None):
            lib().dl_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
