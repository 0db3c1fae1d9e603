"""CPU checks of the C ABI library: it builds for sm_103a, loads, and exports
every function include/dl.h declares (no compute call without a GPU)."""
import os
import re

import pytest

import pdl_persistent_megakernel_gb300 as dl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            txt = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"\b(dl_[a-z_0-9]+)\s*\(", txt))
    return names


def test_library_exports_every_declared_symbol():
    try:
        so = dl.build()
    except (RuntimeError, FileNotFoundError) as e:  # no nvcc here
        pytest.skip(f"cannot build: {e}")
    L = dl.lib()
    declared = _declared()
    assert {"dl_plan_create", "dl_decode_step", "dl_plan_destroy"} <= declared
    missing = [n for n in declared if not hasattr(L, n)]
    assert not missing, missing
    assert set(dl.EXPORTS) <= declared


def test_last_error_is_empty_string_initially():
    L = dl.lib()
    assert isinstance(L.dl_last_error(), bytes)


def test_plan_create_rejects_bad_config_without_gpu():
    # config validation runs before any CUDA call
    from pdl_persistent_megakernel_gb300 import synth
    cfg = synth.DecodeConfig("bad", hidden=256, inter=384, n_q_heads=4, n_kv_heads=2,
                             head_dim=64, n_layers=1, vocab=0, fp8=False, num_requests=1,
                             tokens_per_request=1, context=100, page_size=16)
    import torch
    w = {"layers": [{}]}
    with pytest.raises(dl.DLError) as e:
        dl.Plan(cfg, w)
    assert "head_dim" in str(e.value)


def _cfg(**kw):
    from pdl_persistent_megakernel_gb300 import synth
    base = dict(hidden=256, inter=384, n_q_heads=4, n_kv_heads=2, head_dim=128, n_layers=1,
                vocab=0, fp8=False, num_requests=1, tokens_per_request=1, context=100,
                page_size=16)
    base.update(kw)
    return synth.DecodeConfig("bad", **base)


@pytest.mark.parametrize("kw,plan_kw,msg", [
    (dict(n_q_heads=6, n_kv_heads=4), {}, "n_q_heads % n_kv_heads"),
    (dict(hidden=200), {}, "multiples of 128"),
    (dict(hidden=16384), {}, "hidden > 8192"),
    (dict(vocab=1000), {}, "vocab must be a multiple of 128"),
    (dict(num_requests=65), {}, "more than 64 tokens"),
    (dict(tokens_per_request=16, n_q_heads=32, n_kv_heads=2), {}, "group size > 64"),
    (dict(page_size=48), {}, "page_size must divide 64"),
    (dict(), dict(max_context=400), "max_context"),
    (dict(fp8=True, vocab=128), {}, "layer plans"),
], ids=["gqa", "hidden128", "hidden_max", "vocab128", "tokens", "qrows", "page", "pages",
        "fp8_full"])
def test_plan_create_rejects_each_config_rule_without_gpu(kw, plan_kw, msg):
    """Every rule of the plan's config check, violated alone, is refused with
    its own message before any CUDA call."""
    with pytest.raises(dl.DLError) as e:
        dl.Plan(_cfg(**kw), {"layers": [{}]}, **plan_kw)
    assert msg in str(e.value)


class _Addr:
    """A stand-in tensor: only its address is read (the checks under test
    run before any CUDA call, so nothing dereferences it)."""

    def __init__(self, a):
        self.a = a

    def data_ptr(self):
        return self.a


@pytest.mark.parametrize("kw,call_kw,msg", [
    (dict(head_dim=64), {}, "head_dim must be 128"),
    (dict(n_q_heads=6, n_kv_heads=4), {}, "n_q_heads % n_kv_heads"),
    (dict(), dict(layer=1), "layer out of range"),
    (dict(num_requests=65), {}, "more than 64 tokens"),
    (dict(tokens_per_request=16, n_q_heads=32, n_kv_heads=2), {}, "group size > 64"),
    (dict(page_size=48), {}, "page_size must divide 64"),
    (dict(), dict(max_context=400), "max_pages_per_request * page_size < max_context"),
    (dict(num_requests=64, n_q_heads=65, n_kv_heads=65), {}, "4096"),
    (dict(), dict(q=None), "NULL tensor pointer"),
    (dict(fp8=True), {}, "NULL tensor pointer"),          # FP8 needs out_scale
    (dict(), dict(q=_Addr(0x1008)), "misaligned"),
], ids=["head_dim", "gqa", "layer", "tokens", "qrows", "page", "pages", "pairs", "null",
        "fp8_scale", "align"])
def test_attention_noalloc_rejects_each_rule_without_gpu(kw, call_kw, msg):
    """Every host check of the allocation-free attention entry point,
    violated alone, is refused with its own message before any CUDA call."""
    args = dict(layer=0, q=_Addr(0x10000), kv_pages=_Addr(0x20000),
                block_table=_Addr(0x30000), positions=_Addr(0x40000), out=_Addr(0x50000))
    args.update(call_kw)
    max_context = args.pop("max_context", None)
    with pytest.raises(dl.DLError) as e:
        dl.attention_noalloc(_cfg(**kw), args["layer"], args["q"], args["kv_pages"],
                             args["block_table"], args["positions"], args["out"],
                             max_context=max_context, check=False, stream=0)
    assert msg in str(e.value)


def test_null_plan_is_an_argument_error_everywhere():
    """Every entry point that takes a plan refuses NULL without touching a
    device: a dl_status of DL_ERR_INVALID_ARG, -1 for the counts, NULL for
    the logits pointer, nothing for destroy."""
    import ctypes as C
    L = dl.lib()
    INVALID = 1
    z = None
    assert L.dl_decode_step(z, z, z, z, z, z, z, 0, z) == INVALID
    assert L.dl_decode_step_host(z, z, z, z, z, z, z, 0, z) == INVALID
    assert L.dl_plan_status(z) == INVALID
    p, n = C.c_void_p(), C.c_size_t()
    assert L.dl_plan_debug_buffer(z, 0, C.byref(p), C.byref(n)) == INVALID
    i = C.c_int()
    assert L.dl_plan_mega_info(z, C.byref(i), C.byref(i), C.byref(i)) == INVALID
    assert L.dl_plan_debug_perturb_wait(z, 0, 0, 1) == INVALID
    buf = C.create_string_buffer(32)
    assert L.dl_plan_op_info(z, 0, buf, 32, C.byref(i), C.byref(i)) == INVALID
    assert L.dl_plan_launch_op(z, 0, z) == INVALID
    assert L.dl_plan_launch_ops(z, 0, 1, 0, 0, z) == INVALID
    assert L.dl_plan_trace(z, z, 0, C.byref(i), C.byref(i)) == INVALID
    assert L.dl_plan_kernel_count(z, 0) == -1 and L.dl_plan_op_count(z) == -1
    assert not L.dl_plan_logits(z)
    L.dl_plan_destroy(z)
