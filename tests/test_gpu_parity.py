"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, on
seeded inputs, element by element, for every schedule.

Small cases span several weight tiles and Stream-K splits with a ragged KV
tail; the full-size cases are the Qwen3-0.6B layer (batch 1, ctx 1024) and
the Qwen3-8B FP8 layer (M = 16, ctx 8192) in the launch configuration the
bench times.  Tolerances:
- r' = bf16(x + r) bit for bit; the first norm's FP8 codes bit for bit
  except, by one step, where the oracle's quotient lies within 2^-18 of an
  e4m3 rounding boundary (fp32 versus fp64 norm), its scales within 2^-18;
- every tensor whose inputs are identical on both sides (q after QK-norm +
  RoPE, the new K/V rows of layer 0; in FP8 given the GPU's own first-norm
  codes), every bf16 intermediate,
  and the lm_head given the GPU's own final hidden state:
  |gpu - oracle| <= 1e-2 (1 + |oracle|) element-wise (after RoPE, |oracle|
  is the norm of the element's rotation pair);
- FP8 tensors downstream of a quantised attention or projection input:
  rms(gpu - oracle) <= 5e-2 rms(oracle) per tensor (relative RMS error).
"""
import numpy as np
import pytest
import torch

import oracle

import pdl_persistent_megakernel_gb300 as dl
from pdl_persistent_megakernel_gb300 import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import (Case, as_bf16_np, as_f32_np, as_u8_np, bf16_close,
                             check_fp8_codes_exact, check_lm_head_stagewise, dequant, f64,
                             fp8_qkv_given_gpu_h1, read_debug, rel_rms_close, rope_close)

SMALL = {
    # GEMV (M = 1), 16-token pages, ctx 100 = 64 + a ragged 36
    "bf16_m1": synth.DecodeConfig("bf16_m1", hidden=256, inter=384, n_q_heads=4, n_kv_heads=2,
                                  head_dim=128, n_layers=1, vocab=0, fp8=False, num_requests=1,
                                  tokens_per_request=1, context=100, page_size=16, seed=11),
    # GEMV with 4 tokens (2 requests x 2), GQA group 4
    "bf16_m4": synth.DecodeConfig("bf16_m4", hidden=512, inter=640, n_q_heads=8, n_kv_heads=2,
                                  head_dim=128, n_layers=1, vocab=0, fp8=False, num_requests=2,
                                  tokens_per_request=2, context=150, page_size=16, seed=12),
    # tcgen05 path, bf16, M = 16 (2 x 8), 64-token pages
    "bf16_m16": synth.DecodeConfig("bf16_m16", hidden=512, inter=768, n_q_heads=8, n_kv_heads=2,
                                   head_dim=128, n_layers=1, vocab=0, fp8=False, num_requests=2,
                                   tokens_per_request=8, context=200, page_size=64, seed=13),
    # CUDA-core GEMV path, FP8, M = 4
    "fp8_m4": synth.DecodeConfig("fp8_m4", hidden=512, inter=768, n_q_heads=8, n_kv_heads=2,
                                 head_dim=128, n_layers=1, vocab=0, fp8=True, num_requests=2,
                                 tokens_per_request=2, context=150, page_size=16, seed=16),
    # tcgen05 path, FP8, M = 16
    "fp8_m16": synth.DecodeConfig("fp8_m16", hidden=512, inter=768, n_q_heads=8, n_kv_heads=2,
                                  head_dim=128, n_layers=1, vocab=0, fp8=True, num_requests=2,
                                  tokens_per_request=8, context=200, page_size=64, seed=14),
    # two layers + lm_head + argmax, M = 1
    "step_m1": synth.DecodeConfig("step_m1", hidden=256, inter=384, n_q_heads=4, n_kv_heads=2,
                                  head_dim=128, n_layers=2, vocab=1024, fp8=False,
                                  num_requests=1, tokens_per_request=1, context=70,
                                  page_size=16, seed=15),
}

MODES = [dl.MODE_SERIAL, dl.MODE_PDL_GRAPH, dl.MODE_MEGAKERNEL, dl.MODE_GRAPH_LINEAR,
         dl.MODE_GRAPH_LINEAR_PDL, dl.MODE_GRAPH_DAG]

_cases = {}


def case(name):
    if name not in _cases:
        cfg = SMALL[name] if name in SMALL else synth.CONFIGS[name]
        _cases[name] = Case(cfg)
    return _cases[name]


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("mode", MODES, ids=lambda m: dl.MODE_NAMES[m])
def test_small_layer_all_modes(name, mode):
    c = case(name)
    plan = c.plan()
    out, kv = c.run(plan, mode)
    if c.cfg.vocab:
        ids = out.cpu().numpy()
        logits = c.ref["logits"]
        top2 = np.sort(logits, axis=1)[:, -2:]
        sure = (top2[:, 1] - top2[:, 0]) > 1e-2
        assert np.array_equal(ids[sure], c.ref["ids"][sure]), (ids, c.ref["ids"])
        got = check_lm_head_stagewise(c, plan, f"{name}/{dl.MODE_NAMES[mode]}")
        # the ids are the argmax of the GPU's own logits
        assert np.array_equal(ids, got.argmax(axis=1)), (ids, got.argmax(axis=1))
    else:
        c.check_layer_out(out, f"{name}/{dl.MODE_NAMES[mode]}")
    c.check_kv(kv, f"{name}/{dl.MODE_NAMES[mode]}", plan)
    plan.close()


@pytest.mark.parametrize("name", ["bf16_m1", "bf16_m4", "bf16_m16", "fp8_m4", "fp8_m16"])
def test_small_intermediates(name):
    """Every row of the step against the oracle's intermediates."""
    c = case(name)
    plan = c.plan(modes=1 << dl.MODE_SERIAL)
    out, _ = c.run(plan, dl.MODE_SERIAL)
    _check_intermediates(c, plan, out)
    plan.close()


@pytest.mark.parametrize("name", ["bf16_m4", "bf16_m16", "fp8_m16"])
@pytest.mark.parametrize("num_sms", [5, 7])
def test_small_intermediates_ctas_span_pairs(name, num_sms):
    """With a few CTAs every Stream-K range crosses (request, kv head) pair
    and GEMM tile boundaries: a CTA leaves one pair's partial and starts the
    next, so both split-KV workspace slots and multi-contributor fix-ups are
    exercised."""
    c = case(name)
    plan = c.plan(modes=1 << dl.MODE_SERIAL, num_sms=num_sms)
    out, _ = c.run(plan, dl.MODE_SERIAL)
    _check_intermediates(c, plan, out)
    c.check_layer_out(out, f"{name}/sms{num_sms}")
    plan.close()


def _check_intermediates(c, plan, out):
    cfg = c.cfg
    M, H, I = cfg.M, cfg.hidden, cfg.inter
    QD = cfg.n_q_heads * cfg.head_dim
    # r' = bf16(x + r): one rounding of an exact sum on both sides
    r1 = as_bf16_np(read_debug(plan, "r1"), (M, H))
    nd = int((r1 != c.ref["r1"]).sum())
    assert nd == 0, f"r1: {nd} of {r1.size} values differ"
    q_got = as_bf16_np(read_debug(plan, "q_rot"), (M, QD)).reshape(M, -1, cfg.head_dim)
    if cfg.fp8:
        # the first norm's e4m3 codes and scales (identical inputs; a code may
        # differ only at an e4m3 rounding boundary)
        lw = c.w["layers"][0]
        _, _, hf = oracle.add_rmsnorm(synth.as_u16(c.inp["x"]), synth.as_u16(c.inp["residual"]),
                                      synth.as_u16(lw["ln1_w"]), cfg.eps)
        check_fp8_codes_exact(as_u8_np(read_debug(plan, "h1"), (M, H)),
                              as_f32_np(read_debug(plan, "h1_scales"), (M, H // 128)),
                              c.ref["h1_codes"], c.ref["h1_scales"], hf, "h1")
        # q after QK-norm + RoPE, given the GPU's own h1 codes
        q_want, _, _ = fp8_qkv_given_gpu_h1(c, plan)
        rope_close(q_got, q_want, "q_rot")
    else:
        # q after QK-norm + RoPE: the projection's inputs are identical on
        # both sides (h1 is checked above), so the element bound holds
        rope_close(q_got, c.ref["q_rot"].reshape(M, -1, cfg.head_dim), "q_rot")
    # a layer plan writes the new residual straight into out[1]
    r2 = out[1].view(torch.int16).cpu().numpy().view(np.uint16)
    if cfg.fp8:
        rel_rms_close(f64(r2), f64(c.ref["r2"]), "r2")
    else:
        bf16_close(r2, c.ref["r2"], "r2")
    if cfg.fp8:
        for nm, K in (("h1", H), ("attn", QD), ("h2", H), ("act", I)):
            codes = as_u8_np(read_debug(plan, nm), (M, K))
            sc = as_f32_np(read_debug(plan, nm + "_scales"), (M, K // 128))
            got = dequant(codes, sc)
            want = dequant(c.ref[nm + "_codes"], c.ref[nm + "_scales"])
            rel_rms_close(got, want, nm)
        rel_rms_close(f64(as_bf16_np(read_debug(plan, "o2"), (M, H))), f64(c.ref["o2"]), "o2")
    else:
        bf16_close(as_bf16_np(read_debug(plan, "h1"), (M, H)), c.ref["h1"], "h1")
        bf16_close(as_bf16_np(read_debug(plan, "attn"), (M, QD)), c.ref["attn"], "attn")
        bf16_close(as_bf16_np(read_debug(plan, "o2"), (M, H)), c.ref["o2"], "o2")
        bf16_close(as_bf16_np(read_debug(plan, "h2"), (M, H)), c.ref["h2"], "h2")
        bf16_close(as_bf16_np(read_debug(plan, "act"), (M, I)), c.ref["act"], "act")


@pytest.mark.parametrize("name", ["bf16_m1", "fp8_m16", "step_m1"])
def test_schedules_bitwise_identical(name):
    """Serial and graph (linear, +PDL) launch the same kernels over the same
    work split, so their results are bit-identical; replaying a step with the
    same inputs reproduces it exactly.  The megakernel runs the same
    projection engines and the mma.sync attention engine (the standalone
    kernels run attention on tcgen05): its cache and outputs agree to
    rounding (bf16 tolerance)."""
    c = case(name)
    plan = c.plan()
    outs = {}
    for mode in (dl.MODE_SERIAL, dl.MODE_GRAPH_LINEAR, dl.MODE_GRAPH_LINEAR_PDL,
                 dl.MODE_MEGAKERNEL):
        out, kv = c.run(plan, mode, steps=3)
        outs[mode] = (out.cpu(), kv.cpu())
    base = outs[dl.MODE_SERIAL]
    u16 = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    for mode, (o, k) in outs.items():
        if mode == dl.MODE_MEGAKERNEL:
            # (greedy ids of the full step are checked against the oracle)
            bf16_close(u16(k), u16(base[1]), "megakernel vs serial cache")
            if o.dtype == torch.bfloat16:
                bf16_close(u16(o), u16(base[0]), "megakernel vs serial")
        else:
            assert torch.equal(k, base[1]), dl.MODE_NAMES[mode]
            assert torch.equal(o, base[0]), dl.MODE_NAMES[mode]
    plan.close()


@pytest.mark.parametrize("name", ["q06_layer_b1_ctx1024", "q8_layer_m16_ctx8192_fp8"])
@pytest.mark.parametrize("mode", [dl.MODE_SERIAL, dl.MODE_PDL_GRAPH, dl.MODE_MEGAKERNEL],
                         ids=lambda m: dl.MODE_NAMES[m])
def test_full_size_layer(name, mode):
    c = case(name)
    plan = c.plan(modes=(1 << dl.MODE_SERIAL) | (1 << dl.MODE_PDL_GRAPH) | (1 << dl.MODE_MEGAKERNEL))
    out, kv = c.run(plan, mode)
    c.check_layer_out(out, f"{name}/{dl.MODE_NAMES[mode]}")
    c.check_kv(kv, f"{name}/{dl.MODE_NAMES[mode]}", plan)
    plan.close()


@pytest.mark.parametrize("name", ["q06_layer_b1_ctx1024", "q8_layer_m16_ctx8192_fp8"])
def test_full_size_intermediates(name):
    """The layer output is dominated by the residual, so it can hide a wrong
    attention or projection: check every intermediate at full size too."""
    c = case(name)
    plan = c.plan(modes=1 << dl.MODE_SERIAL)
    out, _ = c.run(plan, dl.MODE_SERIAL)
    _check_intermediates(c, plan, out)
    plan.close()


def test_host_buffer_entry_matches_device_entry():
    """dl_decode_step_host (pinned host buffers in, the result read back to a
    pinned host buffer) gives the bytes of dl_decode_step on the same inputs
    and the same starting cache."""
    from gpu_harness import DEV
    c = case("fp8_m16")
    mode = dl.MODE_GRAPH_LINEAR_PDL
    plan = c.plan(modes=1 << mode)
    out_dev, kv_dev = c.run(plan, mode)
    kv = c.inp["kv_pages"].to(DEV)
    xh, rh = c.inp["x"].pin_memory(), c.inp["residual"].pin_memory()
    bth, posh = c.inp["block_table"].pin_memory(), c.inp["positions"].pin_memory()
    outh = torch.empty(out_dev.shape, dtype=out_dev.dtype).pin_memory()
    plan.step_host(xh, rh, kv, bth, posh, outh, mode=mode)
    torch.cuda.synchronize()
    plan.status()
    assert torch.equal(outh, out_dev.cpu())
    assert torch.equal(kv.cpu(), kv_dev.cpu())
    plan.close()


@pytest.mark.parametrize("name", ["bf16_m1", "fp8_m16", "step_m1", "q8_layer_m16_ctx8192_fp8"])
def test_pdl_ablation_launches_match_serial(name):
    """The per-edge ablation hook (dl_plan_launch_ops) over the whole serial
    list, with programmatic stream serialization off and on and every
    projection waiting on its producer after its first weight stages (0),
    after its prologue (1) or at entry (2), gives the serial step's bytes:
    output and cache.  Moving griddepcontrol.wait must never let a kernel
    read an operand its producer has not finished."""
    c = case(name)
    plan = c.plan(modes=1 << dl.MODE_SERIAL)
    out, kv = c.run(plan, dl.MODE_SERIAL)
    want_out, want_kv = out.clone(), kv.clone()
    kv0 = c.inp["kv_pages"].to(kv.device)
    n = len(plan.ops())
    for pdl in (False, True):
        for gdc_mode in (0, 1, 2):
            # the operands stay bound to this case's tensors: reset them
            kv.copy_(kv0)
            out.fill_(-1 if out.dtype == torch.int32 else 0)
            plan.launch_ops(0, n, pdl, gdc_mode)
            torch.cuda.synchronize()
            plan.status()
            what = f"{name} pdl={int(pdl)} gdc_mode={gdc_mode}"
            assert torch.equal(out, want_out), what
            assert torch.equal(kv, want_kv), what
    plan.close()


@pytest.mark.parametrize("name", ["fp8_m16", "bf16_m4", "step_m1"])
def test_megakernel_per_head_events(name, monkeypatch):
    """The megakernel's per-head events (an attention share waits only for
    the QKV tiles of its kv heads) change when work may start, not what it
    computes: the step is bit-identical to the one whose attention waits for
    the whole projection (DL_MEGA_HEAD_EVENTS=0), and the plan carries one
    event per kv head per layer beyond the per-op events."""
    c = case(name)
    cfg = c.cfg
    plan = c.plan(modes=1 << dl.MODE_MEGAKERNEL)
    out1, kv1 = c.run(plan, dl.MODE_MEGAKERNEL)
    out1, kv1 = out1.cpu(), kv1.cpu()
    _, _, ev1 = plan.mega_info()
    n_ops = len(plan.ops())
    plan.close()
    monkeypatch.setenv("DL_MEGA_HEAD_EVENTS", "0")
    plan0 = c.plan(modes=1 << dl.MODE_MEGAKERNEL)
    out0, kv0 = c.run(plan0, dl.MODE_MEGAKERNEL)
    _, _, ev0 = plan0.mega_info()
    plan0.close()
    assert ev0 == n_ops and ev1 == n_ops + cfg.n_layers * cfg.n_kv_heads, (ev0, ev1, n_ops)
    assert torch.equal(out1, out0.cpu()) and torch.equal(kv1, kv0.cpu())
