"""GPU checks of dl_attention_noalloc, the attention entry point that
allocates no device memory.

It exists for callers that may not allocate device memory where they call
it (a framework that owns the device allocator, or code under an exhausted
memory-pool budget); its scratch is a static 8 MiB device array shared by
every call.  Each case runs one decode step through the plan entry point
(dl_decode_step, serial schedule), then calls the no-alloc entry point twice
in a row on the same query, cache, block table and positions, and checks
both outputs against the plan's attention output with the tolerances of the
parity tests: bf16 |a - b| <= 1e-2 (1 + |b|) element-wise; FP8 (dequantised)
rms(a - b) <= 5e-2 rms(b).  The second call sees the scratch the first call
left behind.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import pdl_persistent_megakernel_gb300 as dl
from pdl_persistent_megakernel_gb300 import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import (DEV, as_bf16_np, as_f32_np, as_u8_np, bf16_close, dequant,
                             read_debug, rel_rms_close, to_dev)

SCRATCH_BYTES = 8 << 20

CASES = {
    # GQA group 4, 2 tokens per request, 16-token pages, ragged 150-key context
    "bf16_m4": synth.DecodeConfig("nb_bf16_m4", hidden=512, inter=640, n_q_heads=8, n_kv_heads=2,
                                  head_dim=128, n_layers=1, vocab=0, fp8=False, num_requests=2,
                                  tokens_per_request=2, context=150, page_size=16, seed=21),
    # 32 query rows per (request, kv head), 64-token pages, two layers
    "bf16_qr32": synth.DecodeConfig("nb_bf16_qr32", hidden=512, inter=768, n_q_heads=8,
                                    n_kv_heads=2, head_dim=128, n_layers=2, vocab=0, fp8=False,
                                    num_requests=2, tokens_per_request=8, context=700,
                                    page_size=64, seed=22),
    # FP8 output (e4m3 codes + per-128 scales)
    "fp8_m16": synth.DecodeConfig("nb_fp8_m16", hidden=512, inter=768, n_q_heads=8, n_kv_heads=2,
                                  head_dim=128, n_layers=1, vocab=0, fp8=True, num_requests=2,
                                  tokens_per_request=8, context=200, page_size=64, seed=23),
    # the Qwen3-8B FP8 layer at M = 16, context 8192 (every SM shares the keys)
    "q8_fp8_full": synth.CONFIGS["q8_layer_m16_ctx8192_fp8"],
}

# 64 query rows per (request, kv head): at every SM the partials need more
# than the 8 MiB scratch, so the call must be refused; with fewer SMs it runs.
QR64 = synth.DecodeConfig("nb_qr64", hidden=512, inter=768, n_q_heads=16, n_kv_heads=2,
                          head_dim=128, n_layers=1, vocab=0, fp8=False, num_requests=2,
                          tokens_per_request=8, context=2048, page_size=64, seed=24)


def _plan_step(cfg, num_sms=0):
    """One serial decode step through the plan entry point; returns the
    device tensors the attention reads and the plan's attention output."""
    w = to_dev(synth.make_weights(cfg))
    inp = {k: v.to(DEV) for k, v in synth.make_inputs(cfg).items()}
    plan = dl.Plan(cfg, w, modes_mask=0, num_sms=num_sms)
    out = torch.zeros((2, cfg.M, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    plan.step(inp["x"], inp["residual"], inp["kv_pages"], inp["block_table"],
              inp["positions"], out, mode=dl.MODE_SERIAL)
    torch.cuda.synchronize()
    plan.status()
    QD = cfg.n_q_heads * cfg.head_dim
    q = read_debug(plan, "q_rot")[:cfg.M * QD * 2].to(DEV)
    attn = read_debug(plan, "attn")
    want = {"attn": attn}
    if cfg.fp8:
        want["scales"] = read_debug(plan, "attn_scales")
    plan.close()
    return inp, q, want


def _compare(cfg, got, got_scales, want, what):
    M, QD = cfg.M, cfg.n_q_heads * cfg.head_dim
    if cfg.fp8:
        g = dequant(got.cpu().numpy().reshape(M, QD), got_scales.cpu().numpy())
        w = dequant(as_u8_np(want["attn"], (M, QD)), as_f32_np(want["scales"], (M, QD // 128)))
        rel_rms_close(g, w, what)
    else:
        g = got.cpu().view(torch.int16).numpy().view(np.uint16).reshape(M, QD)
        bf16_close(g, as_bf16_np(want["attn"], (M, QD)), what)


def _run_twice(cfg, num_sms=0):
    inp, q, want = _plan_step(cfg, num_sms)
    M, QD = cfg.M, cfg.n_q_heads * cfg.head_dim
    for call in range(2):
        # garbage in the outputs, so that a value the call fails to write shows
        if cfg.fp8:
            out = torch.full((M, QD), 0x7F, dtype=torch.uint8, device=DEV)
            sc = torch.full((M, QD // 128), float("nan"), dtype=torch.float32, device=DEV)
        else:
            out = torch.full((M, QD), -1e30, dtype=torch.bfloat16, device=DEV)
            sc = None
        dl.attention_noalloc(cfg, cfg.n_layers - 1, q, inp["kv_pages"], inp["block_table"],
                             inp["positions"], out, sc, num_sms=num_sms, check=True)
        torch.cuda.synchronize()
        _compare(cfg, out, sc, want, f"{cfg.name} call {call + 1}")


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_plan_attention_twice(name):
    _run_twice(CASES[name])


def test_noalloc_rejects_oversized_scratch_and_runs_with_fewer_sms():
    cfg = QR64
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks = -(-cfg.context // 64)
    pairs = cfg.num_requests * cfg.n_kv_heads
    G = min(sms, pairs * blocks, 62 * pairs)
    need = 16896 + G * 2 * 64 * 129 * 4
    if need > SCRATCH_BYTES:
        inp = {k: v.to(DEV) for k, v in synth.make_inputs(cfg).items()}
        QD = cfg.n_q_heads * cfg.head_dim
        q = torch.zeros((cfg.M, QD), dtype=torch.bfloat16, device=DEV)
        out = torch.zeros((cfg.M, QD), dtype=torch.bfloat16, device=DEV)
        with pytest.raises(dl.DLError) as e:
            dl.attention_noalloc(cfg, 0, q, inp["kv_pages"], inp["block_table"],
                                 inp["positions"], out, None, check=True)
        assert e.value.status == 2 and "scratch" in str(e.value), str(e.value)
    # 100 CTAs x 2 x 64 rows x 516 bytes fits
    _run_twice(cfg, num_sms=100)
