"""GPU checks of dl_attention_noalloc, the attention entry point that
allocates no device memory.

It exists for callers that may not allocate device memory where they call
it (a framework that owns the device allocator, or code under an exhausted
memory-pool budget); its scratch is a static 8 MiB device array shared by
every call.  Each case runs one decode step through the plan entry point
(dl_decode_step, serial schedule) so that the cache holds the step's new
K/V and the plan's q (after QK-norm + RoPE) is at hand.  Then:
- two calls in a row, each checked against the oracle's attention given the
  same q, cache, block table and positions (bf16: |gpu - oracle| <= 1e-2
  (1 + |oracle|) element-wise; FP8, dequantised: rms(gpu - oracle) <= 5e-2
  rms(oracle)) and against the plan's own attention output; the second call
  sees the scratch the first one left behind;
- two asynchronous calls (check = 0) queued back to back on one stream with
  different queries and outputs, synchronised once: only the stream order
  keeps the second call's binding upload and counter reset behind the first
  call's kernel;
- a call refused for its scratch size, then a good call;
- a call with a position outside [0, max_context): reported as
  DL_ERR_DEVICE_BOUNDS, after which a good call works.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
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
    device tensors the attention reads, the plan's q and attention output."""
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
    want = {"attn": read_debug(plan, "attn")}
    if cfg.fp8:
        want["scales"] = read_debug(plan, "attn_scales")
    plan.close()
    return inp, q, want


def _oracle_attention(cfg, layer, q, inp):
    """The oracle's attention output (fp64 [M, Hq d]) for the query q (bf16
    device tensor [M, Hq, d]) over the cache as it is on the device: the
    causal softmax over keys 0..p of each token's request, per q head on its
    kv head's K/V rows gathered through the block table."""
    M, Hq, Hkv, d, T = cfg.M, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.tokens_per_request
    G = Hq // Hkv
    qh = oracle.bf16_to_double(q.cpu().view(torch.int16).numpy().view(np.uint16)).reshape(M, Hq, d)
    kv = inp["kv_pages"].cpu().view(torch.int16).numpy().view(np.uint16)
    bt = inp["block_table"].cpu().numpy()
    pos = inp["positions"].cpu().numpy()
    out = np.zeros((M, Hq, d))
    for r in range(cfg.num_requests):
        n = int(pos[r * T + T - 1]) + 1
        for h in range(Hkv):
            K = oracle.kv_gather(kv, bt, Hkv, cfg.page_size, d, layer, r, h, 0, n)
            V = oracle.kv_gather(kv, bt, Hkv, cfg.page_size, d, layer, r, h, 1, n)
            for t in range(T):
                m = r * T + t
                for g in range(G):
                    out[m, h * G + g], _ = oracle.attention_partial(qh[m, h * G + g], K, V, 0, n,
                                                                    int(pos[m]))
    return out.reshape(M, Hq * d)


def _alloc_out(cfg):
    """Outputs filled with garbage, so that a value a call fails to write shows."""
    M, QD = cfg.M, cfg.n_q_heads * cfg.head_dim
    if cfg.fp8:
        out = torch.full((M, QD), 0x7F, dtype=torch.uint8, device=DEV)
        sc = torch.full((M, QD // 128), float("nan"), dtype=torch.float32, device=DEV)
    else:
        out = torch.full((M, QD), -1e30, dtype=torch.bfloat16, device=DEV)
        sc = None
    return out, sc


def _compare(cfg, got, got_scales, want64, plan_attn, what):
    """Against the oracle (given the same q), and against the plan's own
    attention output."""
    M, QD = cfg.M, cfg.n_q_heads * cfg.head_dim
    if cfg.fp8:
        g = dequant(got.cpu().numpy().reshape(M, QD), got_scales.cpu().numpy())
        rel_rms_close(g, want64, f"{what} vs oracle")
        if plan_attn is not None:
            w = dequant(as_u8_np(plan_attn["attn"], (M, QD)),
                        as_f32_np(plan_attn["scales"], (M, QD // 128)))
            rel_rms_close(g, w, f"{what} vs plan")
    else:
        g = got.cpu().view(torch.int16).numpy().view(np.uint16).reshape(M, QD)
        bf16_close(g, oracle.bf16_from_double(want64), f"{what} vs oracle")
        if plan_attn is not None:
            bf16_close(g, as_bf16_np(plan_attn["attn"], (M, QD)), f"{what} vs plan")


def _run_twice(cfg, num_sms=0):
    inp, q, want = _plan_step(cfg, num_sms)
    layer = cfg.n_layers - 1
    ref = _oracle_attention(cfg, layer, q, inp)
    for call in range(2):
        out, sc = _alloc_out(cfg)
        dl.attention_noalloc(cfg, layer, q, inp["kv_pages"], inp["block_table"],
                             inp["positions"], out, sc, num_sms=num_sms, check=True)
        torch.cuda.synchronize()
        _compare(cfg, out, sc, ref, want, f"{cfg.name} call {call + 1}")
    return inp, q


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_oracle_and_plan_twice(name):
    _run_twice(CASES[name])


@pytest.mark.parametrize("name", ["bf16_qr32", "fp8_m16"])
def test_noalloc_async_calls_back_to_back(name):
    """Two calls with check = 0 on one stream, different queries and
    outputs, one synchronisation; each output is checked against the oracle
    given its own query."""
    cfg = CASES[name]
    inp, q1, _ = _plan_step(cfg)
    layer = cfg.n_layers - 1
    g = torch.Generator(device="cpu")
    g.manual_seed(1234)
    q2 = torch.randn(q1.numel() // 2, generator=g).to(torch.bfloat16).to(DEV)
    o1, s1 = _alloc_out(cfg)
    o2, s2 = _alloc_out(cfg)
    stream = torch.cuda.current_stream()
    for q, o, s in ((q1, o1, s1), (q2, o2, s2)):
        dl.attention_noalloc(cfg, layer, q, inp["kv_pages"], inp["block_table"],
                             inp["positions"], o, s, check=False, stream=stream)
    torch.cuda.synchronize()
    for i, (q, o, s) in enumerate(((q1, o1, s1), (q2, o2, s2))):
        _compare(cfg, o, s, _oracle_attention(cfg, layer, q, inp), None,
                 f"{cfg.name} async call {i + 1}")


def test_noalloc_rejects_oversized_scratch_then_runs():
    """At every SM the 64-row case needs more scratch than there is: the call
    is refused (and nothing is launched), a good call right after it works,
    and with fewer SMs the 64-row case itself runs."""
    cfg = QR64
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks = -(-cfg.context // 64)
    pairs = cfg.num_requests * cfg.n_kv_heads
    G = min(sms, pairs * blocks, 62 * pairs)
    need = 17152 + G * 2 * 64 * 129 * 4
    if need > SCRATCH_BYTES:
        inp = {k: v.to(DEV) for k, v in synth.make_inputs(cfg).items()}
        QD = cfg.n_q_heads * cfg.head_dim
        q = torch.zeros((cfg.M, QD), dtype=torch.bfloat16, device=DEV)
        out = torch.zeros((cfg.M, QD), dtype=torch.bfloat16, device=DEV)
        with pytest.raises(dl.DLError) as e:
            dl.attention_noalloc(cfg, 0, q, inp["kv_pages"], inp["block_table"],
                                 inp["positions"], out, None, check=True)
        assert e.value.status == 2 and "scratch" in str(e.value), str(e.value)
        _run_twice(CASES["bf16_m4"])
    # 100 CTAs x 2 x 64 rows x 516 bytes fits
    _run_twice(cfg, num_sms=100)


def test_noalloc_reports_out_of_range_position_then_runs():
    """A position at max_context (one past the last allowed) is reported by
    the kernel's own bounds check as DL_ERR_DEVICE_BOUNDS; the next good call
    on the same scratch gives the right result."""
    cfg = CASES["bf16_m4"]
    inp, q = _run_twice(cfg)
    bad = inp["positions"].clone()
    bad[-1] = cfg.context          # max_context = cfg.context
    out, sc = _alloc_out(cfg)
    with pytest.raises(dl.DLError) as e:
        dl.attention_noalloc(cfg, 0, q, inp["kv_pages"], inp["block_table"], bad, out, sc,
                             check=True)
    assert e.value.status == 7, str(e.value)
    out, sc = _alloc_out(cfg)
    dl.attention_noalloc(cfg, 0, q, inp["kv_pages"], inp["block_table"], inp["positions"], out,
                         sc, check=True)
    torch.cuda.synchronize()
    _compare(cfg, out, sc, _oracle_attention(cfg, 0, q, inp), None, "after the refused call")
