"""Seeded synthetic workloads for the decode step.

This module only draws inputs: shapes, random weights, caches, block tables
and positions.  It holds none of the decode step's arithmetic and is the one
piece of code shared by the CUDA path's tests/bench and the CPU oracle's
harness.

Distributions (the workload recipe):
  * projection and lm_head weights ~ N(0, 0.02) in bf16;
  * RMSNorm weights (ln1, ln2, q_norm, k_norm, final) = 1 + N(0, 0.02): with a
    literal N(0, 0.02) every norm output would collapse to ~0.02 scale and the
    logits would be nearly flat, which makes the greedy-id check vacuous;
  * FP8 configs store each projection as OCP e4m3 codes with one fp32 scale
    per 128x128 block, s = amax(block) / 448 (s = 1 for an all-zero block),
    code = e4m3(w / s) -- the weight format the FP8 configuration names;
  * x, residual ~ N(0, 1) bf16; the paged KV cache ~ N(0, 1) bf16 everywhere;
  * block table: a seeded random permutation of the pages, consumed in order,
    ceil(context / page_size) pages per request; three spare pages are never
    referenced;
  * positions: request r's T new tokens sit at context - T .. context - 1.

Every tensor gets its own generator seeded from (config seed, tensor name),
so a tensor's values do not depend on which other tensors were drawn.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Dict, List, Optional

import torch


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    hidden: int
    inter: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_layers: int
    vocab: int            # 0: single-layer plan, no lm_head
    fp8: bool
    num_requests: int
    tokens_per_request: int
    context: int          # keys per request after this step (= last position + 1)
    page_size: int
    eps: float = 1e-6
    rope_theta: float = 1e6
    seed: int = 1234
    spare_pages: int = 3

    @property
    def M(self) -> int:
        return self.num_requests * self.tokens_per_request

    @property
    def pages_per_request(self) -> int:
        return -(-self.context // self.page_size)

    @property
    def num_pages(self) -> int:
        return self.num_requests * self.pages_per_request + self.spare_pages

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    def replace(self, **kw) -> "DecodeConfig":
        return dataclasses.replace(self, **kw)


Q06 = dict(hidden=1024, inter=3072, n_q_heads=16, n_kv_heads=8, head_dim=128)
Q8 = dict(hidden=4096, inter=12288, n_q_heads=32, n_kv_heads=8, head_dim=128)
VOCAB = 151936

CONFIGS: Dict[str, DecodeConfig] = {
    # Qwen3-0.6B-shaped single layer, batch 1, context 1024, 16-token pages.
    "q06_layer_b1_ctx1024": DecodeConfig(
        "q06_layer_b1_ctx1024", **Q06, n_layers=1, vocab=0, fp8=False,
        num_requests=1, tokens_per_request=1, context=1024, page_size=16,
        seed=1235),
    # Full Qwen3-0.6B-shaped step: 28 layers + final norm + lm_head + argmax.
    "q06_step_b1_ctx4096": DecodeConfig(
        "q06_step_b1_ctx4096", **Q06, n_layers=28, vocab=VOCAB, fp8=False,
        num_requests=1, tokens_per_request=1, context=4096, page_size=16,
        seed=1236),
    # Qwen3-8B-shaped layer, M = 16 (2 requests x 8 tokens), FP8, ctx 8192.
    "q8_layer_m16_ctx8192_fp8": DecodeConfig(
        "q8_layer_m16_ctx8192_fp8", **Q8, n_layers=1, vocab=0, fp8=True,
        num_requests=2, tokens_per_request=8, context=8192, page_size=64,
        seed=1237),
    # Full Qwen3-8B-shaped step: 36 layers, batch 1, ctx 8192, bf16.
    "q8_step_b1_ctx8192": DecodeConfig(
        "q8_step_b1_ctx8192", **Q8, n_layers=36, vocab=VOCAB, fp8=False,
        num_requests=1, tokens_per_request=1, context=8192, page_size=64,
        seed=1238),
}


def sweep_config(batch: int, context: int, fp8: bool) -> DecodeConfig:
    """Crossover sweep cell: Qwen3-8B-shaped layer, `batch` requests of one
    token each at position context - 1, 64-token pages."""
    return DecodeConfig(
        f"q8_layer_b{batch}_ctx{context}_{'fp8' if fp8 else 'bf16'}", **Q8,
        n_layers=1, vocab=0, fp8=fp8, num_requests=batch,
        tokens_per_request=1, context=context, page_size=64,
        seed=1239 + batch * 7 + context // 1024)


def _seed(cfg: DecodeConfig, name: str) -> int:
    h = hashlib.sha256(f"{cfg.seed}/{name}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(cfg: DecodeConfig, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(cfg, name))
    return g


def randn_bf16(cfg: DecodeConfig, name: str, shape, std: float = 1.0,
               mean: float = 0.0, device="cpu") -> torch.Tensor:
    g = _gen(cfg, name, device)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    # draw in fp32 chunks to bound host memory for multi-GB tensors
    flat = out.view(-1)
    step = 1 << 26
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        t = torch.randn(n, generator=g, dtype=torch.float32, device=device)
        flat[i:i + n] = (t * std + mean).to(torch.bfloat16)
    return out


def quantize_blocks_e4m3(w: torch.Tensor):
    """Store a bf16 [N, K] weight as e4m3 codes (uint8 [N, K]) plus one fp32
    scale per 128x128 block ([N/128, K/128]).  Input preparation for the FP8
    weight format; N and K must be multiples of 128."""
    N, K = w.shape
    assert N % 128 == 0 and K % 128 == 0
    codes = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    scales = torch.empty((N // 128, K // 128), dtype=torch.float32,
                         device=w.device)
    rows = 1024
    for n0 in range(0, N, rows):
        blk = w[n0:n0 + rows].float()
        nb = blk.shape[0] // 128
        b4 = blk.view(nb, 128, K // 128, 128)
        amax = b4.abs().amax(dim=(1, 3))
        s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        scales[n0 // 128:n0 // 128 + nb] = s
        q = (b4 / s[:, None, :, None]).view(blk.shape)
        codes[n0:n0 + rows] = q.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scales


def make_layer_weights(cfg: DecodeConfig, layer: int, device="cpu") -> dict:
    H, I, d = cfg.hidden, cfg.inter, cfg.head_dim
    qd = cfg.n_q_heads * d
    pre = f"layer{layer}/"
    w = {
        "ln1_w": randn_bf16(cfg, pre + "ln1_w", (H,), 0.02, 1.0, device),
        "q_norm_w": randn_bf16(cfg, pre + "q_norm_w", (d,), 0.02, 1.0, device),
        "k_norm_w": randn_bf16(cfg, pre + "k_norm_w", (d,), 0.02, 1.0, device),
        "ln2_w": randn_bf16(cfg, pre + "ln2_w", (H,), 0.02, 1.0, device),
    }
    shapes = {"w_qkv": (cfg.qkv_rows, H), "w_o": (H, qd),
              "w_gate_up": (2 * I, H), "w_down": (H, I)}
    for name, shp in shapes.items():
        wt = randn_bf16(cfg, pre + name, shp, 0.02, 0.0, device)
        if cfg.fp8:
            codes, scales = quantize_blocks_e4m3(wt)
            del wt
            w[name] = codes
            w[name + "_scale"] = scales
        else:
            w[name] = wt
            w[name + "_scale"] = None
    return w


def make_weights(cfg: DecodeConfig, device="cpu") -> dict:
    out = {"layers": [make_layer_weights(cfg, l, device)
                      for l in range(cfg.n_layers)]}
    if cfg.vocab > 0:
        out["final_norm_w"] = randn_bf16(cfg, "final_norm_w", (cfg.hidden,),
                                         0.02, 1.0, device)
        out["lm_head_w"] = randn_bf16(cfg, "lm_head_w",
                                      (cfg.vocab, cfg.hidden), 0.02, 0.0,
                                      device)
    else:
        out["final_norm_w"] = None
        out["lm_head_w"] = None
    return out


def make_inputs(cfg: DecodeConfig, device="cpu") -> dict:
    M, H = cfg.M, cfg.hidden
    x = randn_bf16(cfg, "x", (M, H), device=device)
    res = randn_bf16(cfg, "residual", (M, H), device=device)
    kv = randn_bf16(cfg, "kv_pages",
                    (cfg.n_layers, cfg.num_pages, 2, cfg.n_kv_heads,
                     cfg.page_size, cfg.head_dim), device=device)
    g = _gen(cfg, "block_table", "cpu")
    perm = torch.randperm(cfg.num_pages, generator=g, dtype=torch.int64)
    ppr = cfg.pages_per_request
    bt = perm[:cfg.num_requests * ppr].to(torch.int32).view(
        cfg.num_requests, ppr).to(device)
    T = cfg.tokens_per_request
    pos = torch.tensor([cfg.context - T + t for r in range(cfg.num_requests)
                        for t in range(T)], dtype=torch.int32, device=device)
    return {"x": x, "residual": res, "kv_pages": kv, "block_table": bt,
            "positions": pos}


def as_u16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 view (bit pattern), on the CPU."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
