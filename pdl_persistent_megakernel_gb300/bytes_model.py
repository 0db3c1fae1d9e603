"""Byte accounting for the memory-bound decode step (measurement, not compute).

Two models:

* ``algorithmic_bytes(cfg)`` -- the bytes one decode step must move, each
  once: projection weights (FP8 codes plus their fp32 128x128 block scales),
  norm weights, every request's K and V read once (shared by its G*T query
  rows), the step's new K/V written, activations in/out (4*M*H elements per
  layer), and for full steps the lm_head and the fp32 logits.  Re-reads,
  split-KV partials, split-K workspace and counters are excluded.  This is the
  numerator of every achieved-GB/s figure the bench reports.

* ``gap_model(...)`` -- the kernel-per-op accounting of the analytic gap
  model on page "PDL and megakernel" (section on estimating the gaps): each
  of the ten kernels of a layer plus three tail kernels is charged its read +
  write bytes, the step's data time is total bytes / effective bandwidth, and
  every kernel boundary adds a gap g.  It exists to pin our accounting
  against the table that page prints (see tests/golden/decode_gaps.json).
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

from .synth import DecodeConfig


def algorithmic_bytes(cfg: DecodeConfig) -> Dict[str, float]:
    H, I, d = cfg.hidden, cfg.inter, cfg.head_dim
    wb = 1 if cfg.fp8 else 2
    mats = [(cfg.qkv_rows, H), (H, cfg.n_q_heads * d), (2 * I, H), (H, I)]
    w = sum(n * k * wb for n, k in mats)
    if cfg.fp8:
        w += sum((n // 128) * (k // 128) * 4 for n, k in mats)
    w += (2 * H + 2 * d) * 2
    kvd = cfg.n_kv_heads * d
    per_layer = {
        "weights": w,
        "kv_read": cfg.num_requests * cfg.context * kvd * 2 * 2,
        "kv_write": cfg.M * kvd * 2 * 2,
        "activations": 4 * cfg.M * H * 2,
    }
    out = {k: float(v * cfg.n_layers) for k, v in per_layer.items()}
    if cfg.vocab > 0:
        out["lm_head"] = float(cfg.vocab * H * 2 + H * 2)
        out["logits"] = float(cfg.M * cfg.vocab * 4)
    out["total"] = float(sum(out.values()))
    return out


def gap_model_kernels(hidden: int, inter: int, layers: int, heads: int,
                      kv_heads: int, head_dim: int, vocab: int, batch: int,
                      context: int, elem_bytes: int = 2
                      ) -> List[Tuple[str, int]]:
    """(kernel, bytes read + written) for one decode step, vLLM-level fusion:
    residual add + RMSNorm and QK-norm + RoPE are one kernel each."""
    qdim, kvdim = heads * head_dim, kv_heads * head_dim
    act = batch * hidden * elem_bytes          # one activation row set
    per_layer = [
        ("add_rmsnorm", 4 * act),              # x, residual in; residual, h out
        ("qkv_proj", hidden * (qdim + 2 * kvdim) * elem_bytes),
        ("qk_norm_rope", 2 * batch * (qdim + kvdim) * elem_bytes),
        ("kv_cache_write", 2 * batch * kvdim * elem_bytes),
        ("attention", batch * context * 2 * kvdim * elem_bytes),
        ("o_proj", qdim * hidden * elem_bytes),
        ("add_rmsnorm", 4 * act),
        ("gate_up_proj", hidden * 2 * inter * elem_bytes),
        ("silu_mul", 3 * batch * inter * elem_bytes),
        ("down_proj", inter * hidden * elem_bytes),
    ]
    tail = [("final_norm", 2 * act), ("lm_head", hidden * vocab * elem_bytes),
            ("sample", batch * vocab * 4)]
    return per_layer * layers + tail


def gap_model(kernels: Sequence[Tuple[str, int]], bandwidth: float,
              gaps_us: Sequence[float]) -> Dict[str, object]:
    """Data time (us) = sum(bytes) / bandwidth; with a gap g per kernel the
    step takes data + n * g.  Also counts kernels whose own data time is
    under 1 us."""
    n = len(kernels)
    t_data = sum(b for _, b in kernels) / bandwidth * 1e6
    return {
        "kernels": n,
        "data_us": t_data,
        "with_gap_us": [t_data + n * g for g in gaps_us],
        "gap_share": [n * g / (t_data + n * g) for g in gaps_us],
        "under_1us": sum(1 for _, b in kernels if b / bandwidth * 1e6 < 1.0),
        "mean_us": t_data / n,
    }


def op_bytes(cfg: DecodeConfig, name: str) -> float:
    """Algorithmic bytes of one launch of a serial-schedule operation (inputs
    read once, outputs written once, weights once)."""
    H, I, d = cfg.hidden, cfg.inter, cfg.head_dim
    M, R = cfg.M, cfg.num_requests
    qd, kvd = cfg.n_q_heads * d, cfg.n_kv_heads * d
    eb = 1 if cfg.fp8 else 2

    def act(K):  # a quantised (or bf16) activation [M, K]
        return M * K * eb + (M * (K // 128) * 4 if cfg.fp8 else 0)

    def wts(N, K):
        return N * K * eb + ((N // 128) * (K // 128) * 4 if cfg.fp8 else 0)

    if name in ("add_rmsnorm1", "add_rmsnorm2"):
        return 3 * M * H * 2 + act(H) + H * 2
    if name == "final_norm":
        return 3 * M * H * 2 + M * H * 2 + H * 2
    if name == "qkv_rope_kvwrite":
        return wts(cfg.qkv_rows, H) + act(H) + M * qd * 2 + M * 2 * kvd * 2 + 2 * d * 2
    if name == "attention":
        return R * cfg.context * kvd * 2 * 2 + M * qd * 2 + act(qd)
    if name == "o_proj":
        return wts(H, qd) + act(qd) + M * H * 2
    if name == "gate_up_silu":
        return wts(2 * I, H) + act(H) + act(I)
    if name == "down_proj":
        return wts(H, I) + act(I) + M * H * 2
    if name == "lm_head_argmax":
        return cfg.vocab * H * 2 + M * H * 2 + M * cfg.vocab * 4 + M * 4
    raise KeyError(name)
