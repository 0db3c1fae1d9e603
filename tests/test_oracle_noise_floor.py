"""The noise floor of the bf16 materialisation chain, on the CPU.

The layer rounds to bf16 at every materialised tensor (r', h, q/k/v, q^, k^,
attention output, o, r'', h2, g, u, a, y).  Two correct implementations
that accumulate in different precisions (fp64 in the oracle, fp32 in the
kernels) round an intermediate differently wherever its exact value sits
next to a bf16 rounding boundary: a one-ulp flip.  Each later operation sums
these flips, so element-wise agreement within 1e-2 (1 + |oracle|) holds per
operation given identical inputs, but not for the output of a long chain.

This file measures that floor without a GPU.  A vectorised torch
restatement of the layer, with the oracle's materialisation points, runs
with the kernels' arithmetic (fp32 sums, attention probabilities entering
the P.V product as bf16) on the Qwen3-8B-shaped bf16 sweep cell with 4
requests at context 1024, and is compared with the fp64 oracle:
- every projection given the same input meets the element bound;
- the first tensors of the chain (r', h1, q^) agree bit for bit;
- the layer output y breaks the element bound at a few hundred elements or
  fewer with errors of a few hundredths, the order the CUDA path shows
  against the oracle on the same cell (105 of 16384 elements, largest error
  0.0625);
- the relative RMS error of y and of the new residual stays below 1e-2,
  the bound the GPU parity tests hold layer outputs of long chains to.
The same restatement in float64 reproduces the oracle (the cross-check of
test_oracle_layer.py at this size).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from pdl_persistent_megakernel_gb300 import synth

CELL = synth.sweep_config(4, 1024, False)


def f64(b):
    return oracle.bf16_to_double(np.asarray(b))


def torch_layer(cfg, w, inputs, dt, p_bf16=False):
    """The decode layer in torch with arithmetic type `dt`, rounding to bf16
    where the oracle materialises a tensor.  With p_bf16 the attention
    probabilities exp(s - max) enter the P.V product as bf16 numbers (a
    tensor-core PV product takes bf16 operands) and the sum that normalises
    them stays in `dt`.  Returns the materialised tensors by name (as float64
    values of bf16 numbers)."""
    bf = lambda t: t.to(torch.bfloat16).to(dt)
    d, P = cfg.head_dim, cfg.page_size
    Hq, Hkv = cfg.n_q_heads, cfg.n_kv_heads
    G, T, M, I = Hq // Hkv, cfg.tokens_per_request, cfg.M, cfg.inter
    x, res = inputs["x"].to(dt), inputs["residual"].to(dt)
    cache = inputs["kv_pages"].clone()
    out = {}

    def rms(v, wt):
        return v / torch.sqrt((v * v).mean(-1, keepdim=True) + cfg.eps) * wt.to(dt)

    out["r1"] = r1 = bf(x + res)
    out["h1"] = h1 = bf(rms(r1, w["ln1_w"]))
    qkv = bf(h1 @ w["w_qkv"].to(dt).T)
    heads = qkv.view(M, -1, d)
    inv = torch.tensor([cfg.rope_theta ** (-2.0 * i / d) for i in range(d // 2)],
                       dtype=torch.float64)
    pos = inputs["positions"].to(torch.int64)
    ang = pos.double()[:, None] * inv[None, :]
    cos, sin = torch.cos(ang).to(dt)[:, None], torch.sin(ang).to(dt)[:, None]

    def rot(v):
        a, b = v[..., :d // 2], v[..., d // 2:]
        return torch.cat([a * cos - b * sin, b * cos + a * sin], -1)

    out["q_rot"] = q = bf(rot(bf(rms(heads[:, :Hq], w["q_norm_w"]))))
    k = bf(rot(bf(rms(heads[:, Hq:Hq + Hkv], w["k_norm_w"]))))
    v = heads[:, Hq + Hkv:]
    bt = inputs["block_table"].to(torch.int64)
    pg = bt[torch.arange(M) // T, pos // P]
    cache[0, pg, 0, :, pos % P] = k.to(torch.bfloat16)
    cache[0, pg, 1, :, pos % P] = v.to(torch.bfloat16)
    attn = torch.zeros(M, Hq, d, dtype=dt)
    for r in range(cfg.num_requests):
        toks = torch.arange(r * T, (r + 1) * T)
        n = int(pos[toks[-1]]) + 1
        j = torch.arange(n)
        pages = bt[r, j // P]
        K = cache[0, pages, 0, :, j % P].to(dt)        # [n, Hkv, d]
        V = cache[0, pages, 1, :, j % P].to(dt)
        for hk in range(Hkv):
            qq = q[toks, hk * G:(hk + 1) * G]          # [T, G, d]
            s = qq @ K[:, hk].T / math.sqrt(d)          # [T, G, n]
            causal = j[None, :] <= pos[toks][:, None]   # [T, n]
            s = s.masked_fill(~causal[:, None, :], float("-inf"))
            if p_bf16:
                e = torch.exp(s - s.amax(-1, keepdim=True))
                o = bf(e) @ V[:, hk] / e.sum(-1, keepdim=True)
            else:
                o = torch.softmax(s, -1) @ V[:, hk]
            attn[toks, hk * G:(hk + 1) * G] = o
    out["attn"] = attn = bf(attn.view(M, -1))
    out["o2"] = o2 = bf(attn @ w["w_o"].to(dt).T)
    out["r2"] = r2 = bf(o2 + r1)
    out["h2"] = h2 = bf(rms(r2, w["ln2_w"]))
    gu = bf(h2 @ w["w_gate_up"].to(dt).T)
    out["act"] = a = bf(torch.nn.functional.silu(gu[:, :I]) * gu[:, I:])
    out["y"] = bf(a @ w["w_down"].to(dt).T)
    return {k: t.double().reshape(M, -1).numpy() for k, t in out.items()}


def _violations(got, want):
    err = np.abs(got - want)
    return int((err > 1e-2 * (1 + np.abs(want))).sum()), float(err.max())


def _rel_rms(got, want):
    return float(np.sqrt(((got - want) ** 2).mean() / (want ** 2).mean()))


@pytest.fixture(scope="module")
def cell():
    cfg = CELL
    w = synth.make_layer_weights(cfg, 0)
    inputs = synth.make_inputs(cfg)
    ref = oracle.decode_step(cfg, {"layers": [w]}, inputs, trace=True)
    return cfg, w, inputs, ref


def test_float64_restatement_reproduces_the_oracle(cell):
    cfg, w, inputs, ref = cell
    got = torch_layer(cfg, w, inputs, torch.float64)
    for name in ("r1", "h1"):
        assert np.array_equal(got[name], f64(ref[name])), name
    for name in ("q_rot", "attn", "o2", "r2", "h2", "act"):
        assert _violations(got[name], f64(ref[name]))[0] == 0, name
    assert _violations(got["y"], f64(ref["out"][0]))[0] == 0


def test_kernel_arithmetic_noise_floor(cell):
    """fp32 arithmetic and bf16 attention probabilities, as in the kernels."""
    cfg, w, inputs, ref = cell
    got = torch_layer(cfg, w, inputs, torch.float32, p_bf16=True)
    y_want = f64(ref["out"][0])
    # the chain's first tensors have identical inputs and no long sums
    for name in ("r1", "h1", "q_rot"):
        assert np.array_equal(got[name], f64(ref[name])), name
    # every projection, given this side's own input, meets the element bound:
    # the oracle's operation applied to the same input
    I = cfg.inter
    for src, dst, wname in (("attn", "o2", "w_o"), ("h2", "act", "w_gate_up"),
                            ("act", "y", "w_down")):
        want = oracle.gemm_bf16(got[src], synth.as_u16(w[wname]))
        if dst == "act":
            g = f64(oracle.bf16_from_double(want[:, :I]))
            u = f64(oracle.bf16_from_double(want[:, I:]))
            want = oracle.silu(g) * u
        n, e = _violations(got[dst], f64(oracle.bf16_from_double(want)))
        assert n == 0, (dst, n, e)
    # end to end the element bound breaks on y, by the amount the CUDA path
    # shows on this cell (105 of 16384 elements, largest error 0.0625)
    n, e = _violations(got["y"], y_want)
    assert 10 <= n <= 1000, n
    assert 0.01 < e < 0.25, e
    # while the relative RMS error of the layer outputs stays below 1e-2
    assert _rel_rms(got["y"], y_want) < 1e-2
    assert _rel_rms(got["r2"], f64(ref["out"][1])) < 1e-2
