"""CPU checks of the GPU tests' own reference helpers (tests/gpu_harness.py):
each, fed the oracle's own inputs, must reproduce the oracle's result, and
each tolerance helper must flag the mistakes it exists to catch."""
import numpy as np
import pytest
import torch

import oracle
from pdl_persistent_megakernel_gb300 import synth
import gpu_harness as gh

FP8 = synth.DecodeConfig("h_fp8", hidden=256, inter=256, n_q_heads=4, n_kv_heads=2,
                         head_dim=128, n_layers=1, vocab=0, fp8=True, num_requests=2,
                         tokens_per_request=2, context=40, page_size=16, seed=5)


class _Case:
    def __init__(self, cfg):
        self.cfg = cfg
        self.w = synth.make_weights(cfg)
        self.inp = synth.make_inputs(cfg)
        self.ref = oracle.decode_step(cfg, self.w, self.inp, trace=True)


def test_fp8_qkv_from_oracle_h1_reproduces_the_oracle():
    c = _Case(FP8)
    cfg = c.cfg
    q, k, v = gh.fp8_qkv_from_h1(c, c.ref["h1_codes"], c.ref["h1_scales"])
    assert np.array_equal(q.reshape(cfg.M, -1), c.ref["q_rot"])
    assert np.array_equal(k.reshape(cfg.M, -1), c.ref["k_rot"])
    assert np.array_equal(v.reshape(cfg.M, -1), c.ref["v"])


def test_fp8_code_check_accepts_own_codes_and_flags_a_real_difference():
    c = _Case(FP8)
    cfg = c.cfg
    lw = c.w["layers"][0]
    _, _, hf = oracle.add_rmsnorm(synth.as_u16(c.inp["x"]), synth.as_u16(c.inp["residual"]),
                                  synth.as_u16(lw["ln1_w"]), cfg.eps)
    codes, scales = c.ref["h1_codes"], c.ref["h1_scales"]
    gh.check_fp8_codes_exact(codes, scales, codes, scales, hf, "same")
    # a code moved by one step where the quotient is far from a boundary
    q = (hf.reshape(cfg.M, -1, 128) / scales[:, :, None]).reshape(cfg.M, -1)
    mids = gh._e4m3_midpoints()
    aq = np.abs(q)
    j = np.clip(np.searchsorted(mids, aq), 1, len(mids) - 1)
    far = np.minimum(np.abs(aq - mids[j]), np.abs(aq - mids[j - 1])) > 1e-3 * aq
    far &= (codes & 0x7F) > 8
    idx = np.argwhere(far)[0]
    bad = codes.copy()
    bad[tuple(idx)] = bad[tuple(idx)] - 1
    with pytest.raises(AssertionError):
        gh.check_fp8_codes_exact(bad, scales, codes, scales, hf, "moved")
    # a scale off by 1e-4
    with pytest.raises(AssertionError):
        gh.check_fp8_codes_exact(codes, scales * (1 + 1e-4), codes, scales, hf, "scale")


def test_rope_close_pair_bound():
    rng = np.random.default_rng(3)
    w = oracle.bf16_from_double(rng.standard_normal((4, 128)))
    gh.rope_close(w, w, "same")
    # a one-ulp-scale error of a large partner passes, a 5 % error does not
    off = oracle.bf16_from_double(gh.f64(w) * 1.05)
    with pytest.raises(AssertionError):
        gh.rope_close(off, w, "5%")
