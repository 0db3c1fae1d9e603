"""Pins of the oracle's operations against closed forms, invariants, library
routines (numpy / torch float64) and brute force on tiny inputs."""
import math

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(11)


def bf16(a) -> np.ndarray:
    t = torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f64(b) -> np.ndarray:
    return oracle.bf16_to_double(b)


# ----------------------------------------------------- add + RMSNorm (+quant)

def test_residual_add_matches_torch_and_unit_rms():
    M, H = 3, 256
    x = bf16(RNG.standard_normal((M, H)))
    r = bf16(RNG.standard_normal((M, H)))
    ones = bf16(np.ones(H))
    r_out, hb, hf = oracle.add_rmsnorm(x, r, ones, 1e-6)
    tx = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    tr = torch.from_numpy(r.view(np.int16)).view(torch.bfloat16).float()
    want = (tx + tr).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(r_out, want)
    # with w = 1: rms(h) = sqrt(ms / (ms + eps)), ms = mean(r_out^2)
    rr = f64(r_out)
    ms = (rr ** 2).mean(axis=1)
    rms = np.sqrt((hf.astype(np.float64) ** 2).mean(axis=1))
    assert np.allclose(rms, np.sqrt(ms / (ms + 1e-6)), rtol=1e-6)


def test_rmsnorm_constant_row_and_weight():
    H = 128
    for c in (0.5, -3.0, 1e-3):
        x = bf16(np.full((1, H), c))
        z = bf16(np.zeros((1, H)))
        w = bf16(RNG.uniform(0.5, 1.5, H))
        _, _, hf = oracle.add_rmsnorm(x, z, w, 1e-6)
        cc = f64(x)[0, 0]
        want = cc / math.sqrt(cc * cc + 1e-6) * f64(w)
        assert np.allclose(hf[0], want, rtol=1e-6)
    # eps inside the sqrt: an all-zero row stays zero
    _, hb, hf = oracle.add_rmsnorm(bf16(np.zeros((1, H))), bf16(np.zeros((1, H))),
                                   bf16(np.ones(H)), 1e-6)
    assert not hf.any() and not hb.any()


def test_quant_group128_properties():
    M, K = 4, 512
    v = (RNG.standard_normal((M, K)) * np.array([1e-3, 1.0, 30.0, 1.0])[:, None]).astype(np.float32)
    v[3, 128:256] = 0.0                               # an all-zero group
    codes, scales = oracle.quant_group128(v)
    assert scales.shape == (M, K // 128)
    assert scales[3, 1] == 1.0 and not codes[3, 128:256].any()
    deq = oracle.e4m3_decode(codes) * np.repeat(scales, 128, axis=1)
    for m in range(M):
        for g in range(K // 128):
            blk = v[m, g * 128:(g + 1) * 128].astype(np.float64)
            if not blk.any():
                continue
            amax = np.abs(blk).max()
            assert np.isclose(scales[m, g], np.float32(amax) / np.float32(448.0), rtol=0)
            i = int(np.abs(blk).argmax())
            assert (codes[m, g * 128 + i] & 0x7F) == 0x7E     # amax -> 448
            # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normals,
            # absolute error <= 2^-10 * s in the subnormal range
            err = np.abs(deq[m, g * 128:(g + 1) * 128] - blk)
            bound = np.maximum(np.abs(blk) * 2.0 ** -4, 2.0 ** -10 * scales[m, g])
            assert np.all(err <= bound * (1 + 1e-6))
    # library check: codes equal torch's e4m3 cast of v / s (fp32 division)
    q = torch.from_numpy(v) / torch.from_numpy(np.repeat(scales, 128, axis=1))
    want = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, want)


# ----------------------------------------------------------------- GEMMs

def test_gemm_bf16_one_hot_and_numpy():
    M, N, K = 3, 40, 96
    a = f64(bf16(RNG.standard_normal((M, K))))
    w = np.zeros((N, K), np.uint16)
    for n in range(N):
        w[n, (7 * n) % K] = bf16([1.0])[0]
    out = oracle.gemm_bf16(a, w)
    for n in range(N):
        assert np.array_equal(out[:, n], a[:, (7 * n) % K])
    wr = bf16(RNG.standard_normal((N, K)) * 0.05)
    out = oracle.gemm_bf16(a, wr)
    assert np.allclose(out, a @ f64(wr).T, rtol=1e-12, atol=1e-14)


def test_gemm_fp8_matches_dequantized_numpy():
    M, N, K = 5, 256, 384
    a_codes = RNG.integers(0, 256, (M, K), dtype=np.uint8)
    w_codes = RNG.integers(0, 256, (N, K), dtype=np.uint8)
    for c in (a_codes, w_codes):
        c[(c & 0x7F) == 0x7F] = 0x10                  # no NaN codes
    a_s = RNG.uniform(0.01, 2, (M, K // 128)).astype(np.float32)
    w_s = RNG.uniform(0.01, 2, (N // 128, K // 128)).astype(np.float32)
    out = oracle.gemm_fp8(a_codes, a_s, w_codes, w_s)
    dec = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).double().numpy()
    A = dec(a_codes) * np.repeat(a_s.astype(np.float64), 128, axis=1)
    W = dec(w_codes) * np.kron(w_s.astype(np.float64), np.ones((128, 128)))
    want = A @ W.T
    assert np.allclose(out, want, rtol=1e-11, atol=1e-9 * np.abs(want).max())


# --------------------------------------------------------- QK-norm + RoPE

def test_head_rmsnorm_unit_rms():
    d = 128
    v = RNG.standard_normal(d) * 7
    out = oracle.head_rmsnorm(v, bf16(np.ones(d)), 1e-6)
    ms = (v ** 2).mean()
    assert np.isclose(np.sqrt((out ** 2).mean()), np.sqrt(ms / (ms + 1e-6)), rtol=1e-12)


def test_rope_invariants():
    d, theta = 128, 1e6
    q = RNG.standard_normal(d)
    k = RNG.standard_normal(d)
    assert np.array_equal(oracle.rope(q, 0, theta), q)         # p = 0: identity
    for p in (1, 17, 8191, 32767):
        rq = oracle.rope(q, p, theta)
        pn = q[:64] ** 2 + q[64:] ** 2
        assert np.allclose(rq[:64] ** 2 + rq[64:] ** 2, pn, rtol=1e-12)
    # <R_p q, R_s k> depends only on p - s
    a = oracle.rope(q, 100, theta) @ oracle.rope(k, 40, theta)
    b = oracle.rope(q, 5060, theta) @ oracle.rope(k, 5000, theta)
    assert np.isclose(a, b, rtol=1e-9)
    # one-hot e_0 pairs with e_64 at angle p * theta^0 = p (neox half split)
    e0 = np.zeros(d)
    e0[0] = 1.0
    out = oracle.rope(e0, 3, theta)
    assert np.isclose(out[0], math.cos(3)) and np.isclose(out[64], math.sin(3))
    assert np.count_nonzero(np.abs(out) > 1e-15) == 2
    # pair i = 10 rotates by p * theta^(-20/128)
    e = np.zeros(d)
    e[10 + 64] = 1.0
    out = oracle.rope(e, 9, theta)
    ang = 9 * theta ** (-20 / 128)
    assert np.isclose(out[10], -math.sin(ang)) and np.isclose(out[74], math.cos(ang))


# --------------------------------------------------------------- paged KV

def test_kv_gather_matches_numpy_indexing_with_tags():
    L, NP, Hkv, P, d = 2, 9, 2, 4, 8
    cache = np.arange(L * NP * 2 * Hkv * P * d, dtype=np.uint32).astype(np.uint16)
    cache = cache.reshape(L, NP, 2, Hkv, P, d)
    R, ppr = 2, 4
    bt = np.random.default_rng(5).permutation(NP)[:R * ppr].astype(np.int32).reshape(R, ppr)
    for layer in range(L):
        for r in range(R):
            for h in range(Hkv):
                for kv in range(2):
                    n = 13
                    got = oracle.kv_gather(cache, bt, Hkv, P, d, layer, r, h, kv, n)
                    want = np.stack([cache[layer, bt[r, j // P], kv, h, j % P] for j in range(n)])
                    assert np.array_equal(got, want)
    # flat offsets agree with numpy's row-major layout of the 6-D cache
    idx = (1, 7, 1, 1, 3, 5)
    assert oracle.kv_offset(NP, Hkv, P, d, *idx) == np.ravel_multi_index(idx, cache.shape)
    # a block-table entry out of range is rejected
    bad = bt.copy()
    bad[0, 0] = NP
    with pytest.raises(ValueError):
        oracle.kv_gather(cache, bad, Hkv, P, d, 0, 0, 0, 0, 3)


# ------------------------------------------------- attention + LSE combine

def _rand_kv(n, d):
    return bf16(RNG.standard_normal((n, d))), bf16(RNG.standard_normal((n, d)))


def test_attention_one_key_and_equal_keys():
    d = 16
    q = RNG.standard_normal(d)
    K, V = _rand_kv(1, d)
    o, lse = oracle.attention_partial(q, K, V, 0, 1, 0)
    assert np.array_equal(o, f64(V)[0])
    assert np.isclose(lse, q @ f64(K)[0] / math.sqrt(d), rtol=1e-14)
    n = 7
    K = np.repeat(K, n, axis=0)
    V = bf16(RNG.standard_normal((n, d)))
    o, lse = oracle.attention_partial(q, K, V, 0, n, n - 1)
    assert np.allclose(o, f64(V).mean(axis=0), rtol=1e-13)
    assert np.isclose(lse, q @ f64(K)[0] / math.sqrt(d) + math.log(n), rtol=1e-13)


def test_attention_matches_torch_softmax_and_masks():
    d, n = 8, 37
    q = RNG.standard_normal(d)
    K, V = _rand_kv(n, d)
    for last in (n - 1, 20, 0):
        o, lse = oracle.attention_partial(q, K, V, 0, n, last)
        Kt = torch.from_numpy(f64(K)[:last + 1])
        Vt = torch.from_numpy(f64(V)[:last + 1])
        s = torch.from_numpy(q) @ Kt.T / math.sqrt(d)
        want = torch.softmax(s, dim=0) @ Vt
        assert np.allclose(o, want.numpy(), rtol=1e-12, atol=1e-14)
        assert np.isclose(lse, torch.logsumexp(s, 0).item(), rtol=1e-13)
    o, lse = oracle.attention_partial(q, K, V, 25, 37, 20)     # fully masked
    assert lse == -math.inf and not o.any()


def test_lse_combine_equals_unsplit():
    d, n = 16, 300
    q = RNG.standard_normal(d) * 3
    K, V = _rand_kv(n, d)
    last = 271
    o_ref, lse_ref = oracle.attention_partial(q, K, V, 0, n, last)
    for bounds in ([0, n], [0, 64, 128, 192, 256, n], [0, 1, 2, 290, n],
                   [0, 100, 272, 300]):            # last split fully masked
        parts = [oracle.attention_partial(q, K, V, a, b, last)
                 for a, b in zip(bounds[:-1], bounds[1:])]
        o, lse = oracle.lse_combine(np.stack([p[0] for p in parts]),
                                    np.array([p[1] for p in parts]))
        assert np.allclose(o, o_ref, rtol=0, atol=1e-12)
        assert abs(lse - lse_ref) < 1e-12
    o, lse = oracle.lse_combine(np.zeros((2, d)), np.array([-np.inf, -np.inf]))
    assert lse == -math.inf and not o.any()
