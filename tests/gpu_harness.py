"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI and the CPU oracle on the same seeded inputs and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import pdl_persistent_megakernel_gb300 as dl
from pdl_persistent_megakernel_gb300 import synth

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def to_dev(w):
    return {"layers": [{k: (v.to(DEV) if v is not None else None) for k, v in lw.items()}
                       for lw in w["layers"]],
            "final_norm_w": None if w.get("final_norm_w") is None else w["final_norm_w"].to(DEV),
            "lm_head_w": None if w.get("lm_head_w") is None else w["lm_head_w"].to(DEV)}


def f64(b):
    return oracle.bf16_to_double(np.asarray(b))


def bf16_close(got, want, what=""):
    """bf16 paths: |gpu - oracle| <= 1e-2 (1 + |oracle|) element-wise."""
    g, w = f64(got), f64(want)
    err = np.abs(g - w)
    tol = 1e-2 * (1 + np.abs(w))
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} beyond tolerance, max err {err.max():.4g}"


def rope_close(got, want, what=""):
    """Rows after RoPE ([..., d], neox pairs (i, i + d/2)): |gpu - oracle|
    <= 1e-2 (1 + the pair's norm) element-wise.  The rotation mixes each
    element with its partner and keeps the pair's norm, so an element's
    rounding scale is its pair's: a one-ulp rounding difference of a large
    input reaches its small partner through the sine term (the element bound
    of the partner alone would flag that)."""
    g, w = f64(got), f64(want)
    d = w.shape[-1]
    half = d // 2
    partner = np.concatenate([w[..., half:], w[..., :half]], axis=-1)
    pn = np.sqrt(w * w + partner * partner)
    err = np.abs(g - w)
    bad = err > 1e-2 * (1 + pn)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} beyond tolerance, max err {err.max():.4g}"


def rel_rms_close(got, want, what="", tol=5e-2):
    """FP8 path: the relative RMS error rms(gpu - oracle) / rms(oracle) of a
    tensor is at most 5e-2.  (Element-wise maxima are not bounded by it: an
    activation value that sits on an e4m3 rounding boundary may round either
    way on the two sides, a one-code flip of up to 12.5% of that element, and
    flips compound through the four quantised projection inputs.)"""
    g, w = np.asarray(got, np.float64), np.asarray(want, np.float64)
    rms = np.sqrt((w ** 2).mean())
    err = np.sqrt(((g - w) ** 2).mean())
    assert err <= tol * rms, f"{what}: rms err {err:.4g} > {tol} * rms {rms:.4g}"


def dequant(codes, scales):
    c = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()
    return c * np.repeat(np.asarray(scales, np.float64), 128, axis=1)


class _DevView:
    """Zero-copy view of a plan-owned device buffer (CUDA array interface)."""

    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                         "data": (ptr, False), "version": 3}


def read_debug(plan, name):
    """Copy a plan-owned intermediate buffer to a CPU uint8 tensor."""
    ptr, nbytes = plan.debug_buffer(name)
    torch.cuda.synchronize()
    return torch.as_tensor(_DevView(ptr, nbytes), device=DEV).clone().cpu()


def as_bf16_np(u8, shape):
    return u8.numpy().view(np.uint16)[:int(np.prod(shape))].reshape(shape)


def as_f32_np(u8, shape):
    return u8.numpy().view(np.float32)[:int(np.prod(shape))].reshape(shape)


def as_u8_np(u8, shape):
    return u8.numpy()[:int(np.prod(shape))].reshape(shape)


def check_mlp_stagewise(case, plan, out, what=""):
    """bf16 layer: the gate/up + SiLU*mul and down projections, each given
    the GPU's own input (the oracle's operations applied to the GPU's h2 and
    SiLU*mul output), element-wise within the bf16 tolerance.  End to end the
    two chains differ by one-ulp bf16 rounding flips (fp32 versus fp64
    accumulation next to a rounding boundary), and a K = 12288 down
    projection sums a thousand of them; per operation no such flip exists."""
    cfg = case.cfg
    M, H, I = cfg.M, cfg.hidden, cfg.inter
    lw = case.w["layers"][cfg.n_layers - 1]
    h2 = as_bf16_np(read_debug(plan, "h2"), (M, H))
    act = as_bf16_np(read_debug(plan, "act"), (M, I))
    gu = oracle.gemm_bf16(f64(h2), synth.as_u16(lw["w_gate_up"]))
    g = f64(oracle.bf16_from_double(gu[:, :I]))
    u = f64(oracle.bf16_from_double(gu[:, I:]))
    act_want = oracle.bf16_from_double(oracle.silu(g) * u)
    bf16_close(act, act_want, f"{what} silu*mul given the GPU's h2")
    y = out[0].view(torch.int16).cpu().numpy().view(np.uint16)
    y_want = oracle.bf16_from_double(oracle.gemm_bf16(f64(act), synth.as_u16(lw["w_down"])))
    bf16_close(y, y_want, f"{what} down projection given the GPU's act")


def check_lm_head_stagewise(case, plan, what=""):
    """Full steps: the fp32 logits against the oracle's lm_head applied to
    the GPU's own final-norm output, element-wise within 1e-2 (1 + |oracle|).
    The final hidden state ends a chain of every layer's bf16 roundings; given
    it, the lm_head is one operation whose inputs are identical on both
    sides."""
    cfg = case.cfg
    M, H, V = cfg.M, cfg.hidden, cfg.vocab
    hf = as_bf16_np(read_debug(plan, "h_final"), (M, H))
    nbytes = M * V * 4
    got = torch.as_tensor(_DevView(plan.logits_ptr(), nbytes), device=DEV).clone().cpu()
    got = got.numpy().view(np.float32).reshape(M, V).astype(np.float64)
    want = oracle.gemm_bf16(f64(hf), synth.as_u16(case.w["lm_head_w"]))
    err = np.abs(got - want)
    bad = err > 1e-2 * (1 + np.abs(want))
    assert not bad.any(), f"{what} lm_head: {bad.sum()} of {bad.size} beyond tolerance, max err {err.max():.4g}"
    # the greedy ids are the argmax of those logits (lowest index on ties)
    return got


_E4M3_MIDS = None


def _e4m3_midpoints():
    """The rounding boundaries of e4m3 (OCP E4M3FN): midpoints between
    consecutive non-negative codes, from the oracle's decoder."""
    global _E4M3_MIDS
    if _E4M3_MIDS is None:
        v = np.unique(np.abs(oracle.e4m3_decode(np.arange(256, dtype=np.uint8))))
        v = v[np.isfinite(v)]
        _E4M3_MIDS = (v[1:] + v[:-1]) / 2
    return _E4M3_MIDS


def check_fp8_codes_exact(got_codes, got_scales, want_codes, want_scales, want_f32,
                          what="", eps=2.0 ** -18):
    """e4m3 codes of a quantised tensor whose inputs are identical on both
    sides (the first norm of a step), code by code.  The value quantised is
    h / s with h the norm's output and s = amax / 448 of its 128-group: fp32
    on the GPU (an fp32 rsqrt, fp32 products), fp64 rounded to fp32 in the
    oracle (want_f32), a few fp32 ulps apart.  So a code may differ only
    where the oracle's quotient lies within eps (relative) of an e4m3
    rounding boundary, and then only by one step; every other code is equal,
    and the scales agree within eps."""
    gc, wc = np.asarray(got_codes), np.asarray(want_codes)
    gs, ws = np.asarray(got_scales, np.float64), np.asarray(want_scales, np.float64)
    rel = np.abs(gs - ws) / np.abs(ws)
    assert rel.max() <= eps, f"{what}: scale differs by {rel.max():.3g} relative"
    diff = gc != wc
    if not diff.any():
        return
    M, K = gc.shape
    q = (np.asarray(want_f32, np.float32).reshape(M, K // 128, 128) /
         np.asarray(want_scales, np.float32)[:, :, None]).reshape(M, K).astype(np.float64)
    mids = _e4m3_midpoints()
    aq = np.abs(q[diff])
    j = np.clip(np.searchsorted(mids, aq), 1, len(mids) - 1)
    near = np.minimum(np.abs(aq - mids[j]), np.abs(aq - mids[j - 1]))
    ambiguous = near <= eps * aq
    dg = oracle.e4m3_decode(gc[diff])
    dw = oracle.e4m3_decode(wc[diff])
    # neighbours: no representable value strictly between the two
    allv = np.unique(np.abs(oracle.e4m3_decode(np.arange(256, dtype=np.uint8))))
    lo, hi = np.minimum(np.abs(dg), np.abs(dw)), np.maximum(np.abs(dg), np.abs(dw))
    between = np.array([((allv > a) & (allv < b)).any() for a, b in zip(lo, hi)])
    same_sign = np.sign(dg) == np.sign(dw)
    ok = ambiguous & ~between & same_sign
    assert ok.all(), (f"{what}: {int((~ok).sum())} of {gc.size} e4m3 codes differ away from a "
                      f"rounding boundary ({int(diff.sum())} differ in all)")


def fp8_qkv_from_h1(case, codes, scales):
    """FP8 one-layer configs: the oracle's QKV projection, QK-norm and RoPE
    (the oracle's own functions, in the order of its layer) applied to the
    given first-norm e4m3 codes [M, H] and scales [M, H / 128].  Returns q
    after RoPE [M, Hq, d] and the new k (after RoPE) and v rows [M, Hkv, d],
    as bf16 bit patterns."""
    cfg = case.cfg
    M, d = cfg.M, cfg.head_dim
    Hq, Hkv = cfg.n_q_heads, cfg.n_kv_heads
    lw = case.w["layers"][0]
    qkv = oracle.gemm_fp8(np.ascontiguousarray(codes), np.ascontiguousarray(scales),
                          lw["w_qkv"].numpy(), lw["w_qkv_scale"].numpy())
    qkv = f64(oracle.bf16_from_double(qkv)).reshape(M, Hq + 2 * Hkv, d)
    pos = case.inp["positions"].numpy()
    qn, kn = synth.as_u16(lw["q_norm_w"]), synth.as_u16(lw["k_norm_w"])
    q = np.zeros((M, Hq, d), np.uint16)
    k = np.zeros((M, Hkv, d), np.uint16)
    for m in range(M):
        for h in range(Hq + Hkv):
            nrm = f64(oracle.bf16_from_double(
                oracle.head_rmsnorm(qkv[m, h], qn if h < Hq else kn, cfg.eps)))
            rot = oracle.bf16_from_double(oracle.rope(nrm, int(pos[m]), cfg.rope_theta))
            if h < Hq:
                q[m, h] = rot
            else:
                k[m, h - Hq] = rot
    v = oracle.bf16_from_double(qkv[:, Hq + Hkv:])
    return q, k, v


def fp8_qkv_given_gpu_h1(case, plan):
    """fp8_qkv_from_h1 on the GPU's own first-norm codes and scales.  Those
    codes may differ from the oracle's at e4m3 rounding boundaries
    (check_fp8_codes_exact); given the same codes the projection, QK-norm and
    RoPE are operations with identical inputs on both sides."""
    cfg = case.cfg
    M, H = cfg.M, cfg.hidden
    codes = as_u8_np(read_debug(plan, "h1"), (M, H))
    sc = as_f32_np(read_debug(plan, "h1_scales"), (M, H // 128))
    return fp8_qkv_from_h1(case, codes, sc)


class Case:
    """Inputs + oracle result of one configuration (computed once)."""

    def __init__(self, cfg, weights=None, inputs=None, trace=True):
        self.cfg = cfg
        self.w = weights or synth.make_weights(cfg)
        self.inp = inputs or synth.make_inputs(cfg)
        self.ref = oracle.decode_step(cfg, self.w, self.inp, trace=trace)
        self.wd = to_dev(self.w)

    def plan(self, modes=dl.ALL_MODES, **kw):
        return dl.Plan(self.cfg, self.wd, modes_mask=modes, **kw)

    def run(self, plan, mode, steps=1):
        cfg = self.cfg
        kv = self.inp["kv_pages"].to(DEV)
        if cfg.vocab:
            out = torch.full((cfg.M,), -1, dtype=torch.int32, device=DEV)
        else:
            out = torch.zeros((2, cfg.M, cfg.hidden), dtype=torch.bfloat16, device=DEV)
        # the tensors stay referenced (self.last_args) while the step runs
        args = (self.inp["x"].to(DEV), self.inp["residual"].to(DEV), kv,
                self.inp["block_table"].to(DEV), self.inp["positions"].to(DEV), out)
        self.last_args = args
        for _ in range(steps):
            plan.step(*args, mode=mode)
        torch.cuda.synchronize()
        plan.status()
        return out, kv

    def check_layer_out(self, out, what=""):
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        if self.cfg.fp8:
            for i, nm in ((0, "y"), (1, "residual")):
                rel_rms_close(f64(got[i]), f64(self.ref["out"][i]), f"{what} {nm}")
        else:
            bf16_close(got, self.ref["out"], what)

    def check_kv(self, kv, what="", plan=None):
        """Untouched cache bytes identical; the step's new K/V rows of layer
        0 (its inputs are the step's own, so every operation before the cache
        write sees identical inputs on both sides) within the bf16 element
        bound, FP8 included (K rows, after RoPE, relative to their pair's
        norm); later layers' rows (whose inputs carry the
        earlier layers' rounding differences) to the relative RMS bound of
        their path."""
        cfg = self.cfg
        before = synth.as_u16(self.inp["kv_pages"])
        after = kv.view(torch.int16).cpu().numpy().view(np.uint16).reshape(before.shape)
        want = self.ref["kv_pages"].reshape(before.shape)
        bt = self.inp["block_table"].numpy()
        pos = self.inp["positions"].numpy()
        mask = np.zeros(before.shape, bool)
        for m in range(cfg.M):
            pg = bt[m // cfg.tokens_per_request, pos[m] // cfg.page_size]
            mask[:, pg, :, :, pos[m] % cfg.page_size, :] = True
        assert np.array_equal(after[~mask], before[~mask]), f"{what}: untouched cache bytes changed"
        d = cfg.head_dim
        # layer 0: K rows after QK-norm + RoPE (pair bound), V rows plain
        if cfg.fp8 and plan is not None and cfg.n_layers == 1:
            # FP8: given the GPU's own first-norm codes (see fp8_qkv_given_gpu_h1)
            _, kw, vw = fp8_qkv_given_gpu_h1(self, plan)
            for m in range(cfg.M):
                pg = bt[m // cfg.tokens_per_request, pos[m] // cfg.page_size]
                sl = pos[m] % cfg.page_size
                rope_close(after[0, pg, 0, :, sl], kw[m], f"{what} layer-0 new k, token {m}")
                bf16_close(after[0, pg, 1, :, sl], vw[m], f"{what} layer-0 new v, token {m}")
        elif cfg.fp8:
            rel_rms_close(f64(after[0][mask[0]]), f64(want[0][mask[0]]), f"{what} layer-0 new kv")
        else:
            rope_close(after[0, :, 0][mask[0, :, 0]].reshape(-1, d),
                       want[0, :, 0][mask[0, :, 0]].reshape(-1, d), f"{what} layer-0 new k")
            bf16_close(after[0, :, 1][mask[0, :, 1]], want[0, :, 1][mask[0, :, 1]],
                       f"{what} layer-0 new v")
        if cfg.n_layers > 1:
            later = mask.copy()
            later[0] = False
            if cfg.fp8:
                rel_rms_close(f64(after[later]), f64(want[later]), f"{what} new kv")
            else:
                bf16_close(after[later], want[later], f"{what} new kv")
