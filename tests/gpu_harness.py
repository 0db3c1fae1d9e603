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

    def check_kv(self, kv, what=""):
        """Untouched cache bytes identical; the step's new K/V rows close."""
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
        if cfg.fp8:
            rel_rms_close(f64(after[mask]), f64(want[mask]), f"{what} new kv")
        else:
            bf16_close(after[mask], want[mask], f"{what} new kv")
