"""GPU checks of the trace build (DL_TRACE=1 at plan creation): every CTA
share of every op leaves ordered %globaltimer stamps, the shares' work units
add up to the op's units, and ops of the serial schedule follow each other."""
import os

import numpy as np
import pytest
import torch

import pdl_persistent_megakernel_gb300 as dl
from pdl_persistent_megakernel_gb300 import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import DEV, to_dev

CFG = synth.DecodeConfig("trace_m16", hidden=512, inter=768, n_q_heads=8, n_kv_heads=2,
                         head_dim=128, n_layers=2, vocab=0, fp8=True, num_requests=2,
                         tokens_per_request=8, context=300, page_size=64, seed=31)


def _units(cfg, name, grid):
    """Work units of one op (the engines' split), from the op's shape."""
    H, I, d = cfg.hidden, cfg.inter, cfg.head_dim
    kel = 128 if cfg.fp8 else 64
    if name.startswith("add_rmsnorm") or name == "final_norm":
        return cfg.M
    if name == "qkv_rope_kvwrite":
        return (cfg.qkv_rows // 128) * (H // kel)
    if name == "o_proj":
        return (H // 128) * (cfg.n_q_heads * d // kel)
    if name == "gate_up_silu":
        return (I // 128) * (H // kel)
    if name == "down_proj":
        return (H // 128) * (I // kel)
    if name == "attention":
        return cfg.num_requests * cfg.n_kv_heads * (-(-cfg.context // 64))
    return None


@pytest.mark.parametrize("mode", [dl.MODE_SERIAL, dl.MODE_GRAPH_LINEAR, dl.MODE_MEGAKERNEL],
                         ids=lambda m: dl.MODE_NAMES[m])
def test_trace_stamps_ordered_and_units_complete(mode, monkeypatch):
    monkeypatch.setenv("DL_TRACE", "1")
    cfg = CFG
    w = to_dev(synth.make_weights(cfg))
    inp = {k: v.to(DEV) for k, v in synth.make_inputs(cfg).items()}
    plan = dl.Plan(cfg, w, modes_mask=(1 << dl.MODE_GRAPH_LINEAR) | (1 << dl.MODE_MEGAKERNEL))
    out = torch.zeros((2, cfg.M, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    plan.step(inp["x"], inp["residual"], inp["kv_pages"], inp["block_table"],
              inp["positions"], out, mode=mode)
    torch.cuda.synchronize()
    plan.status()
    tr = plan.trace()
    ops = plan.ops()
    assert tr.shape[0] >= len(ops) and tr.shape[2] == 8
    prev_end = 0
    for k, (name, grid, _) in enumerate(ops):
        t = tr[k, :grid].astype(np.int64)
        start, deps, end = t[:, 0], t[:, 1], t[:, 4]
        assert (start > 0).all() and (end > 0).all(), name
        assert (deps >= start).all() and (end >= deps).all(), name
        first, last = t[:, 2], t[:, 3]
        busy = t[:, 5] > 0
        if not name.startswith("add_rmsnorm"):
            assert (first[busy] >= deps[busy]).all(), name
            assert (last[busy] >= first[busy]).all() and (end[busy] >= last[busy]).all(), name
        want = _units(cfg, name, grid)
        if want is not None:
            assert int(t[:, 5].sum()) == want, (name, int(t[:, 5].sum()), want)
        # every share of op k starts its dependent reads after op k-1 ended;
        # in the megakernel an attention share waits only for the QKV tiles
        # of its kv heads (per-head events): after the shares that finish them
        if k > 0 and mode == dl.MODE_MEGAKERNEL and name == "attention":
            _check_head_events(cfg, tr, k, ops)
        elif k > 0 and mode != dl.MODE_SERIAL:
            assert deps.min() >= prev_end - 2000, name   # globaltimer granularity slack
        prev_end = int(end.max())
        assert (tr[k, grid:] == 0).all(), name
    # reading cleared the table
    assert not plan.trace().any()
    plan.close()


def _sk_begin(U, G, c):
    return (U * c) // G


def _sk_owner(U, G, x):
    """The share whose Stream-K range holds unit x."""
    c = min(G - 1, (x * G) // U)
    while c > 0 and _sk_begin(U, G, c) > x:
        c -= 1
    while c + 1 < G and _sk_begin(U, G, c + 1) <= x:
        c += 1
    return c


def _check_head_events(cfg, tr, k, ops):
    """Each attention share's dependent reads start after the QKV shares
    that finish (own the first unit of) every tile of its pairs' kv heads:
    the group's q heads, the k head and the v head."""
    Hq, Hkv = cfg.n_q_heads, cfg.n_kv_heads
    G = Hq // Hkv
    kb = cfg.hidden // (128 if cfg.fp8 else 64)
    nt = Hq + 2 * Hkv
    gq, ga = ops[k - 1][1], ops[k][1]
    uq = nt * kb
    qend = tr[k - 1, :gq, 4].astype(np.int64)
    nb = -(-cfg.context // 64)
    ua = cfg.num_requests * Hkv * nb
    adeps = tr[k, :ga, 1].astype(np.int64)
    for c in range(ga):
        u0, u1 = _sk_begin(ua, ga, c), _sk_begin(ua, ga, c + 1)
        if u1 <= u0:
            continue
        heads = {p % Hkv for p in range(u0 // nb, (u1 - 1) // nb + 1)}
        tiles = [t for h in heads for t in list(range(h * G, h * G + G)) + [Hq + h, Hq + Hkv + h]]
        owners = {_sk_owner(uq, gq, t * kb) for t in tiles}
        assert adeps[c] >= max(qend[o] for o in owners) - 2000, ("attention share", c)


def test_trace_off_is_reported():
    os.environ.pop("DL_TRACE", None)
    cfg = CFG
    w = to_dev(synth.make_weights(cfg))
    plan = dl.Plan(cfg, w, modes_mask=0)
    with pytest.raises(dl.DLError) as e:
        plan.trace()
    assert e.value.status == 2
    plan.close()
