"""GPU: bit-exact paged-KV indexing through the C ABI, and failure detection
of the megakernel's bounded waits (no GPU fault: a wait threshold nothing
can reach expires and the plan reports DL_ERR_TIMEOUT)."""
import numpy as np
import pytest
import torch

import oracle
import pdl_persistent_megakernel_gb300 as dl
from pdl_persistent_megakernel_gb300 import synth

pytestmark = pytest.mark.gpu


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("P,ctx", [(16, 100), (64, 300), (128, 130)])
def test_kv_write_and_gather_bit_exact(P, ctx):
    L, Hkv, d, R, T = 2, 3, 128, 3, 4
    ppr = -(-ctx // P)
    NP = R * ppr + 5
    g = torch.Generator().manual_seed(P + ctx)
    perm = torch.randperm(NP, generator=g)[:R * ppr].to(torch.int32).view(R, ppr)
    # tag-valued cache: every element distinct (int16 bit patterns)
    n = L * NP * 2 * Hkv * P * d
    cache = (torch.arange(n, dtype=torch.int64) % 65521).to(torch.int16).view(L, NP, 2, Hkv, P, d)
    pos = torch.tensor([ctx - T + t for r in range(R) for t in range(T)], dtype=torch.int32)
    src = torch.randint(-30000, 30000, (R * T, 2, Hkv, d), generator=g, dtype=torch.int16)
    dev = torch.device("cuda")
    kv = cache.to(dev)
    layer = 1
    # keep every device tensor referenced while the asynchronous calls use it
    src_d, bt_d, pos_d = src.to(dev), perm.to(dev), pos.to(dev)
    rc = dl.lib().dl_test_kv_write(src_d.data_ptr(), kv.data_ptr(), bt_d.data_ptr(),
                                   pos_d.data_ptr(), layer, R * T, T, Hkv, d, P, NP, ppr,
                                   _stream())
    assert rc == 0
    dst = torch.empty((R, 2, Hkv, ctx, d), dtype=torch.int16, device=dev)
    rc = dl.lib().dl_test_kv_gather(kv.data_ptr(), bt_d.data_ptr(), dst.data_ptr(), layer,
                                    R, ctx, Hkv, d, P, NP, ppr, _stream())
    assert rc == 0
    torch.cuda.synchronize()
    got_cache = kv.cpu().numpy().view(np.uint16)
    # expected cache: the oracle writes the same rows (kv slot math pinned on the CPU)
    want = cache.numpy().view(np.uint16).copy()
    bt = perm.numpy()
    for m in range(R * T):
        p = int(pos[m])
        for kvs in range(2):
            for h in range(Hkv):
                want[layer, bt[m // T, p // P], kvs, h, p % P] = src[m, kvs, h].numpy().view(np.uint16)
    assert np.array_equal(got_cache, want)
    gathered = dst.cpu().numpy().view(np.uint16)
    for r in range(R):
        for kvs in range(2):
            for h in range(Hkv):
                ref = oracle.kv_gather(want, bt, Hkv, P, d, layer, r, h, kvs, ctx)
                assert np.array_equal(gathered[r, kvs, h], ref)


def test_megakernel_wait_timeout_is_reported():
    cfg = synth.DecodeConfig("timeout", hidden=256, inter=384, n_q_heads=4, n_kv_heads=2,
                             head_dim=128, n_layers=1, vocab=0, fp8=False, num_requests=1,
                             tokens_per_request=1, context=100, page_size=16, seed=21)
    w = synth.make_weights(cfg)
    inp = synth.make_inputs(cfg)
    dev = torch.device("cuda")
    wd = {"layers": [{k: (v.to(dev) if v is not None else None) for k, v in lw.items()}
                     for lw in w["layers"]]}
    plan = dl.Plan(cfg, wd, modes_mask=1 << dl.MODE_MEGAKERNEL)
    # the host validator rejects an unsatisfiable threshold
    assert plan.perturb_wait(1000, 20_000_000, validate=True) == 6  # DL_ERR_PLAN_INVALID
    # forced past the validator, the device wait gives up after ~20 ms
    assert plan.perturb_wait(1000, 20_000_000, validate=False) == 0
    out = torch.zeros((2, cfg.M, cfg.hidden), dtype=torch.bfloat16, device=dev)
    args = (inp["x"].to(dev), inp["residual"].to(dev), inp["kv_pages"].to(dev),
            inp["block_table"].to(dev), inp["positions"].to(dev), out)
    plan.step(*args, mode=dl.MODE_MEGAKERNEL)
    torch.cuda.synchronize()
    with pytest.raises(dl.DLError) as e:
        plan.status()
    assert e.value.status == 5   # DL_ERR_TIMEOUT
    # the context stays usable: restore the plan and run a correct step
    assert plan.perturb_wait(0, 0, validate=True) == 0
    ref = oracle.decode_step(cfg, w, inp)
    plan.step(*args, mode=dl.MODE_MEGAKERNEL)
    torch.cuda.synchronize()
    plan.status()
    got = out.float().cpu().numpy()
    want = oracle.bf16_to_double(ref["out"])
    assert (np.abs(got - want) <= 1e-2 * (1 + np.abs(want))).all()
    plan.close()


def test_invalid_arguments_rejected_synchronously():
    cfg = synth.DecodeConfig("args", hidden=256, inter=384, n_q_heads=4, n_kv_heads=2,
                             head_dim=128, n_layers=1, vocab=0, fp8=False, num_requests=1,
                             tokens_per_request=1, context=100, page_size=16, seed=22)
    w = synth.make_weights(cfg)
    dev = torch.device("cuda")
    wd = {"layers": [{k: (v.to(dev) if v is not None else None) for k, v in lw.items()}
                     for lw in w["layers"]]}
    plan = dl.Plan(cfg, wd, modes_mask=1)
    x = torch.zeros((1, 256), dtype=torch.bfloat16, device=dev)
    rc = dl.lib().dl_decode_step(plan._h, None, x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                 x.data_ptr(), x.data_ptr(), 0, None)
    assert rc == 1
    rc = dl.lib().dl_decode_step(plan._h, x.data_ptr() + 2, x.data_ptr(), x.data_ptr(),
                                 x.data_ptr(), x.data_ptr(), x.data_ptr(), 0, None)
    assert rc == 1
    rc = dl.lib().dl_decode_step(plan._h, x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                 x.data_ptr(), x.data_ptr(), x.data_ptr(), 2, None)
    assert rc == 1   # megakernel not prepared for this plan
    plan.close()
    bad = cfg.replace(head_dim=64)
    with pytest.raises(dl.DLError):
        dl.Plan(bad, wd)
