"""GPU parity of the full decode steps at full size: the Qwen3-0.6B-shaped
step (28 layers, batch 1, context 4096, 16-token pages) and the
Qwen3-8B-shaped step (36 layers, batch 1, context 8192, 64-token pages),
both bf16, each ending in the final RMSNorm, the lm_head and the greedy
argmax, in the serial, graph + multistream + PDL and megakernel schedules.

Greedy ids must equal the oracle's wherever its top-2 logit gap exceeds
1e-2, and equal the argmax of the GPU's own logits everywhere.  The lm_head
is checked element-wise (1e-2 (1 + |oracle|)) given the GPU's own final
hidden state.  The rest is checked at the depth where an element-wise bound
holds:
the new K/V rows of layer 0 (whose inputs are the step's own) to the bf16
tolerance |gpu - oracle| <= 1e-2 (1 + |oracle|); every layer's new K/V rows
and the fp32 logits to a relative RMS error of 5e-2, because each layer's
input already carries the bf16 rounding differences of the layers before
it and these compound over depth.  Untouched cache bytes must be unchanged.
"""
import numpy as np
import pytest
import torch

import pdl_persistent_megakernel_gb300 as dl
from pdl_persistent_megakernel_gb300 import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import (DEV, Case, _DevView, bf16_close, check_lm_head_stagewise, f64,
                             rel_rms_close, rope_close)

MODES = [dl.MODE_SERIAL, dl.MODE_PDL_GRAPH, dl.MODE_MEGAKERNEL]
STEPS = ["q06_step_b1_ctx4096", "q8_step_b1_ctx8192"]


@pytest.fixture(scope="module", params=STEPS)
def step_case(request):
    c = Case(synth.CONFIGS[request.param], trace=False)
    plan = c.plan(modes=sum(1 << m for m in MODES))
    yield c, plan
    plan.close()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", MODES, ids=lambda m: dl.MODE_NAMES[m])
def test_full_step_ids_logits_and_cache(step_case, mode):
    c, plan = step_case
    cfg = c.cfg
    ids, kv = c.run(plan, mode)
    ids = ids.cpu().numpy()
    want_logits = c.ref["logits"].astype(np.float64)
    top2 = np.sort(want_logits, axis=1)[:, -2:]
    sure = (top2[:, 1] - top2[:, 0]) > 1e-2
    assert np.array_equal(ids[sure], c.ref["ids"][sure]), (dl.MODE_NAMES[mode], ids, c.ref["ids"])
    nbytes = cfg.M * cfg.vocab * 4
    got = torch.as_tensor(_DevView(plan.logits_ptr(), nbytes), device=DEV).clone().cpu()
    got = got.numpy().view(np.float32).reshape(cfg.M, cfg.vocab).astype(np.float64)
    what = f"{cfg.name}/{dl.MODE_NAMES[mode]}"
    rel_rms_close(got, want_logits, f"{what} logits")
    # given the GPU's own final hidden state the lm_head meets the element
    # bound, and the ids are the argmax of the GPU's logits
    got2 = check_lm_head_stagewise(c, plan, what)
    assert np.array_equal(got2, got)
    assert np.array_equal(ids, got.argmax(axis=1)), (ids, got.argmax(axis=1))
    before = synth.as_u16(c.inp["kv_pages"])
    after = kv.view(torch.int16).cpu().numpy().view(np.uint16).reshape(before.shape)
    want = c.ref["kv_pages"].reshape(before.shape)
    bt, pos = c.inp["block_table"].numpy(), c.inp["positions"].numpy()
    mask = np.zeros(before.shape, bool)
    for m in range(cfg.M):
        pg = bt[m // cfg.tokens_per_request, pos[m] // cfg.page_size]
        mask[:, pg, :, :, pos[m] % cfg.page_size, :] = True
    assert np.array_equal(after[~mask], before[~mask]), f"{what}: untouched cache bytes changed"
    d = cfg.head_dim
    rope_close(after[0, :, 0][mask[0, :, 0]].reshape(-1, d),
               want[0, :, 0][mask[0, :, 0]].reshape(-1, d), f"{what} layer-0 new k")
    bf16_close(after[0, :, 1][mask[0, :, 1]], want[0, :, 1][mask[0, :, 1]],
               f"{what} layer-0 new v")
    rel_rms_close(f64(after[mask]), f64(want[mask]), f"{what} new kv")
