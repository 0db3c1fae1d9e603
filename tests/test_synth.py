"""CPU checks of the seeded synthetic inputs (pdl_persistent_megakernel_gb300.synth), the
one recipe both the CUDA path and the oracle take their inputs from: reproducible,
independent per tensor, and shaped as the design states (block tables, positions, the
norm and projection weight distributions, the FP8 block format)."""
import torch

from pdl_persistent_megakernel_gb300 import synth

CFG = synth.DecodeConfig("synth_check", hidden=512, inter=768, n_q_heads=8, n_kv_heads=2,
                         head_dim=128, n_layers=2, vocab=256, fp8=False, num_requests=3,
                         tokens_per_request=4, context=300, page_size=64, seed=41)


def test_inputs_are_reproducible_and_seed_dependent():
    a, b = synth.make_inputs(CFG), synth.make_inputs(CFG)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    c = synth.make_inputs(CFG.replace(seed=42))
    assert not torch.equal(a["x"], c["x"])
    # every tensor draws from its own stream
    assert not torch.equal(a["x"], a["residual"])


def test_block_table_is_a_permutation_with_spare_pages():
    bt = synth.make_inputs(CFG)["block_table"]
    assert bt.shape == (CFG.num_requests, CFG.pages_per_request) and bt.dtype == torch.int32
    v = bt.flatten().tolist()
    assert len(set(v)) == len(v) and min(v) >= 0 and max(v) < CFG.num_pages
    assert CFG.num_pages - len(v) == CFG.spare_pages
    assert CFG.pages_per_request * CFG.page_size >= CFG.context


def test_positions_are_the_last_tokens_of_each_request():
    pos = synth.make_inputs(CFG)["positions"]
    assert pos.dtype == torch.int32
    pos = pos.view(CFG.num_requests, CFG.tokens_per_request)
    want = list(range(CFG.context - CFG.tokens_per_request, CFG.context))
    for r in range(CFG.num_requests):
        assert pos[r].tolist() == want


def test_weight_distributions_and_shapes():
    w = synth.make_weights(CFG)
    lw = w["layers"][0]
    # norm weights 1 + N(0, 0.02) (a literal N(0, 0.02) would collapse every norm)
    for k in ("ln1_w", "ln2_w", "q_norm_w", "k_norm_w"):
        v = lw[k].float()
        assert abs(v.mean().item() - 1.0) < 0.01 and 0.012 < v.std().item() < 0.028, k
    # projections N(0, 0.02), [out, in]
    shapes = {"w_qkv": (CFG.qkv_rows, CFG.hidden), "w_o": (CFG.hidden, CFG.n_q_heads * 128),
              "w_gate_up": (2 * CFG.inter, CFG.hidden), "w_down": (CFG.hidden, CFG.inter)}
    for k, shp in shapes.items():
        v = lw[k].float()
        assert tuple(v.shape) == shp, k
        assert abs(v.mean().item()) < 2e-3 and abs(v.std().item() - 0.02) < 1e-3, k
        assert lw[k + "_scale"] is None
    assert tuple(w["lm_head_w"].shape) == (CFG.vocab, CFG.hidden)
    assert abs(w["final_norm_w"].float().mean().item() - 1.0) < 0.01
    # layers draw their own weights
    assert not torch.equal(w["layers"][0]["w_o"], w["layers"][1]["w_o"])


def test_fp8_block_format_round_trip():
    wt = synth.randn_bf16(CFG, "probe", (256, 384), 0.02)
    codes, scales = synth.quantize_blocks_e4m3(wt)
    assert codes.dtype == torch.uint8 and tuple(scales.shape) == (2, 3)
    w = wt.float()
    # each 128 x 128 block's largest magnitude maps to 448, the e4m3 maximum
    amax = w.view(2, 128, 3, 128).abs().amax(dim=(1, 3))
    assert torch.allclose(scales, amax / 448)
    deq = (codes.view(torch.float8_e4m3fn).float().view(2, 128, 3, 128)
           * scales[:, None, :, None]).view(256, 384)
    # e4m3 keeps 3 mantissa bits: a rounding error of at most 2^-4 of the
    # value for everything in the normal range (2^-6 of the scale and up)
    normal = w.abs() > scales.max() * 2.0 ** -6
    assert normal.float().mean() > 0.9
    assert ((deq - w).abs()[normal] <= w.abs()[normal] * 2.0 ** -4).all()
    # the FP8 configuration stores exactly these codes and scales
    lw = synth.make_layer_weights(CFG.replace(fp8=True), 0)
    c2, s2 = synth.quantize_blocks_e4m3(synth.randn_bf16(CFG, "layer0/w_o", (CFG.hidden, 1024),
                                                         0.02, 0.0))
    assert torch.equal(lw["w_o"], c2) and torch.equal(lw["w_o_scale"], s2)
