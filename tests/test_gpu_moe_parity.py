"""GPU parity of the MoE layer (routing, permutation, grouped GEMMs, combine partition).

Routing permutation and per-expert counts are compared bit-exactly with the
oracle; the fp32 output within 1e-2 * max|ref| + 1e-3.
"""
import numpy as np
import pytest

import oracle
from seeded_inputs import make_inputs, workload_inputs
from tests.gpu_helpers import assert_close, to_dev_bf16, workspace

pytestmark = pytest.mark.gpu
tl = pytest.importorskip("communication_overlapped_gemm_gb300")


@pytest.fixture(scope="module")
def ctx():
    c = tl.Context(0)
    yield c
    c.close()


def run_moe(ctx, inp, topk):
    import torch
    x = to_dev_bf16(inp["x"])
    logits = torch.from_numpy(np.ascontiguousarray(inp["logits"])).cuda()
    wg, wu, wd = (to_dev_bf16(inp[k]) for k in ("w_gate", "w_up", "w_down"))
    T, H = x.shape
    E, _, F = wg.shape
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    perm = torch.empty(T * topk, dtype=torch.int32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    ws = workspace(tl.tl_moe_workspace_bytes(T, H, E, F, topk))
    tl.tl_moe_combine(ctx, x, logits, topk, wg, wu, wd, out, ws, perm_out=perm, counts_out=counts)
    torch.cuda.synchronize()
    assert ctx.check() == tl.TL_OK
    return out.cpu().numpy().astype(np.float64), perm.cpu().numpy(), counts.cpu().numpy()


@pytest.mark.parametrize("T,H,E,F,k", [(64, 256, 4, 128, 2), (300, 512, 16, 256, 2), (200, 256, 8, 384, 3),
                                       (130, 256, 1, 128, 1), (257, 768, 64, 128, 2)])
def test_moe_matches_oracle(ctx, T, H, E, F, k):
    inp = make_inputs("moe", 70 + E, T=T, H=H, E=E, F=F)
    out, perm, counts = run_moe(ctx, inp, k)
    ref = oracle.moe(inp["x"], inp["logits"], inp["w_gate"], inp["w_up"], inp["w_down"], k)
    assert np.array_equal(perm, ref["perm"]), "routing permutation differs"
    assert np.array_equal(counts, ref["counts"])
    assert_close(out, ref["out"], f"moe T={T} E={E} k={k}")


def test_moe_top2_combine_is_deterministic(ctx):
    inp = make_inputs("moe", 81, T=512, H=512, E=8, F=256)
    a, _, _ = run_moe(ctx, inp, 2)
    b, _, _ = run_moe(ctx, inp, 2)
    assert np.array_equal(a, b)


def test_moe_full_size_routing_exact_and_sampled_rows(ctx):
    """Full MoE layer (T=4096, H=2048, E=64, F=1408, top-2): routing bit-exact, sampled tokens."""
    inp = workload_inputs("moe_64e")
    out, perm, counts = run_moe(ctx, inp, 2)
    ex, _ = oracle.moe_route(inp["logits"], 2)
    c_ref, _, perm_ref, _ = oracle.moe_permute(ex, 64)
    assert np.array_equal(perm, perm_ref)
    assert np.array_equal(counts, c_ref)
    rng = np.random.default_rng(5)
    toks = sorted(set(rng.integers(0, 4096, 40).tolist()) | {0, 4095})
    rows, _, _ = oracle.moe_rows(inp["x"], inp["logits"], inp["w_gate"], inp["w_up"], inp["w_down"], 2, toks)
    assert_close(out[toks], rows, "moe_64e sampled tokens")


@pytest.mark.parametrize("T,H,E,F,k", [(300, 512, 16, 256, 2), (200, 256, 8, 384, 3)])
def test_moe_renormalised_gates_match_oracle(T, H, E, F, k):
    """cfg.moe_renorm = 1: the top-k gates of a token divided by their sum (the other reading
    of the pages' unspecified router), against oracle.moe(..., renorm=True)."""
    inp = make_inputs("moe", 90 + E, T=T, H=H, E=E, F=F)
    with tl.Context(0, moe_renorm=1) as c2:
        out, perm, counts = run_moe(c2, inp, k)
    ref = oracle.moe(inp["x"], inp["logits"], inp["w_gate"], inp["w_up"], inp["w_down"], k, renorm=True)
    assert np.array_equal(perm, ref["perm"]) and np.array_equal(counts, ref["counts"])
    assert_close(out, ref["out"], f"moe renorm T={T} E={E} k={k}")
    plain = oracle.moe(inp["x"], inp["logits"], inp["w_gate"], inp["w_up"], inp["w_down"], k)["out"]
    assert np.max(np.abs(out - plain)) > 0.1 * np.max(np.abs(plain))  # the flag reached the kernel


def test_moe_full_size_on_eight_combine_sms(ctx):
    """The MoE workload as stated (combine kernel on 8 reserved SMs): routing bit-exact,
    sampled tokens against the oracle, and the output bit-identical to a 16-SM partition's
    (top-2 into a zeroed fp32 out: neither the order of the two adds nor which CTA claims a
    y tile matters)."""
    inp = workload_inputs("moe_64e")
    with tl.Context(0, combine_ctas=8) as c8:
        out8, perm, counts = run_moe(c8, inp, 2)
    with tl.Context(0, combine_ctas=16) as c16:
        out16, _, _ = run_moe(c16, inp, 2)
    assert np.array_equal(out8, out16)
    ex, _ = oracle.moe_route(inp["logits"], 2)
    c_ref, _, perm_ref, _ = oracle.moe_permute(ex, 64)
    assert np.array_equal(perm, perm_ref) and np.array_equal(counts, c_ref)
    rng = np.random.default_rng(15)
    toks = sorted(set(rng.integers(0, 4096, 40).tolist()) | {0, 4095})
    rows, _, _ = oracle.moe_rows(inp["x"], inp["logits"], inp["w_gate"], inp["w_up"], inp["w_down"], 2, toks)
    assert_close(out8[toks], rows, "moe_64e on 8 combine SMs, sampled tokens")
    out16, _, _ = run_moe(ctx, inp, 2)
    assert np.array_equal(out8, out16)


@pytest.mark.parametrize("cfg", [dict(combine_ctas=1), dict(grid_ctas=16, combine_ctas=2), dict(grid_ctas=3, combine_ctas=1)])
def test_moe_small_grids_and_partitions(ctx, cfg):
    """The combine's run-time claims with few CTAs: a one-SM partition, and grids of 16 and 3
    CTAs where most y tiles are combined by GEMM CTAs after their last tile.  The result
    matches the oracle and is bit-identical to the default configuration's."""
    inp = make_inputs("moe", 95, T=300, H=512, E=16, F=256)
    ref_out, _, _ = run_moe(ctx, inp, 2)
    with tl.Context(0, **cfg) as c2:
        out, perm, counts = run_moe(c2, inp, 2)
    ref = oracle.moe(inp["x"], inp["logits"], inp["w_gate"], inp["w_up"], inp["w_down"], 2)
    assert np.array_equal(perm, ref["perm"]) and np.array_equal(counts, ref["counts"])
    assert_close(out, ref["out"], f"moe {cfg}")
    assert np.array_equal(out, ref_out)
