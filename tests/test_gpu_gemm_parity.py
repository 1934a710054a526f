"""GPU parity of AllGather+GEMM, GEMM+ReduceScatter and the MLP chain against the fp64 oracle.

Every call goes through the C ABI (via the ctypes binding).  Tolerance for the
bf16-in / fp32-accumulate outputs: max|gpu - ref| <= 1e-2 * max|ref| + 1e-3.
The gather index map is checked bit-exactly; results that the design fixes
bit-for-bit (tile order, swizzle, mover geometry, grid size) are compared with
array_equal.
"""
import numpy as np
import pytest

import oracle
from seeded_inputs import make_inputs, workload_inputs
from tests.gpu_helpers import assert_close, bf16_bits, bf16_to_f64, to_dev_bf16, workspace

pytestmark = pytest.mark.gpu

tl = pytest.importorskip("communication_overlapped_gemm_gb300")


@pytest.fixture(scope="module")
def ctx():
    import torch
    assert torch.cuda.is_available()
    c = tl.Context(0)
    yield c
    c.close()


def run_ag(ctx, inp, rank=0):
    import torch
    a = [to_dev_bf16(x) for x in inp["a_shards"]]
    b = to_dev_bf16(inp["b"])
    W = len(a)
    mpr, k = a[0].shape
    n = b.shape[1]
    c = torch.empty((W * mpr, n), dtype=torch.bfloat16, device="cuda")
    ws = workspace(tl.tl_ag_gemm_workspace_bytes(W, mpr, n, k))
    tl.tl_ag_gemm(ctx, a, b, c, ws, rank=rank)
    torch.cuda.synchronize()
    assert ctx.check() == tl.TL_OK
    return c, ws


def check_gathered(ws, inp, rank):
    """The gathered operand T holds every remote shard at its rank-order slot, bit for bit; the
    self rank's slot is never written by the fused call (the GEMM reads that shard in place),
    so it keeps the workspace's zero fill."""
    import torch
    gath = oracle.ag_gather_bits(inp["a_shards"])
    got = bf16_bits(ws[: gath.size * 2].view(torch.bfloat16).view(gath.shape))
    mpr = inp["a_shards"][0].shape[0]
    for r in range(len(inp["a_shards"])):
        rows = slice(r * mpr, (r + 1) * mpr)
        if r == rank:
            assert not got[rows].any()
        else:
            assert np.array_equal(got[rows], gath[rows])


# ----------------------------------------------------------------------------- AllGather + GEMM
def test_ag_gemm_tiny_matches_oracle(ctx):
    inp = workload_inputs("ag_tiny")
    c, ws = run_ag(ctx, inp)
    ref = oracle.ag_gemm(inp["a_shards"], inp["b"])
    assert_close(bf16_to_f64(c), ref, "ag_tiny")
    # the gathered operand is the rank-order concatenation, bit for bit
    check_gathered(ws, inp, 0)


@pytest.mark.parametrize("W,mpr,n,k", [(1, 128, 256, 64), (3, 256, 200, 136), (4, 128, 520, 328)])
def test_ag_gemm_ragged_matches_oracle(ctx, W, mpr, n, k):
    inp = make_inputs("ag_gemm", 11 + W, W=W, m_per_rank=mpr, n=n, k=k)
    for rank in range(W):
        c, ws = run_ag(ctx, inp, rank=rank)
        assert_close(bf16_to_f64(c), oracle.ag_gemm(inp["a_shards"], inp["b"]), f"ag W={W} rank={rank}")
        check_gathered(ws, inp, rank)  # W = 1: nothing to gather, the region stays zero


def test_ag_gemm_invariant_to_order_and_geometry():
    """Tile order, swizzle, mover chunking, mover warps and grid size do not change a bit."""
    import torch
    inp = make_inputs("ag_gemm", 21, W=4, m_per_rank=256, n=768, k=512)
    outs = []
    for cfg in [dict(swizzle=1), dict(swizzle=0), dict(chunks_per_slab=1, mover_warps=1),
                dict(chunks_per_slab=8, mover_warps=4), dict(grid_ctas=37), dict(pair_ctas=1, grid_ctas=38)]:
        with tl.Context(0, **cfg) as c2:
            for rank in (0, 3):
                c, _ = run_ag(c2, inp, rank=rank)
                outs.append(bf16_bits(c))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    assert_close(bf16_to_f64(torch.from_numpy(outs[0].view(np.int16)).view(torch.bfloat16)),
                 oracle.ag_gemm(inp["a_shards"], inp["b"]), "ag invariance")


def test_mover_k_parts_are_bit_identical():
    """cfg.mover_kparts: tl_ag_gemm's mover cuts each head slab into 2 or 4 K parts and a tile
    waits for each part before its k-blocks in it.  With K long enough for every split (4096:
    64 k-blocks), the AllGather+GEMM gives the same bits with 1, 2 and 4 parts, and the
    gathered operand is exact."""
    import torch
    inp = make_inputs("ag_gemm", 23, W=3, m_per_rank=256, n=264, k=4096)
    outs = []
    for kp, extra in [(1, {}), (2, {}), (4, {}), (4, dict(chunks_per_slab=4)), (4, dict(pair_ctas=1))]:
        with tl.Context(0, mover_kparts=kp, **extra) as c2:
            c, ws = run_ag(c2, inp, rank=1)
            outs.append(bf16_bits(c))
            check_gathered(ws, inp, 1)
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    assert_close(bf16_to_f64(torch.from_numpy(outs[0].view(np.int16)).view(torch.bfloat16)),
                 oracle.ag_gemm(inp["a_shards"], inp["b"]), "ag with K parts")


def test_ag_gemm_llama70b_sampled(ctx):
    """Full-size AllGather+GEMM (W=8, 8192x3584x8192) checked on sampled entries."""
    inp = workload_inputs("ag_70b")
    c, ws = run_ag(ctx, inp, rank=0)
    rng = np.random.default_rng(7)
    rows = np.concatenate([rng.integers(0, 8192, 200), [0, 8191, 1023, 1024, 7 * 1024]])
    cols = np.concatenate([rng.integers(0, 3584, 200), [0, 3583, 255, 256, 3583]])
    got = bf16_to_f64(c)[rows, cols]
    ref = oracle.ag_gemm_entries(inp["a_shards"], inp["b"], rows, cols)
    assert_close(got, ref, "ag_70b sampled")
    # and whole rows of every shard region (several tiles, every rank)
    for r in range(8):
        row = r * 1024 + 517
        ref_row = oracle.ag_gemm_entries(inp["a_shards"], inp["b"], [row] * 3584, np.arange(3584))
        assert_close(bf16_to_f64(c)[row], ref_row, f"ag_70b row {row}")
    check_gathered(ws, inp, 0)


# ----------------------------------------------------------------------------- GEMM + ReduceScatter
def run_rs(ctx, inp):
    import torch
    a = [to_dev_bf16(x) for x in inp["a"]]
    b = [to_dev_bf16(x) for x in inp["b"]]
    W = len(a)
    m, kr = a[0].shape
    n = b[0].shape[1]
    out = [torch.empty((m // W, n), dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    size = tl.tl_gemm_rs_ring_workspace_bytes if ctx.config.rs_ring else tl.tl_gemm_rs_workspace_bytes
    ws = workspace(size(W, m, n, kr))
    tl.tl_gemm_rs(ctx, a, b, out, ws)
    torch.cuda.synchronize()
    assert ctx.check() == tl.TL_OK
    return out


@pytest.mark.parametrize("W,m,n,kr", [(1, 128, 256, 64), (2, 256, 256, 128), (4, 512, 328, 200),
                                      (8, 1024, 264, 72), (2, 512, 264, 136), (3, 768, 520, 3584)])
def test_gemm_rs_matches_oracle(ctx, W, m, n, kr):
    inp = make_inputs("gemm_rs", 31 + W, W=W, m=m, n=n, k_r=kr)
    out = run_rs(ctx, inp)
    ref = oracle.gemm_rs(inp["a"], inp["b"])
    for o in range(W):
        assert_close(bf16_to_f64(out[o]), ref[o], f"rs W={W} owner {o}")


def test_gemm_rs_deterministic_across_orders():
    inp = make_inputs("gemm_rs", 41, W=4, m=1024, n=512, k_r=256)
    outs = []
    for cfg in [dict(swizzle=1), dict(swizzle=0), dict(grid_ctas=23), dict(pair_ctas=0), dict(pair_ctas=1, grid_ctas=46)]:
        with tl.Context(0, **cfg) as c2:
            for _ in range(2):
                outs.append([bf16_bits(o) for o in run_rs(c2, inp)])
    for o in outs[1:]:
        assert all(np.array_equal(x, y) for x, y in zip(o, outs[0]))


@pytest.mark.parametrize("W,m,n,kr", [(1, 128, 256, 64), (2, 256, 256, 128), (4, 512, 328, 200),
                                      (8, 1024, 264, 72), (3, 768, 520, 3584)])
def test_gemm_rs_ring_matches_oracle(W, m, n, kr):
    """Ring reduction (cfg.rs_ring = 1): each owner's partial travels o+1 -> ... -> o, every
    rank adding its own; within tolerance of the oracle and bit-identical run to run and
    across the CTA-pair / single-CTA engines and grid sizes (the ring order is fixed)."""
    inp = make_inputs("gemm_rs", 31 + W, W=W, m=m, n=n, k_r=kr)
    ref = oracle.gemm_rs(inp["a"], inp["b"])
    outs = []
    for cfg in [dict(), dict(pair_ctas=0), dict(grid_ctas=23)]:
        with tl.Context(0, rs_ring=1, **cfg) as c2:
            for _ in range(2):
                out = run_rs(c2, inp)
                outs.append([bf16_bits(o) for o in out])
                for o in range(W):
                    assert_close(bf16_to_f64(out[o]), ref[o], f"ring W={W} owner {o} {cfg}")
    for o in outs[1:]:
        assert all(np.array_equal(x, y) for x, y in zip(o, outs[0]))


def test_gemm_rs_ring_full_size_whole_rows():
    """Full-size ring GEMM+RS (W=8, 8192x8192, K = 8 x 3584): whole rows of every owner."""
    inp = workload_inputs("rs_70b")
    with tl.Context(0, rs_ring=1) as c2:
        out = run_rs(c2, inp)
    for o in range(8):
        rows = [0, 300, 1023]
        ref = oracle.gemm_rs_rows(inp["a"], inp["b"], o, rows)
        assert_close(bf16_to_f64(out[o])[rows], ref, f"ring rs_70b owner {o}")


def test_gemm_rs_full_size_whole_rows(ctx):
    """Full-size GEMM+RS (W=8, A_p 8192x3584, B_p 3584x8192): whole rows of every owner (all
    32 column tiles, every band and every 8-producer chain of those rows), in the launch
    configuration the benchmark times."""
    inp = workload_inputs("rs_70b")
    out = run_rs(ctx, inp)
    rng = np.random.default_rng(9)
    for o in range(8):
        rows = sorted({0, 1023, 255, 256, int(rng.integers(0, 1024))})
        ref = oracle.gemm_rs_rows(inp["a"], inp["b"], o, rows)
        assert_close(bf16_to_f64(out[o])[rows], ref, f"rs_70b owner {o} rows {rows}")


@pytest.mark.parametrize("W,m,n", [(1, 4, 8), (2, 256, 264), (3, 300, 100), (8, 8192, 1024)])
def test_reduce_scatter_alone_matches_oracle_and_its_fixed_order(ctx, W, m, n):
    """tl_reduce_scatter: within tolerance of the fp64 oracle, and bit for bit the documented
    fp32 sum in the order p = 0..W-1 rounded once to bf16."""
    import torch
    from seeded_inputs import f32_to_bf16_bits
    parts = make_inputs("reduce_scatter", 100 + W, W=W, m=m, n=n)["partials"]
    dp = [torch.from_numpy(x).cuda() for x in parts]
    out = [torch.full((m // W, n), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    tl.tl_reduce_scatter(ctx, dp, out)
    torch.cuda.synchronize()
    ref = oracle.reduce_scatter(parts)
    s = parts[0].copy()
    for x in parts[1:]:
        s = s + x  # float32, rank order
    exp = f32_to_bf16_bits(s)
    mo = m // W
    for o in range(W):
        assert_close(bf16_to_f64(out[o]), ref[o], f"reduce_scatter W={W} owner {o}")
        assert np.array_equal(bf16_bits(out[o]), exp[o * mo:(o + 1) * mo])


# ----------------------------------------------------------------------------- MLP chain
def run_mlp2(ctx, inp):
    import torch
    x = [to_dev_bf16(v) for v in inp["x_shards"]]
    w1 = [to_dev_bf16(v) for v in inp["w1"]]
    w2 = [to_dev_bf16(v) for v in inp["w2"]]
    W = len(x)
    tr, h = x[0].shape
    f = w1[0].shape[1]
    out = [torch.empty((tr, h), dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    ws = workspace(tl.tl_mlp2_workspace_bytes(W, tr * W, h, f))
    tl.tl_mlp2(ctx, x, w1, w2, out, ws)
    torch.cuda.synchronize()
    assert ctx.check() == tl.TL_OK
    return out


@pytest.mark.parametrize("W,T,h,f", [(1, 128, 256, 256), (2, 512, 264, 328), (4, 1024, 512, 384)])
def test_mlp2_matches_oracle(ctx, W, T, h, f):
    inp = make_inputs("mlp2", 51 + W, W=W, tokens=T, hidden=h, f_r=f)
    out = run_mlp2(ctx, inp)
    ref = oracle.mlp2(inp["x_shards"], inp["w1"], inp["w2"])
    for o in range(W):
        assert_close(bf16_to_f64(out[o]), ref[o], f"mlp2 W={W} owner {o}")


@pytest.mark.parametrize("W,T,h,f", [(2, 512, 264, 328), (4, 1024, 512, 384), (8, 1024, 136, 256)])
def test_mlp2_push_gather_matches_oracle_and_pull(W, T, h, f):
    """Push-mode AllGather inside the MLP chain (cfg.ag_push = 1: every shard read once and
    written into the other ranks' copies): the gathered copies equal pull's bit for bit (every
    rank's copy holds the other ranks' shards, its own slot untouched), and the output is
    bit-identical to pull's and within tolerance of the oracle."""
    import torch
    inp = make_inputs("mlp2", 61 + W, W=W, tokens=T, hidden=h, f_r=f)
    res = {}
    for push in (0, 1):
        with tl.Context(0, ag_push=push) as c2:
            x = [to_dev_bf16(v) for v in inp["x_shards"]]
            w1 = [to_dev_bf16(v) for v in inp["w1"]]
            w2 = [to_dev_bf16(v) for v in inp["w2"]]
            out = [torch.empty((T // W, h), dtype=torch.bfloat16, device="cuda") for _ in range(W)]
            ws = workspace(tl.tl_mlp2_workspace_bytes(W, T, h, f))
            tl.tl_mlp2(c2, x, w1, w2, out, ws)
            torch.cuda.synchronize()
            assert c2.check() == tl.TL_OK
            xg = bf16_bits(ws[: W * T * h * 2].view(torch.bfloat16).view(W, T, h))
            res[push] = (xg, [bf16_bits(o) for o in out])
    gath = oracle.ag_gather_bits(inp["x_shards"])
    tr = T // W
    for r in range(W):
        for src in range(W):
            rows = slice(src * tr, (src + 1) * tr)
            for push in (0, 1):
                got = res[push][0][r][rows]
                assert (not got.any()) if src == r else np.array_equal(got, gath[rows])
    assert all(np.array_equal(a, b) for a, b in zip(res[0][1], res[1][1]))
    ref = oracle.mlp2(inp["x_shards"], inp["w1"], inp["w2"])
    for o in range(W):
        assert_close((res[1][1][o].astype(np.uint32) << 16).view(np.float32).astype(np.float64), ref[o],
                     f"mlp2 push W={W} owner {o}")


def test_mlp2_full_size_whole_rows(ctx):
    """Full-size MLP chain (W=4, 4096 tokens, hidden 4096, ffn 4 x 3584): whole rows of every
    owner, each through all four ranks' layer-1 tiles, GELU and layer-2 chains."""
    inp = workload_inputs("mlp2_8b")
    out = run_mlp2(ctx, inp)
    rng = np.random.default_rng(11)
    for o in range(4):
        rows = sorted({0, 1023, 511, int(rng.integers(0, 1024))})
        ref = oracle.mlp2_rows(inp["x_shards"], inp["w1"], inp["w2"], o, rows)
        assert_close(bf16_to_f64(out[o])[rows], ref, f"mlp2_8b owner {o} rows {rows}")


def mlp2_h_from_workspace(ws, W, T, h, f):
    """The layer-1 activation H (W ranks x T tokens x f bf16) as documented in include/tl.h:
    it follows the gathered X (W x T x h bf16) at the next 256-byte boundary."""
    import torch
    off = (W * T * h * 2 + 255) // 256 * 256
    return bf16_bits(ws[off:off + W * T * f * 2].view(torch.bfloat16).view(W, T, f))


def test_mlp2_layer1_h_bit_identical_across_orders_engines_and_grids():
    """H_r = GELU(X . W1_r), stored in bf16 between the layers, is the same bits whatever the
    tile order, CTA-pair or single-CTA engine, grid size or mover geometry (each tile's K loop
    is fixed), and matches the oracle's H within tolerance; the outputs too are bit-identical
    (the layer-2 chain sums in the fixed order)."""
    import torch
    W, T, h, f = 2, 1024, 264, 520
    inp = make_inputs("mlp2", 74, W=W, tokens=T, hidden=h, f_r=f)
    hs, outs = [], []
    for cfg in [dict(), dict(swizzle=0), dict(pair_ctas=0), dict(pair_ctas=0, grid_ctas=37),
                dict(grid_ctas=38), dict(chunks_per_slab=4, mover_warps=1), dict(ag_push=1),
                dict(ag_push=1, chunks_per_slab=2, pair_ctas=0)]:
        with tl.Context(0, **cfg) as c2:
            x = [to_dev_bf16(v) for v in inp["x_shards"]]
            w1 = [to_dev_bf16(v) for v in inp["w1"]]
            w2 = [to_dev_bf16(v) for v in inp["w2"]]
            out = [torch.empty((T // W, h), dtype=torch.bfloat16, device="cuda") for _ in range(W)]
            ws = workspace(tl.tl_mlp2_workspace_bytes(W, T, h, f))
            tl.tl_mlp2(c2, x, w1, w2, out, ws)
            torch.cuda.synchronize()
            assert c2.check() == tl.TL_OK
            hs.append(mlp2_h_from_workspace(ws, W, T, h, f))
            outs.append(np.concatenate([bf16_bits(o) for o in out]))
    for x, y in zip(hs[1:], outs[1:]):
        assert np.array_equal(x, hs[0])
        assert np.array_equal(y, outs[0])
    for r in range(W):
        hr = (hs[0][r].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert_close(hr, oracle.mlp2_h(inp["x_shards"], inp["w1"], r), f"mlp2 H_{r}")


# ----------------------------------------------------------------------------- bounded waits
def test_missing_signal_times_out_and_context_survives():
    """A mover chunk that is never signalled makes the consumer's bounded wait run out:
    the call reports TL_ERR_TIMEOUT and the context stays usable."""
    import torch
    inp = make_inputs("ag_gemm", 61, W=2, m_per_rank=128, n=256, k=256)
    with tl.Context(0, debug_skip_chunk=3, timeout_ns=50_000_000) as c2:
        a = [to_dev_bf16(x) for x in inp["a_shards"]]
        b = to_dev_bf16(inp["b"])
        c = torch.empty((256, 256), dtype=torch.bfloat16, device="cuda")
        ws = workspace(tl.tl_ag_gemm_workspace_bytes(2, 128, 256, 256))
        tl.tl_ag_gemm(c2, a, b, c, ws, rank=0)
        torch.cuda.synchronize()
        assert c2.check() == tl.TL_ERR_TIMEOUT
        assert c2.check() == tl.TL_OK  # cleared
    with tl.Context(0) as c3:
        c, _ = run_ag(c3, inp)
        assert_close(bf16_to_f64(c), oracle.ag_gemm(inp["a_shards"], inp["b"]), "after timeout")


@pytest.mark.parametrize("op", ["ag", "rs", "mlp2"])
def test_cta_pair_and_single_cta_paths_agree(op):
    """256-row tiles on CTA pairs (cta_group::2) and on single CTAs give the same result
    within tolerance (both checked against the oracle)."""
    import torch
    outs = []
    for pair in (1, 0):  # 1 forces CTA pairs for every op
        with tl.Context(0, pair_ctas=pair) as c2:
            if op == "ag":
                inp = make_inputs("ag_gemm", 71, W=2, m_per_rank=512, n=520, k=328)
                c, _ = run_ag(c2, inp, rank=1)
                outs.append(bf16_to_f64(c))
                ref = oracle.ag_gemm(inp["a_shards"], inp["b"])
            elif op == "rs":
                inp = make_inputs("gemm_rs", 72, W=2, m=1024, n=520, k_r=200)
                outs.append(np.concatenate([bf16_to_f64(o) for o in run_rs(c2, inp)]))
                ref = np.concatenate(oracle.gemm_rs(inp["a"], inp["b"]))
            else:
                inp = make_inputs("mlp2", 73, W=2, tokens=1024, hidden=264, f_r=520)
                outs.append(np.concatenate([bf16_to_f64(o) for o in run_mlp2(c2, inp)]))
                ref = np.concatenate(oracle.mlp2(inp["x_shards"], inp["w1"], inp["w2"]))
            assert_close(outs[-1], ref, f"{op} pair_ctas={pair}")
    assert_close(outs[0], outs[1], f"{op} pair vs single")
