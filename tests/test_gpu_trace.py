"""GPU checks of the per-CTA trace buffer (tl_ctx_set_trace).

With tracing on, every tile of a fused call appears exactly once in the MMA warp's spans,
once per epilogue warp, every mover chunk once, and every combined y tile of the MoE layer
once; the results are bit-identical to an untraced call.
"""
import numpy as np
import pytest

from seeded_inputs import make_inputs
from tests.gpu_helpers import bf16_bits, to_dev_bf16, workspace

pytestmark = pytest.mark.gpu

tl = pytest.importorskip("communication_overlapped_gemm_gb300")
from communication_overlapped_gemm_gb300 import trace  # noqa: E402

CAP = 512


def traced(ctx, fn):
    """Run fn() untraced, then traced; return (untraced result, traced result, parsed trace)."""
    import torch
    ref = fn()
    buf = torch.zeros(tl.tl_trace_bytes(ctx.num_ctas, CAP), dtype=torch.uint8, device="cuda")
    ctx.set_trace(buf, CAP)
    try:
        got = fn()
    finally:
        ctx.set_trace(None, CAP)
    torch.cuda.synchronize()
    tr = trace.parse(buf.cpu().numpy().tobytes())
    assert tr["dropped"] == 0
    sp = tr["spans"]
    assert sp.size > 0
    assert int(sp["dur"].max()) < 10**9
    span = int(sp["t0"].max()) - int(sp["t0"].min())
    assert 0 <= span < 10**9
    return ref, got, tr


def once_each(sp, kind, n, per=1):
    idx = np.sort(sp["index"][sp["kind"] == kind])
    assert np.array_equal(idx, np.repeat(np.arange(n), per)), (kind, idx[:20], n)


def test_trace_ag_gemm_tiles_and_chunks():
    import torch
    inp = make_inputs("ag_gemm", 91, W=4, m_per_rank=256, n=768, k=512)
    a = [to_dev_bf16(x) for x in inp["a_shards"]]
    b = to_dev_bf16(inp["b"])
    with tl.Context(0) as ctx:
        def run():
            c = torch.empty((4 * 256, 768), dtype=torch.bfloat16, device="cuda")
            ws = workspace(tl.tl_ag_gemm_workspace_bytes(4, 256, 768, 512))
            tl.tl_ag_gemm(ctx, a, b, c, ws)
            torch.cuda.synchronize()
            assert ctx.check() == tl.TL_OK
            return bf16_bits(c)
        ref, got, tr = traced(ctx, run)
        assert np.array_equal(ref, got)
        assert tr["grid"] == ctx.num_ctas
        sp = tr["spans"]
        ntiles = 4 * 1 * 3  # W x 256-row blocks per shard x 256-column blocks
        once_each(sp, 4, ntiles)          # MMA tile
        once_each(sp, 1, ntiles)          # producer tile
        once_each(sp, 7, ntiles, per=8)   # epilogue tile, 8 epilogue warps (one warpgroup per row half)
        once_each(sp, 9, 3 * 2 * 32)      # mover chunk: W-1 remote shards x 128-row slabs x chunks
        assert set(sp["warp"][sp["kind"] == 4].tolist()) == {1}
        assert set(sp["warp"][sp["kind"] == 1].tolist()) == {0}


def test_trace_gemm_rs_on_cta_pairs():
    import torch
    W, m, n, kr = 2, 512, 512, 256
    inp = make_inputs("gemm_rs", 92, W=W, m=m, n=n, k_r=kr)
    a = [to_dev_bf16(x) for x in inp["a"]]
    b = [to_dev_bf16(x) for x in inp["b"]]
    with tl.Context(0) as ctx:
        def run():
            out = [torch.empty((m // W, n), dtype=torch.bfloat16, device="cuda") for _ in range(W)]
            ws = workspace(tl.tl_gemm_rs_workspace_bytes(W, m, n, kr))
            tl.tl_gemm_rs(ctx, a, b, out, ws)
            torch.cuda.synchronize()
            assert ctx.check() == tl.TL_OK
            return np.concatenate([bf16_bits(o) for o in out])
        ref, got, tr = traced(ctx, run)
        assert np.array_equal(ref, got)
        sp = tr["spans"]
        ntiles = W * (m // 256) * (n // 256)
        once_each(sp, 4, ntiles)              # the leader CTA of each pair issues the MMAs
        assert np.all(sp["cta"][sp["kind"] == 4] % 2 == 0)
        once_each(sp, 7, ntiles, per=2 * 4)   # both CTAs' 4 epilogue warps
        once_each(sp, 1, ntiles, per=2)       # both CTAs' producers


def test_trace_moe_side_partition():
    import torch
    T, H, E, F, k = 300, 512, 16, 256, 2
    inp = make_inputs("moe", 93, T=T, H=H, E=E, F=F)
    x = to_dev_bf16(inp["x"])
    logits = torch.from_numpy(np.ascontiguousarray(inp["logits"])).cuda()
    wg, wu, wd = (to_dev_bf16(inp[key]) for key in ("w_gate", "w_up", "w_down"))
    with tl.Context(0) as ctx:
        counts = torch.empty(E, dtype=torch.int32, device="cuda")

        def run():
            out = torch.zeros((T, H), dtype=torch.float32, device="cuda")
            ws = workspace(tl.tl_moe_workspace_bytes(T, H, E, F, k))
            tl.tl_moe_combine(ctx, x, logits, k, wg, wu, wd, out, ws, counts_out=counts)
            torch.cuda.synchronize()
            assert ctx.check() == tl.TL_OK
            return out.cpu().numpy()
        ref, got, tr = traced(ctx, run)
        assert np.array_equal(ref, got)
        m = int(sum((int(c) + 127) // 128 for c in counts.cpu().numpy()))
        n_up, n_down = F // 128, H // 256
        sp = tr["spans"]
        once_each(sp, 10, m * n_down)        # every y tile combined once
        once_each(sp, 4, m * (n_up + n_down))
        # y tiles are claimed at run time by the combine partition and, after their last GEMM
        # tile, by the GEMM partition's CTAs: each is combined exactly once, by some CTA
        side = sp["cta"][sp["kind"] == 10]
        assert side.min() >= 0 and side.max() < ctx.num_ctas
