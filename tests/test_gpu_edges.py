"""Edge cases and limits of the C ABI on the GPU: the standalone AllGather, empty
problems, argument errors, the largest emulated world (W = 8) for every operator and
the MoE layer's limits (E = 256 experts, top-8)."""
import ctypes

import numpy as np
import pytest

import oracle
from seeded_inputs import make_inputs
from tests.gpu_helpers import assert_close, bf16_bits, bf16_to_f64, to_dev_bf16, workspace

pytestmark = pytest.mark.gpu
tl = pytest.importorskip("communication_overlapped_gemm_gb300")


@pytest.fixture(scope="module")
def ctx():
    c = tl.Context(0)
    yield c
    c.close()


@pytest.mark.parametrize("W,mpr,k,rank", [(3, 256, 328, 2), (8, 128, 64, 5), (1, 384, 136, 0), (4, 256, 8192, 1),
                                        (2, 128, 2056, 0)])
@pytest.mark.parametrize("tma", [0, 1])
def test_standalone_allgather_is_bit_exact(W, mpr, k, rank, tma):
    """Both copy engines (the SMs' load/store path and the TMA unit's bulk copies): the gathered
    buffer is the rank-order concatenation bit for bit, and every chunk signal carries the
    call's value.  k = 8192 makes a chunk (4 rows) two 32 KB bulk copies; k = 2056 a chunk
    that is not a whole number of 32 KB stages."""
    import torch
    inp = make_inputs("ag_gemm", 200 + W, W=W, m_per_rank=mpr, n=64, k=k)
    a = [to_dev_bf16(x) for x in inp["a_shards"]]
    ws = workspace(tl.tl_ag_gemm_workspace_bytes(W, mpr, 8, k))
    with tl.Context(0, mover_tma=tma) as c2:
        for _ in range(2):  # a second call on the same workspace: the signals move to the new value
            tl.tl_allgather(c2, a, ws, rank=rank)
        torch.cuda.synchronize()
        assert c2.check() == tl.TL_OK
    gath = oracle.ag_gather_bits(inp["a_shards"])
    got = bf16_bits(ws[: gath.size * 2].view(torch.bfloat16).view(gath.shape))
    if W == 1:  # nothing to gather: a no-op, the zero-filled region stays zero
        assert not got.any()
        return
    assert np.array_equal(got, gath)
    # every chunk signal (W shards x m_per_rank/128 slabs x 32 chunks) holds one and the same
    # nonzero value, the second call's
    off = (gath.size * 2 + 255) // 256 * 256
    sig = ws[off: off + W * (mpr // 128) * 32 * 8].view(torch.int64).cpu().numpy()
    assert sig.min() == sig.max() and sig[0] != 0


def test_empty_problems_are_noops(ctx):
    L = tl.lib()
    ptrs = (ctypes.c_void_p * 8)()
    assert L.tl_ag_gemm(ctx.handle, 2, 0, ptrs, None, None, None, 0, 0, 256, 256, None) == tl.TL_OK
    assert L.tl_ag_gemm(ctx.handle, 2, 0, ptrs, None, None, None, 0, 128, 0, 256, None) == tl.TL_OK
    assert L.tl_gemm_rs(ctx.handle, 2, ptrs, ptrs, ptrs, None, 0, 0, 256, 64, None) == tl.TL_OK
    assert L.tl_mlp2(ctx.handle, 2, ptrs, ptrs, ptrs, ptrs, None, 0, 0, 256, 256, None) == tl.TL_OK
    assert L.tl_allgather(ctx.handle, 2, 0, ptrs, None, 0, 0, 64, None) == tl.TL_OK
    assert L.tl_ag_gemm_static_scratch(ctx.handle, 2, 0, ptrs, None, None, 0, 256, 256, None) == tl.TL_OK


def test_argument_errors(ctx):
    import torch
    L = tl.lib()
    a = [torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    b = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    need = tl.tl_ag_gemm_workspace_bytes(2, 128, 256, 64)
    ws = workspace(need + 64)
    P = lambda ts: (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    st = int(torch.cuda.current_stream().cuda_stream)
    ok = L.tl_ag_gemm(ctx.handle, 2, 0, P(a), b.data_ptr(), c.data_ptr(), ws.data_ptr(), need, 128, 256, 64, st)
    assert ok == tl.TL_OK
    # workspace one byte short
    assert L.tl_ag_gemm(ctx.handle, 2, 0, P(a), b.data_ptr(), c.data_ptr(), ws.data_ptr(), need - 1, 128, 256, 64,
                        st) == tl.TL_ERR_WORKSPACE
    # misaligned operand pointer
    assert L.tl_ag_gemm(ctx.handle, 2, 0, P(a), b.data_ptr() + 2, c.data_ptr(), ws.data_ptr(), need, 128, 256, 64,
                        st) == tl.TL_ERR_INVALID
    # rank out of range, W above 8, rows not a 128 multiple, k not a multiple of 8
    assert L.tl_ag_gemm(ctx.handle, 2, 2, P(a), b.data_ptr(), c.data_ptr(), ws.data_ptr(), need, 128, 256, 64,
                        st) == tl.TL_ERR_INVALID
    assert L.tl_ag_gemm(ctx.handle, 9, 0, P(a * 5), b.data_ptr(), c.data_ptr(), ws.data_ptr(), need, 128, 256, 64,
                        st) == tl.TL_ERR_INVALID
    assert L.tl_ag_gemm(ctx.handle, 2, 0, P(a), b.data_ptr(), c.data_ptr(), ws.data_ptr(), need, 100, 256, 64,
                        st) == tl.TL_ERR_INVALID
    assert L.tl_ag_gemm(ctx.handle, 2, 0, P(a), b.data_ptr(), c.data_ptr(), ws.data_ptr(), need, 128, 256, 60,
                        st) == tl.TL_ERR_INVALID
    torch.cuda.synchronize()
    assert ctx.check() == tl.TL_OK
    # invalid configurations are refused at context creation
    for bad in (dict(mover_warps=0), dict(mover_warps=5), dict(chunks_per_slab=3), dict(swizzle=2),
                dict(pair_ctas=3), dict(timeout_ns=0)):
        with pytest.raises(tl.TLError):
            tl.Context(0, **bad)


def test_world_size_8_every_operator(ctx):
    import torch
    from tests.test_gpu_gemm_parity import run_ag, run_mlp2, run_rs
    inp = make_inputs("ag_gemm", 210, W=8, m_per_rank=256, n=264, k=200)
    c, _ = run_ag(ctx, inp, rank=7)
    assert_close(bf16_to_f64(c), oracle.ag_gemm(inp["a_shards"], inp["b"]), "ag W=8")
    inp = make_inputs("gemm_rs", 211, W=8, m=2048, n=264, k_r=136)
    out = run_rs(ctx, inp)
    ref = oracle.gemm_rs(inp["a"], inp["b"])
    for o in range(8):
        assert_close(bf16_to_f64(out[o]), ref[o], f"rs W=8 owner {o}")
    inp = make_inputs("mlp2", 212, W=8, tokens=2048, hidden=264, f_r=136)
    out = run_mlp2(ctx, inp)
    ref = oracle.mlp2(inp["x_shards"], inp["w1"], inp["w2"])
    for o in range(8):
        assert_close(bf16_to_f64(out[o]), ref[o], f"mlp2 W=8 owner {o}")


@pytest.mark.parametrize("T,H,E,F,k", [(96, 256, 256, 128, 8), (33, 512, 256, 256, 2)])
def test_moe_limits(ctx, T, H, E, F, k):
    from tests.test_gpu_moe_parity import run_moe
    inp = make_inputs("moe", 220 + k, T=T, H=H, E=E, F=F)
    out, perm, counts = run_moe(ctx, inp, k)
    ref = oracle.moe(inp["x"], inp["logits"], inp["w_gate"], inp["w_up"], inp["w_down"], k)
    assert np.array_equal(perm, ref["perm"]) and np.array_equal(counts, ref["counts"])
    assert_close(out, ref["out"], f"moe E={E} k={k}")
