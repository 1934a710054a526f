"""The AllGather + GEMM entry point for callers that cannot allocate device memory.

tl_ag_gemm_static_scratch keeps its scratch in a fixed device array inside the
library instead of a caller-provided workspace, for code being recorded into a
CUDA graph by stream capture, plug-ins without access to an allocator, and
real-time paths that forbid allocation.  Through the C ABI, two calls in a row
are checked against the workspace entry point tl_ag_gemm (and the oracle) within
the suite's tolerance, and a problem too large for the array must be refused.
This file is collected last on purpose.
"""
import pytest

import oracle
from seeded_inputs import make_inputs
from tests.gpu_helpers import assert_close, bf16_to_f64, to_dev_bf16, workspace

pytestmark = pytest.mark.gpu
tl = pytest.importorskip("communication_overlapped_gemm_gb300")


def test_static_scratch_matches_workspace_entry_point_on_two_calls():
    import torch
    with tl.Context(0) as ctx:
        for seed, (W, mpr, n, k) in [(91, (2, 128, 256, 256)), (92, (4, 256, 520, 328))]:
            inp = make_inputs("ag_gemm", seed, W=W, m_per_rank=mpr, n=n, k=k)
            a = [to_dev_bf16(x) for x in inp["a_shards"]]
            b = to_dev_bf16(inp["b"])
            c_ws = torch.empty((W * mpr, n), dtype=torch.bfloat16, device="cuda")
            c_na = torch.full((W * mpr, n), float("nan"), dtype=torch.bfloat16, device="cuda")
            ws = workspace(tl.tl_ag_gemm_workspace_bytes(W, mpr, n, k))
            tl.tl_ag_gemm(ctx, a, b, c_ws, ws, rank=1)
            tl.tl_ag_gemm_static_scratch(ctx, a, b, c_na, rank=1)
            torch.cuda.synchronize()
            assert ctx.check() == tl.TL_OK
            got = bf16_to_f64(c_na)
            assert_close(got, bf16_to_f64(c_ws), f"static scratch vs workspace W={W}")
            assert_close(got, oracle.ag_gemm(inp["a_shards"], inp["b"]), f"static scratch vs oracle W={W}")


def test_static_scratch_after_another_context():
    """Calls from two contexts share the one array: a call in a second context (its own,
    unrelated signal values), then a call in the first, both match the oracle.  Each call
    clears the signal words the other context left."""
    import torch
    inp = make_inputs("ag_gemm", 93, W=4, m_per_rank=128, n=256, k=384)
    ref = oracle.ag_gemm(inp["a_shards"], inp["b"])
    a = [to_dev_bf16(x) for x in inp["a_shards"]]
    b = to_dev_bf16(inp["b"])
    with tl.Context(0) as c1, tl.Context(0) as c2:
        for ctx, rank in ((c2, 2), (c1, 0), (c2, 3), (c1, 1)):
            c = torch.full((4 * 128, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
            tl.tl_ag_gemm_static_scratch(ctx, a, b, c, rank=rank)
            torch.cuda.synchronize()
            assert ctx.check() == tl.TL_OK
            assert_close(bf16_to_f64(c), ref, f"static scratch, rank {rank}")


def test_static_scratch_rejects_too_large_problem():
    import torch
    with tl.Context(0) as ctx:
        W, mpr, n, k = 8, 1024, 256, 2048  # gathered operand 32 MiB > 16 MiB
        a = [torch.zeros((mpr, k), dtype=torch.bfloat16, device="cuda") for _ in range(W)]
        b = torch.zeros((k, n), dtype=torch.bfloat16, device="cuda")
        c = torch.zeros((W * mpr, n), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(tl.TLError) as e:
            tl.tl_ag_gemm_static_scratch(ctx, a, b, c)
        assert e.value.code == tl.TL_ERR_WORKSPACE
