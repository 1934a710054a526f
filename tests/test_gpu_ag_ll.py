"""GPU parity of AllGather+GEMM with the low-latency push gather (cfg.ag_ll = 1).

The owners of the remote shards push them as LL words {bf16 x 2, call signal} and every
output tile reads its rows' words straight into its operand buffer ("Triton-distributed ...",
§3.2 Algorithm 1 and the low-latency AllGather before Algorithm 4).  Checked against the fp64
oracle with the bf16-in / fp32-accumulate tolerance, bit for bit against the pull path where
both issue the same 128-row MMAs, and across calls that reuse the workspace without zeroing it
(a word left by an earlier call must never be taken for this call's).
"""
import numpy as np
import pytest

import oracle
from seeded_inputs import make_inputs, workload_inputs
from tests.gpu_helpers import assert_close, bf16_bits, bf16_to_f64, to_dev_bf16, workspace

pytestmark = pytest.mark.gpu

tl = pytest.importorskip("communication_overlapped_gemm_gb300")


@pytest.fixture(scope="module")
def ctx_ll():
    import torch
    assert torch.cuda.is_available()
    c = tl.Context(0, ag_ll=1)
    yield c
    c.close()


@pytest.fixture(scope="module")
def ctx_pull():
    c = tl.Context(0)
    yield c
    c.close()


def dev(inp):
    return [to_dev_bf16(x) for x in inp["a_shards"]], to_dev_bf16(inp["b"])


def call(ctx, a, b, ws, rank):
    import torch
    W = len(a)
    mpr, k = a[0].shape
    n = b.shape[1]
    c = torch.empty((W * mpr, n), dtype=torch.bfloat16, device="cuda")
    tl.tl_ag_gemm(ctx, a, b, c, ws, rank=rank)
    torch.cuda.synchronize()
    assert ctx.check() == tl.TL_OK
    return c


@pytest.mark.parametrize("W,mpr,n,k,rank", [
    (2, 128, 256, 256, 0),    # the tiny AllGather+GEMM workload
    (2, 128, 256, 256, 1),
    (3, 128, 264, 200, 2),    # ragged n and k (k not a 64 multiple: zero-filled A and B columns)
    (4, 128, 520, 64, 1),     # one k-block, three column blocks
    (8, 128, 256, 1024, 5),   # W = 8, 16 k-blocks through the 4-stage ring
])
def test_ll_matches_oracle_and_pull_bits(ctx_ll, ctx_pull, W, mpr, n, k, rank):
    inp = make_inputs("ag_gemm", 40 + W, W=W, m_per_rank=mpr, n=n, k=k)
    assert tl.tl_ag_gemm_ll_capable(ctx_ll, W, mpr, n, k)
    a, b = dev(inp)
    ws = workspace(tl.tl_ag_gemm_workspace_bytes(W, mpr, n, k))
    c_ll = call(ctx_ll, a, b, ws, rank)
    assert_close(bf16_to_f64(c_ll), oracle.ag_gemm(inp["a_shards"], inp["b"]), f"ll W={W} rank={rank}")
    # the pull path on 128-row tiles issues the same MMAs in the same k order
    c_pull = call(ctx_pull, a, b, workspace(tl.tl_ag_gemm_workspace_bytes(W, mpr, n, k)), rank)
    assert np.array_equal(bf16_bits(c_ll), bf16_bits(c_pull))


def test_ll_256_row_shards_match_oracle(ctx_ll):
    """m_per_rank = 256: the pull path takes 256-row tiles; the LL path still takes two 128-row
    tiles per shard block and must match the oracle."""
    inp = make_inputs("ag_gemm", 51, W=4, m_per_rank=256, n=512, k=256)
    a, b = dev(inp)
    ws = workspace(tl.tl_ag_gemm_workspace_bytes(4, 256, 512, 256))
    for rank in (0, 3):
        c = call(ctx_ll, a, b, ws, rank)
        assert_close(bf16_to_f64(c), oracle.ag_gemm(inp["a_shards"], inp["b"]), f"ll 256 rank={rank}")


def test_ll_reused_workspace_takes_only_this_calls_words(ctx_ll):
    """Three calls on one unzeroed workspace with new shard values each time (and a change of
    rank, which changes which slabs are written): every result is that call's product."""
    ws = workspace(tl.tl_ag_gemm_workspace_bytes(3, 128, 256, 512))
    for seed, rank in ((61, 0), (62, 1), (63, 1)):
        inp = make_inputs("ag_gemm", seed, W=3, m_per_rank=128, n=256, k=512)
        a, b = dev(inp)
        c = call(ctx_ll, a, b, ws, rank)
        assert_close(bf16_to_f64(c), oracle.ag_gemm(inp["a_shards"], inp["b"]), f"ll reuse seed={seed}")


def test_ll_tiny_workload_bits_match_pull(ctx_ll, ctx_pull):
    inp = workload_inputs("ag_tiny")
    a, b = dev(inp)
    W, (mpr, k), n = len(a), a[0].shape, b.shape[1]
    c_ll = call(ctx_ll, a, b, workspace(tl.tl_ag_gemm_workspace_bytes(W, mpr, n, k)), 0)
    c_pull = call(ctx_pull, a, b, workspace(tl.tl_ag_gemm_workspace_bytes(W, mpr, n, k)), 0)
    assert np.array_equal(bf16_bits(c_ll), bf16_bits(c_pull))


def test_ll_refuses_large_problems(ctx_ll):
    """Past 2^20 gathered elements the workspace has no LL slabs: TL_ERR_UNSUPPORTED, nothing run."""
    import torch
    W, mpr, n, k = 8, 128, 256, 1032
    assert not tl.tl_ag_gemm_ll_capable(ctx_ll, W, mpr, n, k)
    a = [torch.zeros((mpr, k), dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    b = torch.zeros((k, n), dtype=torch.bfloat16, device="cuda")
    c = torch.full((W * mpr, n), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = workspace(tl.tl_ag_gemm_workspace_bytes(W, mpr, n, k))
    with pytest.raises(tl.TLError) as e:
        tl.tl_ag_gemm(ctx_ll, a, b, c, ws)
    assert e.value.code == tl.TL_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((c == 7.0).all())


def test_ll_single_rank_is_the_plain_gemm(ctx_ll):
    inp = make_inputs("ag_gemm", 71, W=1, m_per_rank=128, n=256, k=128)
    a, b = dev(inp)
    c = call(ctx_ll, a, b, workspace(tl.tl_ag_gemm_workspace_bytes(1, 128, 256, 128)), 0)
    assert_close(bf16_to_f64(c), oracle.ag_gemm(inp["a_shards"], inp["b"]), "ll W=1")
