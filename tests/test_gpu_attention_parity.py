"""GPU parity of the AllGather KV + self-attention kernel against the fp64 oracle.

Through the C ABI: the kernel's mover warps gather the K/V shards (rank order, bit for
bit) while its tcgen05 flash-attention warps run the rank's queries over them.  Tolerance for
the bf16-in / fp32-accumulate outputs: max|gpu - ref| <= 1e-2 * max|ref| + 1e-3.
"""
import numpy as np
import pytest

import oracle
from seeded_inputs import make_inputs, workload_inputs
from tests.gpu_helpers import assert_close, bf16_bits, bf16_to_f64, to_dev_bf16, workspace

pytestmark = pytest.mark.gpu

tl = pytest.importorskip("communication_overlapped_gemm_gb300")


def run_attn(inp, rank=0, **cfg):
    import torch
    q = to_dev_bf16(inp["q"])
    ks = [to_dev_bf16(x) for x in inp["k_shards"]]
    vs = [to_dev_bf16(x) for x in inp["v_shards"]]
    W = len(ks)
    H, L, d = q.shape
    out = torch.full((H, L, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = workspace(tl.tl_ag_attention_workspace_bytes(W, H, L, d))
    with tl.Context(0, timeout_ns=500_000_000, **cfg) as ctx:
        tl.tl_ag_attention(ctx, q, ks, vs, out, ws, rank=rank)
        torch.cuda.synchronize()
        assert ctx.check() == tl.TL_OK
    kv = W * L * d * H * 2
    kg = bf16_bits(ws[:kv].view(torch.bfloat16).view(W, H, L, d))  # shard-major gathered K
    return out, kg


@pytest.mark.parametrize("W,H,L,rank", [(2, 2, 128, 0), (1, 1, 128, 0), (3, 2, 256, 2), (4, 1, 384, 1), (3, 3, 128, 1),
                                        (8, 1, 128, 7)])
def test_ag_attention_matches_oracle(W, H, L, rank):
    inp = make_inputs("ag_attn", 80 + W, W=W, heads=H, l_r=L, d=128)
    out, kg = run_attn(inp, rank=rank)
    ref = oracle.ag_attention(inp["q"], inp["k_shards"], inp["v_shards"])
    assert_close(bf16_to_f64(out), ref, f"attention W={W} H={H} L={L} rank={rank}")
    # the gathered K holds shard r at r; per head it is the oracle's rank-order gather
    assert np.array_equal(np.concatenate(list(kg), axis=1), oracle.attn_gather(inp["k_shards"]))


@pytest.mark.parametrize("W,H,L,rank", [(3, 2, 200, 1), (2, 1, 100, 0), (1, 1, 72, 0), (4, 2, 130, 3),
                                        (2, 1, 300, 1), (3, 2, 520, 2), (2, 3, 384, 0)])
def test_ag_attention_ragged_lengths(W, H, L, rank):
    """Shard lengths that are not a multiple of the 256-key block: each shard's last key block
    and the last 256-query tile are partial (the absent keys get no weight, the absent rows are
    not stored).  Below 128 the second key half of every block is absent for all rows (its
    group keeps a running max of -inf); 300 and 520 have full blocks before the partial one;
    384 ends half-way through a block and a query tile."""
    inp = make_inputs("ag_attn", 97 + L, W=W, heads=H, l_r=L, d=128)
    out, kg = run_attn(inp, rank=rank)
    ref = oracle.ag_attention(inp["q"], inp["k_shards"], inp["v_shards"])
    assert_close(bf16_to_f64(out), ref, f"attention W={W} H={H} L={L} rank={rank}")
    assert np.array_equal(np.concatenate(list(kg), axis=1), oracle.attn_gather(inp["k_shards"]))


@pytest.mark.parametrize("W,H,L,ctas,rank", [
    (3, 3, 256, 4, 1),   # 3 items on 2 pairs: items 0 and 1 whole, item 2 in halves of 1 and 2 blocks
    (2, 2, 300, 6, 0),   # ragged: 4 items (2 heads x 2 query tiles) on 3 pairs, the last one split
    (4, 5, 256, 8, 3),   # 5 items on 4 pairs, halves of 2 blocks each
    (1, 2, 512, 6, 0),   # one rank: 4 items on 3 pairs, halves of one block
    (3, 3, 512, 8, 2),   # 6 items on 4 pairs, two split; the second half starts inside a remote shard
])
def test_ag_attention_split_tail(W, H, L, ctas, rank):
    """Grids whose last wave the items would fill less than half: the last items run as two
    halves of their keys on two pairs and the half that finishes second combines both.
    Against the oracle, and bit for bit across repeated calls on one workspace (either half
    may finish second; the combine takes half 0 first either way)."""
    import torch
    inp = make_inputs("ag_attn", 120 + W * 10 + H, W=W, heads=H, l_r=L, d=128)
    q = to_dev_bf16(inp["q"])
    ks = [to_dev_bf16(x) for x in inp["k_shards"]]
    vs = [to_dev_bf16(x) for x in inp["v_shards"]]
    ws = workspace(tl.tl_ag_attention_workspace_bytes(W, H, L, 128))
    ref = oracle.ag_attention(inp["q"], inp["k_shards"], inp["v_shards"])
    outs = []
    with tl.Context(0, timeout_ns=500_000_000, grid_ctas=ctas) as ctx:
        for _ in range(3):
            out = torch.full((H, L, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
            tl.tl_ag_attention(ctx, q, ks, vs, out, ws, rank=rank)
            torch.cuda.synchronize()
            assert ctx.check() == tl.TL_OK
            outs.append(bf16_bits(out))
    assert_close(bf16_to_f64(out), ref, f"attention split tail W={W} H={H} L={L} ctas={ctas}")
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


def test_ag_attention_peaked_scores():
    """Large-magnitude queries make the softmax peaked and its running maximum move a lot
    from block to block (the rescale of O in TMEM)."""
    inp = make_inputs("ag_attn", 91, W=2, heads=2, l_r=256, d=128)
    from seeded_inputs import f32_to_bf16_bits
    inp["q"] = f32_to_bf16_bits(oracle.widen_bf16(inp["q"]).astype(np.float32) * 6.0)
    out, _ = run_attn(inp, rank=1)
    ref = oracle.ag_attention(inp["q"], inp["k_shards"], inp["v_shards"])
    assert_close(bf16_to_f64(out), ref, "attention peaked")


def test_ag_attention_growing_scores():
    """Keys scaled up block by block in the order the kernel visits them (the local shard,
    then rank + 1, ...), so that the running maximum of most rows grows by more than 2^8 (in
    base 2) at every block and O is rescaled each time; the odd query rows are zero, so
    their scores stay 0 and, in the same warps, they never rescale."""
    from seeded_inputs import f32_to_bf16_bits
    W, H, L, rank = 3, 1, 256, 1
    inp = make_inputs("ag_attn", 93, W=W, heads=H, l_r=L, d=128)
    q = oracle.widen_bf16(inp["q"]).astype(np.float32)
    q[:, 1::2] = 0.0
    inp["q"] = f32_to_bf16_bits(q)
    ks = []
    for r, k in enumerate(inp["k_shards"]):
        kf = oracle.widen_bf16(k).astype(np.float32)
        step = (r - rank) % W  # the kernel visits shard r at this step
        for b in range(L // 128):
            kf[:, b * 128:(b + 1) * 128] *= 1.0 + 3.0 * (step * (L // 128) + b)
        ks.append(f32_to_bf16_bits(kf))
    inp["k_shards"] = ks
    out, _ = run_attn(inp, rank=rank)
    ref = oracle.ag_attention(inp["q"], inp["k_shards"], inp["v_shards"])
    assert_close(bf16_to_f64(out), ref, "attention growing scores")


def test_ag_attention_16k_sampled():
    """Attn-1 at 16k on 8 ranks (32 heads, 2048 queries per rank), as bench.py runs it;
    sampled query rows of a few heads against the oracle."""
    import torch
    inp = workload_inputs("attn_16k")
    out, kg = run_attn(inp, rank=0)
    heads, rows = [0, 13, 31], [0, 127, 128, 1000, 2047]
    ref = oracle.ag_attention_rows(inp["q"], inp["k_shards"], inp["v_shards"], heads, rows)
    got = bf16_to_f64(out)[heads][:, rows]
    assert_close(got, ref, "attn_16k sampled")
    assert np.array_equal(np.concatenate(list(kg[:, 5:6]), axis=1), oracle.attn_gather([k[5:6] for k in inp["k_shards"]]))
