"""Host-side checks of the C-ABI library (no GPU needed).

The library builds for sm_103a with nvcc, loads, and exports every function that
include/tl.h declares; host-only entry points (config defaults, status strings,
workspace sizes, argument validation, the tile-order maps) behave as documented.
The tile orders are tied to the static tile-centric mapping formulas of
"TileLink: Generating Efficient Compute-Communication Overlapping Kernels using
Tile-Centric Primitives", §4.1 (as restated in the oracle), and to the swizzles of
"Triton-distributed ...", §3.7.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tl():
    import communication_overlapped_gemm_gb300 as tl
    tl.build()
    tl.lib()
    return tl


def header_functions():
    src = open(os.path.join(ROOT, "include", "tl.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tl_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(tl):
    declared = header_functions()
    assert len(declared) >= 19
    L = tl.lib()
    for name in declared:
        assert hasattr(L, name), f"{name} declared in include/tl.h but not exported"
    assert sorted(tl.EXPORTED_SYMBOLS) == declared


def test_built_for_sm103a_only():
    from communication_overlapped_gemm_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_config_defaults_and_strerror(tl):
    c = tl.Config()
    assert tl.lib().tl_config_default(ctypes.byref(c)) == tl.TL_OK
    assert (c.mover_warps, c.chunks_per_slab, c.swizzle, c.grid_ctas, c.combine_ctas) == (4, 32, 1, 0, 8)
    assert c.debug_skip_chunk == -1 and c.timeout_ns == 2_000_000_000 and c.pair_ctas == 2 and c.moe_renorm == 0
    assert c.rs_ring == 0 and c.ag_push == 0 and c.mover_kparts == 0 and c.ag_ll == 0
    assert c.mover_tma == 0
    assert tl.lib().tl_config_default(None) == tl.TL_ERR_INVALID
    for code in (tl.TL_OK, tl.TL_ERR_INVALID, tl.TL_ERR_UNSUPPORTED, tl.TL_ERR_CUDA, tl.TL_ERR_TIMEOUT,
                 tl.TL_ERR_WORKSPACE):
        assert tl.lib().tl_strerror(code)
    assert tl.lib().tl_version() >= 100


def test_workspace_sizes(tl):
    # gathered A (W*m*k*2) + 32 signals of 8 bytes per 128-row slab, each 256-aligned
    assert tl.tl_ag_gemm_workspace_bytes(8, 1024, 3584, 8192) == 8 * 1024 * 8192 * 2 + 8 * 8 * 32 * 8
    assert tl.tl_ag_gemm_workspace_bytes(2, 100, 256, 256) == 0       # m_per_rank not a 128 multiple
    # small problems (W * m_per_rank * k <= 2^20) add the LL slabs: 4 bytes per element
    assert tl.tl_ag_gemm_workspace_bytes(2, 128, 256, 256) == 2 * 128 * 256 * 2 + 2 * 1 * 32 * 8 + 2 * 128 * 256 * 4
    assert tl.tl_ag_gemm_workspace_bytes(8, 128, 256, 1024) == 8 * 128 * 1024 * 2 + 8 * 32 * 8 + 8 * 128 * 1024 * 4
    assert tl.tl_ag_gemm_workspace_bytes(8, 128, 256, 1032) == 8 * 128 * 1032 * 2 + 8 * 32 * 8   # over 2^20
    assert tl.tl_ag_gemm_workspace_bytes(9, 128, 256, 256) == 0       # W > 8
    assert tl.tl_gemm_rs_workspace_bytes(8, 8192, 8192, 3584) == 8192 * 8192 * 4 + 64 * 32 * 8
    assert tl.tl_gemm_rs_workspace_bytes(8, 1000, 256, 64) == 0
    assert tl.tl_mlp2_workspace_bytes(4, 4096, 4096, 3584) > 4 * 4096 * 4096 * 2 + 4 * 4096 * 3584 * 2
    assert tl.tl_moe_workspace_bytes(4096, 2048, 64, 1408, 2) > 0
    assert tl.tl_moe_workspace_bytes(4096, 2000, 64, 1408, 2) == 0    # H not a 256 multiple
    assert tl.tl_moe_workspace_bytes(4096, 2048, 300, 1408, 2) == 0   # E > 256
    al = lambda x: (x + 255) // 256 * 256
    # attention: gathered K and V, one signal per (shard, head, 128-key block) (the last block
    # of a shard partial when l_r is not a multiple of 128), then the split items' partials:
    # min(items, 40) items x 2 halves x 2 CTAs of fp32 O (128 x 128) and (m, l) per row, and
    # one counter per item and CTA
    def tail(items):
        t = min(items, 40)
        return al(t * 4 * 128 * 128 * 4) + al(t * 4 * 128 * 2 * 4) + al(t * 2 * 8)
    assert tl.tl_ag_attention_workspace_bytes(8, 32, 2048, 128) == \
        2 * al(8 * 32 * 2048 * 128 * 2) + al(8 * 32 * 16 * 8) + tail(32 * 8)
    assert tl.tl_ag_attention_workspace_bytes(3, 2, 200, 128) == \
        2 * al(3 * 2 * 200 * 128 * 2) + al(3 * 2 * 2 * 8) + tail(2 * 1)
    assert tl.tl_ag_attention_workspace_bytes(2, 2, 128, 64) == 0    # head dim other than 128
    assert tl.tl_ag_attention_workspace_bytes(9, 2, 128, 128) == 0   # W > 8


def test_argument_validation_needs_no_gpu(tl):
    L = tl.lib()
    ptrs = (ctypes.c_void_p * 2)(16, 32)
    # null context / bad shapes are rejected before any CUDA call
    assert L.tl_ag_gemm(None, 2, 0, ptrs, 16, 16, 16, 1 << 20, 128, 256, 256, None) == tl.TL_ERR_INVALID
    assert L.tl_gemm_rs(None, 2, ptrs, ptrs, ptrs, 16, 1 << 20, 256, 256, 64, None) == tl.TL_ERR_INVALID
    assert L.tl_mlp2(None, 2, ptrs, ptrs, ptrs, ptrs, 16, 1 << 20, 256, 256, 256, None) == tl.TL_ERR_INVALID
    assert L.tl_moe_combine(None, 16, 16, 2, 16, 16, 16, 16, None, None, 16, 1 << 20, 64, 256, 4, 128,
                            None) == tl.TL_ERR_INVALID
    assert L.tl_ag_attention(None, 2, 0, 16, ptrs, ptrs, 16, 16, 1 << 20, 2, 128, 128, None) == tl.TL_ERR_INVALID
    assert L.tl_ag_gemm_static_scratch(None, 2, 0, ptrs, 16, 16, 128, 256, 256, None) == tl.TL_ERR_INVALID
    assert L.tl_allgather(None, 2, 0, ptrs, 16, 1 << 20, 128, 256, None) == tl.TL_ERR_INVALID
    assert L.tl_reduce_scatter(None, 2, ptrs, ptrs, 256, 256, None) == tl.TL_ERR_INVALID
    assert L.tl_ctx_check(None) == tl.TL_ERR_INVALID


@pytest.mark.parametrize("W,rank,mpr,n", [(8, 0, 1024, 3584), (8, 5, 1024, 3584), (2, 1, 128, 256), (3, 2, 256, 520)])
def test_ag_tile_order_is_rank_swizzled_and_matches_static_map(tl, W, rank, mpr, n):
    src, mb, nb = tl.tl_ag_tile_order(W, rank, mpr, n, 1)
    bm = 256 if mpr % 256 == 0 else 128  # tile rows the kernel uses; m_block is in 128-row units
    mps, nbk = mpr // bm, -(-n // 256)
    assert len(src) == W * mps * nbk
    # every tile exactly once
    keys = set(zip(src.tolist(), mb.tolist(), nb.tolist()))
    assert keys == {(s, m * (bm // 128), b) for s in range(W) for m in range(mps) for b in range(nbk)}
    # step s computes with the shard of rank (rank + s) mod W: the local shard first
    per = mps * nbk
    for s in range(W):
        assert set(src[s * per:(s + 1) * per].tolist()) == {(rank + s) % W}
    # the source rank agrees with the pages' static mapping f_R for the tile's global rows
    for t in range(0, len(src), max(1, len(src) // 97)):
        row_tile = (src[t] * mpr) // 128 + mb[t]
        lo, hi, r, _ = oracle.static_tile_map(int(row_tile), W * mpr, W, 1, 128)
        assert r == src[t] and lo == src[t] * mpr + mb[t] * 128
    s0, _, _ = tl.tl_ag_tile_order(W, rank, mpr, n, 0)
    assert s0[:per].tolist() == [0] * per  # identity order starts at rank 0


def _rs_band_order(W, m, n, swizzle, band_rows=2048, band_cols=4096):
    """The documented GEMM+RS walk, restated: bands of band_rows x band_cols of the output in
    row-major order; inside a band producers 0..W-1; a producer's band tiles with the column
    block slowest and the row block fastest, the rows rotated to start at owner (p+1) mod W."""
    bm = 256 if (m // W) % 256 == 0 else 128
    mbo, nbk = m // W // bm, -(-n // 256)
    mt, BR, BC = W * mbo, max(1, band_rows // bm), max(1, band_cols // 256)
    out = []
    for r0 in range(0, mt, BR):
        rows0 = list(range(r0, min(mt, r0 + BR)))
        for c0 in range(0, nbk, BC):
            for q in range(W):
                rows = rows0
                if swizzle:
                    first = [r for r in rows0 if r // mbo == (q + 1) % W]
                    if first:
                        k = rows0.index(first[0])
                        rows = rows0[k:] + rows0[:k]
                for c in range(c0, min(nbk, c0 + BC)):
                    out += [(q, r // mbo, (r % mbo) * (bm // 128), c) for r in rows]
    return out


@pytest.mark.parametrize("W,m,n", [(8, 8192, 8192), (4, 1024, 520), (1, 128, 256), (6, 1536, 768), (5, 640, 300),
                                   (8, 1024, 264), (2, 8192, 8200)])
def test_rs_tile_order_banded_and_owner_swizzled(tl, W, m, n):
    bm = 256 if (m // W) % 256 == 0 else 128
    mbo, nbk = m // W // bm, -(-n // 256)
    for swz in (1, 0):
        p, o, mb, nb = tl.tl_rs_tile_order(W, m, n, swz)
        got = list(zip(p.tolist(), o.tolist(), mb.tolist(), nb.tolist()))
        assert len(got) == W * W * mbo * nbk and len(set(got)) == len(got)
        assert got == _rs_band_order(W, m, n, swz)
        # every output tile's W partials come in the producer order 0..W-1 (the fixed fp32
        # summation order the peer signals chain)
        seen = {}
        for q, oo, r, c in got:
            assert seen.get((oo, r, c), -1) == q - 1
            seen[(oo, r, c)] = q


@pytest.mark.parametrize("W,m,n", [(8, 8192, 8192), (4, 1024, 520), (1, 128, 256), (3, 768, 520), (5, 640, 296)])
def test_rs_ring_tile_order(tl, W, m, n):
    """The ring: owner by owner, bands of 2048 x 4096, hops 0..W-1 inside a band, column block
    slowest inside a hop; hop s of owner o is computed by producer (o + 1 + s) mod W, the owner
    last, and each tile's hops come in order."""
    bm = 256 if (m // W) % 256 == 0 else 128
    mbo, nbk = m // W // bm, -(-n // 256)
    p, o, mb, nb, hop = tl.tl_rs_ring_tile_order(W, m, n)
    got = list(zip(p.tolist(), o.tolist(), mb.tolist(), nb.tolist(), hop.tolist()))
    BR, BC = max(1, 2048 // bm), 4096 // 256
    exp = []
    for oo in range(W):
        for r0 in range(0, mbo, BR):
            for c0 in range(0, nbk, BC):
                for sh in range(W):
                    for c in range(c0, min(nbk, c0 + BC)):
                        exp += [((oo + 1 + sh) % W, oo, r * (bm // 128), c, sh) for r in range(r0, min(mbo, r0 + BR))]
    assert got == exp
    seen = {}
    for q, oo, r, c, sh in got:
        assert seen.get((oo, r, c), -1) == sh - 1
        seen[(oo, r, c)] = sh
    assert all(v == W - 1 for v in seen.values()) and len(seen) == W * mbo * nbk
    al = lambda x: (x + 255) // 256 * 256
    assert tl.tl_gemm_rs_ring_workspace_bytes(W, m, n, 64) == al(W * m * n * 4) + al((m // 128) * nbk * 8)


def test_tile_order_rejects_bad_shapes(tl):
    with pytest.raises(tl.TLError):
        tl.tl_ag_tile_order(2, 2, 128, 256, 1)
    with pytest.raises(tl.TLError):
        tl.tl_rs_tile_order(3, 1000, 256, 1)


def test_static_scratch_binding_checks_shapes_before_any_call(tl):
    """A wrong-shaped output or an uneven shard is refused by the binding itself, before the
    library (or the GPU) sees the call: the kernel's tensor maps would otherwise be built for
    shapes the buffers do not have."""
    import torch
    a = [torch.zeros((128, 256), dtype=torch.bfloat16) for _ in range(2)]
    b = torch.zeros((256, 256), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="inconsistent shapes"):
        tl.tl_ag_gemm_static_scratch(None, a, b, torch.zeros((128, 256), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="inconsistent shapes"):
        tl.tl_ag_gemm_static_scratch(None, [a[0], torch.zeros((256, 256), dtype=torch.bfloat16)], b,
                                     torch.zeros((256, 256), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="inconsistent shapes"):
        tl.tl_ag_gemm_static_scratch(None, a, torch.zeros((128, 256), dtype=torch.bfloat16),
                                     torch.zeros((256, 256), dtype=torch.bfloat16))


@pytest.mark.parametrize("T,H,E,F,k,m", [(4096, 2048, 64, 1408, 2, 96), (4096, 2048, 64, 1408, 2, 127),
                                         (4096, 2048, 64, 1408, 2, 1), (300, 512, 16, 256, 2, 13),
                                         (96, 256, 256, 128, 8, 1), (200, 256, 8, 384, 3, 7),
                                         (64, 256, 4, 128, 2, 0)])
def test_moe_tile_order(tl, T, H, E, F, k, m):
    """The persistent MoE kernel's tile order ([TL] §4.1 dynamic mapping, its closed form):
    every up and down tile exactly once; every down tile after all up tiles of its row tile,
    so a co-resident grid taking tiles in this order never waits on a later tile; every up tile
    before the first down tile; the down tiles in the order the combine claims them, and for
    each column block their row tiles ascending (the tile of a token's lower expert comes
    first)."""
    n_up, n_down = F // 128, H // 256
    kind, row, col = tl.tl_moe_tile_order(T, H, E, F, k, m)
    tiles = list(zip(kind.tolist(), row.tolist(), col.tolist()))
    assert len(tiles) == m * (n_up + n_down)
    assert sorted(tiles) == sorted([(1, r, c) for r in range(m) for c in range(n_up)] +
                                   [(2, r, c) for r in range(m) for c in range(n_down)])
    pos = {t: i for i, t in enumerate(tiles)}
    for r in range(m):
        last_up = max(pos[(1, r, c)] for c in range(n_up))
        assert all(pos[(2, r, c)] > last_up for c in range(n_down))
    assert kind.tolist() == sorted(kind.tolist())  # all up tiles (1) before all down tiles (2)
    crow, ccol = tl.tl_moe_combine_order(T, H, E, F, k, m)
    downs = [(r, c) for (kk, r, c) in tiles if kk == 2]
    assert list(zip(crow.tolist(), ccol.tolist())) == downs
    for c in range(n_down):
        rows_c = [r for (r, cc) in downs if cc == c]
        assert rows_c == sorted(rows_c)


def test_moe_tile_order_refuses_bad_queries(tl):
    rmax_tiles = -(-(4096 * 2 + 127 * 64) // 128)  # the row-tile bound the workspace is sized for
    assert tl.tl_moe_tile_order(4096, 2048, 64, 1408, 2, rmax_tiles)[0].size == rmax_tiles * (11 + 8)
    for bad in ((4096, 2048, 64, 1408, 2, rmax_tiles + 1), (4096, 2048, 64, 1408, 2, -1),
                (4096, 2000, 64, 1408, 2, 4)):
        with pytest.raises(tl.TLError):
            tl.tl_moe_tile_order(*bad)
        with pytest.raises(tl.TLError):
            tl.tl_moe_combine_order(*bad)
