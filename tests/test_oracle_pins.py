"""Pins of the fp64 CPU oracle against things other than itself.

Hand-derived fixtures (tests/golden/*.json, each citing its passage), pure-Python
brute-force loops on tiny shapes, special cases that reduce to a textbook GEMM,
closed forms (column-concatenated GEMM for the reduce-scatter, unsharded GEMM for
the all-gather), textbook constants for GELU/SiLU, and bijection/stability of
the MoE permutation.  No GPU needed.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from seeded_inputs import f32_to_bf16_bits, make_inputs, normal_bf16, normal_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _py(bits):
    """bf16 bits -> nested Python floats (decode via struct-free bit math)."""
    arr = np.asarray(bits, dtype=np.uint16)
    f = (arr.astype(np.uint32) << 16).view(np.float32)
    return f.astype(float).tolist()


# ----------------------------------------------------------------------------- golden fixtures
def test_golden_ag_gemm_hand():
    g = _load("ag_gemm_w2_hand.json")
    c = oracle.ag_gemm([_bits(a) for a in g["a_shards"]], _bits(g["b"]))
    assert np.array_equal(c, np.array(g["c"], dtype=np.float64))


def test_golden_gemm_rs_hand():
    g = _load("gemm_rs_w2_hand.json")
    outs = oracle.gemm_rs([_bits(a) for a in g["a"]], [_bits(b) for b in g["b"]])
    for o, exp in zip(outs, g["out"]):
        assert np.array_equal(o, np.array(exp, dtype=np.float64))


def test_golden_activations():
    g = _load("activations_textbook.json")
    for x, y in g["gelu"]:
        assert abs(float(oracle.gelu(np.array([x]))[0]) - y) <= 1e-15 * max(1.0, abs(y))
    for x, y in g["silu"]:
        assert abs(float(oracle.silu(np.array([x]))[0]) - y) <= 1e-15 * max(1.0, abs(y))


def test_gelu_limits():
    x = np.array([-40.0, -10.0, 10.0, 40.0])
    y = oracle.gelu(x)
    assert abs(y[0]) < 1e-300 and abs(y[1]) < 1e-20
    assert y[2] == pytest.approx(10.0, rel=1e-15) and y[3] == 40.0


def test_golden_moe_hand():
    g = _load("moe_t2_e3_hand.json")
    logits = np.array(g["logits"], dtype=np.float32)
    res = oracle.moe(_bits(g["x"]), logits, _bits(g["w_gate"]), _bits(g["w_up"]),
                     _bits(g["w_down"]), g["topk"])
    assert res["experts"].tolist() == g["experts"]
    assert np.allclose(res["gates"], np.array(g["gates"]), rtol=0, atol=g["gate_tol"])
    assert res["perm"].tolist() == g["perm"]
    assert res["counts"].tolist() == g["counts"]
    assert res["offsets"].tolist() == g["offsets"]
    assert res["inv"].tolist() == g["inv"]
    assert np.allclose(res["out"], np.array(g["out"]), rtol=2e-6, atol=0)


def test_golden_static_map():
    g = _load("static_map_hand.json")
    for tid, lo, hi, rank, ch in g["cases"]:
        assert oracle.static_tile_map(tid, g["M"], g["R"], g["C"], g["Tm"]) == (lo, hi, rank, ch)


# ----------------------------------------------------------------------------- brute force
def _bf_matmul(A, B):
    n, k = len(A), len(A[0])
    m = len(B[0])
    return [[sum(A[i][t] * B[t][j] for t in range(k)) for j in range(m)] for i in range(n)]


@pytest.mark.parametrize("W", [1, 2, 3])
def test_ag_gemm_brute_force(W):
    shards = [normal_bf16(900 + r, (2, 5), 1.0) for r in range(W)]
    b = normal_bf16(950, (5, 4), 1.0)
    A = [row for s in shards for row in _py(s)]
    ref = _bf_matmul(A, _py(b))
    got = oracle.ag_gemm(shards, b)
    assert np.allclose(got, np.array(ref), rtol=1e-13, atol=1e-13)


def test_ag_gemm_w1_is_plain_gemm():
    a = normal_bf16(11, (64, 48), 1.0)
    b = normal_bf16(12, (48, 40), 1.0)
    got = oracle.ag_gemm([a], b)
    ref = oracle.widen_bf16(a) @ oracle.widen_bf16(b)
    assert np.array_equal(got, ref)


def test_ag_gemm_equals_unsharded_and_gather_bits():
    full = normal_bf16(21, (96, 32), 1.0)
    b = normal_bf16(22, (32, 24), 1.0)
    shards = [full[i * 24:(i + 1) * 24] for i in range(4)]
    assert np.array_equal(oracle.ag_gather_bits(shards), full)
    assert np.allclose(oracle.ag_gemm(shards, b), _bf_matmul(_py(full), _py(b)), rtol=1e-13, atol=1e-13)


def test_ag_gemm_entries_match_full():
    inp = make_inputs("ag_gemm", 1, W=2, m_per_rank=128, n=256, k=256)
    full = oracle.ag_gemm(inp["a_shards"], inp["b"])
    rng = np.random.default_rng(0)
    rows = rng.integers(0, 256, 40)
    cols = rng.integers(0, 256, 40)
    got = oracle.ag_gemm_entries(inp["a_shards"], inp["b"], rows, cols)
    assert np.allclose(got, full[rows, cols], rtol=1e-12, atol=1e-12)


def test_gemm_rs_brute_force_and_closed_form():
    W, m, kr, n = 3, 6, 4, 5
    a = [normal_bf16(300 + p, (m, kr), 1.0) for p in range(W)]
    b = [normal_bf16(400 + p, (kr, n), 1.0) for p in range(W)]
    outs = oracle.gemm_rs(a, b)
    # brute force: sum over producers of each partial, then take the owner's rows
    S = [[0.0] * n for _ in range(m)]
    for p in range(W):
        P = _bf_matmul(_py(a[p]), _py(b[p]))
        for i in range(m):
            for j in range(n):
                S[i][j] += P[i][j]
    mo = m // W
    for o in range(W):
        assert np.allclose(outs[o], np.array(S[o * mo:(o + 1) * mo]), rtol=1e-13, atol=1e-13)
    # closed form: one GEMM with K = W*k_r on column-concat A and row-concat B
    Acat = np.concatenate([oracle.widen_bf16(x) for x in a], axis=1)
    Bcat = np.concatenate([oracle.widen_bf16(x) for x in b], axis=0)
    assert np.allclose(np.concatenate(outs, axis=0), Acat @ Bcat, rtol=1e-13, atol=1e-13)


def test_reduce_scatter_hand_brute_force_and_gemm_rs():
    # hand case, W = 2: owner 0 keeps row 0 of the sum, owner 1 row 1 (a swapped owner or a
    # dropped rank fails)
    p0 = np.array([[1.0, -2.0], [3.0, 4.0]], dtype=np.float32)
    p1 = np.array([[10.0, 20.0], [-30.0, 0.5]], dtype=np.float32)
    out = oracle.reduce_scatter([p0, p1])
    assert [o.tolist() for o in out] == [[[11.0, 18.0]], [[-27.0, 4.5]]]
    # brute force, W = 3, every element a sum over ranks in a Python loop
    rng = np.random.default_rng(3)
    parts = [rng.standard_normal((6, 5)).astype(np.float32) for _ in range(3)]
    out = oracle.reduce_scatter(parts)
    for o in range(3):
        for i in range(2):
            for j in range(5):
                acc = 0.0
                for p in range(3):
                    acc += float(parts[p][o * 2 + i][j])
                assert out[o][i][j] == acc
    # with the ranks' products as partials it is the GEMM + ReduceScatter (whose own pins are
    # the brute force and the column-concatenated GEMM above)
    inp = make_inputs("gemm_rs", 5, W=2, m=4, n=3, k_r=8)
    prods = [(oracle.widen_bf16(a) @ oracle.widen_bf16(b)).astype(np.float32) for a, b in zip(inp["a"], inp["b"])]
    for x, y in zip(oracle.reduce_scatter(prods), oracle.gemm_rs(inp["a"], inp["b"])):
        assert np.allclose(x, y, rtol=1e-6, atol=1e-7)


def test_gemm_rs_entries_match_full():
    W, m, kr, n = 4, 64, 32, 48
    a = [normal_bf16(500 + p, (m, kr), 1.0) for p in range(W)]
    b = [normal_bf16(600 + p, (kr, n), 1.0) for p in range(W)]
    outs = oracle.gemm_rs(a, b)
    rows = np.arange(0, 16, 3)
    cols = np.arange(0, 48, 7)[: len(rows)]
    for o in range(W):
        got = oracle.gemm_rs_entries(a, b, o, rows, cols)
        assert np.allclose(got, outs[o][rows, cols], rtol=1e-12, atol=1e-12)
        assert np.allclose(oracle.gemm_rs_rows(a, b, o, [5, 0, 15]), outs[o][[5, 0, 15]], rtol=1e-12, atol=1e-12)


def test_mlp2_brute_force():
    W, T, h, fr = 2, 4, 6, 3
    x = [normal_bf16(700 + r, (T // W, h), 1.0) for r in range(W)]
    w1 = [normal_bf16(710 + r, (h, fr), 0.5) for r in range(W)]
    w2 = [normal_bf16(720 + r, (fr, h), 0.5) for r in range(W)]
    outs = oracle.mlp2(x, w1, w2)
    X = [row for s in x for row in _py(s)]
    S = [[0.0] * h for _ in range(T)]
    for r in range(W):
        Hm = _bf_matmul(X, _py(w1[r]))
        Hm = [[0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in row] for row in Hm]
        P = _bf_matmul(Hm, _py(w2[r]))
        for i in range(T):
            for j in range(h):
                S[i][j] += P[i][j]
    mo = T // W
    for o in range(W):
        assert np.allclose(outs[o], np.array(S[o * mo:(o + 1) * mo]), rtol=1e-12, atol=1e-14)
    rows = [0, 1]
    cols = [2, 5]
    for o in range(W):
        got = oracle.mlp2_entries(x, w1, w2, o, rows, cols)
        assert np.allclose(got, outs[o][rows, cols], rtol=1e-12, atol=1e-14)
        # whole rows: the row sampler against the brute-force S
        assert np.allclose(oracle.mlp2_rows(x, w1, w2, o, [1, 0]), np.array(S[o * mo:(o + 1) * mo])[[1, 0]],
                           rtol=1e-12, atol=1e-14)
    # H_r against the brute-force GELU(X . W1_r)
    for r in range(W):
        Hm = [[0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in row] for row in _bf_matmul(X, _py(w1[r]))]
        assert np.allclose(oracle.mlp2_h(x, w1, r), np.array(Hm), rtol=1e-12, atol=1e-14)


def test_moe_route_ties_and_gates():
    logits = np.array([[1.0, 3.0, 3.0, 0.5], [2.0, 2.0, 2.0, 2.0]], dtype=np.float32)
    ex, g = oracle.moe_route(logits, 2)
    assert ex.tolist() == [[1, 2], [0, 1]]
    p0 = np.exp(np.array([1.0, 3.0, 3.0, 0.5]) - 3.0)
    p0 /= p0.sum()
    assert np.allclose(g[0], p0[[1, 2]], rtol=1e-15)
    assert np.allclose(g[1], [0.25, 0.25], rtol=1e-15)
    _, g2 = oracle.moe_route(logits, 2, renorm=True)
    assert np.allclose(g2.sum(axis=1), 1.0)


def test_moe_permute_bijection_and_stability():
    rng = np.random.default_rng(3)
    T, k, E = 300, 2, 16
    logits = rng.standard_normal((T, E)).astype(np.float32)
    ex, _ = oracle.moe_route(logits, k)
    counts, offsets, perm, inv = oracle.moe_permute(ex, E)
    assert counts.sum() == T * k and offsets[-1] == T * k
    assert sorted(perm.tolist()) == list(range(T * k))
    assert np.array_equal(inv[perm], np.arange(T * k))
    flat = ex.reshape(-1)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)  # stable: (t, j) order kept inside an expert
    # each token's two experts are distinct
    assert np.all(ex[:, 0] != ex[:, 1])


def test_moe_single_expert_is_dense_gated_mlp():
    T, H, F = 8, 16, 8
    x = normal_bf16(800, (T, H), 1.0)
    logits = normal_f32(801, (T, 1), 1.0)
    wg = normal_bf16(802, (1, H, F), 0.3)
    wu = normal_bf16(803, (1, H, F), 0.3)
    wd = normal_bf16(804, (1, F, H), 0.3)
    res = oracle.moe(x, logits, wg, wu, wd, topk=1)
    X = oracle.widen_bf16(x)
    dense = (oracle.silu(X @ oracle.widen_bf16(wg[0])) * (X @ oracle.widen_bf16(wu[0]))) @ oracle.widen_bf16(wd[0])
    assert np.allclose(res["gates"], 1.0)
    assert np.allclose(res["out"], dense, rtol=1e-13, atol=1e-13)


def test_moe_brute_force_tiny():
    T, H, E, F, k = 8, 16, 4, 8, 2
    x = normal_bf16(810, (T, H), 1.0)
    logits = normal_f32(811, (T, E), 1.0)
    wg = normal_bf16(812, (E, H, F), 0.3)
    wu = normal_bf16(813, (E, H, F), 0.3)
    wd = normal_bf16(814, (E, F, H), 0.3)
    res = oracle.moe(x, logits, wg, wu, wd, topk=k)
    X = _py(x)
    L = logits.astype(float).tolist()
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-L[t][e], e))[:k]
        mx = max(L[t])
        Z = sum(math.exp(v - mx) for v in L[t])
        acc = [0.0] * H
        for e in order:
            gate = math.exp(L[t][e] - mx) / Z
            G, U, D = _py(wg[e]), _py(wu[e]), _py(wd[e])
            hvec = []
            for f in range(F):
                gv = sum(X[t][i] * G[i][f] for i in range(H))
                uv = sum(X[t][i] * U[i][f] for i in range(H))
                hvec.append(gv / (1.0 + math.exp(-gv)) * uv)
            for j in range(H):
                acc[j] += gate * sum(hvec[f] * D[f][j] for f in range(F))
        assert np.allclose(res["out"][t], acc, rtol=1e-12, atol=1e-13)
    rows, ex2, g2 = oracle.moe_rows(x, logits, wg, wu, wd, k, [0, 5, 7])
    assert np.allclose(rows, res["out"][[0, 5, 7]], rtol=1e-12, atol=1e-13)


def test_static_map_brute_force():
    # brute force: walk the rows of each rank/channel and check the affine formulas
    for M, R, C, Tm in [(1024, 8, 2, 64), (8192, 8, 1, 128), (256, 2, 4, 32)]:
        mpr = M // R
        mpc = M // (R * C)
        for tid in range(M // Tm):
            lo, hi, rank, ch = oracle.static_tile_map(tid, M, R, C, Tm)
            rows = range(lo, hi)
            assert {r // mpr for r in rows} == {rank}
            assert {r // mpc for r in rows} == {ch}


def test_round_bf16_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to the even mantissa (1.0)
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5])
    assert oracle.round_bf16(x).tolist() == [1.0, 1.0 + 2.0 ** -6, -2.5]


def test_seeded_inputs_deterministic_and_scaled():
    a1 = make_inputs("ag_gemm", 1, W=2, m_per_rank=128, n=256, k=256)
    a2 = make_inputs("ag_gemm", 1, W=2, m_per_rank=128, n=256, k=256)
    assert all(np.array_equal(x, y) for x, y in zip(a1["a_shards"], a2["a_shards"]))
    assert np.array_equal(a1["b"], a2["b"])
    assert not np.array_equal(a1["a_shards"][0], a1["a_shards"][1])
    v = oracle.widen_bf16(a1["b"])
    assert abs(v.std() - 1.0 / 16.0) < 0.002 and abs(v.mean()) < 0.002


# ----------------------------------------------------------------------------- AG KV + self-attention
def _attn_brute(q, ks, vs):
    """Per-query loops with math.exp: softmax(q k^T / sqrt(d)) v over the rank-order gather."""
    Q = oracle.widen_bf16(q)
    K = np.concatenate([oracle.widen_bf16(k) for k in ks], axis=1)
    V = np.concatenate([oracle.widen_bf16(v) for v in vs], axis=1)
    H, L, d = Q.shape
    out = np.zeros_like(Q)
    for h in range(H):
        for i in range(L):
            s = [sum(Q[h, i, c] * K[h, j, c] for c in range(d)) / math.sqrt(d) for j in range(K.shape[1])]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            z = sum(w)
            for c in range(d):
                out[h, i, c] = sum(w[j] * V[h, j, c] for j in range(K.shape[1])) / z
    return out


def test_attention_matches_brute_force():
    inp = make_inputs("ag_attn", 41, W=3, heads=2, l_r=3, d=4)
    got = oracle.ag_attention(inp["q"], inp["k_shards"], inp["v_shards"])
    ref = _attn_brute(inp["q"], inp["k_shards"], inp["v_shards"])
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_attention_gather_is_rank_order_concatenation():
    inp = make_inputs("ag_attn", 42, W=4, heads=3, l_r=5, d=8)
    g = oracle.attn_gather(inp["k_shards"])
    assert g.shape == (3, 20, 8)
    for r in range(4):
        assert np.array_equal(g[:, 5 * r:5 * (r + 1)], inp["k_shards"][r])


def test_attention_zero_query_is_mean_of_values():
    inp = make_inputs("ag_attn", 43, W=2, heads=2, l_r=6, d=8)
    q = np.zeros_like(inp["q"])
    got = oracle.ag_attention(q, inp["k_shards"], inp["v_shards"])
    V = oracle.widen_bf16(oracle.attn_gather(inp["v_shards"]))
    assert np.allclose(got, np.broadcast_to(V.mean(axis=1, keepdims=True), got.shape), rtol=0, atol=1e-14)


def test_attention_dominant_key_selects_its_value():
    # one key is 64 times the query direction: its score exceeds every other by > 100,
    # so the output is that key's value row to within exp(-100)
    from seeded_inputs import f32_to_bf16_bits
    inp = make_inputs("ag_attn", 44, W=2, heads=1, l_r=4, d=16)
    qf = oracle.widen_bf16(inp["q"])
    ks = [oracle.widen_bf16(k).copy() for k in inp["k_shards"]]
    ks[1][0, 2] = 64.0 * qf[0, 1]
    kb = [f32_to_bf16_bits(k.astype(np.float32)) for k in ks]
    got = oracle.ag_attention(inp["q"], kb, inp["v_shards"])
    assert np.allclose(got[0, 1], oracle.widen_bf16(inp["v_shards"][1])[0, 2], atol=1e-12)


def test_attention_invariant_to_duplicated_context_and_shard_order():
    inp = make_inputs("ag_attn", 45, W=3, heads=2, l_r=4, d=8)
    q, ks, vs = inp["q"], inp["k_shards"], inp["v_shards"]
    base = oracle.ag_attention(q, ks, vs)
    assert np.allclose(oracle.ag_attention(q, ks + ks, vs + vs), base, rtol=1e-12, atol=1e-13)
    order = [2, 0, 1]
    assert np.allclose(oracle.ag_attention(q, [ks[i] for i in order], [vs[i] for i in order]), base,
                       rtol=1e-12, atol=1e-13)


def test_attention_rows_match_full():
    inp = make_inputs("ag_attn", 46, W=2, heads=3, l_r=8, d=8)
    full = oracle.ag_attention(inp["q"], inp["k_shards"], inp["v_shards"])
    part = oracle.ag_attention_rows(inp["q"], inp["k_shards"], inp["v_shards"], [2, 0], [5, 1])
    assert np.allclose(part, full[[2, 0]][:, [5, 1]], rtol=1e-13, atol=1e-14)
