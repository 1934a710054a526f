"""Plain CPU oracle in float64 for the tile-centric overlapped GEMM path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.  It
shares no code with the CUDA path and never runs on the product path.

Every function states the passage it follows.  Pages:
  [TL]  "TileLink: Generating Efficient Compute-Communication Overlapping Kernels
         using Tile-Centric Primitives" (ar5iv 2503.20313)
  [TD]  "Triton-distributed: Programming Overlapping Kernels on Distributed AI
         Systems with the Triton Compiler" (arXiv 2504.19442)
  [RA]  "Resource-aware Computation-Communication Overlap for multi-GPU ML
         Workloads" (three abstracts: CTA-pipelining, CommFuse, MoE tile overlap)

Arithmetic: bf16 inputs are widened exactly to float64; products of two bf16
values are exact in float64; sums are float64.  Matrix products use numpy's
float64 matmul as the one library primitive (no blocking or reordering of our
own).  The transcendental steps (erf, exp) use scipy/numpy float64 routines.

Pinning (tests/test_oracle_pins.py): brute-force loops on tiny shapes, the W=1
reduction to a plain GEMM, equality with the unsharded GEMM, the column-concat
closed form of the reduce-scatter, hand-derived integer fixtures in
tests/golden/, textbook values of Phi(1) and the logistic function, and
bijection/ordering checks of the MoE permutation.  No function here is
"parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

try:  # erf for exact GELU; scipy is present on both the build host and the GPU host
    from scipy.special import erf as _erf
except Exception:  # pragma: no cover - fallback keeps the oracle usable without scipy
    _erf = np.vectorize(math.erf, otypes=[np.float64])

__all__ = [
    "widen_bf16", "ag_gather_bits", "ag_gemm", "ag_gemm_entries", "gemm_rs", "reduce_scatter",
    "gemm_rs_entries", "gemm_rs_rows", "gelu", "silu", "mlp2", "mlp2_entries", "mlp2_rows", "mlp2_h", "moe_route", "moe_permute",
    "moe", "moe_rows", "static_tile_map", "round_bf16", "attn_gather", "ag_attention", "ag_attention_rows",
]


# ----------------------------------------------------------------------------- decoding
def widen_bf16(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly (sign/exponent/8-bit mantissa kept)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(x) -> np.ndarray:
    """float64 -> nearest bf16 value (ties to even), returned as float64.

    Used only for the optional 'mirror' diagnosis of the MLP chain (the GPU keeps
    the intermediate activation in bf16); the default oracle never rounds.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------- AllGather + GEMM
def ag_gather_bits(a_shards) -> np.ndarray:
    """The gathered operand of AllGather, as raw bf16 bits.

    [TD] §3.2 Alg. 2 (pull-mode one-sided AllGather): shard r lands at offset
    r*|L| of the symmetric buffer, i.e. the gathered matrix is the row
    concatenation of the shards in rank order.  Bit copy, no arithmetic.
    """
    return np.concatenate([np.ascontiguousarray(a, dtype=np.uint16) for a in a_shards], axis=0)


def ag_gemm(a_shards, b) -> np.ndarray:
    """C = AllGather(A) . B in float64.

    [TL] §2.1 (tensor-parallel FFN: input gathered from every rank, then GEMM
    with the local weight shard) and [TD] §3.2 Alg. 2 (rank-order placement):
    A = [A_0; A_1; ...; A_{W-1}],  C[i, j] = sum_k A[i, k] * B[k, j].
    """
    A = widen_bf16(ag_gather_bits(a_shards))
    B = widen_bf16(b)
    return A @ B


def ag_gemm_entries(a_shards, b, rows, cols) -> np.ndarray:
    """Selected entries C[rows[i], cols[i]] of ag_gemm, each as its own dot product."""
    m_per = np.asarray(a_shards[0]).shape[0]
    out = np.empty(len(rows), dtype=np.float64)
    B = b
    for i, (r, c) in enumerate(zip(rows, cols)):
        shard = a_shards[r // m_per]
        arow = widen_bf16(shard[r % m_per])
        bcol = widen_bf16(np.ascontiguousarray(B[:, c]))
        out[i] = float(np.dot(arow, bcol))
    return out


# ----------------------------------------------------------------------------- GEMM + ReduceScatter
def gemm_rs(a_list, b_list) -> list:
    """out_o = rows [o*M/W, (o+1)*M/W) of S = sum_p A_p . B_p, float64.

    [TD] §3.3 Alg. 3 (one-sided push-mode ReduceScatter): every rank's partial
    is pushed to the owner's slot and the owner sums R = R + T[r] over all r;
    [TL] §2.1 (tensor-parallel FFN: partial results reduced and scattered).
    """
    W = len(a_list)
    S = None
    for p in range(W):
        P = widen_bf16(a_list[p]) @ widen_bf16(b_list[p])
        S = P if S is None else S + P
    M = S.shape[0]
    assert M % W == 0
    mo = M // W
    return [S[o * mo:(o + 1) * mo] for o in range(W)]


def reduce_scatter(partials) -> list:
    """out_o = rows [o*M/W, (o+1)*M/W) of P_0 + P_1 + ... + P_{W-1}, float64.

    [TD] §3.3 Alg. 3 (one-sided push-mode ReduceScatter) without a GEMM in
    front of it: rank p's partial T[p] reaches the owner, which accumulates
    R = R + T[p] over every rank and keeps its own rows.  The partials are
    float32 arrays (the GPU path's message precision), widened exactly.
    """
    W = len(partials)
    S = None
    for p in range(W):
        P = np.asarray(partials[p], dtype=np.float32).astype(np.float64)
        S = P if S is None else S + P
    M = S.shape[0]
    assert M % W == 0
    mo = M // W
    return [S[o * mo:(o + 1) * mo] for o in range(W)]


def gemm_rs_entries(a_list, b_list, owner, rows, cols) -> np.ndarray:
    """Selected entries out_owner[rows[i], cols[i]], each summed over producers p = 0..W-1."""
    W = len(a_list)
    M = np.asarray(a_list[0]).shape[0]
    mo = M // W
    out = np.zeros(len(rows), dtype=np.float64)
    for i, (r, c) in enumerate(zip(rows, cols)):
        gr = owner * mo + r
        acc = 0.0
        for p in range(W):
            acc += float(np.dot(widen_bf16(a_list[p][gr]), widen_bf16(np.ascontiguousarray(b_list[p][:, c]))))
        out[i] = acc
    return out


def gemm_rs_rows(a_list, b_list, owner, rows) -> np.ndarray:
    """Whole rows out_owner[rows[i], :], each the plain sum over producers p = 0..W-1 of
    (row of A_p) . B_p (the definition of gemm_rs, one row at a time)."""
    W = len(a_list)
    mo = np.asarray(a_list[0]).shape[0] // W
    gr = [owner * mo + r for r in rows]
    out = None
    for p in range(W):
        part = widen_bf16(np.asarray(a_list[p])[gr]) @ widen_bf16(b_list[p])
        out = part if out is None else out + part
    return out


# ----------------------------------------------------------------------------- activations
def gelu(x) -> np.ndarray:
    """Exact GELU, 0.5 * x * (1 + erf(x / sqrt(2))), float64.

    [TL] §7.2 names a GELU activation between the two MLP GEMMs; the exact
    (erf) form is the definition of GELU.
    """
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))


def silu(z) -> np.ndarray:
    """SiLU(z) = z / (1 + exp(-z)), float64 ([TL] §7.2 names SiLUMul)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


# ----------------------------------------------------------------------------- 2-layer MLP chain
def mlp2(x_shards, w1, w2, mirror_bf16_h: bool = False) -> list:
    """Tensor-parallel 2-layer MLP: AG + GEMM -> GELU -> GEMM + RS, float64.

    [TL] §2.1 (FFN = AllGather + GEMM with column-sharded W1, activation, GEMM
    with row-sharded W2, ReduceScatter) and [RA] CTA-pipelining (2-layer GEMM
    representing the MLP).  X = [X_0; ...; X_{W-1}];  H_r = GELU(X . W1_r);
    S = sum_r H_r . W2_r;  out_o = rows o of S.
    """
    X = widen_bf16(ag_gather_bits(x_shards))
    W = len(w1)
    S = None
    for r in range(W):
        H = gelu(X @ widen_bf16(w1[r]))
        if mirror_bf16_h:
            H = round_bf16(H)
        P = H @ widen_bf16(w2[r])
        S = P if S is None else S + P
    mo = S.shape[0] // W
    return [S[o * mo:(o + 1) * mo] for o in range(W)]


def mlp2_entries(x_shards, w1, w2, owner, rows, cols) -> np.ndarray:
    """Selected entries of out_owner: the full GELU row of H_r is formed for each needed row."""
    W = len(w1)
    T_per = np.asarray(x_shards[0]).shape[0]
    out = np.zeros(len(rows), dtype=np.float64)
    cache = {}
    for i, (r, c) in enumerate(zip(rows, cols)):
        gr = owner * T_per + r          # row of S == row of the gathered X
        if gr not in cache:
            xrow = widen_bf16(x_shards[gr // T_per][gr % T_per])
            cache[gr] = [gelu(xrow @ widen_bf16(w1[q])) for q in range(W)]
        acc = 0.0
        for q in range(W):
            acc += float(np.dot(cache[gr][q], widen_bf16(np.ascontiguousarray(w2[q][:, c]))))
        out[i] = acc
    return out


def mlp2_rows(x_shards, w1, w2, owner, rows) -> np.ndarray:
    """Whole rows out_owner[rows[i], :]: for each row the gathered X row, its GELU rows of
    every H_r, and sum_r H_r row . W2_r (the definition of mlp2, one row at a time)."""
    W = len(w1)
    T_per = np.asarray(x_shards[0]).shape[0]
    X = widen_bf16(np.stack([np.asarray(x_shards[(owner * T_per + r) // T_per])[(owner * T_per + r) % T_per]
                             for r in rows]))
    out = None
    for q in range(W):
        part = gelu(X @ widen_bf16(w1[q])) @ widen_bf16(w2[q])
        out = part if out is None else out + part
    return out


def mlp2_h(x_shards, w1, rank) -> np.ndarray:
    """The intermediate H_rank = GELU(X . W1_rank) of the MLP chain, float64 ([TL] §2.1)."""
    X = widen_bf16(ag_gather_bits(x_shards))
    return gelu(X @ widen_bf16(w1[rank]))


# ----------------------------------------------------------------------------- MoE
def moe_route(logits, topk: int, renorm: bool = False):
    """Top-k expert choice and softmax gates per token.

    The pages leave the router open ([TL] §4.1 dynamic mapping: "dynamic routing
    determines the data distribution"; [TD] Table 4 gives only E and topk).
    Reading taken: experts = the k largest logits, descending, ties to the lower
    expert index; p = softmax over all E logits (float64, max-subtracted);
    gate_k = p[expert_k]; no renormalisation unless renorm=True.
    Returns (experts int32 [T, k], gates float64 [T, k]).
    """
    L = np.asarray(logits, dtype=np.float32)
    T, E = L.shape
    experts = np.empty((T, topk), dtype=np.int32)
    gates = np.empty((T, topk), dtype=np.float64)
    for t in range(T):
        row = L[t]
        # stable sort of -logit: equal logits keep ascending expert order
        order = np.argsort(-row.astype(np.float64), kind="stable")
        sel = order[:topk]
        z = row.astype(np.float64)
        p = np.exp(z - z.max())
        p = p / p.sum()
        g = p[sel]
        if renorm:
            g = g / g.sum()
        experts[t] = sel
        gates[t] = g
    return experts, gates


def moe_permute(experts, E: int):
    """Stable expert-major permutation of the T*k assignments.

    [TL] §4.1 dynamic mapping (lookup tables f_S_low/f_S_high/f_R filled at run
    time by the routing).  Assignment a = t*k + j goes to expert experts[t, j];
    assignments are ordered by (expert, t, j).  Returns counts[E],
    offsets[E+1] (exclusive scan), perm[T*k] (perm[pos] = a) and inv[T*k]
    (inv[a] = pos).
    """
    ex = np.asarray(experts, dtype=np.int64).reshape(-1)
    n = ex.shape[0]
    counts = np.zeros(E, dtype=np.int64)
    for e in ex:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:-1].copy()
    perm = np.empty(n, dtype=np.int64)
    inv = np.empty(n, dtype=np.int64)
    for a in range(n):          # a increases in (t, j) order -> stable within an expert
        e = ex[a]
        pos = fill[e]
        fill[e] += 1
        perm[pos] = a
        inv[a] = pos
    return counts, offsets, perm, inv


def moe(x, logits, w_gate, w_up, w_down, topk: int, renorm: bool = False):
    """MoE layer with SiLU-gated experts and gate-weighted combine, float64.

    [TL] §7.2 (MoE = Gather + GroupGEMM, then GroupGEMM + Scatter + TopK
    reduce); [RA] MoE tile-signalled overlap (expert compute, then the return
    step puts each expert output row back at its token).  For every assignment
    a = (t, j) with expert e:  y_a = (SiLU(x_t Wg_e) * (x_t Wu_e)) Wd_e;
    out[t] = sum_j gate[t, j] * y_(t, j).
    Returns dict(out [T,H], experts, gates, counts, offsets, perm, inv, y [T*k,H] in assignment order).
    """
    X = widen_bf16(x)
    T, H = X.shape
    E = np.asarray(w_gate).shape[0]
    experts, gates = moe_route(logits, topk, renorm)
    counts, offsets, perm, inv = moe_permute(experts, E)
    y = np.zeros((T * topk, H), dtype=np.float64)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        assign = perm[lo:hi]
        toks = assign // topk
        Xe = X[toks]
        Wg = widen_bf16(w_gate[e]); Wu = widen_bf16(w_up[e]); Wd = widen_bf16(w_down[e])
        h = silu(Xe @ Wg) * (Xe @ Wu)
        y[assign] = h @ Wd
    out = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for j in range(topk):
            out[t] += gates[t, j] * y[t * topk + j]
    return dict(out=out, experts=experts, gates=gates, counts=counts, offsets=offsets,
                perm=perm, inv=inv, y=y)


def moe_rows(x, logits, w_gate, w_up, w_down, topk: int, tokens, renorm: bool = False):
    """out[t] for selected tokens only (same definition as moe(), one token at a time)."""
    X = widen_bf16(x)
    experts, gates = moe_route(np.asarray(logits)[list(tokens)], topk, renorm)
    rows = []
    for i, t in enumerate(tokens):
        acc = np.zeros(X.shape[1], dtype=np.float64)
        for j in range(topk):
            e = int(experts[i, j])
            h = silu(X[t] @ widen_bf16(w_gate[e])) * (X[t] @ widen_bf16(w_up[e]))
            acc += gates[i, j] * (h @ widen_bf16(w_down[e]))
        rows.append(acc)
    return np.stack(rows), experts, gates


# ----------------------------------------------------------------------------- tile-centric mapping
def static_tile_map(tile_id: int, M: int, R: int, C: int, Tm: int):
    """Static (affine) tile-centric mapping for pull-mode AllGather + GEMM.

    [TL] §4.1, static mapping equations: M_per_rank = ceil(M / R),
    M_per_channel = ceil(M / (R*C)), range_M = [id*Tm, id*Tm + Tm),
    src_rank = floor(id / floor(M_per_rank / Tm)),
    channel = floor(id / floor(M_per_channel / Tm)).
    Returns (range_lo, range_hi, src_rank, channel).
    """
    m_per_rank = -(-M // R)
    m_per_channel = -(-M // (R * C))
    lo = tile_id * Tm
    hi = lo + Tm
    src_rank = tile_id // (m_per_rank // Tm)
    channel = tile_id // (m_per_channel // Tm)
    return lo, hi, src_rank, channel


# ----------------------------------------------------------------------------- AG KV + self-attention
def attn_gather(shards) -> np.ndarray:
    """Sequence-parallel context gather: K (or V) shards [heads, L_r, d] of ranks 0..W-1
    concatenated along the sequence in rank order, per head ([TL] §5, AllGather KV +
    self-attention: the KV cache sequence S split into W equal parts, one per rank).
    Returns the bf16 bit patterns [heads, W * L_r, d]."""
    return np.concatenate([np.ascontiguousarray(x, dtype=np.uint16) for x in shards], axis=1)


def ag_attention(q, k_shards, v_shards) -> np.ndarray:
    """Self-attention of one rank's queries over the gathered context ([TL] §2 and §7.2,
    sequence-parallel self-attention; the pages give no mask, read as non-causal):
        O[h] = softmax(Q[h] K[h]^T / sqrt(d)) V[h],  K, V = attn_gather(shards).
    q: bf16 bits [heads, L_q, d]; shards: bf16 bits [heads, L_r, d].  float64, softmax
    with the row maximum subtracted."""
    Q = widen_bf16(q)
    K = widen_bf16(attn_gather(k_shards))
    V = widen_bf16(attn_gather(v_shards))
    d = Q.shape[-1]
    S = np.matmul(Q, np.swapaxes(K, 1, 2)) / math.sqrt(d)
    S -= S.max(axis=-1, keepdims=True)
    P = np.exp(S)
    P /= P.sum(axis=-1, keepdims=True)
    return np.matmul(P, V)


def ag_attention_rows(q, k_shards, v_shards, heads, rows) -> np.ndarray:
    """ag_attention at the query rows `rows` of the heads `heads` only (same arithmetic);
    returns [len(heads), len(rows), d]."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    hs = list(heads)
    sub = lambda x: np.ascontiguousarray(x, dtype=np.uint16)[hs]
    return ag_attention(sub(q)[:, list(rows)], [sub(k) for k in k_shards], [sub(v) for v in v_shards])
