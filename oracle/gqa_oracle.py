"""fp64 oracle of grouped-query attention (GQA) under head sharding.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA library never
imports or calls this module.

H query heads share Hkv key/value heads (H % Hkv == 0); query head t uses key/value
head t // (H / Hkv) -- consecutive query heads form a group [张量并行 notes, §相关分析,
GQA]. The tensor-parallel degree N may go up to H (H % N == 0). When N <= Hkv
(Hkv % N == 0) shard i owns H/N query heads and Hkv/N key/value heads. When N > Hkv
(N % Hkv == 0) each key/value head is replicated on r = N / Hkv shards: shard i owns
H/N query heads, all in group i // r, and a copy of that group's key/value weights;
the replicas' weight gradients are summed (an all-reduce among them) so the copies
stay identical -- the synchronisation the notes call for.

Sharded weight layout (P2's per-rank column-parallel QKV, whose output is reshaped to
[3, heads_per_rank, head_dim]): shard i's columns are one block
[W_q of its query heads | W_k of its key/value heads | W_v of the same], the blocks in
shard order.
"""
from __future__ import annotations

import math

import numpy as np

from . import tp_oracle as T


def gqa_split(H, Hkv, N):
    """(query heads per shard, key/value heads per shard, replication factor r)."""
    if H % Hkv or H % N:
        raise ValueError("need H % Hkv == 0 and H % N == 0")
    if N <= Hkv:
        if Hkv % N:
            raise ValueError("N <= Hkv needs Hkv % N == 0")
        return H // N, Hkv // N, 1
    if N % Hkv:
        raise ValueError("N > Hkv needs N % Hkv == 0")
    return H // N, 1, N // Hkv


def shard_heads(H, Hkv, N, i):
    """Global query heads and key/value heads of shard i."""
    hq, hkv, r = gqa_split(H, Hkv, N)
    q = list(range(i * hq, (i + 1) * hq))
    kv = list(range(i * hkv, (i + 1) * hkv)) if r == 1 else [i // r]
    return q, kv


def gqa_pack(Wq, Wk, Wv, H, Hkv, N):
    """Sharded QKV weight (h, N * (hq + 2 hkv) * d) from the full W_q (h, H d),
    W_k, W_v (h, Hkv d); replicated key/value heads are copied into every replica."""
    d = Wq.shape[1] // H
    blocks = []
    for i in range(N):
        q, kv = shard_heads(H, Hkv, N, i)
        cols = lambda W, heads: [W[:, t * d:(t + 1) * d] for t in heads]
        blocks += cols(Wq, q) + cols(Wk, kv) + cols(Wv, kv)
    return np.concatenate(blocks, axis=1)


def gqa_attention_unsplit(xn, Wq, Wk, Wv, b, s, H, Hkv, causal=False):
    """Single-device GQA: Q = xn W_q, K = xn W_k, V = xn W_v; query head t attends
    with key/value head t // (H / Hkv). Returns O (M, H d)."""
    d = Wq.shape[1] // H
    g = H // Hkv
    Q, K, V = xn @ Wq, xn @ Wk, xn @ Wv
    O = np.zeros((xn.shape[0], H * d))
    for t in range(H):
        j = t // g
        for bb in range(b):
            r = slice(bb * s, (bb + 1) * s)
            O[r, t * d:(t + 1) * d] = T.attention_head_fwd(
                Q[r, t * d:(t + 1) * d], K[r, j * d:(j + 1) * d], V[r, j * d:(j + 1) * d],
                causal)[0]
    return O


def gqa_block_unsplit(x, b, s, gamma, beta, Wq, Wk, Wv, Wo, H, Hkv, causal=False):
    """out = x + GQA(LN(x)) W_o on one device."""
    xn = T.layernorm_fwd(x, gamma, beta)[0]
    return x + gqa_attention_unsplit(xn, Wq, Wk, Wv, b, s, H, Hkv, causal) @ Wo


def _shard_views(H, Hkv, N, d):
    hq, hkv, _ = gqa_split(H, Hkv, N)
    Ws = (hq + 2 * hkv) * d
    return hq, hkv, Ws


def gqa_attention_fwd(QKV, b, s, H, Hkv, N, causal=False):
    """The attention core on the sharded QKV (M, N S): shard i's local query head tl
    attends with its local key/value head tl // g, every batch element on its own, each
    head by `tp_oracle.attention_head_fwd` [Megatron-LM 实战 04, TPAttention; 张量并行
    notes, §相关分析, GQA]. Returns O (M, H d), the heads in order."""
    M = QKV.shape[0]
    hq, hkv, _ = gqa_split(H, Hkv, N)
    d = QKV.shape[1] // (N * (hq + 2 * hkv))
    Ws = (hq + 2 * hkv) * d
    g = hq // hkv
    O = np.zeros((M, H * d))
    for i in range(N):
        Qi = QKV[:, i * Ws:(i + 1) * Ws]
        for tl in range(hq):
            kl = tl // g
            for bb in range(b):
                r = slice(bb * s, (bb + 1) * s)
                q = Qi[r, tl * d:(tl + 1) * d]
                k = Qi[r, (hq + kl) * d:(hq + kl + 1) * d]
                v = Qi[r, (hq + hkv + kl) * d:(hq + hkv + kl + 1) * d]
                O[r, (i * hq + tl) * d:(i * hq + tl + 1) * d] = T.attention_head_fwd(
                    q, k, v, causal)[0]
    return O


def gqa_attention_bwd(QKV, dO, b, s, H, Hkv, N, causal=False):
    """Backward of `gqa_attention_fwd`: dQKV (M, N S) in the same layout, each head by
    `tp_oracle.attention_head_bwd`; a key/value head's gradient sums the contributions
    of its shard's query heads that use it (a replica's share when N > Hkv; the
    replicas' all-reduce is the block's, in `gqa_block_bwd`)."""
    d = dO.shape[1] // H
    hq, hkv, Ws = _shard_views(H, Hkv, N, d)
    g = hq // hkv
    dQKV = np.zeros_like(QKV)
    for i in range(N):
        Qi = QKV[:, i * Ws:(i + 1) * Ws]
        dQi = dQKV[:, i * Ws:(i + 1) * Ws]
        dOi = dO[:, i * hq * d:(i + 1) * hq * d]
        for tl in range(hq):
            kl = tl // g
            qc = slice(tl * d, (tl + 1) * d)
            kc = slice((hq + kl) * d, (hq + kl + 1) * d)
            vc = slice((hq + hkv + kl) * d, (hq + hkv + kl + 1) * d)
            for bb in range(b):
                rr = slice(bb * s, (bb + 1) * s)
                dq, dk, dv = T.attention_head_bwd(Qi[rr, qc], Qi[rr, kc], Qi[rr, vc],
                                                  dOi[rr, qc], causal)
                dQi[rr, qc] += dq
                dQi[rr, kc] += dk
                dQi[rr, vc] += dv
    return dQKV


def gqa_block_fwd(x, b, s, gamma, beta, Wsh, Wo, H, Hkv, N, causal=False):
    """Head-sharded GQA block, shard by shard: QKV_i = LN(x) Wsh_i (column-parallel),
    attention on shard i's query heads with its (possibly replicated) key/value heads,
    Z_i = O_i W_o,i (row block i), out = x + sum_i Z_i. Returns xn, QKV (all shards'
    blocks side by side), O (heads in order), out."""
    d = Wo.shape[0] // H
    hq, hkv, Ws = _shard_views(H, Hkv, N, d)
    xn = T.layernorm_fwd(x, gamma, beta)[0]
    QKV = np.concatenate([xn @ Wsh[:, i * Ws:(i + 1) * Ws] for i in range(N)], axis=1)
    O = gqa_attention_fwd(QKV, b, s, H, Hkv, N, causal)
    rows = lambda i: slice(i * hq * d, (i + 1) * hq * d)
    parts = [O[:, rows(i)] @ Wo[rows(i), :] for i in range(N)]
    return {"xn": xn, "QKV": QKV, "O": O, "out": T.shard_reduce(parts, residual=x)}


def gqa_block_bwd(x, b, s, gamma, beta, Wsh, Wo, H, Hkv, N, dout, causal=False):
    """Backward of `gqa_block_fwd`, shard by shard. Shard i: dO_i = dout W_o,i^T;
    attention backward over its query heads -- a key/value head's gradient sums the
    contributions of the shard's query heads that use it; dWsh_i = xn^T dQKV_i;
    dW_o,i = O_i^T dout. The f-backward sums dxn = sum_i dQKV_i Wsh_i^T over the shards,
    then LN backward (+ dout). Finally the replicas of each key/value head add their
    weight gradients and every replica takes the sum (the all-reduce that keeps the
    copies identical)."""
    d = Wo.shape[0] // H
    hq, hkv, Ws = _shard_views(H, Hkv, N, d)
    _, _, r = gqa_split(H, Hkv, N)
    f = gqa_block_fwd(x, b, s, gamma, beta, Wsh, Wo, H, Hkv, N, causal)
    xn, QKV, O = f["xn"], f["QKV"], f["O"]
    rows = lambda i: slice(i * hq * d, (i + 1) * hq * d)
    dWo = np.zeros_like(Wo)
    dO = np.zeros_like(O)
    for i in range(N):
        dO[:, rows(i)] = dout @ Wo[rows(i), :].T
        dWo[rows(i), :] = O[:, rows(i)].T @ dout
    dQKV = gqa_attention_bwd(QKV, dO, b, s, H, Hkv, N, causal)
    dWsh = np.zeros_like(Wsh)
    dxparts = []
    for i in range(N):
        dQi = dQKV[:, i * Ws:(i + 1) * Ws]
        dWsh[:, i * Ws:(i + 1) * Ws] = xn.T @ dQi
        dxparts.append(dQi @ Wsh[:, i * Ws:(i + 1) * Ws].T)
    dxn = T.shard_reduce(dxparts)
    dx, dg, db = T.layernorm_bwd(x, gamma, dxn)
    if r > 1:  # all-reduce of each replicated key/value head's weight gradient
        for j in range(Hkv):
            reps = [i for i in range(N) if i // r == j]
            for off in (hq * d, (hq + hkv) * d):
                cols = [slice(i * Ws + off, i * Ws + off + d) for i in reps]
                tot = T.shard_reduce([dWsh[:, c] for c in cols])
                for c in cols:
                    dWsh[:, c] = tot
    return {"dx": dx + dout, "dgamma": dg, "dbeta": db, "dWqkv": dWsh, "dWo": dWo}


def gqa_unpack_grad(dWsh, H, Hkv, N, d):
    """Full dW_q, dW_k, dW_v from the sharded gradient (any replica's copy of a
    key/value head: after the all-reduce they are equal)."""
    hq, hkv, Ws = _shard_views(H, Hkv, N, d)
    h = dWsh.shape[0]
    dWq, dWk, dWv = np.zeros((h, H * d)), np.zeros((h, Hkv * d)), np.zeros((h, Hkv * d))
    for i in range(N):
        q, kv = shard_heads(H, Hkv, N, i)
        B = dWsh[:, i * Ws:(i + 1) * Ws]
        for a, t in enumerate(q):
            dWq[:, t * d:(t + 1) * d] = B[:, a * d:(a + 1) * d]
        for a, j in enumerate(kv):
            dWk[:, j * d:(j + 1) * d] = B[:, (hq + a) * d:(hq + a + 1) * d]
            dWv[:, j * d:(j + 1) * d] = B[:, (hq + hkv + a) * d:(hq + hkv + a + 1) * d]
    return dWq, dWk, dWv
