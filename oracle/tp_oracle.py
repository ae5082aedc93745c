"""fp64 oracle: the Megatron-style tensor-parallel linear block, written out plainly.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA library never
imports or calls this module.

Conventions (all arrays float64, row-major):
  X : (M, h) activations, M = b*s tokens               -- "X: (b, s, h), W: (h, h')"
  W : (h, h') weights, Y = X @ W                        [张量并行 notes, §基本思想]
  column shard i of W  = columns [i*h'/N, (i+1)*h'/N)   [张量并行 notes, §两个矩阵相乘, column split of B]
  row shard i of W     = rows    [i*h/N,  (i+1)*h/N)    [张量并行 notes, §两个矩阵相乘, row split of A]
Shards are contiguous blocks taken in shard order; every shard is a slice of one
seeded full weight, so the sharded result must equal the unsplit one.

Where the pages leave a step open, the reading taken is stated at the function.
"""
from __future__ import annotations

import math

import numpy as np

try:  # scipy is on both machines; keep a slow exact fallback anyway
    from scipy.special import erf as _erf
except Exception:  # pragma: no cover
    _erf = np.vectorize(math.erf, otypes=[np.float64])

SQRT2 = math.sqrt(2.0)
INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)
LN_EPS = 1e-5


# ---------------------------------------------------------------- elementwise

def gelu(x):
    """Exact GELU: x * Phi(x) = x * 1/2 * [1 + erf(x / sqrt(2))].

    [张量并行 notes, §MLP 层的并行化, "GELU 的标准计算公式"]. The erf form is used,
    not the tanh approximation.
    """
    x = np.asarray(x, dtype=np.float64)
    return x * 0.5 * (1.0 + _erf(x / SQRT2))


def gelu_prime(x):
    """d/dx GELU(x) = Phi(x) + x * phi(x), phi the standard normal density.

    Differentiates the formula of [张量并行 notes, §MLP 层的并行化].
    """
    x = np.asarray(x, dtype=np.float64)
    cdf = 0.5 * (1.0 + _erf(x / SQRT2))
    pdf = INV_SQRT_2PI * np.exp(-0.5 * x * x)
    return cdf + x * pdf


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    ex = np.exp(x[~pos])
    out[~pos] = ex / (1.0 + ex)
    return out


def silu(x):
    """SiLU(x) = x * sigmoid(x).

    The pages name the SwiGLU weights W_gate / W_up without writing the
    function out [20260402-parallelism, §1 Tensor Parallelism]; the reading
    taken is the usual one: A = SiLU(X W_gate) * (X W_up), elementwise.
    """
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


# ---------------------------------------------------------------- shards

def col_shards(W, N):
    """Column blocks W_1..W_N of W (h x h'), in shard order.

    [张量并行 notes, §基本思想, "按列拆分 B"]; [Infra: Tensor Parallel, Column-wise TP].
    """
    W = np.asarray(W)
    if W.shape[1] % N:
        raise ValueError("h' must be divisible by N")
    w = W.shape[1] // N
    return [W[:, i * w:(i + 1) * w] for i in range(N)]


def row_shards(W, N):
    """Row blocks W_1..W_N of W (h x h'), in shard order.

    [张量并行 notes, §基本思想, "按行拆分 A"]; [Infra: Tensor Parallel, Row-wise TP].
    """
    W = np.asarray(W)
    if W.shape[0] % N:
        raise ValueError("h must be divisible by N")
    w = W.shape[0] // N
    return [W[i * w:(i + 1) * w, :] for i in range(N)]


# ---------------------------------------------------------------- linear layers

def col_linear(X, W, N):
    """Column-parallel linear: every shard reads the whole X (broadcast) and
    computes Y_i = X W_i; the concatenation [Y_1 ... Y_N] is the all-gather.

    [张量并行 notes, §并行化矩阵乘法运算, 列并行]; [Infra: Tensor Parallel, Column-wise TP].
    Returns the list of shard outputs.
    """
    return [X @ Wi for Wi in col_shards(W, N)]


def row_partials(X, W, N):
    """Row-parallel linear before the reduction: X is split by column
    (scatter), W by row, shard i computes X_i W_i.

    [张量并行 notes, §并行化矩阵乘法运算, 行并行]; [Infra: Tensor Parallel, Row-wise TP].
    """
    return [Xi @ Wi for Xi, Wi in zip(col_shards(X, N), row_shards(W, N))]


def shard_reduce(partials, residual=None):
    """The all-reduce stand-in: Z = sum_i Z_i, shards summed in order 0..N-1,
    plus an optional residual.

    [张量并行 notes, §MLP 层的并行化, "g 的 forward 计算 ... all-reduce，相加得到 Z"].
    """
    Z = np.zeros_like(np.asarray(partials[0], dtype=np.float64))
    for P in partials:
        Z = Z + P
    if residual is not None:
        Z = Z + residual
    return Z


def row_linear(X, W, N, residual=None):
    """sum_i X_i W_i (+ residual)."""
    return shard_reduce(row_partials(X, W, N), residual)


def col_linear_bwd(X, W, dYs, N):
    """Column-parallel backward: dW_i = X^T dY_i, dX = sum_i dY_i W_i^T.

    [Infra: Tensor Parallel, Column-wise TP, backward]. (The same statement on the
    张量并行 notes is garbled by extraction; this page's form is taken.)
    """
    Ws = col_shards(W, N)
    dW = np.concatenate([X.T @ dYi for dYi in dYs], axis=1)
    dX = shard_reduce([dYi @ Wi.T for dYi, Wi in zip(dYs, Ws)])
    return dX, dW


def row_linear_bwd(X, W, dY, N):
    """Row-parallel backward: dW_i = X_i^T dY, dX_i = dY W_i^T, dX = [dX_1 ... dX_N].

    [Infra: Tensor Parallel, Row-wise TP, backward];
    [张量并行 notes, §并行化矩阵乘法运算, 行并行, "f 的反向传播 ... concat"].
    """
    Xs, Ws = col_shards(X, N), row_shards(W, N)
    dW = np.concatenate([Xi.T @ dY for Xi in Xs], axis=0)
    dX = np.concatenate([dY @ Wi.T for Wi in Ws], axis=1)
    return dX, dW


# ---------------------------------------------------------------- MLP, GELU

def mlp_gelu_fwd(X, W1, W2, N, residual=None):
    """Megatron MLP: W1 split by column, GELU on each shard, W2 split by row,
    one sum at the end: Z = sum_i GELU(X W1_i) W2_i.

    [张量并行 notes, §MLP 层的并行化, "A 列切 + B 行切的完整公式"];
    [Infra: Tensor Parallel, MLP]. Returns Y (pre-activation), H = GELU(Y), Z.
    """
    Ys = col_linear(X, W1, N)
    Hs = [gelu(Y) for Y in Ys]
    Zs = [Hi @ W2i for Hi, W2i in zip(Hs, row_shards(W2, N))]
    return {"Y": np.concatenate(Ys, axis=1), "H": np.concatenate(Hs, axis=1),
            "Z": shard_reduce(Zs, residual)}


def mlp_gelu_fwd_unsplit(X, W1, W2):
    """Single-device reference GELU(X W1) W2 [Infra: Tensor Parallel, MLP(x) = sigma(X W1) W2]."""
    return gelu(X @ W1) @ W2


def mlp_gelu_row_then_col(X, A, B, N):
    """The scheme the notes reject: A split by row, B by column, so the sum of
    the shards' X_i A_i must be taken before GELU.

    [张量并行 notes, §两个矩阵相乘]. Returns (correct, wrong) where `wrong`
    applies GELU per shard before summing -- the result the non-additivity of
    GELU forbids.
    """
    parts = [Xi @ Ai for Xi, Ai in zip(col_shards(X, N), row_shards(A, N))]
    correct = gelu(shard_reduce(parts)) @ B
    wrong = shard_reduce([gelu(P) for P in parts]) @ B
    return correct, wrong


def mlp_gelu_bwd(X, W1, W2, dZ, N):
    """Backward of the Megatron GELU MLP, shard by shard.

    g-backward is the identity: every shard gets the whole dZ
    [张量并行 notes, §MLP 层的并行化, "g 的 backward 计算"]. Then per shard:
      dH_i  = dZ W2_i^T                       (row-parallel, dX_i = dY W_i^T)
      dY_i  = dH_i * GELU'(Y_i)
      dW2_i = H_i^T dZ                        (row-parallel, dW_i = X_i^T dY)
      dW1_i = X^T dY_i                        (column-parallel)
    and f-backward sums dX = sum_i dY_i W1_i^T [张量并行 notes, "f 的 backward 计算 ...
    all-reduce"; Infra: Tensor Parallel, Column-wise and Row-wise TP backward].
    """
    Ys = col_linear(X, W1, N)
    W1s, W2s = col_shards(W1, N), row_shards(W2, N)
    dYs, dW1s, dW2s, dXs = [], [], [], []
    for Yi, W1i, W2i in zip(Ys, W1s, W2s):
        Hi = gelu(Yi)
        dHi = dZ @ W2i.T
        dYi = dHi * gelu_prime(Yi)
        dYs.append(dYi)
        dW2s.append(Hi.T @ dZ)
        dW1s.append(X.T @ dYi)
        dXs.append(dYi @ W1i.T)
    return {"dY": np.concatenate(dYs, axis=1), "dX": shard_reduce(dXs),
            "dW1": np.concatenate(dW1s, axis=1), "dW2": np.concatenate(dW2s, axis=0)}


def mlp_gelu_dW_cols(X, W1, W2, dZ, cols):
    """dW1[:, cols] and dW2[cols, :] for a set of hidden (ffn) indices `cols`.

    GELU acts column by column [张量并行 notes, §MLP 层的并行化, "满足列 / 通道可分性"],
    so these entries need only the columns `cols` of Y; it is the backward above
    restricted to those columns (used to sample very large workloads).
    """
    cols = np.asarray(cols)
    Yc = X @ W1[:, cols]
    dYc = (dZ @ W2[cols, :].T) * gelu_prime(Yc)
    return {"dW1": X.T @ dYc, "dW2": gelu(Yc).T @ dZ}


# ---------------------------------------------------------------- MLP, SwiGLU

def mlp_swiglu_fwd(X, Wg, Wu, Wd, N, residual=None):
    """SwiGLU MLP with W_gate and W_up split by column and W_down by row
    [20260402-parallelism, §1 Tensor Parallelism]:
      G_i = X Wg_i, U_i = X Wu_i, A_i = SiLU(G_i) * U_i, Z = sum_i A_i Wd_i.
    Gate and up shards cover the same column range.
    """
    Gs, Us = col_linear(X, Wg, N), col_linear(X, Wu, N)
    As = [silu(G) * U for G, U in zip(Gs, Us)]
    Zs = [Ai @ Wdi for Ai, Wdi in zip(As, row_shards(Wd, N))]
    return {"G": np.concatenate(Gs, axis=1), "U": np.concatenate(Us, axis=1),
            "A": np.concatenate(As, axis=1), "Z": shard_reduce(Zs, residual)}


def mlp_swiglu_fwd_unsplit(X, Wg, Wu, Wd):
    return (silu(X @ Wg) * (X @ Wu)) @ Wd


def _swiglu_grads(dA, G, U):
    """dG = dA * U * s * (1 + G (1 - s)), dU = dA * G * s, s = sigmoid(G)
    (derivative of SiLU(g) = g s(g) is s(g) (1 + g (1 - s(g))))."""
    s = sigmoid(G)
    return dA * U * s * (1.0 + G * (1.0 - s)), dA * G * s


def mlp_swiglu_bwd(X, Wg, Wu, Wd, dZ, N):
    """Backward of the SwiGLU MLP shard by shard (same operator algebra as the
    GELU MLP): dA_i = dZ Wd_i^T, (dG_i, dU_i) from the SwiGLU derivative,
    dWd_i = A_i^T dZ, dWg_i = X^T dG_i, dWu_i = X^T dU_i,
    dX = sum_i (dG_i Wg_i^T + dU_i Wu_i^T).
    """
    Gs, Us = col_linear(X, Wg, N), col_linear(X, Wu, N)
    Wgs, Wus, Wds = col_shards(Wg, N), col_shards(Wu, N), row_shards(Wd, N)
    out = {k: [] for k in ("dG", "dU", "dWg", "dWu", "dWd")}
    dXs = []
    for Gi, Ui, Wgi, Wui, Wdi in zip(Gs, Us, Wgs, Wus, Wds):
        Ai = silu(Gi) * Ui
        dAi = dZ @ Wdi.T
        dGi, dUi = _swiglu_grads(dAi, Gi, Ui)
        out["dG"].append(dGi)
        out["dU"].append(dUi)
        out["dWd"].append(Ai.T @ dZ)
        out["dWg"].append(X.T @ dGi)
        out["dWu"].append(X.T @ dUi)
        dXs.append(dGi @ Wgi.T + dUi @ Wui.T)
    res = {k: np.concatenate(v, axis=0 if k == "dWd" else 1) for k, v in out.items()}
    res["dX"] = shard_reduce(dXs)
    return res


def mlp_swiglu_dW_cols(X, Wg, Wu, Wd, dZ, cols):
    """dWg[:, cols], dWu[:, cols], dWd[cols, :] (column-restricted backward)."""
    cols = np.asarray(cols)
    G, U = X @ Wg[:, cols], X @ Wu[:, cols]
    dA = dZ @ Wd[cols, :].T
    dG, dU = _swiglu_grads(dA, G, U)
    return {"dWg": X.T @ dG, "dWu": X.T @ dU, "dWd": (silu(G) * U).T @ dZ}


# ---------------------------------------------------------------- LayerNorm

def layernorm_fwd(x, gamma, beta, eps=LN_EPS):
    """LN(x) = gamma * (x - mu) / sqrt(sigma^2 + eps) + beta over the full hidden
    width, biased variance [张量并行 notes, §相关分析, LayerNorm formula].
    eps = 1e-5 is the reading taken (the pages leave it open; the listing uses
    the framework default). Returns (y, mu, rstd)."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    return gamma * ((x - mu) * rstd) + beta, mu[..., 0], rstd[..., 0]


def layernorm_bwd(x, gamma, dy, eps=LN_EPS):
    """Gradients of LN: dbeta = sum dy, dgamma = sum dy * xhat,
    dx = rstd * (g - mean(g) - xhat * mean(g * xhat)) with g = dy * gamma.
    Sums run over all rows (every rank holds the same x, so gamma/beta grads need
    no all-reduce [张量并行 notes, §相关分析])."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mu) * rstd
    g = dy * gamma
    dx = rstd * (g - g.mean(axis=-1, keepdims=True)
                 - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    red = tuple(range(x.ndim - 1))
    return dx, (dy * xhat).sum(axis=red), dy.sum(axis=red)


def shard_reduce_ln(partials, residual, gamma, beta, eps=LN_EPS):
    """The shard sum, then LayerNorm of its full-width result.

    x = sum_i Z_i (+ residual) is what the all-reduce leaves on every rank; LN
    needs the statistics of the whole hidden width, so it can only run after the
    sum [张量并行 notes, §相关分析, forward bottleneck before LayerNorm]. Shards are
    summed in order 0..N-1 (`shard_reduce`), then `layernorm_fwd`.
    Returns (x, y, mu, rstd).
    """
    x = shard_reduce(partials, residual)
    y, mu, rstd = layernorm_fwd(x, gamma, beta, eps)
    return x, y, mu, rstd


# ---------------------------------------------------------------- attention

def softmax_rows(S):
    S = S - S.max(axis=-1, keepdims=True)
    E = np.exp(S)
    return E / E.sum(axis=-1, keepdims=True)


def attention_head_fwd(Q, K, V, causal=False):
    """One head: O = softmax(Q K^T / sqrt(d)) V (rows of the score matrix).

    Scale 1/sqrt(head_dim) and no mask follow [Megatron-LM 实战 04 张量并行实现, 核心实现,
    TPAttention.forward]; `causal` is an option the listing does not use.
    """
    d = Q.shape[-1]
    S = (Q @ K.T) / math.sqrt(d)
    if causal:
        S = S + np.triu(np.full(S.shape, -np.inf), k=1)
    P = softmax_rows(S)
    return P @ V, P


def attention_head_bwd(Q, K, V, dO, causal=False):
    """dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dP * P)),
    dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d)."""
    d = Q.shape[-1]
    O, P = attention_head_fwd(Q, K, V, causal)
    dV = P.T @ dO
    dP = dO @ V.T
    dS = P * (dP - (dP * P).sum(axis=-1, keepdims=True))
    return dS @ K / math.sqrt(d), dS.T @ Q / math.sqrt(d), dV


def qkv_shard_columns(h, n_heads, N, i):
    """Column indices of W_qkv = [W_q | W_k | W_v] (h x 3h) that shard i owns.

    Heads are split across shards (heads % N == 0, [Infra: Tensor Parallel,
    attention]); head t occupies columns t*d .. t*d+d-1 of each of the three
    blocks. Shard i takes its heads' columns from all three blocks -- the reading
    of the listing's per-shard [3, heads/tp, head_dim] output layout
    [Megatron-LM 实战 04 张量并行实现, 核心实现, TPAttention].
    """
    hs = h // N
    base = np.arange(i * hs, (i + 1) * hs)
    return np.concatenate([base, h + base, 2 * h + base])


def attn_block_fwd(x, b, s, gamma, beta, Wqkv, Wo, n_heads, N, causal=False,
                   eps=LN_EPS):
    """x1 = x + sum_i O_i Wo_i with O_i the outputs of shard i's heads on LN(x).

    Heads are independent [张量并行 notes, §Multi-Head Attention 的并行化]; each shard
    owns heads/N heads and the matching row block of W_o; no gather of the
    heads is needed because the shard output feeds the row-split W_o directly
    [20260402-parallelism, §1 Tensor Parallelism; Infra: Tensor Parallel, attention].
    x: (M, h) with M = b*s; the s rows of one sequence are consecutive.
    Returns dict with xn (LN output), QKV, O (heads concatenated), out.
    """
    M, h = x.shape
    if h % n_heads or n_heads % N:
        raise ValueError("need h % heads == 0 and heads % N == 0")
    d = h // n_heads
    xn, mu, rstd = layernorm_fwd(x, gamma, beta, eps)
    QKV = np.zeros((M, 3 * h))
    O = np.zeros((M, h))
    partials = []
    hs = h // N
    for i in range(N):
        cols = qkv_shard_columns(h, n_heads, N, i)
        QKVi = xn @ Wqkv[:, cols]  # column-parallel, shard i
        QKV[:, cols] = QKVi
        Oi = np.zeros((M, hs))
        for tl in range(n_heads // N):
            for bb in range(b):
                r = slice(bb * s, (bb + 1) * s)
                c = slice(tl * d, (tl + 1) * d)
                q = QKVi[r, c]
                k = QKVi[r, hs + tl * d: hs + (tl + 1) * d]
                v = QKVi[r, 2 * hs + tl * d: 2 * hs + (tl + 1) * d]
                Oi[r, c] = attention_head_fwd(q, k, v, causal)[0]
        O[:, i * hs:(i + 1) * hs] = Oi
        partials.append(Oi @ Wo[i * hs:(i + 1) * hs, :])  # row-parallel W_o
    out = shard_reduce(partials, residual=x)
    return {"xn": xn, "QKV": QKV, "O": O, "out": out}


def attn_block_fwd_unsplit(x, b, s, gamma, beta, Wqkv, Wo, n_heads, causal=False):
    """Single-device multi-head attention block (heads concatenated, then W_o)."""
    M, h = x.shape
    d = h // n_heads
    xn = layernorm_fwd(x, gamma, beta)[0]
    Q, K, V = xn @ Wqkv[:, :h], xn @ Wqkv[:, h:2 * h], xn @ Wqkv[:, 2 * h:]
    O = np.zeros((M, h))
    for t in range(n_heads):
        c = slice(t * d, (t + 1) * d)
        for bb in range(b):
            r = slice(bb * s, (bb + 1) * s)
            O[r, c] = attention_head_fwd(Q[r, c], K[r, c], V[r, c], causal)[0]
    return x + O @ Wo


def attn_block_bwd(x, b, s, gamma, beta, Wqkv, Wo, n_heads, N, dout, causal=False,
                      eps=LN_EPS):
    """Backward of attn_block_fwd. Returns dx, dgamma, dbeta, dWqkv, dWo."""
    M, h = x.shape
    d = h // n_heads
    hs = h // N
    f = attn_block_fwd(x, b, s, gamma, beta, Wqkv, Wo, n_heads, N, causal, eps)
    xn, QKV, O = f["xn"], f["QKV"], f["O"]
    dWo = np.zeros_like(Wo)
    dQKV = np.zeros_like(QKV)
    for i in range(N):
        rows = slice(i * hs, (i + 1) * hs)
        dWo[rows, :] = O[:, rows].T @ dout       # dW_i = X_i^T dY (row-parallel)
        dOi = dout @ Wo[rows, :].T               # dX_i = dY W_i^T
        cols = qkv_shard_columns(h, n_heads, N, i)
        QKVi = QKV[:, cols]
        dQKVi = np.zeros_like(QKVi)
        for tl in range(n_heads // N):
            for bb in range(b):
                r = slice(bb * s, (bb + 1) * s)
                cq = slice(tl * d, (tl + 1) * d)
                ck = slice(hs + tl * d, hs + (tl + 1) * d)
                cv = slice(2 * hs + tl * d, 2 * hs + (tl + 1) * d)
                dq, dk, dv = attention_head_bwd(QKVi[r, cq], QKVi[r, ck], QKVi[r, cv],
                                                dOi[r, cq], causal)
                dQKVi[r, cq], dQKVi[r, ck], dQKVi[r, cv] = dq, dk, dv
        dQKV[:, cols] = dQKVi
    dWqkv = xn.T @ dQKV
    dxn = shard_reduce([dQKV[:, qkv_shard_columns(h, n_heads, N, i)]
                        @ Wqkv[:, qkv_shard_columns(h, n_heads, N, i)].T for i in range(N)])
    dx_ln, dgamma, dbeta = layernorm_bwd(x, gamma, dxn, eps)
    return {"dx": dout + dx_ln, "dgamma": dgamma, "dbeta": dbeta,
            "dWqkv": dWqkv, "dWo": dWo, "dQKV": dQKV}


def layer_fwd(x, b, s, p, n_heads, N, causal=False):
    """Pre-LN transformer layer: x1 = x + Attn(LN1(x)); out = x1 + MLP(LN2(x1))
    [Megatron-LM 实战 04 张量并行实现, 核心实现, TPTransformerLayer.forward].
    p: dict with gamma1, beta1, Wqkv, Wo, gamma2, beta2, W1, W2."""
    a = attn_block_fwd(x, b, s, p["gamma1"], p["beta1"], p["Wqkv"], p["Wo"],
                          n_heads, N, causal)
    x1 = a["out"]
    xn2, _, _ = layernorm_fwd(x1, p["gamma2"], p["beta2"])
    m = mlp_gelu_fwd(xn2, p["W1"], p["W2"], N, residual=x1)
    return {"x1": x1, "xn2": xn2, "out": m["Z"], "attn": a, "mlp": m}


def layer_bwd(x, b, s, p, n_heads, N, dout, causal=False):
    f = layer_fwd(x, b, s, p, n_heads, N, causal)
    x1, xn2 = f["x1"], f["xn2"]
    g = mlp_gelu_bwd(xn2, p["W1"], p["W2"], dout, N)
    dx1_ln, dgamma2, dbeta2 = layernorm_bwd(x1, p["gamma2"], g["dX"])
    dx1 = dout + dx1_ln
    a = attn_block_bwd(x, b, s, p["gamma1"], p["beta1"], p["Wqkv"], p["Wo"],
                          n_heads, N, dx1, causal)
    return {"dx": a["dx"], "dgamma1": a["dgamma"], "dbeta1": a["dbeta"],
            "dWqkv": a["dWqkv"], "dWo": a["dWo"], "dgamma2": dgamma2, "dbeta2": dbeta2,
            "dW1": g["dW1"], "dW2": g["dW2"]}


# ---------------------------------------------------------------- sequence parallelism

def seq_slices(M, N):
    """Rows that virtual rank r holds in the sequence-parallel regions:
    [r*M/N, (r+1)*M/N). Reading taken: token rows are ordered so that each rank's
    piece of the sequence is one contiguous block (M % N == 0)."""
    if M % N:
        raise ValueError("sequence parallelism needs M % N == 0")
    m = M // N
    return [slice(r * m, (r + 1) * m) for r in range(N)]


def _sp_mlp(xn, W1, W2, N, act, W1u):
    if act == "gelu":
        return mlp_gelu_fwd(xn, W1, W2, N)
    return mlp_swiglu_fwd(xn, W1, W1u, W2, N)


def sp_mlp_block_fwd(x, gamma, beta, W1, W2, N, act="gelu", W1u=None, eps=LN_EPS):
    """Pre-LN MLP sub-block, out = x + MLP(LN(x)), in its sequence-parallel form
    [20260402-parallelism, §5 Sequence Parallelism]:
      rank r holds only its rows x_r of the LayerNorm / residual activations and
      normalises them (LN on 1/N of the rows); an all-gather assembles the full
      LN output for the tensor-parallel MLP (column split, then row split); the
      all-reduce that would end the MLP is split into its reduce-scatter half, so
      rank r receives only its rows of sum_i Z_i and adds its residual rows.
    Returns xn (gathered), mean, rstd, the MLP's saved activations and out (the
    ranks' slices stacked in rank order)."""
    sl = seq_slices(x.shape[0], N)
    ln = [layernorm_fwd(x[q], gamma, beta, eps) for q in sl]           # LN(1/N) per rank
    xn = np.concatenate([t[0] for t in ln], axis=0)                     # all-gather
    m = _sp_mlp(xn, W1, W2, N, act, W1u)                                # TP MLP, per shard
    out = np.concatenate([m["Z"][q] + x[q] for q in sl], axis=0)        # reduce-scatter + x_r
    return {"xn": xn, "mean": np.concatenate([t[1] for t in ln]),
            "rstd": np.concatenate([t[2] for t in ln]), "mlp": m, "out": out}


def sp_mlp_block_bwd(x, gamma, beta, W1, W2, N, dout, act="gelu", W1u=None, eps=LN_EPS):
    """Backward of `sp_mlp_block_fwd`. The backward of the reduce-scatter is an
    all-gather of dout (every shard reads the whole dZ); the backward of the
    all-gather is a reduce-scatter of the MLP's input gradient, so rank r gets
    dxn_r = (sum_i dX_i)[rows of r]; LN backward runs per rank on its rows, plus
    the residual's dout_r. Each rank's LN parameters only see its own rows, so
    the ranks' gamma / beta gradients differ and are summed over the ranks (an
    all-reduce) -- unlike the replicated LN of plain tensor parallelism, whose
    gradients agree on every rank [张量并行 notes, §相关分析]."""
    f = sp_mlp_block_fwd(x, gamma, beta, W1, W2, N, act, W1u, eps)
    sl = seq_slices(x.shape[0], N)
    dZ = np.concatenate([dout[q] for q in sl], axis=0)                   # all-gather
    if act == "gelu":
        g = mlp_gelu_bwd(f["xn"], W1, W2, dZ, N)
        res = {"dW1": g["dW1"], "dW2": g["dW2"]}
    else:
        g = mlp_swiglu_bwd(f["xn"], W1, W1u, W2, dZ, N)
        res = {"dW1": g["dWg"], "dW1u": g["dWu"], "dW2": g["dWd"]}
    dx, dgr, dbr = [], [], []
    for q in sl:
        dxr, dg, db = layernorm_bwd(x[q], gamma, g["dX"][q], eps)      # reduce-scatter rows
        dx.append(dxr + dout[q])
        dgr.append(dg)
        dbr.append(db)
    res.update({"dx": np.concatenate(dx, axis=0), "dgamma_ranks": np.stack(dgr),
                "dbeta_ranks": np.stack(dbr), "dgamma": shard_reduce(dgr),
                "dbeta": shard_reduce(dbr)})
    return res


def rel_err(got, ref):
    """max|got - ref| / max|ref| -- the parity metric."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(got - ref)) if ref.size else 0.0
    return float(num / den) if den > 0 else float(num)
