"""fp64 oracle of the vocabulary-parallel embedding and cross-entropy, and of the
small tensor-parallel GPT trained with them.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA library never
imports or calls this module.

Shapes: token ids (b, s) flattened to M = b*s rows, the s rows of one sequence
consecutive; E (v, h) is the word embedding, shared with the output layer
(logits = x E^T). Vocabulary shard i owns rows [i*v/N, (i+1)*v/N) of E -- the
contiguous-block reading of the other splits.
"""
from __future__ import annotations

import math

import numpy as np

from . import tp_oracle as T


def vocab_range(v, N, i):
    """Rows [lo, hi) of the vocabulary that shard i owns."""
    if v % N:
        raise ValueError("vocabulary size must be divisible by N")
    return i * (v // N), (i + 1) * (v // N)


# ---------------------------------------------------------------- embedding

def vocab_embed_fwd(ids, E, N):
    """Vocabulary-parallel lookup: shard i returns E[id] for the ids it owns and a
    zero row for the others; the all-reduce of the shards' results is the input
    [张量并行 notes, §嵌入层的并行化, input layer]. Shards summed in order 0..N-1."""
    ids = np.asarray(ids).reshape(-1)
    v, h = E.shape
    parts = []
    for i in range(N):
        lo, hi = vocab_range(v, N, i)
        P = np.zeros((ids.size, h))
        for t, tok in enumerate(ids):
            if lo <= tok < hi:
                P[t] = E[tok]
        parts.append(P)
    return T.shard_reduce(parts)


def vocab_embed_bwd(ids, dx, v, N):
    """Gradient of the lookup: shard i adds dx[t] to row id_t of its block for the
    ids it owns (tokens in order); the blocks stacked are dE (v, h)."""
    ids = np.asarray(ids).reshape(-1)
    h = dx.shape[1]
    blocks = []
    for i in range(N):
        lo, hi = vocab_range(v, N, i)
        B = np.zeros((hi - lo, h))
        for t, tok in enumerate(ids):
            if lo <= tok < hi:
                B[tok - lo] += dx[t]
        blocks.append(B)
    return np.concatenate(blocks, axis=0)


# ---------------------------------------------------------------- cross-entropy

def vocab_ce_fwd(logits, targets, N):
    """Cross-entropy over a vocabulary split into N column blocks, without gathering
    the logits [张量并行 notes, §损失计算层的并行化]:
      every shard takes its row maxima, an all-reduce (max) gives m; every shard sums
      exp(l - m) over its columns, an all-reduce (sum) gives the softmax denominator
      S; the shard holding a row's target takes -log p = log S + m - l_target; each
      shard sums those over its rows and a last all-reduce adds the N scalars.
    The loss is the mean over the M rows (the listing's cross-entropy default).
    Returns (loss, lse, row_loss, shard_loss) with lse = m + log S."""
    targets = np.asarray(targets).reshape(-1)
    M, v = logits.shape
    rng = [vocab_range(v, N, i) for i in range(N)]
    m = np.max(np.stack([logits[:, lo:hi].max(axis=1) for lo, hi in rng]), axis=0)
    S = T.shard_reduce([np.exp(logits[:, lo:hi] - m[:, None]).sum(axis=1) for lo, hi in rng])
    lse = m + np.log(S)
    row_loss = np.zeros(M)
    shard_loss = np.zeros(N)
    for i, (lo, hi) in enumerate(rng):
        own = (targets >= lo) & (targets < hi)
        r = np.nonzero(own)[0]
        row_loss[r] = lse[r] - logits[r, targets[r]]
        shard_loss[i] = row_loss[r].sum()
    return float(T.shard_reduce(list(shard_loss)) / M), lse, row_loss, shard_loss


def vocab_ce_bwd(logits, targets, lse, N, scale):
    """d(loss)/d(logits) block by block: softmax - one_hot(target), times `scale`
    (1/M for the mean); each shard needs only its columns, m and S."""
    targets = np.asarray(targets).reshape(-1)
    M, v = logits.shape
    blocks = []
    for i in range(N):
        lo, hi = vocab_range(v, N, i)
        P = np.exp(logits[:, lo:hi] - lse[:, None])
        own = np.nonzero((targets >= lo) & (targets < hi))[0]
        P[own, targets[own] - lo] -= 1.0
        blocks.append(P * scale)
    return np.concatenate(blocks, axis=1)


# ---------------------------------------------------------------- the model

LAYER_KEYS = ("gamma1", "beta1", "Wqkv", "Wo", "gamma2", "beta2", "W1", "W2")


def gpt_forward(params, ids, targets, cfg):
    """SmallGPT [Megatron-LM 实战 04 张量并行实现, 核心实现, SmallGPT]: embedding,
    `layers` pre-LN tensor-parallel layers, final LN, output layer tied to the
    embedding, cross-entropy. The embedding and the output layer are split by
    vocabulary over the N shards [张量并行 notes, §嵌入层的并行化]: the output layer is
    column-parallel (shard i: logits_i = x_f E_i^T) and feeds the vocabulary-parallel
    cross-entropy directly."""
    b, s, N, heads = cfg["b"], cfg["s"], cfg["N"], cfg["heads"]
    E = params["E"]
    v = E.shape[0]
    x = vocab_embed_fwd(ids, E, N)
    xs = [x]
    for L in params["layers"]:
        x = T.layer_fwd(x, b, s, L, heads, N)["out"]
        xs.append(x)
    xf, _, _ = T.layernorm_fwd(x, params["gammaf"], params["betaf"])
    logits = np.concatenate([xf @ E[lo:hi].T for lo, hi in
                             (vocab_range(v, N, i) for i in range(N))], axis=1)
    loss, lse, _, _ = vocab_ce_fwd(logits, targets, N)
    return {"loss": loss, "logits": logits, "lse": lse, "xs": xs, "xf": xf}


def gpt_backward(params, ids, targets, cfg):
    """Loss and gradients of every parameter. The output layer's input gradient is
    summed over the vocabulary shards (an all-reduce); the shared embedding's
    gradient is the output layer's plus the input layer's
    [张量并行 notes, §嵌入层的并行化, grad_total = grad_in + grad_out]."""
    b, s, N, heads = cfg["b"], cfg["s"], cfg["N"], cfg["heads"]
    E = params["E"]
    v = E.shape[0]
    f = gpt_forward(params, ids, targets, cfg)
    M = f["logits"].shape[0]
    dlog = vocab_ce_bwd(f["logits"], targets, f["lse"], N, 1.0 / M)
    rng = [vocab_range(v, N, i) for i in range(N)]
    dxf = T.shard_reduce([dlog[:, lo:hi] @ E[lo:hi] for lo, hi in rng])
    dE_out = np.concatenate([dlog[:, lo:hi].T @ f["xf"] for lo, hi in rng], axis=0)
    dx, dgf, dbf = T.layernorm_bwd(f["xs"][-1], params["gammaf"], dxf)
    lgrads = [None] * len(params["layers"])
    for li in reversed(range(len(params["layers"]))):
        g = T.layer_bwd(f["xs"][li], b, s, params["layers"][li], heads, N, dx)
        dx = g["dx"]
        lgrads[li] = {k: g["d" + k] for k in LAYER_KEYS}
    dE_in = vocab_embed_bwd(ids, dx, v, N)
    return f["loss"], {"E": dE_in + dE_out, "layers": lgrads, "gammaf": dgf, "betaf": dbf}


# ---------------------------------------------------------------- optimiser

ADAMW = {"lr": 3e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.01}


def adamw_step(p, g, m, v, t, lr, beta1, beta2, eps, weight_decay):
    """AdamW with decoupled weight decay (Loshchilov & Hutter, "Decoupled Weight Decay
    Regularization", ICLR 2019), bias-corrected moments, step t >= 1:
      p <- p (1 - lr wd);  m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;
      p <- p - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps).
    The listing trains with AdamW(lr=3e-4) and the framework's defaults
    (betas 0.9 / 0.999, eps 1e-8, weight decay 0.01) -- the reading taken."""
    p = p * (1.0 - lr * weight_decay)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    mh = m / (1.0 - beta1 ** t)
    vh = v / (1.0 - beta2 ** t)
    return p - lr * mh / (np.sqrt(vh) + eps), m, v


def _flatten(tree):
    """Parameters in a fixed order: E, each layer's tensors, gammaf, betaf."""
    keys = LAYER_KEYS
    out = [("E", tree["E"])]
    for li, L in enumerate(tree["layers"]):
        out += [(f"L{li}.{k}", L[k]) for k in keys]
    out += [("gammaf", tree["gammaf"]), ("betaf", tree["betaf"])]
    return out


def _unflatten(items, n_layers):
    d = dict(items)
    keys = LAYER_KEYS
    return {"E": d["E"], "gammaf": d["gammaf"], "betaf": d["betaf"],
            "layers": [{k: d[f"L{li}.{k}"] for k in keys} for li in range(n_layers)]}


def gpt_train(params, ids, targets, cfg, steps, opt=ADAMW):
    """The listing's loop: loss, backward, optimiser step, `steps` times on the same
    batch. Returns the loss of every step (taken before that step's update) and the
    final parameters."""
    nl = len(params["layers"])
    items = [(k, np.array(a, dtype=np.float64)) for k, a in _flatten(params)]
    ms = {k: np.zeros_like(a) for k, a in items}
    vs = {k: np.zeros_like(a) for k, a in items}
    losses = []
    for t in range(1, steps + 1):
        cur = _unflatten(items, nl)
        loss, grads = gpt_backward(cur, ids, targets, cfg)
        losses.append(loss)
        gitems = dict(_flatten(grads))
        new = []
        for k, p in items:
            p2, ms[k], vs[k] = adamw_step(p, gitems[k], ms[k], vs[k], t, **opt)
            new.append((k, p2))
        items = new
    return losses, _unflatten(items, nl)
