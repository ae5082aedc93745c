"""Pins of the vocabulary-parallel embedding / cross-entropy oracle and of the small
GPT trained with it: textbook special cases (plain lookup, one-hot products, the
log-sum-exp cross-entropy), closed forms (uniform logits give log v; AdamW's first
step), finite differences of every gradient, and the pages' own check that one and
two shards give the same loss trajectory."""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import gpt_oracle as G
from oracle import tp_oracle as T
from tests.test_oracle_pins import _fd


def _rng(seed):
    return np.random.default_rng(seed)


@pytest.mark.parametrize("N", [1, 2, 4])
def test_vocab_embed_is_lookup_and_onehot_transpose(N):
    r = _rng(60)
    v, h, M = 16, 5, 11
    E, ids, dx = r.normal(size=(v, h)), r.integers(0, v, size=M), r.normal(size=(M, h))
    assert np.array_equal(G.vocab_embed_fwd(ids, E, N), E[ids])
    onehot = np.zeros((M, v))
    onehot[np.arange(M), ids] = 1.0
    assert np.allclose(G.vocab_embed_bwd(ids, dx, v, N), onehot.T @ dx, rtol=0, atol=1e-14)


@pytest.mark.parametrize("N", [1, 2, 4])
def test_vocab_ce_is_logsumexp_cross_entropy(N):
    r = _rng(61)
    M, v = 7, 12
    L, tg = 3.0 * r.normal(size=(M, v)), r.integers(0, v, size=M)
    loss, lse, rows, shards = G.vocab_ce_fwd(L, tg, N)
    ref_rows = logsumexp(L, axis=1) - L[np.arange(M), tg]
    assert np.allclose(rows, ref_rows, rtol=1e-14, atol=1e-14)
    assert abs(loss - ref_rows.mean()) <= 1e-14 * abs(loss)
    assert np.allclose(lse, logsumexp(L, axis=1), rtol=1e-15)
    assert abs(shards.sum() - rows.sum()) <= 1e-13


def test_vocab_ce_closed_forms():
    """Uniform logits give log v; a row shift changes nothing."""
    v = 256
    loss = G.vocab_ce_fwd(np.full((3, v), 0.7), np.array([0, 100, 255]), 4)[0]
    assert abs(loss - math.log(v)) <= 1e-14
    r = _rng(62)
    L, tg = r.normal(size=(4, 8)), np.array([1, 7, 3, 0])
    l0 = G.vocab_ce_fwd(L, tg, 2)[0]
    l1 = G.vocab_ce_fwd(L + np.array([[3.0], [-1.0], [0.5], [40.0]]), tg, 2)[0]
    assert abs(l0 - l1) <= 1e-13


@pytest.mark.parametrize("N", [1, 2])
def test_vocab_ce_bwd_fd(N):
    r = _rng(63)
    M, v = 5, 8
    L, tg = r.normal(size=(M, v)), r.integers(0, v, size=M)
    _, lse, _, _ = G.vocab_ce_fwd(L, tg, N)
    g = G.vocab_ce_bwd(L, tg, lse, N, 1.0 / M)
    assert T.rel_err(g, _fd(lambda: G.vocab_ce_fwd(L, tg, N)[0], L)) <= 1e-8


def _tiny(seed, v=8, h=8, heads=2, f=16, layers=1):
    r = _rng(seed)
    lay = lambda: {"gamma1": 1 + 0.1 * r.normal(size=h), "beta1": 0.1 * r.normal(size=h),
                   "Wqkv": 0.3 * r.normal(size=(h, 3 * h)), "Wo": 0.3 * r.normal(size=(h, h)),
                   "gamma2": 1 + 0.1 * r.normal(size=h), "beta2": 0.1 * r.normal(size=h),
                   "W1": 0.3 * r.normal(size=(h, f)), "W2": 0.3 * r.normal(size=(f, h))}
    return {"E": r.normal(size=(v, h)), "layers": [lay() for _ in range(layers)],
            "gammaf": 1 + 0.1 * r.normal(size=h), "betaf": 0.1 * r.normal(size=h)}


def test_gpt_backward_fd():
    cfg = dict(b=2, s=3, heads=2, N=2)
    p = _tiny(64)
    r = _rng(65)
    ids, tg = r.integers(0, 8, size=(2, 3)), r.integers(0, 8, size=(2, 3))
    loss_fn = lambda: G.gpt_forward(p, ids, tg, cfg)["loss"]
    _, g = G.gpt_backward(p, ids, tg, cfg)
    assert T.rel_err(g["E"], _fd(loss_fn, p["E"])) <= 1e-7          # tied: input + output
    assert T.rel_err(g["gammaf"], _fd(loss_fn, p["gammaf"])) <= 1e-7
    assert T.rel_err(g["betaf"], _fd(loss_fn, p["betaf"])) <= 1e-7
    for k in ("Wqkv", "W1", "gamma1"):
        assert T.rel_err(g["layers"][0][k], _fd(loss_fn, p["layers"][0][k])) <= 1e-7


def test_adamw_first_steps_closed_form():
    p, g = np.array([0.5, -2.0, 0.0]), np.array([0.1, -3.0, 1e-3])
    o = G.ADAMW
    p1, m1, v1 = G.adamw_step(p, g, np.zeros(3), np.zeros(3), 1, **o)
    # step 1: bias-corrected moments are g and g^2, so the step is lr * g / (|g| + eps)
    ref = p * (1 - o["lr"] * o["weight_decay"]) - o["lr"] * g / (np.abs(g) + o["eps"])
    assert np.allclose(p1, ref, rtol=1e-15, atol=1e-18)
    # step 2 with the same gradient: m = 0.19 g, v = 0.001999 g^2 before correction
    p2, _, _ = G.adamw_step(p1, g, m1, v1, 2, **o)
    mh, vh = 0.19 * g / (1 - 0.81), 0.001999 * g * g / (1 - 0.998001)
    ref2 = p1 * (1 - o["lr"] * o["weight_decay"]) - o["lr"] * mh / (np.sqrt(vh) + o["eps"])
    assert np.allclose(p2, ref2, rtol=1e-13, atol=1e-18)


def test_one_and_two_shards_train_identically():
    """The pages' check: the same seed and data give the same loss at every step with
    one shard and with two [Megatron-LM 实战 04 张量并行实现, 验证方法]."""
    p = _tiny(66, v=8, h=8, heads=2, f=16, layers=2)
    r = _rng(67)
    ids, tg = r.integers(0, 8, size=(2, 4)), r.integers(0, 8, size=(2, 4))
    l1, _ = G.gpt_train(p, ids, tg, dict(b=2, s=4, heads=2, N=1), 6)
    l2, _ = G.gpt_train(p, ids, tg, dict(b=2, s=4, heads=2, N=2), 6)
    assert np.max(np.abs(np.array(l1) - np.array(l2))) <= 1e-12
    assert l1[-1] < l1[0]
