"""Pins of the grouped-query attention oracle under head sharding: it reduces to the
(already pinned) multi-head oracle when every query head has its own key/value head,
the grouping is checked head by head against the textbook softmax, the sharded block
(with replicated key/value heads when N > Hkv) equals the single-device block, and
every gradient -- the replicas' all-reduced key/value gradients included -- matches
finite differences of the single-device block."""
import numpy as np
import pytest

from oracle import gqa_oracle as Q
from oracle import tp_oracle as T
from tests.test_oracle_pins import _fd

CASES = [(4, 2, 1), (4, 2, 2), (4, 2, 4), (8, 2, 8), (6, 3, 3), (4, 1, 2), (4, 4, 2)]


def _inputs(seed, H, Hkv, d=2, b=2, s=3):
    r = np.random.default_rng(seed)
    h = H * d
    return dict(x=r.normal(size=(b * s, h)), g=1 + 0.2 * r.normal(size=h),
                be=0.2 * r.normal(size=h), Wq=0.5 * r.normal(size=(h, H * d)),
                Wk=0.5 * r.normal(size=(h, Hkv * d)), Wv=0.5 * r.normal(size=(h, Hkv * d)),
                Wo=0.5 * r.normal(size=(H * d, h)), dout=r.normal(size=(b * s, h)), b=b, s=s, d=d)


@pytest.mark.parametrize("N", [1, 2])
def test_gqa_reduces_to_mha_oracle(N):
    H = 4
    p = _inputs(70, H, H)
    Wqkv = np.concatenate([p["Wq"], p["Wk"], p["Wv"]], axis=1)
    ref = T.attn_block_fwd(p["x"], p["b"], p["s"], p["g"], p["be"], Wqkv, p["Wo"], H, N)["out"]
    Wsh = Q.gqa_pack(p["Wq"], p["Wk"], p["Wv"], H, H, N)
    got = Q.gqa_block_fwd(p["x"], p["b"], p["s"], p["g"], p["be"], Wsh, p["Wo"], H, H, N)["out"]
    assert T.rel_err(got, ref) <= 1e-13


def test_gqa_grouping_head_by_head():
    """Query head t attends with key/value head t // (H / Hkv): textbook softmax rows."""
    H, Hkv, d, b, s = 6, 2, 3, 1, 4
    r = np.random.default_rng(71)
    xn = r.normal(size=(s, 5))
    Wq, Wk, Wv = r.normal(size=(5, H * d)), r.normal(size=(5, Hkv * d)), r.normal(size=(5, Hkv * d))
    O = Q.gqa_attention_unsplit(xn, Wq, Wk, Wv, b, s, H, Hkv)
    for t in range(H):
        j = t // 3
        q, k, v = xn @ Wq[:, t * d:(t + 1) * d], xn @ Wk[:, j * d:(j + 1) * d], xn @ Wv[:, j * d:(j + 1) * d]
        for i in range(s):
            e = [np.exp(sum(q[i, c] * k[jj, c] for c in range(d)) / np.sqrt(d)) for jj in range(s)]
            row = sum(e[jj] * v[jj] for jj in range(s)) / sum(e)
            assert np.allclose(O[i, t * d:(t + 1) * d], row, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("H,Hkv,N", CASES)
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_sharded_equals_unsplit(H, Hkv, N, causal):
    p = _inputs(72, H, Hkv)
    ref = Q.gqa_block_unsplit(p["x"], p["b"], p["s"], p["g"], p["be"], p["Wq"], p["Wk"], p["Wv"],
                              p["Wo"], H, Hkv, causal)
    Wsh = Q.gqa_pack(p["Wq"], p["Wk"], p["Wv"], H, Hkv, N)
    got = Q.gqa_block_fwd(p["x"], p["b"], p["s"], p["g"], p["be"], Wsh, p["Wo"], H, Hkv, N, causal)
    assert T.rel_err(got["out"], ref) <= 1e-13


@pytest.mark.parametrize("H,Hkv,N", CASES)
def test_gqa_bwd_fd(H, Hkv, N):
    p = _inputs(73, H, Hkv)
    x, g, be, Wq, Wk, Wv, Wo, dout = (p[k] for k in ("x", "g", "be", "Wq", "Wk", "Wv", "Wo", "dout"))
    b, s, d = p["b"], p["s"], p["d"]
    loss = lambda: float(np.sum(Q.gqa_block_unsplit(x, b, s, g, be, Wq, Wk, Wv, Wo, H, Hkv) * dout))
    Wsh = Q.gqa_pack(Wq, Wk, Wv, H, Hkv, N)
    gr = Q.gqa_block_bwd(x, b, s, g, be, Wsh, Wo, H, Hkv, N, dout)
    dWq, dWk, dWv = Q.gqa_unpack_grad(gr["dWqkv"], H, Hkv, N, d)
    for got, arr in ((dWq, Wq), (dWk, Wk), (dWv, Wv), (gr["dWo"], Wo), (gr["dx"], x),
                     (gr["dgamma"], g), (gr["dbeta"], be)):
        assert T.rel_err(got, _fd(loss, arr)) <= 1e-7
    # after the all-reduce every replica holds the same key/value gradient
    hq, hkv, r = Q.gqa_split(H, Hkv, N)
    Ws = (hq + 2 * hkv) * d
    if r > 1:
        for i in range(N):
            base = (i // r) * r
            assert np.array_equal(gr["dWqkv"][:, i * Ws + hq * d:(i + 1) * Ws],
                                  gr["dWqkv"][:, base * Ws + hq * d:(base + 1) * Ws])


@pytest.mark.parametrize("H,Hkv,N", [(4, 2, 2), (4, 2, 4), (4, 4, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_core_bwd_fd(H, Hkv, N, causal):
    """The attention core alone: gqa_attention_bwd is the gradient of
    sum(gqa_attention_fwd(QKV) * dO) with respect to every entry of the sharded QKV,
    each replica's key/value columns being inputs of their own."""
    r = np.random.default_rng(74)
    b, s, d = 2, 3, 2
    hq, hkv, _ = Q.gqa_split(H, Hkv, N)
    QKV = r.normal(size=(b * s, N * (hq + 2 * hkv) * d))
    dO = r.normal(size=(b * s, H * d))
    loss = lambda: float(np.sum(Q.gqa_attention_fwd(QKV, b, s, H, Hkv, N, causal) * dO))
    got = Q.gqa_attention_bwd(QKV, dO, b, s, H, Hkv, N, causal)
    assert T.rel_err(got, _fd(loss, QKV)) <= 1e-7


def test_gqa_split_rules():
    assert Q.gqa_split(32, 8, 4) == (8, 2, 1)
    assert Q.gqa_split(32, 8, 16) == (2, 1, 2)
    assert Q.gqa_split(32, 8, 32) == (1, 1, 4)
    for bad in ((32, 8, 3), (32, 8, 12), (8, 3, 2)):
        with pytest.raises(ValueError):
            Q.gqa_split(*bad)
