"""Pins of the fp64 oracle against what the pages and mathematics fix.

Each check ties an oracle function to something other than itself: closed-form
values (tests/golden), brute-force loops in plain Python on tiny inputs, the
block-matrix identities, the Megatron MLP invariant, the GELU counter-example,
and central finite differences for every backward.
"""
import math
import os

import numpy as np
import pytest

from oracle import tp_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                k, x, v = line.split()
                rows.append((k, float(x), float(v)))
    return rows


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- elementwise

def test_gelu_phi_table():
    """GELU(x) = x Phi(x) and GELU'(x) = Phi(x) + x phi(x) at table values."""
    g = _golden("normal_cdf_closed_forms.txt")
    phi = {x: v for k, x, v in g if k == "phi"}
    for k, x, v in g:
        if k == "Phi":
            assert abs(O.gelu(np.array([x]))[0] - x * v) <= 1e-15 * max(1, abs(x))
            if x in phi:
                assert abs(O.gelu_prime(np.array([x]))[0] - (v + x * phi[x])) <= 1e-15


def test_gelu_symmetric_sum_68_95_997():
    """GELU(x) + GELU(-x) = x erf(x / sqrt 2): the 68-95-99.7 rule values."""
    for k, x, v in _golden("normal_cdf_closed_forms.txt"):
        if k == "erf_k_over_sqrt2":
            s = O.gelu(np.array([x]))[0] + O.gelu(np.array([-x]))[0]
            assert abs(s - x * v) <= 2e-15 * x


def test_gelu_counterexample_nonadditive():
    """GELU(1 + (-1)) = 0 but GELU(1) + GELU(-1) = erf(1/sqrt 2) = 0.6826894921370859."""
    assert O.gelu(np.array([0.0]))[0] == 0.0
    s = O.gelu(np.array([1.0]))[0] + O.gelu(np.array([-1.0]))[0]
    assert abs(s - 0.6826894921370859) < 1e-15


def test_gelu_limits_and_separability():
    x = np.array([40.0, -40.0, 0.0])
    y = O.gelu(x)
    assert y[0] == 40.0 and abs(y[1]) < 1e-300 and y[2] == 0.0
    a = _rng(0).normal(size=(3, 8))
    assert np.array_equal(O.gelu(a), np.concatenate([O.gelu(a[:, :3]), O.gelu(a[:, 3:])], 1))


def test_sigmoid_silu_values():
    for k, x, v in _golden("normal_cdf_closed_forms.txt"):
        if k == "sigmoid":
            assert abs(O.sigmoid(np.array([x]))[0] - v) <= 1e-16
            assert abs(O.silu(np.array([x]))[0] - x * v) <= 1e-16 * max(1, abs(x))
    # stable at both tails
    assert O.sigmoid(np.array([-800.0]))[0] == 0.0
    assert O.sigmoid(np.array([800.0]))[0] == 1.0


def test_gelu_prime_is_derivative():
    x = np.linspace(-6, 6, 241)
    e = 1e-6
    fd = (O.gelu(x + e) - O.gelu(x - e)) / (2 * e)
    assert np.max(np.abs(fd - O.gelu_prime(x))) < 1e-8


# ---------------------------------------------------------------- brute force linear

def _py_matmul(A, B):
    n, k = len(A), len(A[0])
    m = len(B[0])
    return [[sum(A[i][t] * B[t][j] for t in range(k)) for j in range(m)] for i in range(n)]


@pytest.mark.parametrize("N", [1, 2, 3])
def test_col_linear_bruteforce(N):
    r = _rng(1)
    X, W = r.normal(size=(3, 4)), r.normal(size=(4, 6))
    Ys = O.col_linear(X, W, N)
    w = 6 // N
    for i, Yi in enumerate(Ys):
        Wi = [[W[k][i * w + j] for j in range(w)] for k in range(4)]
        ref = _py_matmul(X.tolist(), Wi)
        assert np.allclose(Yi, ref, rtol=0, atol=1e-14)


@pytest.mark.parametrize("N", [1, 2, 3])
def test_row_linear_bruteforce(N):
    r = _rng(2)
    X, W = r.normal(size=(3, 6)), r.normal(size=(6, 5))
    w = 6 // N
    ref = [[0.0] * 5 for _ in range(3)]
    for i in range(N):
        Xi = [[X[m][i * w + k] for k in range(w)] for m in range(3)]
        Wi = [[W[i * w + k][j] for j in range(5)] for k in range(w)]
        P = _py_matmul(Xi, Wi)
        ref = [[ref[m][j] + P[m][j] for j in range(5)] for m in range(3)]
    assert np.allclose(O.row_linear(X, W, N), ref, rtol=0, atol=1e-14)


def test_block_identities():
    """X [W1 .. WN] = [X W1 .. X WN] (exactly: same dot products), and
    [X1 .. XN] [W1; ..; WN] = sum Xi Wi to 1e-12."""
    r = _rng(3)
    X, W = r.normal(size=(17, 32)), r.normal(size=(32, 48))
    for N in (1, 2, 4, 8):
        cat = np.concatenate(O.col_linear(X, W, N), axis=1)
        assert O.rel_err(cat, X @ W) <= 1e-12
    W2 = r.normal(size=(48, 24))
    Y = r.normal(size=(17, 48))
    for N in (1, 2, 3, 4, 6, 8):
        assert O.rel_err(O.row_linear(Y, W2, N), Y @ W2) <= 1e-12


def test_shard_reduce_exact_integers():
    r = _rng(4)
    P = r.integers(-1000, 1000, size=(5, 7, 9)).astype(np.float64)
    R = r.integers(-1000, 1000, size=(7, 9)).astype(np.float64)
    want = [[sum(int(P[i, a, b]) for i in range(5)) + int(R[a, b]) for b in range(9)] for a in range(7)]
    assert np.array_equal(O.shard_reduce(list(P), R), np.array(want, dtype=np.float64))


# ---------------------------------------------------------------- MLP forward

def test_mlp_gelu_bruteforce_tiny():
    r = _rng(5)
    X, W1, W2 = r.normal(size=(2, 3)), r.normal(size=(3, 4)), r.normal(size=(4, 3))
    H = [[0.0] * 4 for _ in range(2)]
    for m in range(2):
        for j in range(4):
            y = sum(X[m][k] * W1[k][j] for k in range(3))
            H[m][j] = y * 0.5 * (1 + math.erf(y / math.sqrt(2)))
    Z = _py_matmul(H, W2.tolist())
    for N in (1, 2, 4):
        got = O.mlp_gelu_fwd(X, W1, W2, N)
        assert np.allclose(got["H"], H, rtol=0, atol=1e-14)
        assert np.allclose(got["Z"], Z, rtol=0, atol=1e-13)


def test_megatron_invariant():
    """sum_i GELU(X W1_i) W2_i = GELU(X W1) W2 to 1e-12 for every shard count."""
    r = _rng(6)
    X, W1, W2 = r.normal(size=(9, 16)), r.normal(size=(16, 24)), r.normal(size=(24, 16))
    ref = O.mlp_gelu_fwd_unsplit(X, W1, W2)
    for N in (1, 2, 3, 4, 6, 8, 12, 24):
        assert O.rel_err(O.mlp_gelu_fwd(X, W1, W2, N)["Z"], ref) <= 1e-12
    Wg, Wu, Wd = r.normal(size=(16, 24)), r.normal(size=(16, 24)), r.normal(size=(24, 16))
    ref = O.mlp_swiglu_fwd_unsplit(X, Wg, Wu, Wd)
    for N in (1, 2, 4, 8):
        assert O.rel_err(O.mlp_swiglu_fwd(X, Wg, Wu, Wd, N)["Z"], ref) <= 1e-12


def test_swiglu_bruteforce_tiny():
    r = _rng(7)
    X, Wg, Wu, Wd = (r.normal(size=s) for s in [(2, 3), (3, 4), (3, 4), (4, 2)])
    A = [[0.0] * 4 for _ in range(2)]
    for m in range(2):
        for j in range(4):
            g = sum(X[m][k] * Wg[k][j] for k in range(3))
            u = sum(X[m][k] * Wu[k][j] for k in range(3))
            A[m][j] = g / (1 + math.exp(-g)) * u
    Z = _py_matmul(A, Wd.tolist())
    got = O.mlp_swiglu_fwd(X, Wg, Wu, Wd, 2)
    assert np.allclose(got["A"], A, rtol=0, atol=1e-14)
    assert np.allclose(got["Z"], Z, rtol=0, atol=1e-13)


def test_row_then_col_needs_sum_before_gelu():
    """The rejected scheme: correct only when the shard sum precedes GELU."""
    r = _rng(8)
    X, A, B = r.normal(size=(5, 8)), r.normal(size=(8, 6)), r.normal(size=(6, 4))
    correct, wrong = O.mlp_gelu_row_then_col(X, A, B, 2)
    assert O.rel_err(correct, O.mlp_gelu_fwd_unsplit(X, A, B)) <= 1e-12
    assert O.rel_err(wrong, correct) > 1e-2


# ---------------------------------------------------------------- finite differences

def _fd(fun, arr, eps=1e-6):
    g = np.zeros_like(arr)
    for idx in np.ndindex(arr.shape):
        old = arr[idx]
        arr[idx] = old + eps
        lp = fun()
        arr[idx] = old - eps
        lm = fun()
        arr[idx] = old
        g[idx] = (lp - lm) / (2 * eps)
    return g


def fd_errors_mlp_gelu(N, seed=10):
    r = _rng(seed)
    X, W1, W2 = r.normal(size=(3, 4)), r.normal(size=(4, 8)), r.normal(size=(8, 4))
    dZ = r.normal(size=(3, 4))
    g = O.mlp_gelu_bwd(X, W1, W2, dZ, N)
    loss = lambda: float(np.sum(O.mlp_gelu_fwd(X, W1, W2, N)["Z"] * dZ))
    return {k: O.rel_err(g[k], _fd(loss, a)) for k, a in (("dX", X), ("dW1", W1), ("dW2", W2))}


@pytest.mark.parametrize("N", [1, 2, 4])
def test_mlp_gelu_bwd_fd(N):
    for k, e in fd_errors_mlp_gelu(N).items():
        assert e <= 1e-7, (k, e)


def test_mlp_gelu_bwd_dY():
    """dY = (dZ W2^T) * GELU'(X W1), checked by perturbing Y directly."""
    r = _rng(11)
    Y, W2, dZ = r.normal(size=(3, 8)), r.normal(size=(8, 4)), r.normal(size=(3, 4))
    loss = lambda: float(np.sum((O.gelu(Y) @ W2) * dZ))
    X = np.eye(3)  # Y = X W1 with W1 = Y
    g = O.mlp_gelu_bwd(X, Y.copy(), W2, dZ, 2)
    assert O.rel_err(g["dY"], _fd(loss, Y)) <= 1e-7


def fd_errors_mlp_swiglu(N, seed=12):
    r = _rng(seed)
    X, Wg, Wu, Wd = (r.normal(size=s) for s in [(3, 4), (4, 8), (4, 8), (8, 4)])
    dZ = r.normal(size=(3, 4))
    g = O.mlp_swiglu_bwd(X, Wg, Wu, Wd, dZ, N)
    loss = lambda: float(np.sum(O.mlp_swiglu_fwd(X, Wg, Wu, Wd, N)["Z"] * dZ))
    return {k: O.rel_err(g[k], _fd(loss, a))
            for k, a in (("dX", X), ("dWg", Wg), ("dWu", Wu), ("dWd", Wd))}


@pytest.mark.parametrize("N", [1, 2, 4])
def test_mlp_swiglu_bwd_fd(N):
    for k, e in fd_errors_mlp_swiglu(N).items():
        assert e <= 1e-7, (k, e)


def test_dW_cols_match_full_backward():
    r = _rng(13)
    X, W1, W2, dZ = (r.normal(size=s) for s in [(6, 4), (4, 16), (16, 4), (6, 4)])
    full = O.mlp_gelu_bwd(X, W1, W2, dZ, 4)
    cols = np.array([0, 5, 6, 15])
    part = O.mlp_gelu_dW_cols(X, W1, W2, dZ, cols)
    assert O.rel_err(part["dW1"], full["dW1"][:, cols]) <= 1e-13
    assert O.rel_err(part["dW2"], full["dW2"][cols, :]) <= 1e-13
    Wg, Wu = r.normal(size=(4, 16)), r.normal(size=(4, 16))
    full = O.mlp_swiglu_bwd(X, Wg, Wu, W2, dZ, 2)
    part = O.mlp_swiglu_dW_cols(X, Wg, Wu, W2, dZ, cols)
    for k, ax in (("dWg", 1), ("dWu", 1), ("dWd", 0)):
        ref = full[k][:, cols] if ax == 1 else full[k][cols, :]
        assert O.rel_err(part[k], ref) <= 1e-13


# ---------------------------------------------------------------- LayerNorm

def test_layernorm_invariants():
    r = _rng(14)
    x = r.normal(size=(5, 16)) * 3 + 1
    y, mu, rstd = O.layernorm_fwd(x, np.ones(16), np.zeros(16))
    assert np.allclose(y.mean(axis=1), 0, atol=1e-14)
    var = x.var(axis=1)
    assert np.allclose((y ** 2).mean(axis=1), var / (var + 1e-5), atol=1e-14)
    # x = [1, 2, 3, 4]: mean 2.5, biased variance 1.25
    y, mu, rstd = O.layernorm_fwd(np.array([[1.0, 2, 3, 4]]), np.ones(4), np.zeros(4), eps=0.0)
    assert mu[0] == 2.5 and abs(rstd[0] - 1 / math.sqrt(1.25)) < 1e-15
    assert np.allclose(y[0], np.array([-1.5, -0.5, 0.5, 1.5]) / math.sqrt(1.25), atol=1e-15)


def test_layernorm_bwd_fd():
    r = _rng(15)
    x, gamma, beta, dy = r.normal(size=(3, 6)), r.normal(size=6), r.normal(size=6), r.normal(size=(3, 6))
    dx, dg, db = O.layernorm_bwd(x, gamma, dy)
    loss = lambda: float(np.sum(O.layernorm_fwd(x, gamma, beta)[0] * dy))
    assert O.rel_err(dx, _fd(loss, x)) <= 1e-7
    assert O.rel_err(dg, _fd(loss, gamma)) <= 1e-7
    assert O.rel_err(db, _fd(loss, beta)) <= 1e-7


def _ln_row_loops(v, g, b, eps):
    """LayerNorm of one row in scalar Python: mean, biased variance, normalise."""
    n = len(v)
    mu = sum(v) / n
    var = sum((t - mu) * (t - mu) for t in v) / n
    rs = 1.0 / math.sqrt(var + eps)
    return [g[c] * (v[c] - mu) * rs + b[c] for c in range(n)], mu, rs


def test_shard_reduce_ln_bruteforce():
    """Sum of the shards and LN of the result, element by element in plain loops."""
    r = _rng(40)
    N, M, h = 3, 4, 8
    P = [r.normal(size=(M, h)) for _ in range(N)]
    R, g, b = r.normal(size=(M, h)), r.normal(size=h), r.normal(size=h)
    x, y, mu, rstd = O.shard_reduce_ln(P, R, g, b)
    for m in range(M):
        row = [sum(P[i][m, c] for i in range(N)) + R[m, c] for c in range(h)]
        yr, mr, rr = _ln_row_loops(row, g, b, 1e-5)
        assert max(abs(x[m, c] - row[c]) for c in range(h)) <= 1e-14
        assert max(abs(y[m, c] - yr[c]) for c in range(h)) <= 1e-12
        assert abs(mu[m] - mr) <= 1e-14 and abs(rstd[m] - rr) <= 1e-12 * rr


def test_shard_reduce_ln_equals_ln_of_unsplit_row_gemm():
    """LN after the all-reduce of the row-parallel partials = LN of the unsplit
    product (block identity of the row split, then the same LN)."""
    r = _rng(41)
    H, W, R = r.normal(size=(6, 12)), r.normal(size=(12, 8)), r.normal(size=(6, 8))
    g, b = r.normal(size=8), r.normal(size=8)
    for N in (1, 2, 3, 4):
        x, y, _, _ = O.shard_reduce_ln(O.row_partials(H, W, N), R, g, b)
        Z = H @ W + R
        assert O.rel_err(x, Z) <= 1e-13
        yr = np.array([_ln_row_loops(list(Z[m]), g, b, 1e-5)[0] for m in range(6)])
        assert O.rel_err(y, yr) <= 1e-12


def test_shard_reduce_ln_shift_and_constant_rows():
    """LN ignores a constant added to a whole row (through any shard), and maps a
    constant row to beta."""
    r = _rng(42)
    P = [r.normal(size=(3, 16)) for _ in range(2)]
    g, b = r.normal(size=16), r.normal(size=16)
    _, y0, mu0, rs0 = O.shard_reduce_ln(P, None, g, b)
    Q = [P[0], P[1] + np.array([[5.0], [-2.0], [0.25]])]
    x1, y1, mu1, rs1 = O.shard_reduce_ln(Q, None, g, b)
    assert O.rel_err(y1, y0) <= 1e-12 and np.allclose(rs1, rs0, rtol=1e-12)
    assert np.allclose(mu1 - mu0, [5.0, -2.0, 0.25], atol=1e-13)
    C = [np.full((2, 16), 0.75), np.full((2, 16), -2.0)]
    _, yc, muc, _ = O.shard_reduce_ln(C, np.full((2, 16), 0.5), g, b)
    assert np.allclose(muc, -0.75, atol=1e-15) and np.allclose(yc, b, atol=1e-15)


# ---------------------------------------------------------------- attention

def test_attention_closed_forms():
    r = _rng(16)
    V = r.normal(size=(5, 4))
    Q = r.normal(size=(5, 4))
    # zero keys: every score equal, so each output row is the mean of V
    O1, P = O.attention_head_fwd(Q, np.zeros((5, 4)), V)
    assert np.allclose(O1, np.tile(V.mean(axis=0), (5, 1)), atol=1e-15)
    assert np.allclose(P.sum(axis=1), 1, atol=1e-15)
    # causal: row 0 sees only key 0
    O2, _ = O.attention_head_fwd(Q, r.normal(size=(5, 4)), V, causal=True)
    assert np.allclose(O2[0], V[0], atol=1e-15)
    # a dominant key: scores 40*sqrt(d) apart -> output equals that value row
    K = np.zeros((5, 4)); K[3, 0] = 1.0
    Qd = np.zeros((5, 4)); Qd[:, 0] = 80.0
    O3, _ = O.attention_head_fwd(Qd, K, V)
    assert np.allclose(O3, np.tile(V[3], (5, 1)), atol=1e-12)


def test_attention_textbook_loops():
    r = _rng(17)
    Q, K, V = r.normal(size=(4, 2)), r.normal(size=(4, 2)), r.normal(size=(4, 2))
    out = []
    for i in range(4):
        s = [sum(Q[i][t] * K[j][t] for t in range(2)) / math.sqrt(2) for j in range(4)]
        m = max(s)
        e = [math.exp(v - m) for v in s]
        z = sum(e)
        out.append([sum(e[j] / z * V[j][t] for j in range(4)) for t in range(2)])
    assert np.allclose(O.attention_head_fwd(Q, K, V)[0], out, atol=1e-15)


def test_attention_bwd_fd():
    r = _rng(18)
    Q, K, V, dO = (r.normal(size=(5, 3)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = O.attention_head_bwd(Q, K, V, dO, causal)
        loss = lambda: float(np.sum(O.attention_head_fwd(Q, K, V, causal)[0] * dO))
        assert O.rel_err(dq, _fd(loss, Q)) <= 1e-7
        assert O.rel_err(dk, _fd(loss, K)) <= 1e-7
        assert O.rel_err(dv, _fd(loss, V)) <= 1e-7


def _layer_params(r, h, f):
    return {"gamma1": 1 + 0.1 * r.normal(size=h), "beta1": 0.1 * r.normal(size=h),
            "Wqkv": r.normal(size=(h, 3 * h)) * 0.5, "Wo": r.normal(size=(h, h)) * 0.5,
            "gamma2": 1 + 0.1 * r.normal(size=h), "beta2": 0.1 * r.normal(size=h),
            "W1": r.normal(size=(h, f)) * 0.5, "W2": r.normal(size=(f, h)) * 0.5}


def test_attn_block_split_equals_unsplit():
    r = _rng(19)
    b, s, h, heads = 2, 5, 8, 4
    p = _layer_params(r, h, 16)
    x = r.normal(size=(b * s, h))
    ref = O.attn_block_fwd_unsplit(x, b, s, p["gamma1"], p["beta1"], p["Wqkv"], p["Wo"], heads)
    for N in (1, 2, 4):
        got = O.attn_block_fwd(x, b, s, p["gamma1"], p["beta1"], p["Wqkv"], p["Wo"], heads, N)
        assert O.rel_err(got["out"], ref) <= 1e-12


def test_layer_bwd_fd():
    r = _rng(20)
    b, s, h, heads, f, N = 2, 3, 4, 2, 8, 2
    p = _layer_params(r, h, f)
    x = r.normal(size=(b * s, h))
    dout = r.normal(size=(b * s, h))
    g = O.layer_bwd(x, b, s, p, heads, N, dout)
    loss = lambda: float(np.sum(O.layer_fwd(x, b, s, p, heads, N)["out"] * dout))
    assert O.rel_err(g["dx"], _fd(loss, x)) <= 1e-7
    for k in ("gamma1", "beta1", "Wqkv", "Wo", "gamma2", "beta2", "W1", "W2"):
        assert O.rel_err(g["d" + k], _fd(loss, p[k])) <= 1e-7, k


def test_qkv_shard_columns_cover_once():
    h, heads = 16, 8
    for N in (1, 2, 4, 8):
        cols = np.concatenate([O.qkv_shard_columns(h, heads, N, i) for i in range(N)])
        assert sorted(cols.tolist()) == list(range(3 * h))


# ---------------------------------------------------------------- sequence parallelism

def _block_unsplit(x, g, b, W1, W2, act, W1u):
    """x + MLP(LN(x)) on one device, written with the plain operators."""
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    xn = g * (x - mu) / np.sqrt(var + 1e-5) + b
    if act == "gelu":
        return x + O.gelu(xn @ W1) @ W2
    return x + (O.silu(xn @ W1) * (xn @ W1u)) @ W2


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("N", [1, 2, 4])
def test_sp_mlp_block_equals_unsplit_and_fd(act, N):
    r = _rng(50)
    M, h, f = 8, 4, 8
    x, g, b = r.normal(size=(M, h)), r.normal(size=h), r.normal(size=h)
    W1, W2, W1u = r.normal(size=(h, f)), r.normal(size=(f, h)), r.normal(size=(h, f))
    dout = r.normal(size=(M, h))
    u = W1u if act == "swiglu" else None
    fw = O.sp_mlp_block_fwd(x, g, b, W1, W2, N, act, u)
    assert O.rel_err(fw["out"], _block_unsplit(x, g, b, W1, W2, act, u)) <= 1e-13
    bw = O.sp_mlp_block_bwd(x, g, b, W1, W2, N, dout, act, u)
    loss = lambda: float(np.sum(_block_unsplit(x, g, b, W1, W2, act, u) * dout))
    assert O.rel_err(bw["dx"], _fd(loss, x)) <= 1e-7
    assert O.rel_err(bw["dgamma"], _fd(loss, g)) <= 1e-7
    assert O.rel_err(bw["dbeta"], _fd(loss, b)) <= 1e-7
    assert O.rel_err(bw["dW1"], _fd(loss, W1)) <= 1e-7
    assert O.rel_err(bw["dW2"], _fd(loss, W2)) <= 1e-7
    if act == "swiglu":
        assert O.rel_err(bw["dW1u"], _fd(loss, W1u)) <= 1e-7


def test_sp_rank_gradients_are_per_rank_parameter_gradients():
    """dgamma_ranks[r] is the gradient with respect to rank r's own copy of gamma
    (every rank normalises its rows with its copy), checked by finite differences
    on a block whose LN uses a separate gamma / beta per row slice."""
    r = _rng(51)
    M, h, f, N = 6, 4, 6, 3
    x, W1, W2 = r.normal(size=(M, h)), r.normal(size=(h, f)), r.normal(size=(f, h))
    gs, bs = r.normal(size=(N, h)), r.normal(size=(N, h))
    dout = r.normal(size=(M, h))

    def loss():
        rows = np.concatenate([np.repeat(gs[k][None], M // N, 0) for k in range(N)])
        brow = np.concatenate([np.repeat(bs[k][None], M // N, 0) for k in range(N)])
        return float(np.sum(_block_unsplit(x, rows, brow, W1, W2, "gelu", None) * dout))
    # with equal copies the per-copy gradients are the oracle's per-rank partials
    gs[:] = gs[0]
    bs[:] = bs[0]
    bw = O.sp_mlp_block_bwd(x, gs[0].copy(), bs[0].copy(), W1, W2, N, dout)
    assert O.rel_err(bw["dgamma_ranks"], _fd(loss, gs)) <= 1e-7
    assert O.rel_err(bw["dbeta_ranks"], _fd(loss, bs)) <= 1e-7
    assert np.allclose(bw["dgamma_ranks"].sum(axis=0), bw["dgamma"], rtol=1e-13, atol=1e-13)


def test_sp_output_rows_depend_only_on_own_rank_rows():
    """LN and the MLP act token by token, so rank r's output rows depend only on
    its own input rows (the reduce-scatter hands each rank exactly those)."""
    r = _rng(52)
    M, h, f, N = 8, 4, 8, 4
    x, g, b = r.normal(size=(M, h)), r.normal(size=h), r.normal(size=h)
    W1, W2 = r.normal(size=(h, f)), r.normal(size=(f, h))
    o0 = O.sp_mlp_block_fwd(x, g, b, W1, W2, N)["out"]
    x2 = x.copy()
    x2[2:4] += 1.5  # rank 1's rows
    o1 = O.sp_mlp_block_fwd(x2, g, b, W1, W2, N)["out"]
    assert np.array_equal(o0[:2], o1[:2]) and np.array_equal(o0[4:], o1[4:])
    assert not np.allclose(o0[2:4], o1[2:4])
    with pytest.raises(ValueError):
        O.seq_slices(7, 2)
