"""GPU parity of every entry point against the fp64 oracle, element by element,
on seeded inputs whose sizes span several tiles and end in ragged tails.

Bar: max|gpu - oracle| / max|oracle| <= 1e-2 (bf16 inputs, fp32 accumulation) and
<= 1e-5 (fp32 path), per output tensor."""
import numpy as np
import pytest
import torch

from attention_gemms_gb300 import tpmlp as T
from oracle import tp_oracle as O
from tests.helpers import (BF16_TOL, F32_TOL, empty, gemm_tiles, guard_intact, guarded, host,
                           rel, tensor)

pytestmark = pytest.mark.gpu
BF = T.DType.BF16
bf16 = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    T.lib()
    torch.cuda.set_device(0)
    T.tp_set_wait_timeout_ns(1_000_000_000)  # a legitimate stage wait takes microseconds
    yield
    T.tp_set_wait_timeout_ns(0)
    assert T.tp_check_status() == 0


def _ws(nbytes):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")


# ---------------------------------------------------------------- shard sum

@pytest.mark.parametrize("N", [1, 3, 8])
@pytest.mark.parametrize("n", [64, 100])
@pytest.mark.parametrize("out_dt", [T.DType.F32, T.DType.BF16])
@pytest.mark.parametrize("with_res", [False, True])
def test_shard_reduce(N, n, out_dt, with_res):
    M = 77
    Po, P = tensor((N, M, n), 101, dtype="f32")
    tdt = torch.float32 if out_dt == T.DType.F32 else bf16
    Ro, R = tensor((M, n), 102, dtype="f32" if out_dt == T.DType.F32 else "bf16")
    out, full = guarded((M, n), tdt)
    T.tp_shard_reduce(P, R if with_res else None, out, N, M, n, out_dt)
    torch.cuda.synchronize()
    ref = O.shard_reduce(list(Po), Ro if with_res else None)
    tol = 1e-6 if out_dt == T.DType.F32 else 4e-3
    assert rel(host(out), ref) <= tol
    assert guard_intact(full, M)


# ---------------------------------------------------------------- column / row linear

@pytest.mark.parametrize("act", [T.Act.NONE, T.Act.GELU, T.Act.SWIGLU])
@pytest.mark.parametrize("N", [1, 2, 4])
@pytest.mark.parametrize("M", [1, 333])
def test_col_linear(act, N, M):
    h, f = 192, 512
    Xo, X = tensor((M, h), 201)
    Wo, W = tensor((h, f), 202, 0.05)
    Wuo, Wu = tensor((h, f), 203, 0.05)
    out, full = guarded((M, f), bf16)
    Y, Yu = empty((M, f), bf16), empty((M, f), bf16)
    T.tp_col_linear(X, W, Wu if act == T.Act.SWIGLU else None, Y, Yu, out, M, h, f, N, BF, act)
    torch.cuda.synchronize()
    G = np.concatenate(O.col_linear(Xo, Wo, N), axis=1)
    if act == T.Act.NONE:
        assert rel(host(out), G) <= BF16_TOL
    elif act == T.Act.GELU:
        assert rel(host(Y), G) <= BF16_TOL
        assert rel(host(out), O.gelu(G)) <= BF16_TOL
    else:
        U = np.concatenate(O.col_linear(Xo, Wuo, N), axis=1)
        assert rel(host(Y), G) <= BF16_TOL
        assert rel(host(Yu), U) <= BF16_TOL
        assert rel(host(out), O.silu(G) * U) <= BF16_TOL
    assert guard_intact(full, M)


@pytest.mark.parametrize("mode", [T.Reduce.BUFFERS, T.Reduce.SPLITK])
@pytest.mark.parametrize("N", [1, 2, 4])
@pytest.mark.parametrize("with_res", [False, True])
def test_row_linear(mode, N, with_res):
    M, k, n = 333, 512, 192
    Xo, X = tensor((M, k), 301)
    Wo, W = tensor((k, n), 302, 0.05)
    Ro, R = tensor((M, n), 303)
    out, full = guarded((M, n), bf16)
    wsz = T.tp_workspace_size(T.Op.ROW_LINEAR, M, k, n, N, BF, T.Act.NONE, mode)
    ws = _ws(wsz)
    T.tp_row_linear(X, W, R if with_res else None, out, M, k, n, N, BF, mode, ws, ws.numel())
    torch.cuda.synchronize()
    ref = O.row_linear(Xo, Wo, N, Ro if with_res else None)
    assert rel(host(out), ref) <= BF16_TOL
    assert guard_intact(full, M)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_row_linear_buffers_in_two_row_blocks(dtype):
    """From 2048 rows on, variant A runs the row GEMM as two row blocks (whole 256-row
    tiles, then the ragged rest) and sums the first block's partials beside the second
    block's GEMM: every row of the sum, residual included, against the oracle."""
    M, k, n, N = 2100, 256, 192, 4
    dt = BF if dtype == "bf16" else T.DType.F32
    tdt = bf16 if dtype == "bf16" else torch.float32
    Xo, X = tensor((M, k), 311, dtype=dtype)
    Wo, W = tensor((k, n), 312, 0.05, dtype=dtype)
    Ro, R = tensor((M, n), 313, dtype=dtype)
    out, full = guarded((M, n), tdt)
    ws = _ws(T.tp_workspace_size(T.Op.ROW_LINEAR, M, k, n, N, dt, T.Act.NONE, T.Reduce.BUFFERS))
    T.tp_row_linear(X, W, R, out, M, k, n, N, dt, T.Reduce.BUFFERS, ws, ws.numel())
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    ref = O.row_linear(Xo, Wo, N, Ro)
    tol = BF16_TOL if dtype == "bf16" else F32_TOL
    assert rel(host(out), ref) <= tol
    assert rel(host(out)[1280:], ref[1280:]) <= tol    # the second block on its own
    assert guard_intact(full, M)


# ---------------------------------------------------------------- MLP forward + backward

def _mlp_run(act, mode, N, M, h, f, dtype="bf16", seed0=400, sigma=0.05):
    tdt = bf16 if dtype == "bf16" else torch.float32
    dt = BF if dtype == "bf16" else T.DType.F32
    Xo, X = tensor((M, h), seed0 + 1, dtype=dtype)
    W1o, W1 = tensor((h, f), seed0 + 2, sigma, dtype=dtype)
    Wuo, Wu = tensor((h, f), seed0 + 3, sigma, dtype=dtype)
    W2o, W2 = tensor((f, h), seed0 + 4, sigma, dtype=dtype)
    dZo, dZ = tensor((M, h), seed0 + 5, dtype=dtype)
    sw = act == T.Act.SWIGLU
    Y, Yu, H = empty((M, f), tdt), empty((M, f), tdt), empty((M, f), tdt)
    Z, fullZ = guarded((M, h), tdt)
    dX, fulldX = guarded((M, h), tdt)
    dW1, dWu, dW2 = empty((h, f), tdt), empty((h, f), tdt), empty((f, h), tdt)
    ws = _ws(max(T.tp_workspace_size(T.Op.MLP_FWD, M, h, f, N, dt, act, mode),
                 T.tp_workspace_size(T.Op.MLP_BWD, M, h, f, N, dt, act, mode)))
    T.tp_mlp_fwd(X, W1, Wu if sw else None, W2, None, Y, Yu if sw else None, H, Z, M, h, f, N,
                 dt, act, mode, ws, ws.numel())
    T.tp_mlp_bwd(X, W1, Wu if sw else None, W2, Y, Yu if sw else None, H, dZ, dX, dW1,
                 dWu if sw else None, dW2, M, h, f, N, dt, act, mode, ws, ws.numel())
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    assert guard_intact(fullZ, M) and guard_intact(fulldX, M)
    if sw:
        fr = O.mlp_swiglu_fwd(Xo, W1o, Wuo, W2o, N)
        br = O.mlp_swiglu_bwd(Xo, W1o, Wuo, W2o, dZo, N)
        got = {"G": Y, "U": Yu, "A": H, "Z": Z, "dX": dX, "dWg": dW1, "dWu": dWu, "dWd": dW2}
        ref = {"G": fr["G"], "U": fr["U"], "A": fr["A"], "Z": fr["Z"], "dX": br["dX"],
               "dWg": br["dWg"], "dWu": br["dWu"], "dWd": br["dWd"]}
    else:
        fr = O.mlp_gelu_fwd(Xo, W1o, W2o, N)
        br = O.mlp_gelu_bwd(Xo, W1o, W2o, dZo, N)
        got = {"Y": Y, "H": H, "Z": Z, "dX": dX, "dW1": dW1, "dW2": dW2}
        ref = {"Y": fr["Y"], "H": fr["H"], "Z": fr["Z"], "dX": br["dX"], "dW1": br["dW1"],
               "dW2": br["dW2"]}
    return {k: rel(host(got[k]), ref[k]) for k in got}, {k: host(v) for k, v in got.items()}


@pytest.mark.parametrize("act", [T.Act.GELU, T.Act.SWIGLU])
@pytest.mark.parametrize("mode", [T.Reduce.BUFFERS, T.Reduce.SPLITK])
@pytest.mark.parametrize("N", [1, 2, 4])
def test_mlp_bf16(act, mode, N):
    errs, _ = _mlp_run(act, mode, N, M=333, h=192, f=512)
    for k, e in errs.items():
        assert e <= BF16_TOL, (k, e)


@pytest.mark.parametrize("wide", [0, 2], ids=["pair256", "pair512"])
@pytest.mark.parametrize("act", [T.Act.GELU, T.Act.SWIGLU])
@pytest.mark.parametrize("mode", [T.Reduce.BUFFERS, T.Reduce.SPLITK])
def test_mlp_bf16_pair_tiles(act, mode, wide):
    """Every GEMM of the step on the CTA-pair kernel in one tile width: the paired
    gate/up operands, MN-major weight-gradient operands, the two-segment dX, per-shard
    K-groups and the epilogues that read saved activations."""
    with gemm_tiles(2, wide):
        errs, _ = _mlp_run(act, mode, 2, M=600, h=512, f=1024)
    for k, e in errs.items():
        assert e <= BF16_TOL, (k, e)


@pytest.mark.parametrize("wide", [0, 2], ids=["pair256", "pair512"])
@pytest.mark.parametrize("act", [T.Act.GELU, T.Act.SWIGLU])
def test_mlp_bf16_pair_tiles_many(act, wide):
    """Enough tiles per SM pair that the column GEMM and dA take the TMA-store epilogue
    (at least two tiles per pair), with a ragged M."""
    with gemm_tiles(2, wide):
        errs, _ = _mlp_run(act, T.Reduce.SPLITK, 2, M=2600, h=256, f=4096)
    for k, e in errs.items():
        assert e <= BF16_TOL, (k, e)


@pytest.mark.parametrize("act", [T.Act.GELU, T.Act.SWIGLU])
def test_mlp_bf16_buffers_staged_partials(act):
    """Per-shard fp32 partials (variant A) through the staged TMA-store epilogue: the row
    GEMM and dX have enough tiles (K-groups x 11 x 8) for it, with a ragged M, so the
    partials' 3-D store map (columns, rows, shard) and its clipped last row tile are
    exercised."""
    errs, _ = _mlp_run(act, T.Reduce.BUFFERS, 2, M=2600, h=2048, f=1024)
    for k, e in errs.items():
        assert e <= BF16_TOL, (k, e)


def test_mlp_bf16_multi_tile_k():
    """Several 64-wide K blocks per shard and several M/N tiles with a ragged M tail."""
    errs, _ = _mlp_run(T.Act.GELU, T.Reduce.BUFFERS, 2, M=700, h=384, f=1024)
    for k, e in errs.items():
        assert e <= BF16_TOL, (k, e)


@pytest.mark.parametrize("act", [T.Act.GELU, T.Act.SWIGLU])
@pytest.mark.parametrize("mode", [T.Reduce.BUFFERS, T.Reduce.SPLITK])
def test_mlp_fp32_tiny_config(act, mode):
    """The tiny fp32 workload: X (2, 16, 128), W1 128x512, W2 512x128, N = 2,
    W ~ N(0, 0.02^2), exact erf GELU; FFMA on CUDA cores."""
    errs, _ = _mlp_run(act, mode, 2, M=32, h=128, f=512, dtype="f32", seed0=1000, sigma=0.02)
    for k, e in errs.items():
        assert e <= F32_TOL, (k, e)


def test_mlp_fp32_ragged():
    errs, _ = _mlp_run(T.Act.GELU, T.Reduce.BUFFERS, 3, M=45, h=37, f=99, dtype="f32")
    for k, e in errs.items():
        assert e <= F32_TOL, (k, e)


def test_split_equals_unsplit_on_gpu():
    """N = 4 shards and N = 1 (unsplit) agree on the GPU within the bf16 bound."""
    for act in (T.Act.GELU, T.Act.SWIGLU):
        _, a = _mlp_run(act, T.Reduce.BUFFERS, 4, M=333, h=192, f=512)
        _, b = _mlp_run(act, T.Reduce.SPLITK, 1, M=333, h=192, f=512)
        for k in a:
            assert rel(a[k], b[k]) <= BF16_TOL, (act, k)


def test_deterministic():
    _, a = _mlp_run(T.Act.SWIGLU, T.Reduce.BUFFERS, 2, M=333, h=192, f=512)
    _, b = _mlp_run(T.Act.SWIGLU, T.Reduce.BUFFERS, 2, M=333, h=192, f=512)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


# ---------------------------------------------------------------- bounded waits

def test_wait_timeout_reports_and_recovers():
    """A GEMM whose MMA warp waits on a barrier nothing arrives on stops after the
    time limit, reports TP_ERR_TIMEOUT, and the context stays usable."""
    M, h, f, N = 256, 128, 256, 2
    Xo, X = tensor((M, h), 501)
    Wo, W = tensor((h, f), 502, 0.05)
    out = empty((M, f), bf16)
    T.tp_set_wait_timeout_ns(2_000_000)
    T.tp_debug_inject_wait_fault(True)
    try:
        T.tp_col_linear(X, W, None, None, None, out, M, h, f, N, BF, T.Act.NONE)
        assert T.tp_check_status() == T.Status.TIMEOUT
    finally:
        T.tp_debug_inject_wait_fault(False)
        T.tp_set_wait_timeout_ns(1_000_000_000)
    T.tp_col_linear(X, W, None, None, None, out, M, h, f, N, BF, T.Act.NONE)
    assert T.tp_check_status() == 0
    assert rel(host(out), Xo @ Wo) <= BF16_TOL


# ---------------------------------------------------------------- decode-sized forward

@pytest.mark.parametrize("T_", [1, 8, 32, 64])
@pytest.mark.parametrize("act", [T.Act.GELU, T.Act.SWIGLU])
@pytest.mark.parametrize("mode", [T.Reduce.BUFFERS, T.Reduce.SPLITK])
def test_decode_forward(T_, act, mode):
    M, h, f, N = T_, 256, 1024, 4
    sw = act == T.Act.SWIGLU
    Xo, X = tensor((M, h), 801)
    W1o, W1 = tensor((h, f), 802, 0.05)
    Wuo, Wu = tensor((h, f), 803, 0.05)
    W2o, W2 = tensor((f, h), 804, 0.05)
    H = empty((M, f), bf16)
    Z, full = guarded((M, h), bf16)
    ws = _ws(T.tp_workspace_size(T.Op.MLP_FWD, M, h, f, N, BF, act, mode))
    T.tp_mlp_fwd(X, W1, Wu if sw else None, W2, None, None, None, H, Z, M, h, f, N, BF, act, mode,
                 ws, ws.numel())
    torch.cuda.synchronize()
    ref = O.mlp_swiglu_fwd(Xo, W1o, Wuo, W2o, N) if sw else O.mlp_gelu_fwd(Xo, W1o, W2o, N)
    assert rel(host(H), ref["A"] if sw else ref["H"]) <= BF16_TOL
    assert rel(host(Z), ref["Z"]) <= BF16_TOL
    assert guard_intact(full, M)


# ---------------------------------------------------------------- GELU epilogue precision
#
# The bf16 epilogues compute Phi by an approximation of erf with an absolute error below
# 1.5e-7 on the special-function unit. These inputs make the accumulator of every output
# exactly one chosen bf16 value v (X = a column of ones, W1 holding v in its first row), so
# the epilogue's result can be held to the bf16 rounding of the exact value: |got - ref|
# <= 2^-8 |ref| + 1e-6 (bf16 keeps 8 significant bits; round to nearest). The backward's
# dY = dH * GELU'(Y) reaches dW1 = X^T dY unrounded for M a power of two (dH = 1
# exactly: dZ and W2 hold ones in their first column).

def _gelu_sweep_inputs(M, h, f):
    v = torch.linspace(-9.0, 9.0, f).to(torch.bfloat16)
    X = torch.zeros(M, h, dtype=torch.bfloat16)
    X[:, 0] = 1.0
    W1 = torch.zeros(h, f, dtype=torch.bfloat16)
    W1[0] = v
    W2 = torch.zeros(f, h, dtype=torch.bfloat16)
    W2[:, 0] = 1.0
    dZ = torch.zeros(M, h, dtype=torch.bfloat16)
    dZ[:, 0] = 1.0
    return v.double().numpy(), X.cuda(), W1.cuda(), W2.cuda(), dZ.cuda()


@pytest.mark.parametrize("M,pair,wide", [(128, 1, 1), (256, 2, 0), (256, 2, 2), (4096, 2, 0)],
                         ids=["one-cta", "pair256", "pair512", "pair256-tma"])
def test_gelu_epilogue_precision(M, pair, wide):
    h, f = 64, 4096
    v, X, W1, W2, dZ = _gelu_sweep_inputs(M, h, f)
    e = lambda *s: torch.empty(*s, dtype=bf16, device="cuda")
    Y, H, Z, dX, dW1, dW2 = e(M, f), e(M, f), e(M, h), e(M, h), e(h, f), e(f, h)
    md = T.Reduce.SPLITK
    ws = _ws(max(T.tp_workspace_size(T.Op.MLP_FWD, M, h, f, 1, BF, T.Act.GELU, md),
                 T.tp_workspace_size(T.Op.MLP_BWD, M, h, f, 1, BF, T.Act.GELU, md)))
    with gemm_tiles(pair, wide):
        T.tp_mlp_fwd(X, W1, None, W2, None, Y, None, H, Z, M, h, f, 1, BF, T.Act.GELU, md, ws,
                     ws.numel())
        T.tp_mlp_bwd(X, W1, None, W2, Y, None, H, dZ, dX, dW1, None, dW2, M, h, f, 1, BF,
                     T.Act.GELU, md, ws, ws.numel())
        torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    assert np.array_equal(host(Y[[0, M - 1]]), np.stack([v, v]))
    g, gp = O.gelu(v), O.gelu_prime(v)
    for got in (host(H[0]), host(H[M - 1])):
        assert np.all(np.abs(got - g) <= 2.0 ** -8 * np.abs(g) + 1e-6), np.max(np.abs(got - g))
    if M & (M - 1) == 0:
        got = host(dW1[0]) / M
        assert np.all(np.abs(got - gp) <= 2.0 ** -8 * np.abs(gp) + 1e-6), np.max(np.abs(got - gp))
