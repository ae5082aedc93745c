"""GPU parity of the shard sum fused with LayerNorm (tp_shard_reduce_ln) and of the
row-parallel linear feeding it (tp_row_linear_ln) against the fp64 oracle, element
by element. Widths cover every row-group shape of the kernel (one warp for 8 rows
up to eight warps holding 8 chunks each), ragged row counts and the largest width."""
import numpy as np
import pytest
import torch

from attention_gemms_gb300 import tpmlp as T
from oracle import tp_oracle as O
from tests.helpers import BF16_TOL, F32_TOL, guard_intact, guarded, host, rel, tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    T.lib()
    torch.cuda.set_device(0)
    T.tp_set_wait_timeout_ns(1_000_000_000)
    yield
    T.tp_set_wait_timeout_ns(0)
    assert T.tp_check_status() == 0


def _ws(nbytes):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")


def _gb(h, seed):
    go, g = tensor((h,), seed, 0.5, dtype="f32")
    bo, b = tensor((h,), seed + 1, 0.5, dtype="f32")
    return go + 1.0, (g + 1.0).contiguous(), bo, b


def _dts(dtype):
    if dtype == "bf16":
        return T.DType.BF16, torch.bfloat16, BF16_TOL
    return T.DType.F32, torch.float32, F32_TOL


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N,M,h", [(1, 9, 8), (2, 37, 128), (3, 41, 200), (4, 19, 1032),
                                   (8, 13, 4096), (4, 11, 8192), (2, 5, 16384)])
def test_shard_reduce_ln(dtype, N, M, h):
    dt, tdt, tol = _dts(dtype)
    Po, P = tensor((N, M, h), 3001, dtype="f32")
    Ro, R = tensor((M, h), 3002, dtype=dtype)
    go, g, bo, b = _gb(h, 3003)
    S, Sf = guarded((M, h), tdt)
    Y, Yf = guarded((M, h), tdt)
    mean, meanf = guarded((M,), torch.float32)
    rstd, rstdf = guarded((M,), torch.float32)
    T.tp_shard_reduce_ln(P, R, g, b, S, Y, mean, rstd, N, M, h, 1e-5, dt)
    torch.cuda.synchronize()
    x, y, mu, rs = O.shard_reduce_ln(list(Po), Ro, go, bo)
    assert rel(host(S), x) <= (4e-3 if dtype == "bf16" else 1e-6)
    assert rel(host(Y), y) <= tol
    assert rel(host(mean), mu) <= tol and rel(host(rstd), rs) <= tol
    for full, rows in ((Sf, M), (Yf, M), (meanf, M), (rstdf, M)):
        assert guard_intact(full, rows)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_shard_reduce_ln_optional_outputs(dtype):
    """No residual, no sum_out, no statistics: y alone, still LN of the rounded sum."""
    dt, tdt, tol = _dts(dtype)
    N, M, h = 3, 50, 512
    Po, P = tensor((N, M, h), 3011, dtype="f32")
    go, g, bo, b = _gb(h, 3012)
    Y, Yf = guarded((M, h), tdt)
    T.tp_shard_reduce_ln(P, None, g, b, None, Y, None, None, N, M, h, 1e-5, dt)
    torch.cuda.synchronize()
    assert rel(host(Y), O.shard_reduce_ln(list(Po), None, go, bo)[1]) <= tol
    assert guard_intact(Yf, M)


def test_shard_reduce_ln_constant_rows_give_beta():
    """A row whose sum is constant normalises to beta (variance 0, eps keeps rstd finite)."""
    N, M, h = 2, 4, 256
    P = torch.full((N, M, h), 0.375, dtype=torch.float32, device="cuda")
    go, g, bo, b = _gb(h, 3021)
    Y = torch.empty((M, h), dtype=torch.float32, device="cuda")
    T.tp_shard_reduce_ln(P, None, g, b, None, Y, None, None, N, M, h, 1e-5, T.DType.F32)
    torch.cuda.synchronize()
    assert np.allclose(host(Y), np.broadcast_to(bo, (M, h)), atol=1e-6)


def test_shard_reduce_ln_empty_and_errors():
    g = torch.ones(64, dtype=torch.float32, device="cuda")
    P = torch.zeros((2, 1, 64), dtype=torch.float32, device="cuda")
    Y = torch.empty((1, 64), dtype=torch.float32, device="cuda")
    n0 = T.tp_launch_count()
    T.tp_shard_reduce_ln(P, None, g, g, None, Y, None, None, 2, 0, 64, 1e-5, T.DType.F32)
    assert T.tp_launch_count() == n0  # M = 0: nothing to do, nothing launched
    with pytest.raises(T.TpError) as e:
        T.tp_shard_reduce_ln(P, None, g, g, None, Y, None, None, 2, 1, 60, 1e-5, T.DType.F32)
    assert e.value.status == T.Status.SHAPE
    with pytest.raises(T.TpError) as e:
        T.tp_shard_reduce_ln(P, None, g, g, None, Y, None, None, 2, 1, 16392, 1e-5, T.DType.F32)
    assert e.value.status == T.Status.SHAPE
    with pytest.raises(T.TpError) as e:
        T.tp_shard_reduce_ln(P, None, g, g, None, None, None, None, 2, 1, 64, 1e-5, T.DType.F32)
    assert e.value.status == T.Status.INVALID_ARG


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mode", ["buffers", "splitk"])
@pytest.mark.parametrize("N,M,k,n", [(2, 333, 256, 192), (4, 200, 512, 1024)])
def test_row_linear_ln(dtype, mode, N, M, k, n):
    dt, tdt, tol = _dts(dtype)
    md = T.Reduce.SPLITK if mode == "splitk" else T.Reduce.BUFFERS
    Xo, X = tensor((M, k), 3101, dtype=dtype)
    Wo, W = tensor((k, n), 3102, 0.05, dtype=dtype)
    Ro, R = tensor((M, n), 3103, dtype=dtype)
    go, g, bo, b = _gb(n, 3104)
    S, Sf = guarded((M, n), tdt)
    Y, Yf = guarded((M, n), tdt)
    mean = torch.empty(M, dtype=torch.float32, device="cuda")
    rstd = torch.empty(M, dtype=torch.float32, device="cuda")
    ws = _ws(T.tp_workspace_size(T.Op.ROW_LINEAR, M, k, n, N, dt, T.Act.NONE, md))
    T.tp_row_linear_ln(X, W, R, g, b, S, Y, mean, rstd, M, k, n, N, 1e-5, dt, md, ws, ws.numel())
    torch.cuda.synchronize()
    x, y, mu, rs = O.shard_reduce_ln(O.row_partials(Xo, Wo, N), Ro, go, bo)
    assert rel(host(S), x) <= tol
    assert rel(host(Y), y) <= tol
    assert rel(host(mean), mu) <= tol and rel(host(rstd), rs) <= tol
    assert guard_intact(Sf, M) and guard_intact(Yf, M)


def test_row_linear_ln_modes_agree_with_unfused_path():
    """Buffers mode (fused) and the unfused row linear + LayerNorm give the same sum
    bit for bit (same GEMM partials, same shard order) and LN within rounding."""
    N, M, k, n = 4, 256, 1024, 512
    dt = T.DType.BF16
    X = tensor((M, k), 3201)[1]
    W = tensor((k, n), 3202, 0.05)[1]
    R = tensor((M, n), 3203)[1]
    g, b = _gb(n, 3204)[1], _gb(n, 3204)[3]
    ws = _ws(T.tp_workspace_size(T.Op.ROW_LINEAR, M, k, n, N, dt, T.Act.NONE, T.Reduce.BUFFERS))
    S1, Y1 = torch.empty((M, n), dtype=torch.bfloat16, device="cuda"), torch.empty((M, n), dtype=torch.bfloat16, device="cuda")
    T.tp_row_linear_ln(X, W, R, g, b, S1, Y1, None, None, M, k, n, N, 1e-5, dt, T.Reduce.BUFFERS,
                       ws, ws.numel())
    S2, Y2 = torch.empty_like(S1), torch.empty_like(Y1)
    T.tp_row_linear(X, W, R, S2, M, k, n, N, dt, T.Reduce.BUFFERS, ws, ws.numel())
    T.tp_layernorm_fwd(S2, g, b, Y2, None, None, M, n, 1e-5, dt)
    torch.cuda.synchronize()
    assert torch.equal(S1, S2)
    assert rel(host(Y1), host(Y2)) <= 4e-3
