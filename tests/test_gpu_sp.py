"""GPU parity of the sequence-parallel pre-LN MLP sub-block (tp_sp_mlp_fwd / _bwd)
against the fp64 oracle, element by element: per-rank LN, the tensor-parallel MLP,
the reduce-scatter with the residual rows, and in the backward the reduce-scattered
input gradient, per-rank LN parameter gradients and their sum over the ranks."""
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


def _run(M, h, f, N, act, mode, dtype="bf16", seed=4000):
    dt = T.DType.BF16 if dtype == "bf16" else T.DType.F32
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    A = T.Act.SWIGLU if act == "swiglu" else T.Act.GELU
    md = T.Reduce.SPLITK if mode == "splitk" else T.Reduce.BUFFERS
    sw = act == "swiglu"
    xo, x = tensor((M, h), seed, dtype=dtype)
    go, g = tensor((h,), seed + 1, 0.3, dtype="f32")
    bo, b = tensor((h,), seed + 2, 0.3, dtype="f32")
    go, g = go + 1.0, (g + 1.0).contiguous()
    W1o, W1 = tensor((h, f), seed + 3, 0.05, dtype=dtype)
    Wuo, Wu = tensor((h, f), seed + 4, 0.05, dtype=dtype)
    W2o, W2 = tensor((f, h), seed + 5, 0.05, dtype=dtype)
    do, dout = tensor((M, h), seed + 6, dtype=dtype)
    e = lambda *s, dty=tdt: torch.empty(s, dtype=dty, device="cuda")
    f32 = torch.float32
    xn, mean, rstd = e(M, h), e(M, dty=f32), e(M, dty=f32)
    Y, Yu, H = e(M, f), (e(M, f) if sw else None), e(M, f)
    out, out_full = guarded((M, h), tdt)
    ws = _ws(max(T.tp_workspace_size(T.Op.SP_MLP_FWD, M, h, f, N, dt, A, md),
                 T.tp_workspace_size(T.Op.SP_MLP_BWD, M, h, f, N, dt, A, md)))
    T.tp_sp_mlp_fwd(x, g, b, W1, Wu if sw else None, W2, xn, mean, rstd, Y, Yu, H, out, M, h, f,
                    N, dt, A, md, ws, ws.numel())
    dx, dx_full = guarded((M, h), tdt)
    dg, db = e(h, dty=f32), e(h, dty=f32)
    dgr, dbr = e(N, h, dty=f32), e(N, h, dty=f32)
    dW1, dWu, dW2 = e(h, f), (e(h, f) if sw else None), e(f, h)
    T.tp_sp_mlp_bwd(x, g, W1, Wu if sw else None, W2, xn, mean, rstd, Y, Yu, H, dout, dx, dg, db,
                    dgr, dbr, dW1, dWu, dW2, M, h, f, N, dt, A, md, ws, ws.numel())
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    assert guard_intact(out_full, M) and guard_intact(dx_full, M)
    u = Wuo if sw else None
    fr = O.sp_mlp_block_fwd(xo, go, bo, W1o, W2o, N, act, u)
    br = O.sp_mlp_block_bwd(xo, go, bo, W1o, W2o, N, do, act, u)
    got = {"xn": xn, "mean": mean, "rstd": rstd, "out": out, "dx": dx, "dgamma": dg,
           "dbeta": db, "dgamma_ranks": dgr, "dbeta_ranks": dbr, "dW1": dW1, "dW2": dW2}
    ref = {"xn": fr["xn"], "mean": fr["mean"], "rstd": fr["rstd"], "out": fr["out"],
           "dx": br["dx"], "dgamma": br["dgamma"], "dbeta": br["dbeta"],
           "dgamma_ranks": br["dgamma_ranks"], "dbeta_ranks": br["dbeta_ranks"],
           "dW1": br["dW1"], "dW2": br["dW2"]}
    if sw:
        got["dW1u"], ref["dW1u"] = dWu, br["dW1u"]
    errs = {k: rel(host(got[k]), ref[k]) for k in got}
    return errs, dg, dgr, db, dbr


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("mode", ["buffers", "splitk"])
@pytest.mark.parametrize("N", [2, 4])
def test_sp_mlp_bf16(act, mode, N):
    errs, *_ = _run(M=4 * 97, h=256, f=512, N=N, act=act, mode=mode)
    for k, v in errs.items():
        assert v <= BF16_TOL, (k, v)


def test_sp_mlp_f32():
    errs, *_ = _run(M=3 * 40, h=96, f=192, N=3, act="gelu", mode="buffers", dtype="f32")
    for k, v in errs.items():
        assert v <= F32_TOL, (k, v)


def test_sp_rank_gradients_sum_in_rank_order():
    """dgamma is the fp32 sum of the per-rank gradients taken in rank order."""
    _, dg, dgr, db, dbr = _run(M=8 * 40, h=128, f=512, N=8, act="gelu", mode="splitk")
    for tot, per in ((dg, dgr), (db, dbr)):
        p = per.cpu().numpy()
        acc = np.zeros(p.shape[1], dtype=np.float32)
        for r in range(p.shape[0]):
            acc = acc + p[r]
        assert np.array_equal(acc, tot.cpu().numpy())


def test_sp_one_rank_equals_plain_block():
    """N = 1: LN then the ordinary tensor-parallel MLP with the residual, bit for bit."""
    M, h, f = 200, 128, 256
    dt, A, md = T.DType.BF16, T.Act.GELU, T.Reduce.SPLITK
    x = tensor((M, h), 4101)[1]
    g = torch.ones(h, device="cuda")
    b = torch.zeros(h, device="cuda")
    W1, W2 = tensor((h, f), 4102, 0.05)[1], tensor((f, h), 4103, 0.05)[1]
    e = lambda *s, dty=torch.bfloat16: torch.empty(s, dtype=dty, device="cuda")
    xn, mean, rstd, Y, H, out = e(M, h), e(M, dty=torch.float32), e(M, dty=torch.float32), e(M, f), e(M, f), e(M, h)
    ws = _ws(T.tp_workspace_size(T.Op.SP_MLP_FWD, M, h, f, 1, dt, A, md))
    T.tp_sp_mlp_fwd(x, g, b, W1, None, W2, xn, mean, rstd, Y, None, H, out, M, h, f, 1, dt, A, md,
                    ws, ws.numel())
    xn2, Y2, H2, out2 = e(M, h), e(M, f), e(M, f), e(M, h)
    T.tp_layernorm_fwd(x, g, b, xn2, None, None, M, h, 1e-5, dt)
    T.tp_mlp_fwd(xn2, W1, None, W2, x, Y2, None, H2, out2, M, h, f, 1, dt, A, md, ws, ws.numel())
    torch.cuda.synchronize()
    assert torch.equal(xn, xn2) and torch.equal(H, H2) and torch.equal(out, out2)


def test_sp_rows_must_split_over_ranks():
    dt, A, md = T.DType.BF16, T.Act.GELU, T.Reduce.SPLITK
    t = torch.empty(64 * 256, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(128, device="cuda")
    with pytest.raises(T.TpError) as e:
        T.tp_sp_mlp_fwd(t, g, g, t, None, t, t, g, g, t, None, t, t, 10, 128, 256, 4, dt, A, md,
                        None, 0)
    assert e.value.status == T.Status.SHAPE
