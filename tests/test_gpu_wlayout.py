"""The (out, in) weight layout of the Megatron listing (ColumnParallelLinear /
RowParallelLinear keep W for F.linear, Y = X W^T) at the linear entry points:
the MLP forward and backward with TP_W_OUT_IN weights against the fp64 oracle,
which computes with the pages' (in, out) W -- the transpose of the stored matrix.
Gradients come back in the weights' own (out, in) order.

Token counts cover the kernel configurations that read a K-major weight: the decode
configuration (M <= 64, incl. one token), the one-CTA 128 x 256 tile and the
CTA-pair 256 x 256 tile, each with gate/up paired tiles for SwiGLU.
Bar: max|gpu - oracle| / max|oracle| <= 1e-2 (bf16), <= 1e-5 (fp32)."""
import pytest
import torch

from attention_gemms_gb300 import tpmlp as T
from oracle import tp_oracle as O
from tests.helpers import BF16_TOL, F32_TOL, empty, guard_intact, guarded, host, rel, tensor

pytestmark = pytest.mark.gpu
OUT_IN = T.WLayout.OUT_IN


@pytest.fixture(scope="module", autouse=True)
def _lib():
    T.lib()
    torch.cuda.set_device(0)
    T.tp_set_wait_timeout_ns(1_000_000_000)
    yield
    T.tp_set_wait_timeout_ns(0)
    assert T.tp_check_status() == 0


def _run(act, mode, N, M, h, f, dtype="bf16", seed0=900, sigma=0.05):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dt = T.DType.BF16 if dtype == "bf16" else T.DType.F32
    sw = act == T.Act.SWIGLU
    Xo, X = tensor((M, h), seed0 + 1, dtype=dtype)
    W1o, W1 = tensor((h, f), seed0 + 2, sigma, dtype=dtype)     # the pages' (in, out) W1
    Wuo, Wu = tensor((h, f), seed0 + 3, sigma, dtype=dtype)
    W2o, W2 = tensor((f, h), seed0 + 4, sigma, dtype=dtype)
    dZo, dZ = tensor((M, h), seed0 + 5, dtype=dtype)
    W1t, Wut, W2t = (w.t().contiguous() for w in (W1, Wu, W2))  # stored (out, in)
    Y, Yu, H = empty((M, f), tdt), empty((M, f), tdt), empty((M, f), tdt)
    Z, fullZ = guarded((M, h), tdt)
    dX, fulldX = guarded((M, h), tdt)
    dW1, dWu, dW2 = empty((f, h), tdt), empty((f, h), tdt), empty((h, f), tdt)
    nb = max(T.tp_workspace_size(T.Op.MLP_FWD, M, h, f, N, dt, act, mode),
             T.tp_workspace_size(T.Op.MLP_BWD, M, h, f, N, dt, act, mode))
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    T.tp_mlp_fwd(X, W1t, Wut if sw else None, W2t, None, Y, Yu if sw else None, H, Z, M, h, f, N,
                 dt, act, mode, ws, ws.numel(), w_layout=OUT_IN)
    T.tp_mlp_bwd(X, W1t, Wut if sw else None, W2t, Y, Yu if sw else None, H, dZ, dX, dW1,
                 dWu if sw else None, dW2, M, h, f, N, dt, act, mode, ws, ws.numel(),
                 w_layout=OUT_IN)
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    assert guard_intact(fullZ, M) and guard_intact(fulldX, M)
    if sw:
        fr = O.mlp_swiglu_fwd(Xo, W1o, Wuo, W2o, N)
        br = O.mlp_swiglu_bwd(Xo, W1o, Wuo, W2o, dZo, N)
        got = {"G": Y, "U": Yu, "A": H, "Z": Z, "dX": dX, "dWg": dW1, "dWu": dWu, "dWd": dW2}
        ref = {"G": fr["G"], "U": fr["U"], "A": fr["A"], "Z": fr["Z"], "dX": br["dX"],
               "dWg": br["dWg"].T, "dWu": br["dWu"].T, "dWd": br["dWd"].T}
    else:
        fr = O.mlp_gelu_fwd(Xo, W1o, W2o, N)
        br = O.mlp_gelu_bwd(Xo, W1o, W2o, dZo, N)
        got = {"Y": Y, "H": H, "Z": Z, "dX": dX, "dW1": dW1, "dW2": dW2}
        ref = {"Y": fr["Y"], "H": fr["H"], "Z": fr["Z"], "dX": br["dX"], "dW1": br["dW1"].T,
               "dW2": br["dW2"].T}
    return {k: rel(host(got[k]), ref[k]) for k in got}


@pytest.mark.parametrize("act", [T.Act.GELU, T.Act.SWIGLU])
@pytest.mark.parametrize("mode", [T.Reduce.BUFFERS, T.Reduce.SPLITK])
@pytest.mark.parametrize("M", [1, 40, 200, 333])
def test_mlp_out_in_weights_bf16(act, mode, M):
    errs = _run(act, mode, 2 if M < 300 else 4, M, 192, 512)
    assert max(errs.values()) <= BF16_TOL, errs


@pytest.mark.parametrize("act", [T.Act.GELU, T.Act.SWIGLU])
def test_mlp_out_in_weights_f32(act):
    errs = _run(act, T.Reduce.BUFFERS, 2, 37, 96, 160, dtype="f32", seed0=950)
    assert max(errs.values()) <= F32_TOL, errs


def test_row_linear_out_in_matches_in_out():
    """One row-parallel call in each layout on the same values: both agree with the
    oracle, and with each other within the same bound."""
    M, k, n, N = 300, 512, 256, 4
    Xo, X = tensor((M, k), 981)
    Wo, W = tensor((k, n), 982, 0.05)
    out_a = torch.empty((M, n), dtype=torch.bfloat16, device="cuda")
    out_b = torch.empty_like(out_a)
    for mode in (T.Reduce.BUFFERS, T.Reduce.SPLITK):
        nb = T.tp_workspace_size(T.Op.ROW_LINEAR, M, k, n, N, T.DType.BF16, T.Act.NONE, mode)
        ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
        T.tp_row_linear(X, W, None, out_a, M, k, n, N, T.DType.BF16, mode, ws, ws.numel())
        T.tp_row_linear(X, W.t().contiguous(), None, out_b, M, k, n, N, T.DType.BF16, mode, ws,
                        ws.numel(), w_layout=OUT_IN)
        torch.cuda.synchronize()
        ref = O.row_linear(Xo, Wo, N)
        assert rel(host(out_a), ref) <= BF16_TOL
        assert rel(host(out_b), ref) <= BF16_TOL
        assert rel(host(out_b), host(out_a)) <= BF16_TOL
