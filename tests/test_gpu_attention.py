"""GPU parity of LayerNorm, the head-sharded attention block and the pre-LN layer
against the fp64 oracle (every output, element by element). The layer test runs
the page-2 layer's exact configuration: b=8, s=128, h=128, 8 heads (d=16),
ffn=512, N=2, bf16, weights ~N(0, 0.02^2)."""
import numpy as np
import pytest
import torch

from attention_gemms_gb300 import tpmlp as T
from oracle import tp_oracle as O
from tests.helpers import BF16_TOL, F32_TOL, empty, host, rel, tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    T.lib()
    T.tp_set_wait_timeout_ns(1_000_000_000)
    yield
    T.tp_set_wait_timeout_ns(0)
    assert T.tp_check_status() == 0


def _ws(n):
    return torch.empty(max(int(n), 256), dtype=torch.uint8, device="cuda")


def _gb(h, seed):
    go, g = tensor((h,), seed, 0.1, dtype="f32")
    bo, b = tensor((h,), seed + 1, 0.1, dtype="f32")
    return 1.0 + go, (g + 1.0).contiguous(), bo, b


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
# up to 512 rows the parameter gradients are summed in one cluster launch (512: eight
# chunks of 64 rows), up to 1024 in a 16-CTA cluster where the device places one, above
# it by the partial + final kernels
@pytest.mark.parametrize("Mh", [(100, 128), (33, 200), (1, 8192), (512, 256), (513, 64),
                                (1024, 128), (1025, 64)])
def test_layernorm(dtype, Mh):
    M, h = Mh
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dt = T.DType.BF16 if dtype == "bf16" else T.DType.F32
    tol = BF16_TOL if dtype == "bf16" else F32_TOL
    xo, x = tensor((M, h), 1101, 2.0, dtype=dtype)
    go, g, bo, b = _gb(h, 1102)
    dyo, dy = tensor((M, h), 1104, dtype=dtype)
    ro, r = tensor((M, h), 1105, dtype=dtype)
    y = empty((M, h), tdt)
    mean, rstd = empty((M,), torch.float32), empty((M,), torch.float32)
    T.tp_layernorm_fwd(x, g, b, y, mean, rstd, M, h, 1e-5, dt)
    dx = empty((M, h), tdt)
    dg, db = empty((h,), torch.float32), empty((h,), torch.float32)
    ws = _ws(T.tp_workspace_size(T.Op.LAYERNORM_BWD, M, h, 0, 1, dt))
    T.tp_layernorm_bwd(x, g, mean, rstd, dy, r, dx, dg, db, M, h, dt, ws, ws.numel())
    torch.cuda.synchronize()
    yr, mr, rr = O.layernorm_fwd(xo, go, bo)
    dxr, dgr, dbr = O.layernorm_bwd(xo, go, dyo)
    assert rel(host(y), yr) <= tol
    assert rel(host(mean), mr) <= tol and rel(host(rstd), rr) <= tol
    assert rel(host(dx), dxr + ro) <= tol
    assert rel(host(dg), dgr) <= tol and rel(host(db), dbr) <= tol


def _attn_case(b, s, h, heads, N, causal, mode, dtype="bf16", seed=1200):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dt = T.DType.BF16 if dtype == "bf16" else T.DType.F32
    M = b * s
    xo, x = tensor((M, h), seed, dtype=dtype)
    go, g, bo, bb = _gb(h, seed + 1)
    Wqkvo, Wqkv = tensor((h, 3 * h), seed + 3, 0.1, dtype=dtype)
    Woo, Wo = tensor((h, h), seed + 4, 0.1, dtype=dtype)
    douto, dout = tensor((M, h), seed + 5, dtype=dtype)
    xn, qkv, o, out = empty((M, h), tdt), empty((M, 3 * h), tdt), empty((M, h), tdt), empty((M, h), tdt)
    mean, rstd = empty((M,), torch.float32), empty((M,), torch.float32)
    lse = empty((b, heads, s), torch.float32)
    md = T.Reduce.SPLITK if mode == "splitk" else T.Reduce.BUFFERS
    ws = _ws(max(T.tp_workspace_size(T.Op.ATTN_PROJ_FWD, M, h, 0, N, dt, T.Act.NONE, md),
                 T.tp_workspace_size(T.Op.ATTN_PROJ_BWD, M, h, 0, N, dt, T.Act.NONE, md)))
    T.tp_attn_proj_fwd(x, g, bb, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, out, b, s, h, heads, N,
                       causal, dt, md, ws, ws.numel())
    dx = empty((M, h), tdt)
    dg, db = empty((h,), torch.float32), empty((h,), torch.float32)
    dWqkv, dWo = empty((h, 3 * h), tdt), empty((h, h), tdt)
    T.tp_attn_proj_bwd(x, g, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, dout, dx, dg, db, dWqkv, dWo,
                       b, s, h, heads, N, causal, dt, md, ws, ws.numel())
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    fr = O.attn_block_fwd(xo, b, s, go, bo, Wqkvo, Woo, heads, N, causal)
    br = O.attn_block_bwd(xo, b, s, go, bo, Wqkvo, Woo, heads, N, douto, causal)
    got = {"xn": xn, "QKV": qkv, "O": o, "out": out, "dx": dx, "dgamma": dg, "dbeta": db,
           "dWqkv": dWqkv, "dWo": dWo}
    ref = {"xn": fr["xn"], "QKV": fr["QKV"], "O": fr["O"], "out": fr["out"], "dx": br["dx"],
           "dgamma": br["dgamma"], "dbeta": br["dbeta"], "dWqkv": br["dWqkv"], "dWo": br["dWo"]}
    return {k: rel(host(got[k]), ref[k]) for k in got}


@pytest.mark.parametrize("heads", [8, 4, 2])          # head_dim 16, 32, 64
@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("mode", ["buffers", "splitk"])
def test_attn_block_bf16(heads, causal, mode):
    errs = _attn_case(b=2, s=80, h=128, heads=heads, N=2, causal=causal, mode=mode)
    for k, e in errs.items():
        assert e <= BF16_TOL, (k, e)


@pytest.mark.parametrize("causal", [0, 1])
def test_attn_block_bf16_multi_tile(causal):
    """head_dim 64 (the tensor-core kernels) over three 128-row tiles, the last ragged."""
    errs = _attn_case(b=2, s=300, h=128, heads=2, N=2, causal=causal, mode="buffers")
    for k, e in errs.items():
        assert e <= BF16_TOL, (k, e)


def test_attn_block_f32():
    errs = _attn_case(b=2, s=70, h=64, heads=4, N=2, causal=0, mode="buffers", dtype="f32")
    for k, e in errs.items():
        assert e <= F32_TOL, (k, e)


@pytest.mark.parametrize("mode", ["buffers", "splitk"])
def test_page2_layer_fwd_bwd(mode):
    """The page-2 transformer layer at its own size, forward and backward."""
    b, s, h, heads, f, N = 8, 128, 128, 8, 512, 2
    M = b * s
    dt, tdt = T.DType.BF16, torch.bfloat16
    c = 2000
    xo, x = tensor((M, h), c + 1)
    g1o, g1, b1o, b1 = _gb(h, c + 8)
    g2o, g2, b2o, b2 = _gb(h, c + 10)
    Wqkvo, Wqkv = tensor((h, 3 * h), c + 6, 0.02)
    Woo, Wo = tensor((h, h), c + 7, 0.02)
    W1o, W1 = tensor((h, f), c + 2, 0.02)
    W2o, W2 = tensor((f, h), c + 4, 0.02)
    douto, dout = tensor((M, h), c + 5)
    e = lambda *sh, dty=tdt: empty(sh, dty)
    f32 = torch.float32
    sv = dict(xn1=e(M, h), mean1=e(M, dty=f32), rstd1=e(M, dty=f32), qkv=e(M, 3 * h), o=e(M, h),
              lse=e(b, heads, s, dty=f32), x1=e(M, h), xn2=e(M, h), mean2=e(M, dty=f32),
              rstd2=e(M, dty=f32), y=e(M, f), hh=e(M, f))
    gr = dict(dWqkv=e(h, 3 * h), dWo=e(h, h), dW1=e(h, f), dW2=e(f, h), dgamma1=e(h, dty=f32),
              dbeta1=e(h, dty=f32), dgamma2=e(h, dty=f32), dbeta2=e(h, dty=f32))
    W = T.make_struct(T.LayerWeights, Wqkv=Wqkv, Wo=Wo, W1=W1, W2=W2, gamma1=g1, beta1=b1,
                      gamma2=g2, beta2=b2)
    S = T.make_struct(T.LayerSaved, **sv)
    G = T.make_struct(T.LayerGrads, **gr)
    md = T.Reduce.SPLITK if mode == "splitk" else T.Reduce.BUFFERS
    ws = _ws(max(T.tp_workspace_size(T.Op.LAYER_FWD, M, h, f, N, dt, T.Act.GELU, md),
                 T.tp_workspace_size(T.Op.LAYER_BWD, M, h, f, N, dt, T.Act.GELU, md)))
    out, dx = e(M, h), e(M, h)
    T.tp_layer_fwd(x, W, S, out, b, s, h, f, heads, N, 0, dt, md, ws, ws.numel())
    T.tp_layer_bwd(x, W, S, dout, dx, G, b, s, h, f, heads, N, 0, dt, md, ws, ws.numel())
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    p = {"gamma1": g1o, "beta1": b1o, "Wqkv": Wqkvo, "Wo": Woo, "gamma2": g2o, "beta2": b2o,
         "W1": W1o, "W2": W2o}
    fr = O.layer_fwd(xo, b, s, p, heads, N)
    br = O.layer_bwd(xo, b, s, p, heads, N, douto)
    errs = {"out": rel(host(out), fr["out"]), "x1": rel(host(sv["x1"]), fr["x1"]),
            "dx": rel(host(dx), br["dx"])}
    for k in ("dWqkv", "dWo", "dW1", "dW2", "dgamma1", "dbeta1", "dgamma2", "dbeta2"):
        errs[k] = rel(host(gr[k]), br[k])
    for k, v in errs.items():
        assert v <= BF16_TOL, (mode, k, v)
