"""Parity at the full benchmark sizes, in the launch configuration bench.py times
(tp_col_linear -> tp_row_linear -> tp_mlp_bwd), on sampled outputs the oracle
computes one by one:
  * token rows of Y/G, U, H/A, Z and dX (each needs only that row's inputs),
  * hidden (ffn) columns of dW1/dWg, dWu and rows of dW2/dWd (the column-restricted
    backward of the oracle),
including tile edges and shard boundaries. Bar: 1e-2 relative to max|oracle| of
the sampled block."""
import numpy as np
import pytest
import torch

import bench
from attention_gemms_gb300 import synth
from attention_gemms_gb300 import tpmlp as T
from oracle import tp_oracle as O
from tests.helpers import BF16_TOL, host, rel

pytestmark = pytest.mark.gpu


def _sample(n, k, extra, seed):
    r = np.random.default_rng(seed)
    s = set(int(x) for x in r.choice(n, size=k, replace=False)) | {e for e in extra if 0 <= e < n}
    return np.array(sorted(s))


@pytest.mark.parametrize("workload", ["c5", "c3"])
@pytest.mark.parametrize("mode", ["splitk", "buffers"])
def test_full_size_parity(workload, mode):
    T.lib()
    w = bench.WORKLOADS[workload]
    M, h, f, N = w["b"] * w["s"], w["h"], w["f"], w["N"]
    sw = w["act"] == "swiglu"
    act = T.Act.SWIGLU if sw else T.Act.GELU
    md = T.Reduce.SPLITK if mode == "splitk" else T.Reduce.BUFFERS
    BF = T.DType.BF16
    dev = torch.device("cuda", 0)
    d, hostin = bench.make_inputs(w, 0, dev)
    e = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device=dev)
    Y, Yu, H, Z, dX = e(M, f), (e(M, f) if sw else None), e(M, f), e(M, h), e(M, h)
    dW1, dW1u, dW2 = e(h, f), (e(h, f) if sw else None), e(f, h)
    wsb = max(T.tp_workspace_size(T.Op.ROW_LINEAR, M, f, h, N, BF, T.Act.NONE, md),
              T.tp_workspace_size(T.Op.MLP_BWD, M, h, f, N, BF, act, md))
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    T.tp_col_linear(d["X"], d["W1"], d["W1u"], Y, Yu, H, M, h, f, N, BF, act)
    T.tp_row_linear(H, d["W2"], None, Z, M, f, h, N, BF, md, ws, ws.numel())
    T.tp_mlp_bwd(d["X"], d["W1"], d["W1u"], d["W2"], Y, Yu, H, d["dZ"], dX, dW1, dW1u, dW2,
                 M, h, f, N, BF, act, md, ws, ws.numel())
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0

    rows = _sample(M, 40, [0, 1, 127, 128, 255, M // 2, M - 129, M - 128, M - 1], 11)
    fs = f // N
    cols = _sample(f, 40, [0, 127, 128, fs - 1, fs, 2 * fs - 1, f - 1], 12)
    f64 = lambda a: synth.to_f64(a, "bf16")
    X = f64(hostin["X"])
    dZ = f64(hostin["dZ"])
    W1, W2 = f64(hostin["W1"]), f64(hostin["W2"])
    W1u = f64(hostin["W1u"]) if sw else None
    ri = torch.as_tensor(rows, device=dev)
    ci = torch.as_tensor(cols, device=dev)
    if sw:
        fr = O.mlp_swiglu_fwd(X[rows], W1, W1u, W2, N)
        br = O.mlp_swiglu_bwd(X[rows], W1, W1u, W2, dZ[rows], N)
        dw = O.mlp_swiglu_dW_cols(X, W1, W1u, W2, dZ, cols)
        checks = {"G": (Y, fr["G"]), "U": (Yu, fr["U"]), "A": (H, fr["A"]), "Z": (Z, fr["Z"]),
                  "dX": (dX, br["dX"])}
        wchk = {"dWg": (dW1, dw["dWg"], 1), "dWu": (dW1u, dw["dWu"], 1), "dWd": (dW2, dw["dWd"], 0)}
    else:
        fr = O.mlp_gelu_fwd(X[rows], W1, W2, N)
        br = O.mlp_gelu_bwd(X[rows], W1, W2, dZ[rows], N)
        dw = O.mlp_gelu_dW_cols(X, W1, W2, dZ, cols)
        checks = {"Y": (Y, fr["Y"]), "H": (H, fr["H"]), "Z": (Z, fr["Z"]), "dX": (dX, br["dX"])}
        wchk = {"dW1": (dW1, dw["dW1"], 1), "dW2": (dW2, dw["dW2"], 0)}
    errs = {}
    for k, (g, ref) in checks.items():
        errs[k] = rel(host(g.index_select(0, ri)), ref)
    for k, (g, ref, axis) in wchk.items():
        got = g.index_select(1, ci) if axis == 1 else g.index_select(0, ci)
        errs[k] = rel(host(got), ref)
    for k, v in errs.items():
        assert v <= BF16_TOL, (workload, mode, k, v)


@pytest.mark.parametrize("T_", [1, 8, 32, 64])
def test_decode_full_size_parity(T_):
    """The decode sweep's shapes (h=8192, ffn=28672, N=8, SwiGLU) in bench.py's launch
    configuration (tp_col_linear -> tp_row_linear with fp32 shard partials); the
    oracle computes every output."""
    T.lib()
    w = bench.DECODE
    h, f, N, c = w["h"], w["f"], w["N"], w["cfg"]
    BF = T.DType.BF16
    dev = torch.device("cuda", 0)
    arrs = {k: synth.normal(s, synth.seed_of(c, n) + ex, sg, "bf16")
            for k, s, n, sg, ex in [("X", (T_, h), "X", 1.0, T_), ("Wg", (h, f), "Wg", 0.02, 0),
                                    ("Wu", (h, f), "Wu", 0.02, 0), ("Wd", (f, h), "Wd", 0.02, 0)]}
    d = {k: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev) for k, a in arrs.items()}
    A = torch.empty((T_, f), dtype=torch.bfloat16, device=dev)
    Z = torch.empty((T_, h), dtype=torch.bfloat16, device=dev)
    wsb = T.tp_workspace_size(T.Op.ROW_LINEAR, T_, f, h, N, BF, T.Act.NONE, T.Reduce.BUFFERS)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    T.tp_col_linear(d["X"], d["Wg"], d["Wu"], None, None, A, T_, h, f, N, BF, T.Act.SWIGLU)
    T.tp_row_linear(A, d["Wd"], None, Z, T_, f, h, N, BF, T.Reduce.BUFFERS, ws, wsb)
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    f64 = {k: synth.to_f64(a, "bf16") for k, a in arrs.items()}
    ref = O.mlp_swiglu_fwd(f64["X"], f64["Wg"], f64["Wu"], f64["Wd"], N)
    assert rel(host(A), ref["A"]) <= BF16_TOL
    assert rel(host(Z), ref["Z"]) <= BF16_TOL
