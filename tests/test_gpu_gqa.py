"""GPU parity of the head-sharded grouped-query attention block (tp_gqa_*) against the
fp64 oracle, element by element: the packed sharded weight, forward (xn, qkv, O, out)
and backward (dx, dgamma, dbeta, dWqkv with the replicas' all-reduced key/value
gradients, dWo), for shard counts below, at and above the key/value head count."""
import numpy as np
import pytest
import torch

from attention_gemms_gb300 import tpmlp as T
from oracle import gqa_oracle as Q
from tests.helpers import BF16_TOL, F32_TOL, host, rel, tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    T.lib()
    torch.cuda.set_device(0)
    T.tp_set_wait_timeout_ns(1_000_000_000)
    yield
    T.tp_set_wait_timeout_ns(0)
    assert T.tp_check_status() == 0


def _run(b, s, h, H, Hkv, N, dtype, mode, causal, seed=6000):
    dt = T.DType.BF16 if dtype == "bf16" else T.DType.F32
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    md = T.Reduce.SPLITK if mode == "splitk" else T.Reduce.BUFFERS
    d, M = h // H, b * s
    W = T.tp_gqa_qkv_cols(h, H, Hkv, N)
    assert W > 0
    xo, x = tensor((M, h), seed, dtype=dtype)
    go, g = tensor((h,), seed + 1, 0.2, dtype="f32")
    go, g = go + 1.0, (g + 1.0).contiguous()
    bo, be = tensor((h,), seed + 2, 0.2, dtype="f32")
    sig = 1.0 / np.sqrt(h)  # Q, K, V of unit scale whatever h (bf16 rounding of sharply
    # peaked scores would otherwise dominate the comparison with the unrounded oracle)
    Wqo, Wq = tensor((h, H * d), seed + 3, sig, dtype=dtype)
    Wko, Wk = tensor((h, Hkv * d), seed + 4, sig, dtype=dtype)
    Wvo, Wv = tensor((h, Hkv * d), seed + 5, sig, dtype=dtype)
    Woo, Wo = tensor((h, h), seed + 6, sig, dtype=dtype)
    do, dout = tensor((M, h), seed + 7, dtype=dtype)
    e = lambda *sh, dty=tdt: torch.empty(sh, dtype=dty, device="cuda")
    f32 = torch.float32
    Wsh = e(h, W)
    T.tp_gqa_pack_qkv(Wq, Wk, Wv, Wsh, h, H, Hkv, N, dt)
    xn, mean, rstd, qkv, o, lse, out = (e(M, h), e(M, dty=f32), e(M, dty=f32), e(M, W), e(M, h),
                                        e(b, H, s, dty=f32), e(M, h))
    ws = torch.empty(max(T.tp_gqa_workspace_size(1, M, h, H, Hkv, N, dt, md),
                         T.tp_gqa_workspace_size(0, M, h, H, Hkv, N, dt, md), 256),
                     dtype=torch.uint8, device="cuda")
    T.tp_gqa_attn_proj_fwd(x, g, be, Wsh, Wo, xn, mean, rstd, qkv, o, lse, out, b, s, h, H, Hkv,
                           N, causal, dt, md, ws, ws.numel())
    dx, dg, db, dW, dWo = e(M, h), e(h, dty=f32), e(h, dty=f32), e(h, W), e(h, h)
    T.tp_gqa_attn_proj_bwd(x, g, Wsh, Wo, xn, mean, rstd, qkv, o, lse, dout, dx, dg, db, dW, dWo,
                           b, s, h, H, Hkv, N, causal, dt, md, ws, ws.numel())
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    Wsho = Q.gqa_pack(Wqo, Wko, Wvo, H, Hkv, N)
    assert np.array_equal(host(Wsh), Wsho)                       # a copy: exact
    fr = Q.gqa_block_fwd(xo, b, s, go, bo, Wsho, Woo, H, Hkv, N, bool(causal))
    br = Q.gqa_block_bwd(xo, b, s, go, bo, Wsho, Woo, H, Hkv, N, do, bool(causal))
    got = {"xn": xn, "QKV": qkv, "O": o, "out": out, "dx": dx, "dgamma": dg, "dbeta": db,
           "dWqkv": dW, "dWo": dWo}
    ref = {"xn": fr["xn"], "QKV": fr["QKV"], "O": fr["O"], "out": fr["out"], "dx": br["dx"],
           "dgamma": br["dgamma"], "dbeta": br["dbeta"], "dWqkv": br["dWqkv"], "dWo": br["dWo"]}
    return {k: rel(host(got[k]), ref[k]) for k in got}, host(dW), Hkv, N, W, h, H, d


CASES_BF16 = [  # (h, H, Hkv, N): N below, at and above the key/value head count; MQA
    (256, 8, 2, 2), (256, 8, 4, 4), (256, 8, 2, 4), (512, 8, 2, 8), (256, 8, 1, 4)]


@pytest.mark.parametrize("h,H,Hkv,N", CASES_BF16)
@pytest.mark.parametrize("mode", ["buffers", "splitk"])
@pytest.mark.parametrize("causal", [0, 1])
def test_gqa_block_bf16(h, H, Hkv, N, mode, causal):
    errs, *_ = _run(2, 80, h, H, Hkv, N, "bf16", mode, causal)
    for k, v in errs.items():
        assert v <= BF16_TOL, (k, v)


CORE_CASES = [(4, 4, 1), (8, 2, 2), (8, 4, 2), (8, 2, 4)]  # (H, Hkv, N) at head_dim 64


@pytest.mark.parametrize("H,Hkv,N", CORE_CASES)
@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("s", [300, 64, 1])
def test_gqa_attention_core_bf16(H, Hkv, N, causal, s):
    """The attention core alone at head_dim 64 in bf16, over several 128-row tiles and a
    ragged tail: the forward, and the backward with its scratch (tensor cores) and
    without it (CUDA cores), each against the fp64 oracle on the same bf16 qkv. (H, Hkv,
    N) = (4, 4, 1) is the multi-head layout; (8, 2, 4) replicates each key/value head."""
    b, d = 2, 64
    h, M = H * d, b * s
    W = T.tp_gqa_qkv_cols(h, H, Hkv, N)
    BF = T.DType.BF16
    qo, qkv = tensor((M, W), 6100 + s, dtype="bf16")
    do, dO = tensor((M, h), 6200 + s, dtype="bf16")
    o = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((b, H, s), dtype=torch.float32, device="cuda")
    T.tp_gqa_attention_fwd(qkv, o, lse, b, s, h, H, Hkv, N, causal, BF)
    wsb = T.tp_gqa_attention_bwd_workspace_size(b, s, H)
    assert wsb >= 8 * b * s * H
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    nan = lambda: torch.full((M, W), float("nan"), dtype=torch.bfloat16, device="cuda")
    d_tc, d_cc = nan(), nan()  # every element of dqkv is written
    T.tp_gqa_attention_bwd(qkv, o, lse, dO, d_tc, b, s, h, H, Hkv, N, causal, BF, ws, wsb)
    T.tp_gqa_attention_bwd(qkv, o, lse, dO, d_cc, b, s, h, H, Hkv, N, causal, BF)
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    O_ref = Q.gqa_attention_fwd(qo, b, s, H, Hkv, N, bool(causal))
    d_ref = Q.gqa_attention_bwd(qo, do, b, s, H, Hkv, N, bool(causal))
    assert rel(host(o), O_ref) <= BF16_TOL
    assert rel(host(d_tc), d_ref) <= BF16_TOL
    assert rel(host(d_cc), d_ref) <= BF16_TOL


@pytest.mark.parametrize("H,Hkv,N", [(6, 3, 3), (6, 3, 6), (6, 2, 2)])
def test_gqa_block_f32(H, Hkv, N):
    errs, *_ = _run(2, 70, 16 * H, H, Hkv, N, "f32", "buffers", 0)
    for k, v in errs.items():
        assert v <= F32_TOL, (k, v)


def test_gqa_replicas_hold_equal_gradients():
    """With N > Hkv the key/value columns of every replica are bitwise equal after the
    all-reduce among the replicas."""
    _, dW, Hkv, N, W, h, H, d = _run(2, 64, 256, 8, 2, 8 // 2 * 2, "f32", "splitk", 0)
    hq, hkv, r = Q.gqa_split(H, Hkv, N)
    S = W // N
    assert r > 1
    for i in range(N):
        base = (i // r) * r
        assert np.array_equal(dW[:, i * S + hq * d:(i + 1) * S], dW[:, base * S + hq * d:(base + 1) * S])


def test_gqa_shape_errors():
    assert T.tp_gqa_qkv_cols(256, 8, 3, 2) == 0          # H % Hkv
    assert T.tp_gqa_qkv_cols(256, 8, 4, 3) == 0          # H % N
    assert T.tp_gqa_qkv_cols(256, 8, 2, 4) == 4 * (2 + 2) * 32
    t = torch.empty(1024, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(256, device="cuda")
    with pytest.raises(T.TpError) as e:                   # bf16: (hq + 2 hkv) d = 96 columns
        T.tp_gqa_attn_proj_fwd(t, g, g, t, t, t, g, g, t, t, g, t, 1, 4, 256, 8, 2, 8, 0,
                               T.DType.BF16, T.Reduce.SPLITK, None, 0)
    assert e.value.status == T.Status.SHAPE


def test_gqa_block_graph_replay_matches_eager():
    """The backward runs its weight gradients on a side stream forked from and joined
    back to the caller's stream with events. Captured into a CUDA graph (after an eager
    call created that stream) and replayed, the block gives the eager call's outputs
    bit for bit, and so does a second eager call."""
    b, s, h, H, Hkv, N = 2, 200, 512, 8, 2, 4          # head_dim 64, replicated K/V heads
    BF, md = T.DType.BF16, T.Reduce.BUFFERS
    d, M, W = h // H, b * s, T.tp_gqa_qkv_cols(h, H, Hkv, N)
    _, x = tensor((M, h), 6301)
    g = torch.ones(h, device="cuda")
    be = torch.zeros(h, device="cuda")
    sig = 1.0 / np.sqrt(h)
    _, Wq = tensor((h, H * d), 6302, sig)
    _, Wk = tensor((h, Hkv * d), 6303, sig)
    _, Wv = tensor((h, Hkv * d), 6304, sig)
    _, Wo = tensor((h, h), 6305, sig)
    _, dout = tensor((M, h), 6306)
    e = lambda *sh, dty=torch.bfloat16: torch.zeros(sh, dtype=dty, device="cuda")
    f32 = torch.float32
    Wsh = e(h, W)
    T.tp_gqa_pack_qkv(Wq, Wk, Wv, Wsh, h, H, Hkv, N, BF)
    ws = torch.empty(max(T.tp_gqa_workspace_size(1, M, h, H, Hkv, N, BF, md),
                         T.tp_gqa_workspace_size(0, M, h, H, Hkv, N, BF, md)),
                     dtype=torch.uint8, device="cuda")
    outs = dict(xn=e(M, h), mean=e(M, dty=f32), rstd=e(M, dty=f32), qkv=e(M, W), o=e(M, h),
                lse=e(b, H, s, dty=f32), out=e(M, h), dx=e(M, h), dg=e(h, dty=f32),
                db=e(h, dty=f32), dW=e(h, W), dWo=e(h, h))

    def step(stream):
        q = outs
        T.tp_gqa_attn_proj_fwd(x, g, be, Wsh, Wo, q["xn"], q["mean"], q["rstd"], q["qkv"], q["o"],
                               q["lse"], q["out"], b, s, h, H, Hkv, N, 0, BF, md, ws, ws.numel(),
                               stream)
        T.tp_gqa_attn_proj_bwd(x, g, Wsh, Wo, q["xn"], q["mean"], q["rstd"], q["qkv"], q["o"],
                               q["lse"], dout, q["dx"], q["dg"], q["db"], q["dW"], q["dWo"], b, s,
                               h, H, Hkv, N, 0, BF, md, ws, ws.numel(), stream)

    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in outs.items()}
    for v in outs.values():
        v.zero_()
    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    for k in outs:
        assert torch.equal(outs[k], ref[k]), k
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(torch.cuda.current_stream())
    for v in outs.values():
        v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    for k in outs:
        assert torch.equal(outs[k], ref[k]), k
