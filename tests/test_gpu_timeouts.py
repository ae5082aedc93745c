"""Bounded device waits and concurrent callers.

Every kernel family with mbarrier waits is made to time out on purpose: the test hook
tp_debug_inject_wait_fault makes each launch's MMA thread wait on a barrier nothing
arrives on, with a short limit. The kernel must stop by itself (no fault, no trap),
report TP_ERR_TIMEOUT through tp_check_status, and leave the context usable: a clean
call right after must match the fp64 oracle. Families: the one-CTA 128 x 256 GEMM,
its decode configuration (M <= 64), the CTA-pair GEMM in both tile widths, the tensor-core attention
forward, and the tensor-core attention backward (dK/dV and dQ kernels).

The header promises that calls may come from several host threads: two threads run
the MLP forward + backward (variant A, whose backward forks a side stream) and the
attention block forward + backward (weight gradients on side streams) on their own
streams at the same time, each result checked against the oracle."""
import threading
import time

import numpy as np
import pytest
import torch

from attention_gemms_gb300 import tpmlp as T
from oracle import gqa_oracle as Q
from oracle import tp_oracle as O
from tests.helpers import BF16_TOL, empty, gemm_tiles, host, rel, tensor

pytestmark = pytest.mark.gpu
BF = T.DType.BF16
bf16 = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    T.lib()
    torch.cuda.set_device(0)
    T.tp_set_wait_timeout_ns(1_000_000_000)
    yield
    T.tp_debug_inject_wait_fault(False)
    T.tp_set_wait_timeout_ns(0)
    assert T.tp_check_status() == 0


def _expect_timeout(call, limit_ns=2_000_000):
    """Run `call` with the wait fault injected and a short limit: the status must be
    TP_ERR_TIMEOUT. Returns the host wall time of the call up to its completion."""
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    T.tp_set_wait_timeout_ns(limit_ns)
    T.tp_debug_inject_wait_fault(True)
    try:
        t0 = time.perf_counter()
        call()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert T.tp_check_status() == T.Status.TIMEOUT
    finally:
        T.tp_debug_inject_wait_fault(False)
        T.tp_set_wait_timeout_ns(1_000_000_000)
    assert T.tp_check_status() == 0       # the status word was cleared by the read
    return dt


def _col_case(M, act, seed):
    h, f, N = 128, 512, 2
    Xo, X = tensor((M, h), seed)
    Wo, W = tensor((h, f), seed + 1, 0.05)
    Wuo, Wu = tensor((h, f), seed + 2, 0.05)
    out = empty((M, f), bf16)
    sw = act == T.Act.SWIGLU
    call = lambda: T.tp_col_linear(X, W, Wu if sw else None, None, None, out, M, h, f, N, BF, act)
    G = Xo @ Wo
    ref = O.silu(G) * (Xo @ Wuo) if sw else O.gelu(G)
    return call, out, ref


@pytest.mark.parametrize("M,act,wide", [(128, T.Act.GELU, 1),     # one-CTA 128 x 256 tile
                                        (8, T.Act.SWIGLU, 1),     # decode configuration
                                        (40, T.Act.GELU, 1),      # decode configuration
                                        (512, T.Act.SWIGLU, 0),   # CTA pair, 256 x 256
                                        (512, T.Act.SWIGLU, 2)])  # CTA pair, 256 x 512
def test_gemm_wait_timeout_reports_and_recovers(M, act, wide):
    call, out, ref = _col_case(M, act, 7300 + M)
    with gemm_tiles(1, wide):
        _expect_timeout(call)
        call()
        torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    assert rel(host(out), ref) <= BF16_TOL


def test_wait_limit_is_a_time_not_a_poll_count():
    """The limit counts SM clock cycles at 2 per ns, so a wait gives up after about the
    limit (longer when the clock runs below 2 GHz, shorter by at most the 2.07/2 ratio
    above it), whatever the polling rate."""
    call, _, _ = _col_case(512, T.Act.GELU, 7400)
    call()
    torch.cuda.synchronize()
    limit = 50_000_000  # 50 ms
    dt = _expect_timeout(call, limit)
    assert 0.9 * limit * 1e-9 <= dt <= 4 * limit * 1e-9 + 0.2, dt


def _attn_core(causal, seed):
    b, s, H, Hkv, N, d = 1, 200, 4, 2, 2, 64
    h, M = H * d, b * s
    W = T.tp_gqa_qkv_cols(h, H, Hkv, N)
    qo, qkv = tensor((M, W), seed)
    do, dO = tensor((M, h), seed + 1)
    o = torch.empty((M, h), dtype=bf16, device="cuda")
    lse = torch.empty((b, H, s), dtype=torch.float32, device="cuda")
    wsb = T.tp_gqa_attention_bwd_workspace_size(b, s, H)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    dq = torch.empty((M, W), dtype=bf16, device="cuda")
    fwd = lambda: T.tp_gqa_attention_fwd(qkv, o, lse, b, s, h, H, Hkv, N, causal, BF)
    bwd = lambda: T.tp_gqa_attention_bwd(qkv, o, lse, dO, dq, b, s, h, H, Hkv, N, causal, BF,
                                         ws, wsb)
    refs = lambda: (Q.gqa_attention_fwd(qo, b, s, H, Hkv, N, bool(causal)),
                    Q.gqa_attention_bwd(qo, do, b, s, H, Hkv, N, bool(causal)))
    return fwd, bwd, o, dq, refs


@pytest.mark.parametrize("causal", [0, 1])
def test_attention_tc_wait_timeout_reports_and_recovers(causal):
    fwd, bwd, o, dq, refs = _attn_core(causal, 7500 + causal)
    _expect_timeout(fwd)                  # the forward kernel
    fwd()                                 # a clean forward for the backward's inputs
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    _expect_timeout(bwd)                  # the dK/dV and dQ kernels
    fwd()
    bwd()
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    O_ref, d_ref = refs()
    assert rel(host(o), O_ref) <= BF16_TOL
    assert rel(host(dq), d_ref) <= BF16_TOL


# ---------------------------------------------------------------- several host threads

def _mlp_job(stream, seed, errs):
    M, h, f, N = 384, 256, 1024, 4
    act, mode = T.Act.SWIGLU, T.Reduce.BUFFERS
    with torch.cuda.stream(stream):
        Xo, X = tensor((M, h), seed)
        W1o, W1 = tensor((h, f), seed + 1, 0.05)
        Wuo, Wu = tensor((h, f), seed + 2, 0.05)
        W2o, W2 = tensor((f, h), seed + 3, 0.05)
        dZo, dZ = tensor((M, h), seed + 4)
        Y, Yu, A = (torch.empty((M, f), dtype=bf16, device="cuda") for _ in range(3))
        Z, dX = (torch.empty((M, h), dtype=bf16, device="cuda") for _ in range(2))
        dWg, dWu = (torch.empty((h, f), dtype=bf16, device="cuda") for _ in range(2))
        dWd = torch.empty((f, h), dtype=bf16, device="cuda")
        nb = max(T.tp_workspace_size(T.Op.MLP_FWD, M, h, f, N, BF, act, mode),
                 T.tp_workspace_size(T.Op.MLP_BWD, M, h, f, N, BF, act, mode))
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    for _ in range(5):
        T.tp_mlp_fwd(X, W1, Wu, W2, None, Y, Yu, A, Z, M, h, f, N, BF, act, mode, ws, nb, stream)
        T.tp_mlp_bwd(X, W1, Wu, W2, Y, Yu, A, dZ, dX, dWg, dWu, dWd, M, h, f, N, BF, act, mode,
                     ws, nb, stream)
    stream.synchronize()
    fr = O.mlp_swiglu_fwd(Xo, W1o, Wuo, W2o, N)
    br = O.mlp_swiglu_bwd(Xo, W1o, Wuo, W2o, dZo, N)
    got = {"Z": Z, "dX": dX, "dWg": dWg, "dWu": dWu, "dWd": dWd}
    ref = {"Z": fr["Z"], "dX": br["dX"], "dWg": br["dWg"], "dWu": br["dWu"], "dWd": br["dWd"]}
    errs.update({f"mlp{seed}.{k}": rel(host(got[k]), ref[k]) for k in got})


def _attn_job(stream, seed, errs):
    b, s, h, heads, N, causal = 2, 256, 256, 4, 2, 1      # head_dim 64: tensor-core attention
    M = b * s
    md = T.Reduce.BUFFERS
    with torch.cuda.stream(stream):
        xo, x = tensor((M, h), seed)
        go, g = tensor((h,), seed + 1, 0.1, dtype="f32")
        bo, bb = tensor((h,), seed + 2, 0.1, dtype="f32")
        g = (g + 1.0).contiguous()
        go = go + 1.0
        Wqkvo, Wqkv = tensor((h, 3 * h), seed + 3, 0.1)
        Woo, Wo = tensor((h, h), seed + 4, 0.1)
        douto, dout = tensor((M, h), seed + 5)
        e = lambda *sh: torch.empty(sh, dtype=bf16, device="cuda")
        xn, qkv, o, out, dx = e(M, h), e(M, 3 * h), e(M, h), e(M, h), e(M, h)
        mean, rstd = (torch.empty(M, device="cuda") for _ in range(2))
        lse = torch.empty((b, heads, s), device="cuda")
        dg, db = (torch.empty(h, device="cuda") for _ in range(2))
        dWqkv, dWo = e(h, 3 * h), e(h, h)
        nb = max(T.tp_workspace_size(T.Op.ATTN_PROJ_FWD, M, h, 0, N, BF, T.Act.NONE, md),
                 T.tp_workspace_size(T.Op.ATTN_PROJ_BWD, M, h, 0, N, BF, T.Act.NONE, md))
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    for _ in range(5):
        T.tp_attn_proj_fwd(x, g, bb, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, out, b, s, h, heads,
                           N, causal, BF, md, ws, nb, stream)
        T.tp_attn_proj_bwd(x, g, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, dout, dx, dg, db, dWqkv,
                           dWo, b, s, h, heads, N, causal, BF, md, ws, nb, stream)
    stream.synchronize()
    fr = O.attn_block_fwd(xo, b, s, go, bo, Wqkvo, Woo, heads, N, bool(causal))
    br = O.attn_block_bwd(xo, b, s, go, bo, Wqkvo, Woo, heads, N, douto, bool(causal))
    got = {"out": out, "dx": dx, "dgamma": dg, "dbeta": db, "dWqkv": dWqkv, "dWo": dWo}
    ref = {"out": fr["out"], "dx": br["dx"], "dgamma": br["dgamma"], "dbeta": br["dbeta"],
           "dWqkv": br["dWqkv"], "dWo": br["dWo"]}
    errs.update({f"attn{seed}.{k}": rel(host(got[k]), ref[k]) for k in got})


def test_two_host_threads_on_two_streams():
    errs, failures = {}, []

    def run(job, seed):
        try:
            job(torch.cuda.Stream(), seed, errs)
        except Exception as e:  # noqa: BLE001 -- reported by the main thread
            failures.append(repr(e))

    jobs = [(_mlp_job, 7601), (_attn_job, 7701), (_mlp_job, 7801), (_attn_job, 7901)]
    threads = [threading.Thread(target=run, args=j) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads)
    assert not failures, failures
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    assert len(errs) == 2 * 5 + 2 * 6
    bad = {k: v for k, v in errs.items() if not v <= BF16_TOL}
    assert not bad, bad
    assert np.isfinite(list(errs.values())).all()
