"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, the binding covers them, and argument errors come back as status codes
before anything touches the device."""
import os
import re

import pytest

from attention_gemms_gb300 import build as B
from attention_gemms_gb300 import tpmlp as T

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "tpmlp.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return T.lib()


def header_functions():
    src = open(HEADER).read()
    return re.findall(r"^TP_API\s+[\w\s\*]+?\b(tp_\w+)\s*\(", src, flags=re.M)


def test_exports_every_declared_symbol(L):
    names = header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    assert sorted(names) == sorted(T.exported_names())


def test_version_and_strings(L):
    assert T.tp_version() == 2
    for s in T.Status:
        assert T.tp_status_string(s) == "TP_" + ("OK" if s == 0 else "ERR_" + s.name)


def _status(call):
    try:
        call()
    except T.TpError as e:
        return e.status
    return T.Status.OK


BF = T.DType.BF16
A16 = 1 << 20  # a fake, 16-byte-aligned address: never dereferenced (validation fails first)


def test_col_linear_argument_errors(L):
    c = lambda **kw: (lambda: T.tp_col_linear(**{**dict(X=A16, W=A16, W_up=None, Y=None, Y_up=None,
                                                           out=A16, M=10, h=128, f=256, N=2,
                                                           dtype=BF, act=T.Act.GELU), **kw}))
    assert _status(c(X=None)) == T.Status.INVALID_ARG
    assert _status(c(N=0)) == T.Status.INVALID_ARG
    assert _status(c(M=-1)) == T.Status.INVALID_ARG
    assert _status(c(f=250)) == T.Status.SHAPE          # f % N
    assert _status(c(h=100)) == T.Status.SHAPE          # bf16 tile rule on h
    assert _status(c(f=192, N=2)) == T.Status.SHAPE     # f/N = 96 not a multiple of 64
    assert _status(c(act=T.Act.SWIGLU)) == T.Status.INVALID_ARG   # no W_up
    assert _status(c(X=A16 + 8)) == T.Status.ALIGNMENT
    assert _status(c(dtype=7)) == T.Status.DTYPE
    assert _status(c(act=9)) == T.Status.INVALID_ARG
    assert _status(c(M=0)) == T.Status.OK              # empty input: nothing launched
    assert "h' (f) must be divisible" in T.tp_last_error() or True


def test_row_and_mlp_argument_errors(L):
    r = lambda **kw: (lambda: T.tp_row_linear(**{**dict(Xs=A16, W=A16, residual=None, out=A16, M=10,
                                                          k=256, n=128, N=2, dtype=BF,
                                                          mode=T.Reduce.BUFFERS, ws=None,
                                                          ws_bytes=0), **kw}))
    assert _status(r()) == T.Status.WORKSPACE
    assert _status(r(mode=5)) == T.Status.INVALID_ARG
    assert _status(r(n=100)) == T.Status.SHAPE
    assert _status(r(k=200)) == T.Status.SHAPE
    m = lambda **kw: (lambda: T.tp_mlp_fwd(**{**dict(X=A16, W1=A16, W1_up=None, W2=A16, residual=None,
                                                       Y=None, Y_up=None, H=None, Z=A16, M=10, h=128,
                                                       f=256, N=2, dtype=BF, act=T.Act.GELU,
                                                       mode=T.Reduce.SPLITK, ws=None, ws_bytes=0),
                                                  **kw}))
    assert _status(m()) == T.Status.WORKSPACE     # H = NULL needs workspace
    assert _status(m(act=T.Act.NONE)) == T.Status.INVALID_ARG
    assert _status(m(W2=None)) == T.Status.INVALID_ARG
    b = lambda **kw: (lambda: T.tp_mlp_bwd(**{**dict(X=A16, W1=A16, W1_up=None, W2=A16, Y=A16, Y_up=None,
                                                       H=A16, dZ=A16, dX=A16, dW1=A16, dW1_up=None,
                                                       dW2=A16, M=10, h=128, f=256, N=2, dtype=BF,
                                                       act=T.Act.SWIGLU, mode=T.Reduce.SPLITK,
                                                       ws=A16, ws_bytes=1 << 30), **kw}))
    assert _status(b()) == T.Status.INVALID_ARG   # SwiGLU without W1_up / Y_up / dW1_up
    assert _status(b(act=T.Act.GELU, ws_bytes=10)) == T.Status.WORKSPACE
    s = lambda **kw: (lambda: T.tp_shard_reduce(**{**dict(partials=A16, residual=None, out=A16, N=0,
                                                            M=4, n=8, out_dtype=BF), **kw}))
    assert _status(s()) == T.Status.INVALID_ARG
    assert _status(s(N=2, out=A16 + 4)) == T.Status.ALIGNMENT
    rl = lambda **kw: (lambda: T.tp_shard_reduce_ln(**{**dict(
        partials=A16, residual=None, gamma=A16, beta=A16, sum_out=None, y=A16, mean=None,
        rstd=None, N=2, M=4, h=64, eps=1e-5, dtype=BF), **kw}))
    assert _status(rl(y=None)) == T.Status.INVALID_ARG
    assert _status(rl(h=60)) == T.Status.SHAPE            # h % 8
    assert _status(rl(h=16384 + 8)) == T.Status.SHAPE     # wider than one row group holds
    assert _status(rl(eps=-1.0)) == T.Status.INVALID_ARG
    assert _status(rl(gamma=A16 + 4)) == T.Status.ALIGNMENT
    rr = lambda **kw: (lambda: T.tp_row_linear_ln(**{**dict(
        Xs=A16, W=A16, residual=None, gamma=A16, beta=A16, sum_out=A16, y=A16, mean=None,
        rstd=None, M=10, k=256, n=128, N=2, eps=1e-5, dtype=BF, mode=T.Reduce.BUFFERS, ws=None,
        ws_bytes=0), **kw}))
    assert _status(rr()) == T.Status.WORKSPACE             # buffers mode needs the partials
    assert _status(rr(sum_out=None)) == T.Status.INVALID_ARG
    assert _status(rr(k=250)) == T.Status.SHAPE            # k % N
    assert _status(rr(n=100)) == T.Status.SHAPE            # bf16 tile rule / n % 8
    spf = lambda **kw: (lambda: T.tp_sp_mlp_fwd(**{**dict(
        x=A16, gamma=A16, beta=A16, W1=A16, W1_up=None, W2=A16, xn=A16, mean=A16, rstd=A16,
        Y=A16, Y_up=None, H=A16, out=A16, M=12, h=128, f=256, N=4, dtype=BF, act=T.Act.GELU,
        mode=T.Reduce.BUFFERS, ws=None, ws_bytes=0), **kw}))
    assert _status(spf(M=10)) == T.Status.SHAPE           # M % N
    assert _status(spf(H=None)) == T.Status.INVALID_ARG
    assert _status(spf()) == T.Status.WORKSPACE           # buffers mode needs the partials
    spb = lambda **kw: (lambda: T.tp_sp_mlp_bwd(**{**dict(
        x=A16, gamma=A16, W1=A16, W1_up=None, W2=A16, xn=A16, mean=A16, rstd=A16, Y=A16,
        Y_up=None, H=A16, dout=A16, dx=A16, dgamma=A16, dbeta=A16, dgamma_ranks=None,
        dbeta_ranks=None, dW1=A16, dW1_up=None, dW2=A16, M=12, h=128, f=256, N=4, dtype=BF,
        act=T.Act.GELU, mode=T.Reduce.SPLITK, ws=A16, ws_bytes=1 << 30), **kw}))
    assert _status(spb(dgamma=None)) == T.Status.INVALID_ARG
    assert _status(spb(ws_bytes=16)) == T.Status.WORKSPACE
    assert _status(spb(M=14)) == T.Status.SHAPE
    assert _status(lambda: T.tp_vocab_embed_fwd(A16, A16, A16, 4, 10, 8, 3, BF)) == T.Status.SHAPE
    assert T.tp_gqa_qkv_cols(2048, 32, 8, 16) == 16 * (2 + 2) * 64 and \
        T.tp_gqa_qkv_cols(2048, 32, 8, 12) == 0 and T.tp_gqa_qkv_cols(4096, 32, 8, 8) == 0
    assert T.tp_gqa_workspace_size(1, 64, 256, 8, 2, 4, BF, T.Reduce.BUFFERS) == 4 * 64 * 256 * 4
    assert _status(lambda: T.tp_gqa_pack_qkv(A16, A16, None, A16, 256, 8, 2, 4, BF)) == \
        T.Status.INVALID_ARG
    assert _status(lambda: T.tp_vocab_ce_fwd(A16, A16, A16, A16, None, None, 4, 12, 3, BF)) == \
        T.Status.INVALID_ARG                                # loss pointer missing
    assert _status(lambda: T.tp_adamw_step(A16, A16, A16, A16, 10, 0, 1e-3, 0.9, 0.999, 1e-8,
                                           0.0)) == T.Status.INVALID_ARG   # step 0
    cfg = T.GptConfig(256, 128, 8, 512, 2, 4, 32, 2)
    assert T.tp_gpt_workspace_size(cfg, T.DType.F32, T.Reduce.BUFFERS) > 0
    assert T.tp_gpt_workspace_size(cfg, BF, T.Reduce.BUFFERS) == 0        # fp32 only
    assert T.tp_gpt_workspace_size(T.GptConfig(250, 128, 8, 512, 2, 4, 32, 3), T.DType.F32,
                                   T.Reduce.BUFFERS) == 0                 # vocab % N
    w, g = T.GptWeights(A16, A16, A16, None), T.GptGrads(A16, A16, A16, None)
    assert _status(lambda: T.tp_gpt_fwd_bwd(cfg, w, g, A16, A16, A16, BF, T.Reduce.BUFFERS, A16,
                                            1 << 30)) == T.Status.DTYPE
    assert _status(lambda: T.tp_gpt_fwd_bwd(cfg, w, g, A16, A16, A16, T.DType.F32,
                                            T.Reduce.BUFFERS, A16, 1 << 30)) == \
        T.Status.INVALID_ARG                                # layer arrays missing


def test_attention_core_bwd_workspace_errors(L):
    need = T.tp_gqa_attention_bwd_workspace_size(1, 8, 4)
    assert need >= 8 * 8 * 4 and T.tp_gqa_attention_bwd_workspace_size(1, 8, 0) == 0
    a = lambda **kw: (lambda: T.tp_gqa_attention_bwd(**{**dict(
        qkv=A16, o=A16, lse=A16, dO=A16, dqkv=A16, b=1, s=8, h=256, n_heads=4, n_kv_heads=4,
        N=1, causal=0, dtype=BF, ws=A16, ws_bytes=need), **kw}))
    assert _status(a(ws_bytes=need - 1)) == T.Status.WORKSPACE
    assert _status(a(ws=A16 + 8)) == T.Status.ALIGNMENT
    assert _status(a(dO=None)) == T.Status.INVALID_ARG
    assert _status(a(n_kv_heads=3)) == T.Status.SHAPE


def test_workspace_sizes(L):
    M, h, f, N = 1000, 256, 1024, 4
    assert T.tp_workspace_size(T.Op.COL_LINEAR, M, h, f, N, BF) == 0
    assert T.tp_workspace_size(T.Op.ROW_LINEAR, M, f, h, N, BF, mode=T.Reduce.BUFFERS) == N * M * h * 4
    assert T.tp_workspace_size(T.Op.ROW_LINEAR, M, f, h, N, BF, mode=T.Reduce.SPLITK) == 0
    fwd = T.tp_workspace_size(T.Op.MLP_FWD, M, h, f, N, BF, T.Act.GELU, T.Reduce.BUFFERS)
    assert fwd == M * f * 2 + N * M * h * 4
    bwd = T.tp_workspace_size(T.Op.MLP_BWD, M, h, f, N, BF, T.Act.SWIGLU, T.Reduce.SPLITK)
    assert bwd == 2 * M * f * 2
    assert T.tp_workspace_size(T.Op.MLP_FWD, M, h, f, 0, BF) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(T, "_lib", None)
    monkeypatch.setattr(T, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        T.lib()


def test_weight_layout_and_size_errors(L):
    """The (out, in) weight layout of the Megatron listing (ColumnParallelLinear /
    RowParallelLinear store W for F.linear) is an argument of the four linear entry
    points; an unknown value, and sizes whose byte counts would not fit in 64 bits, are
    rejected before anything is launched."""
    OUT_IN = T.WLayout.OUT_IN
    c = lambda **kw: (lambda: T.tp_col_linear(**{**dict(X=A16, W=A16, W_up=None, Y=None, Y_up=None,
                                                           out=A16, M=10, h=128, f=256, N=2,
                                                           dtype=BF, act=T.Act.GELU), **kw}))
    assert _status(c(w_layout=2)) == T.Status.INVALID_ARG
    assert _status(c(w_layout=OUT_IN, f=250)) == T.Status.SHAPE        # f % N in either layout
    assert _status(c(w_layout=OUT_IN, act=T.Act.SWIGLU)) == T.Status.INVALID_ARG
    assert _status(c(w_layout=OUT_IN, M=0)) == T.Status.OK
    assert _status(c(M=1 << 40)) == T.Status.SHAPE                     # extent >= 2^31
    r = lambda **kw: (lambda: T.tp_row_linear(**{**dict(Xs=A16, W=A16, residual=None, out=A16, M=10,
                                                          k=256, n=128, N=2, dtype=BF,
                                                          mode=T.Reduce.BUFFERS, ws=None,
                                                          ws_bytes=0), **kw}))
    assert _status(r(w_layout=-1)) == T.Status.INVALID_ARG
    assert _status(r(w_layout=OUT_IN, k=200)) == T.Status.SHAPE
    assert _status(r(w_layout=OUT_IN)) == T.Status.WORKSPACE
    # N*M*n*4 with M*n = 2^40 elements and N = 2^16 would pass 2^64 in a plain product
    assert _status(r(M=1 << 30, n=1 << 10, k=1 << 16, N=1 << 16)) == T.Status.SHAPE
    assert T.tp_workspace_size(T.Op.ROW_LINEAR, 1 << 40, 128, 128, 2, BF) == 0
    m = lambda **kw: (lambda: T.tp_mlp_fwd(**{**dict(X=A16, W1=A16, W1_up=None, W2=A16, residual=None,
                                                       Y=None, Y_up=None, H=A16, Z=A16, M=10, h=128,
                                                       f=256, N=2, dtype=BF, act=T.Act.GELU,
                                                       mode=T.Reduce.SPLITK, ws=None, ws_bytes=0),
                                                  **kw}))
    assert _status(m(w_layout=3)) == T.Status.INVALID_ARG
    assert _status(m(w_layout=OUT_IN, M=0)) == T.Status.OK
    b = lambda **kw: (lambda: T.tp_mlp_bwd(**{**dict(X=A16, W1=A16, W1_up=None, W2=A16, Y=A16, Y_up=None,
                                                       H=A16, dZ=A16, dX=A16, dW1=A16, dW1_up=None,
                                                       dW2=A16, M=10, h=128, f=256, N=2, dtype=BF,
                                                       act=T.Act.GELU, mode=T.Reduce.SPLITK,
                                                       ws=A16, ws_bytes=10), **kw}))
    assert _status(b(w_layout=7)) == T.Status.INVALID_ARG
    assert _status(b(w_layout=OUT_IN)) == T.Status.WORKSPACE
    assert _status(b(w_layout=OUT_IN, act=T.Act.SWIGLU)) == T.Status.INVALID_ARG


def test_device_step_argument_errors(L):
    """The device-side step counter and the AdamW that reads it: argument errors come back
    before any launch."""
    adv = lambda **kw: (lambda: T.tp_train_step_advance(**{**dict(step=A16, loss=A16, loss_hist=A16,
                                                                   hist_len=50), **kw}))
    assert _status(adv(step=None)) == T.Status.INVALID_ARG
    assert _status(adv(loss=None)) == T.Status.INVALID_ARG        # loss and loss_hist go together
    assert _status(adv(hist_len=0)) == T.Status.INVALID_ARG
    assert _status(adv(step=A16 + 2)) == T.Status.ALIGNMENT
    ad = lambda **kw: (lambda: T.tp_adamw_step_device(**{**dict(p=A16, g=A16, m=A16, v=A16, n=10,
                                                                step=A16, lr=1e-3, beta1=0.9,
                                                                beta2=0.999, eps=1e-8,
                                                                weight_decay=0.01), **kw}))
    assert _status(ad(step=None)) == T.Status.INVALID_ARG
    assert _status(ad(beta1=1.0)) == T.Status.INVALID_ARG
    assert _status(ad(n=-1)) == T.Status.INVALID_ARG
    assert _status(ad(m=A16 + 1)) == T.Status.ALIGNMENT
    assert _status(ad(n=0)) == T.Status.OK
