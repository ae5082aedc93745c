"""The GEMM engine on its own (tp_gemm): every operand-major combination the
layers use, single-tile and multi-tile sizes with ragged M / N / K tails, against
float64 products of the same (exactly representable) inputs."""
import numpy as np
import pytest
import torch

from attention_gemms_gb300 import tpmlp as T
from tests.helpers import BF16_TOL, F32_TOL, gemm_tiles, guard_intact, guarded, host, rel, tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    T.lib()
    T.tp_set_wait_timeout_ns(1_000_000_000)
    yield
    T.tp_set_wait_timeout_ns(0)
    assert T.tp_check_status() == 0


def _run(M, N, K, at, bt, dtype="bf16", seed=600):
    Ao, A = tensor((K, M) if at else (M, K), seed, dtype=dtype)
    Bo, B = tensor((N, K) if bt else (K, N), seed + 1, 0.1, dtype=dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    C, full = guarded((M, N), tdt)
    T.tp_gemm(A, B, C, M, N, K, at, bt, T.DType.BF16 if dtype == "bf16" else T.DType.F32)
    torch.cuda.synchronize()
    assert T.tp_check_status() == 0
    ref = (Ao.T if at else Ao) @ (Bo.T if bt else Bo)
    return rel(host(C), ref), guard_intact(full, M)


@pytest.mark.parametrize("at", [False, True])
@pytest.mark.parametrize("bt", [False, True])
@pytest.mark.parametrize("MNK", [(128, 128, 64), (128, 256, 64), (256, 512, 192), (200, 264, 136),
                                 (1, 64, 64), (77, 1000, 520),
                                 # few tiles at M >= 256: one-CTA 128 x 64 tiles instead of
                                 # 256 x 256 pairs (the page-2 layer's QKV and MLP shapes)
                                 (1024, 384, 128), (1024, 512, 128), (1000, 136, 520),
                                 # few narrow tiles with a long K (weight-gradient shapes of small layers)
                                 # (ragged M, N and K in the second)
                                 (128, 128, 1024), (200, 192, 680)])
def test_gemm_bf16(at, bt, MNK):
    M, N, K = MNK
    if at and M % 8:
        # a stored (K, M) operand needs 16-byte rows for TMA: rejected before launch
        with pytest.raises(T.TpError) as ei:
            _run(M, N, K, at, bt)
        assert ei.value.status == T.Status.SHAPE
        return
    e, ok = _run(M, N, K, at, bt)
    assert e <= BF16_TOL and ok, e


@pytest.mark.parametrize("at", [False, True])
@pytest.mark.parametrize("bt", [False, True])
def test_gemm_f32(at, bt):
    e, ok = _run(67, 45, 33, at, bt, dtype="f32")
    assert e <= F32_TOL and ok, e


# ---- the CTA-pair kernel in both tile widths (256 x 256 and 256 x 512), forced onto
# small shapes: every operand-major combination; one K block, fewer K blocks than the
# wide form's four stages, more of them, and ragged M / N / K; a second tile half that
# lies wholly or partly past N

@pytest.mark.parametrize("wide", [0, 2], ids=["pair256", "pair512"])
@pytest.mark.parametrize("at", [False, True])
@pytest.mark.parametrize("bt", [False, True])
@pytest.mark.parametrize("MNK", [(256, 512, 64), (256, 512, 128), (512, 1024, 320),
                                 (600, 1288, 520), (768, 264, 192), (256, 256, 512),
                                 # at least two tiles per SM pair: the epilogue's
                                 # TMA-store path, ragged rows and columns
                                 (4000, 5128, 200)])
def test_pair_gemm_forms(wide, at, bt, MNK):
    M, N, K = MNK
    with gemm_tiles(2, wide):
        e, ok = _run(M, N, K, at, bt, seed=640)
    assert e <= BF16_TOL and ok, e


# ---- the CTA-pair kernel's epilogue paths: 256-bit stores / loads when the outputs
# (inputs) are 32-byte aligned, 128-bit otherwise, and the 8-column tail when N % 16 == 8

@pytest.mark.parametrize("wide", [0, 2], ids=["pair256", "pair512"])
@pytest.mark.parametrize("MNK", [(384, 264, 192), (512, 520, 128)])
def test_pair_gemm_ragged_columns(MNK, wide):
    M, N, K = MNK
    with gemm_tiles(2, wide):
        e, ok = _run(M, N, K, False, False)
    assert e <= BF16_TOL and ok, e


@pytest.mark.parametrize("wide", [0, 2], ids=["pair256", "pair512"])
def test_pair_gemm_output_only_16_byte_aligned(wide):
    with gemm_tiles(2, wide):
        _output_only_16_byte_aligned()


def _output_only_16_byte_aligned():
    M, N, K = 512, 512, 256
    A = tensor((M, K), 610)[1]
    B = tensor((K, N), 611, 0.1)[1]
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    buf = torch.empty(M * N + 16, dtype=torch.bfloat16, device="cuda")
    C16 = buf[8:8 + M * N].view(M, N)  # 16 bytes past a 256-byte boundary
    T.tp_gemm(A, B, C, M, N, K, False, False, T.DType.BF16)
    T.tp_gemm(A, B, C16, M, N, K, False, False, T.DType.BF16)
    torch.cuda.synchronize()
    assert C16.data_ptr() % 32 == 16
    assert torch.equal(C, C16)


@pytest.mark.parametrize("wide", [0, 2], ids=["pair256", "pair512"])
def test_pair_gemm_epilogue_inputs_only_16_byte_aligned(wide):
    """The GELU MLP backward reads Y in its epilogue: a Y 16 bytes off a 32-byte boundary
    gives the same gradients bit for bit."""
    with gemm_tiles(2, wide):
        _epilogue_inputs_only_16_byte_aligned()


def _epilogue_inputs_only_16_byte_aligned():
    M, h, f, N = 512, 256, 512, 2
    BF, A = T.DType.BF16, T.Act.GELU
    X = tensor((M, h), 620)[1]
    W1 = tensor((h, f), 621, 0.05)[1]
    W2 = tensor((f, h), 622, 0.05)[1]
    dZ = tensor((M, h), 623)[1]
    e = lambda *s: torch.empty(s, dtype=torch.bfloat16, device="cuda")
    Y, H, Z = e(M, f), e(M, f), e(M, h)
    ws = torch.empty(max(T.tp_workspace_size(T.Op.MLP_FWD, M, h, f, N, BF, A, T.Reduce.SPLITK),
                         T.tp_workspace_size(T.Op.MLP_BWD, M, h, f, N, BF, A, T.Reduce.SPLITK)),
                     dtype=torch.uint8, device="cuda")
    T.tp_mlp_fwd(X, W1, None, W2, None, Y, None, H, Z, M, h, f, N, BF, A, T.Reduce.SPLITK, ws,
                 ws.numel())
    buf = e(M * f + 16)
    Y16 = buf[8:8 + M * f].view(M, f)
    Y16.copy_(Y)
    outs = []
    for Yin in (Y, Y16):
        dX, dW1, dW2 = e(M, h), e(h, f), e(f, h)
        T.tp_mlp_bwd(X, W1, None, W2, Yin, None, H, dZ, dX, dW1, None, dW2, M, h, f, N, BF, A,
                     T.Reduce.SPLITK, ws, ws.numel())
        outs.append((dX, dW1, dW2))
    torch.cuda.synchronize()
    assert Y16.data_ptr() % 32 == 16
    for a, b in zip(*outs):
        assert torch.equal(a, b)
