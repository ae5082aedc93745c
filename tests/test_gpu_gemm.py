"""The GEMM engine on its own (tp_gemm): every operand-major combination the
layers use, single-tile and multi-tile sizes with ragged M / N / K tails, against
float64 products of the same (exactly representable) inputs."""
import numpy as np
import pytest
import torch

from attention_gemms_gb300 import tpmlp as T
from tests.helpers import BF16_TOL, F32_TOL, guard_intact, guarded, host, rel, tensor

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
                                 (1, 64, 64), (77, 1000, 520)])
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
