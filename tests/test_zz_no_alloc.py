"""tp_row_linear_noalloc: the row-parallel linear for callers that cannot allocate
device memory (their device memory belongs to their own pool allocator or a fixed
budget, so they can neither cudaMalloc nor hand over a workspace). Its fp32
partials live in a fixed 32 MiB array inside the library.

Checked through the C ABI on two calls in a row -- the second with other sizes and
inputs, so stale contents of the shared array would show -- in bf16 and in fp32:
bit for bit against the existing workspace-based entry point (tp_row_linear,
TP_REDUCE_BUFFERS: the same GEMM and reduction kernels in the same order), and
against the oracle's row_linear on the same float64 inputs within the parity
tolerance. Also the size limit. This file is collected last, and passes alone in a
fresh process too.
"""
import pytest
import torch

from attention_gemms_gb300 import tpmlp as T
from oracle import tp_oracle as O
from tests.helpers import BF16_TOL, F32_TOL, host, rel, tensor

pytestmark = pytest.mark.gpu

DT = {"bf16": (T.DType.BF16, torch.bfloat16, BF16_TOL),
      "f32": (T.DType.F32, torch.float32, F32_TOL)}


def _existing(X, W, R, M, k, n, N, dt, tdt):
    out = torch.empty((M, n), dtype=tdt, device="cuda")
    wsz = T.tp_workspace_size(T.Op.ROW_LINEAR, M, k, n, N, dt, T.Act.NONE, T.Reduce.BUFFERS)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    T.tp_row_linear(X, W, R, out, M, k, n, N, dt, T.Reduce.BUFFERS, ws, wsz)
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(dtype):
    T.lib()
    dt, tdt, tol = DT[dtype]
    cases = [(333, 512, 192, 4, 7001, True), (64, 1024, 8192, 8, 7101, False)]
    for M, k, n, N, seed, with_res in cases:
        Xo, X = tensor((M, k), seed, dtype=dtype)
        Wo, W = tensor((k, n), seed + 1, 0.05, dtype=dtype)
        Ro, R = tensor((M, n), seed + 2, dtype=dtype)
        res = R if with_res else None
        got = torch.full((M, n), float("nan"), dtype=tdt, device="cuda")
        T.tp_row_linear_noalloc(X, W, res, got, M, k, n, N, dt)
        want = _existing(X, W, res, M, k, n, N, dt, tdt)
        torch.cuda.synchronize()
        assert T.tp_check_status() == 0
        assert torch.equal(got, want)
        ref = O.row_linear(Xo, Wo, N, Ro if with_res else None)
        assert rel(host(got), ref) <= tol


def test_noalloc_rejects_sizes_beyond_its_scratch():
    T.lib()
    M, k, n, N = 1024, 512, 8192, 2   # 2 * 1024 * 8192 * 4 B = 64 MiB > 32 MiB
    _, X = tensor((M, k), 7201)
    _, W = tensor((k, n), 7202, 0.05)
    out = torch.empty((M, n), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(T.TpError) as ei:
        T.tp_row_linear_noalloc(X, W, None, out, M, k, n, N, T.DType.BF16)
    assert ei.value.status == T.Status.WORKSPACE
    assert "32 MiB" in str(ei.value)
