"""tp_row_linear_noalloc: the row-parallel linear for callers that cannot allocate
device memory (their device memory belongs to their own pool allocator or a fixed
budget, so they can neither cudaMalloc nor hand over a workspace). Its fp32
partials live in a fixed 32 MiB array inside the library.

Checked through the C ABI against the existing workspace-based entry point
(tp_row_linear, TP_REDUCE_BUFFERS) on two calls in a row -- the second with other
sizes and inputs, so stale contents of the shared array would show -- and the
size limit. This file is collected last, and passes alone in a fresh process too.
"""
import pytest
import torch

from attention_gemms_gb300 import tpmlp as T
from tests.helpers import BF16_TOL, host, rel, tensor

pytestmark = pytest.mark.gpu
BF = T.DType.BF16


def _existing(X, W, R, M, k, n, N):
    out = torch.empty((M, n), dtype=torch.bfloat16, device="cuda")
    wsz = T.tp_workspace_size(T.Op.ROW_LINEAR, M, k, n, N, BF, T.Act.NONE, T.Reduce.BUFFERS)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    T.tp_row_linear(X, W, R, out, M, k, n, N, BF, T.Reduce.BUFFERS, ws, wsz)
    return out


def test_noalloc_matches_workspace_entry_point_twice():
    T.lib()
    cases = [(333, 512, 192, 4, 7001, True), (64, 1024, 8192, 8, 7101, False)]
    for M, k, n, N, seed, with_res in cases:
        _, X = tensor((M, k), seed)
        _, W = tensor((k, n), seed + 1, 0.05)
        _, R = tensor((M, n), seed + 2)
        res = R if with_res else None
        got = torch.full((M, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        T.tp_row_linear_noalloc(X, W, res, got, M, k, n, N, BF)
        want = _existing(X, W, res, M, k, n, N)
        torch.cuda.synchronize()
        assert T.tp_check_status() == 0
        assert rel(host(got), host(want)) <= BF16_TOL


def test_noalloc_rejects_sizes_beyond_its_scratch():
    T.lib()
    M, k, n, N = 1024, 512, 8192, 2   # 2 * 1024 * 8192 * 4 B = 64 MiB > 32 MiB
    _, X = tensor((M, k), 7201)
    _, W = tensor((k, n), 7202, 0.05)
    out = torch.empty((M, n), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(T.TpError) as ei:
        T.tp_row_linear_noalloc(X, W, None, out, M, k, n, N, BF)
    assert ei.value.status == T.Status.WORKSPACE
    assert "32 MiB" in str(ei.value)
