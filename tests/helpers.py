"""Shared helpers of the GPU tests: seeded inputs as (exact float64 copy for the
oracle, device tensor for the library), and the parity metric."""
import numpy as np
import torch

from attention_gemms_gb300 import synth

BF16_TOL = 1e-2   # max|gpu - oracle| / max|oracle|, bf16 inputs with fp32 accumulation
F32_TOL = 1e-5    # fp32 path (FFMA, no TF32)


def tensor(shape, seed, sigma=1.0, dtype="bf16", device="cuda"):
    """Seeded N(0, sigma^2) tensor: returns (float64 numpy copy, device tensor)."""
    a = synth.normal(shape, seed, sigma, dtype)
    if dtype == "bf16":
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    return synth.to_f64(a, dtype), t.to(device)


def host(t):
    return t.detach().float().cpu().double().numpy()


def rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-300))


def empty(shape, dtype, device="cuda", fill=float("nan")):
    """Output buffer pre-filled with a sentinel, so unwritten elements show up."""
    return torch.full(shape, fill, dtype=dtype, device=device)


def guarded(shape, dtype, guard_rows=2, device="cuda"):
    """(view, full): `view` is the first shape[0] rows of a buffer with extra guard
    rows after it, filled with a sentinel that the kernels must not touch."""
    full = torch.full((shape[0] + guard_rows,) + tuple(shape[1:]), -768.0, dtype=dtype,
                      device=device)
    return full[:shape[0]], full


def guard_intact(full, rows):
    return bool(torch.all(full[rows:] == -768.0).item())


class gemm_tiles:
    """Context manager: GEMM kernel selection for a test (pair: 0 one-CTA only,
    1 automatic, 2 the CTA-pair kernel wherever it can run; wide: 0 256 x 256 pair
    tiles, 1 automatic, 2 256 x 512 pair tiles), restored to automatic on exit."""

    def __init__(self, pair, wide):
        self.pair, self.wide = pair, wide

    def __enter__(self):
        from attention_gemms_gb300 import tpmlp as T
        T.tp_set_gemm_pair_mode(self.pair)
        T.tp_set_gemm_wide_mode(self.wide)
        return self

    def __exit__(self, *exc):
        from attention_gemms_gb300 import tpmlp as T
        T.tp_set_gemm_pair_mode(1)
        T.tp_set_gemm_wide_mode(1)
        return False
