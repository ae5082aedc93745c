"""ctypes binding of libtpmlp (include/tpmlp.h): the same entry points under the
same names, argument marshalling only. Tensors may be passed as torch tensors
(their data_ptr is used), raw integer device addresses, or None (NULL). `stream`
defaults to torch's current CUDA stream.

The library must have been built (python -m attention_gemms_gb300.build); loading
fails loudly otherwise -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import enum
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtpmlp.so")


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    SHAPE = 2
    DTYPE = 3
    ALIGNMENT = 4
    WORKSPACE = 5
    CUDA = 6
    TIMEOUT = 7
    UNSUPPORTED = 8


class DType(enum.IntEnum):
    F32 = 0
    BF16 = 1


class Act(enum.IntEnum):
    NONE = 0
    GELU = 1
    SWIGLU = 2


class Reduce(enum.IntEnum):
    BUFFERS = 0
    SPLITK = 1


class WLayout(enum.IntEnum):
    """tp_wlayout: weights stored (in, out) -- the pages' W -- or (out, in)."""
    IN_OUT = 0
    OUT_IN = 1


class Op(enum.IntEnum):
    COL_LINEAR = 0
    ROW_LINEAR = 1
    MLP_FWD = 2
    MLP_BWD = 3
    ATTN_PROJ_FWD = 4
    ATTN_PROJ_BWD = 5
    LAYERNORM_BWD = 6
    LAYER_FWD = 7
    LAYER_BWD = 8
    SP_MLP_FWD = 9
    SP_MLP_BWD = 10


class LayerWeights(ctypes.Structure):
    """tp_layer_weights"""
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("Wqkv", "Wo", "W1", "W2", "gamma1", "beta1", "gamma2", "beta2")]


class LayerSaved(ctypes.Structure):
    """tp_layer_saved"""
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("xn1", "mean1", "rstd1", "qkv", "o", "lse", "x1", "xn2", "mean2", "rstd2",
                 "y", "hh")]


class LayerGrads(ctypes.Structure):
    """tp_layer_grads"""
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("dWqkv", "dWo", "dW1", "dW2", "dgamma1", "dbeta1", "dgamma2", "dbeta2")]


class GptConfig(ctypes.Structure):
    """tp_gpt_config"""
    _fields_ = [("vocab", ctypes.c_int64), ("hidden", ctypes.c_int64), ("heads", ctypes.c_int64),
                ("ffn", ctypes.c_int64), ("layers", ctypes.c_int64), ("batch", ctypes.c_int64),
                ("seq", ctypes.c_int64), ("shards", ctypes.c_int32)]


class GptWeights(ctypes.Structure):
    """tp_gpt_weights"""
    _fields_ = [("E", ctypes.c_void_p), ("gammaf", ctypes.c_void_p), ("betaf", ctypes.c_void_p),
                ("layers", ctypes.POINTER(LayerWeights))]


class GptGrads(ctypes.Structure):
    """tp_gpt_grads"""
    _fields_ = [("dE", ctypes.c_void_p), ("dgammaf", ctypes.c_void_p), ("dbetaf", ctypes.c_void_p),
                ("layers", ctypes.POINTER(LayerGrads))]


def make_struct(cls, **tensors):
    """Fill one of the layer structs from tensors / addresses / None by field name."""
    return cls(**{k: _ptr(v) for k, v in tensors.items()})


class TpError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = Status(status)
        super().__init__(f"{self.status.name}: {detail}")


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_ST = ctypes.c_int
_SZ = ctypes.c_size_t

# name -> (restype, argtypes), in header order
_SIGS = {
    "tp_version": (ctypes.c_int, []),
    "tp_status_string": (ctypes.c_char_p, [_ST]),
    "tp_last_error": (ctypes.c_char_p, []),
    "tp_check_status": (_ST, [_P]),
    "tp_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "tp_set_gemm_pair_mode": (None, [ctypes.c_int]),
    "tp_set_gemm_wide_mode": (None, [ctypes.c_int]),
    "tp_launch_count": (ctypes.c_uint64, []),
    "tp_workspace_size": (_SZ, [_ST, _I64, _I64, _I64, _I32, _ST, _ST, _ST]),
    "tp_gemm": (_ST, [_P, _P, _P, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, _ST, _P]),
    "tp_col_linear": (_ST, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _ST, _ST, _ST, _P]),
    "tp_row_linear": (_ST, [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _ST, _ST, _P, _SZ, _ST, _P]),
    "tp_shard_reduce": (_ST, [_P, _P, _P, _I32, _I64, _I64, _ST, _P]),
    "tp_shard_reduce_ln": (_ST, [_P] * 8 + [_I32, _I64, _I64, ctypes.c_float, _ST, _P]),
    "tp_row_linear_ln": (_ST, [_P] * 9 + [_I64, _I64, _I64, _I32, ctypes.c_float, _ST, _ST, _P,
                                          _SZ, _P]),
    "tp_mlp_fwd": (_ST, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _ST, _ST,
                         _ST, _P, _SZ, _ST, _P]),
    "tp_mlp_bwd": (_ST, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32,
                         _ST, _ST, _ST, _P, _SZ, _ST, _P]),
    "tp_layernorm_fwd": (_ST, [_P, _P, _P, _P, _P, _P, _I64, _I64, ctypes.c_float, _ST, _P]),
    "tp_layernorm_bwd": (_ST, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _ST, _P, _SZ, _P]),
    "tp_attn_proj_fwd": (_ST, [_P] * 12 + [_I64, _I64, _I64, _I32, _I32, ctypes.c_int, _ST, _ST,
                                           _P, _SZ, _P]),
    "tp_attn_proj_bwd": (_ST, [_P] * 16 + [_I64, _I64, _I64, _I32, _I32, ctypes.c_int, _ST, _ST,
                                           _P, _SZ, _P]),
    "tp_gqa_qkv_cols": (_I64, [_I64, _I32, _I32, _I32]),
    "tp_gqa_workspace_size": (_SZ, [ctypes.c_int, _I64, _I64, _I32, _I32, _I32, _ST, _ST]),
    "tp_gqa_pack_qkv": (_ST, [_P] * 4 + [_I64, _I32, _I32, _I32, _ST, _P]),
    "tp_gqa_attention_fwd": (_ST, [_P] * 3 + [_I64, _I64, _I64, _I32, _I32, _I32, ctypes.c_int,
                                              _ST, _P]),
    "tp_gqa_attention_bwd_workspace_size": (_SZ, [_I64, _I64, _I32]),
    "tp_gqa_attention_bwd": (_ST, [_P] * 5 + [_I64, _I64, _I64, _I32, _I32, _I32, ctypes.c_int,
                                              _ST, _P, _SZ, _P]),
    "tp_gqa_attn_proj_fwd": (_ST, [_P] * 12 + [_I64, _I64, _I64, _I32, _I32, _I32, ctypes.c_int,
                                               _ST, _ST, _P, _SZ, _P]),
    "tp_gqa_attn_proj_bwd": (_ST, [_P] * 16 + [_I64, _I64, _I64, _I32, _I32, _I32, ctypes.c_int,
                                               _ST, _ST, _P, _SZ, _P]),
    "tp_sp_mlp_fwd": (_ST, [_P] * 13 + [_I64, _I64, _I64, _I32, _ST, _ST, _ST, _P, _SZ, _P]),
    "tp_sp_mlp_bwd": (_ST, [_P] * 20 + [_I64, _I64, _I64, _I32, _ST, _ST, _ST, _P, _SZ, _P]),
    "tp_layer_fwd": (_ST, [_P, ctypes.POINTER(LayerWeights), ctypes.POINTER(LayerSaved), _P, _I64,
                           _I64, _I64, _I64, _I32, _I32, ctypes.c_int, _ST, _ST, _P, _SZ, _P]),
    "tp_layer_bwd": (_ST, [_P, ctypes.POINTER(LayerWeights), ctypes.POINTER(LayerSaved), _P, _P,
                           ctypes.POINTER(LayerGrads), _I64, _I64, _I64, _I64, _I32, _I32,
                           ctypes.c_int, _ST, _ST, _P, _SZ, _P]),
    "tp_vocab_embed_fwd": (_ST, [_P, _P, _P, _I64, _I64, _I64, _I32, _ST, _P]),
    "tp_vocab_embed_bwd": (_ST, [_P, _P, _P, _I64, _I64, _I64, _I32, ctypes.c_int, _ST, _P]),
    "tp_vocab_ce_fwd": (_ST, [_P] * 6 + [_I64, _I64, _I32, _ST, _P]),
    "tp_vocab_ce_bwd": (_ST, [_P] * 4 + [_I64, _I64, _I32, ctypes.c_float, _ST, _P]),
    "tp_adamw_step": (_ST, [_P] * 4 + [_I64, _I64] + [ctypes.c_float] * 5 + [_P]),
    "tp_train_step_advance": (_ST, [_P, _P, _P, _I64, _P]),
    "tp_adamw_step_device": (_ST, [_P] * 4 + [_I64, _P] + [ctypes.c_float] * 5 + [_P]),
    "tp_gpt_workspace_size": (_SZ, [ctypes.POINTER(GptConfig), _ST, _ST]),
    "tp_gpt_fwd_bwd": (_ST, [ctypes.POINTER(GptConfig), ctypes.POINTER(GptWeights),
                             ctypes.POINTER(GptGrads), _P, _P, _P, _ST, _ST, _P, _SZ, _P]),
    "tp_row_linear_noalloc": (_ST, [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _ST, _P]),
    "tp_debug_inject_wait_fault": (None, [ctypes.c_int]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m attention_gemms_gb300.build` "
                               "(or __graft_entry__.build()). There is no fallback implementation.")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_names():
    return list(_SIGS)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dtype_of(t) -> DType:
    import torch
    if t.dtype == torch.bfloat16:
        return DType.BF16
    if t.dtype == torch.float32:
        return DType.F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check(status: int):
    if status != 0:
        raise TpError(status, lib().tp_last_error().decode(errors="replace"))


# ---------------------------------------------------------------- utilities

def tp_version() -> int:
    return lib().tp_version()


def tp_status_string(s: int) -> str:
    return lib().tp_status_string(int(s)).decode()


def tp_last_error() -> str:
    return lib().tp_last_error().decode(errors="replace")


def tp_check_status(stream=None) -> int:
    """Returns the status code (does not raise): OK, TIMEOUT or CUDA."""
    return lib().tp_check_status(_stream(stream))


def tp_set_wait_timeout_ns(ns: int) -> None:
    lib().tp_set_wait_timeout_ns(int(ns))


def tp_set_gemm_pair_mode(enable) -> None:
    """False/0: one-CTA kernel only; True/1: automatic; 2: pair kernel whenever it can run."""
    lib().tp_set_gemm_pair_mode(int(enable))


def tp_set_gemm_wide_mode(mode: int) -> None:
    lib().tp_set_gemm_wide_mode(int(mode))


def tp_launch_count() -> int:
    return int(lib().tp_launch_count())


def tp_workspace_size(op, M, h, f, N, dtype, act=Act.NONE, mode=Reduce.BUFFERS) -> int:
    return int(lib().tp_workspace_size(int(op), M, h, f, N, int(dtype), int(act), int(mode)))


def tp_debug_inject_wait_fault(enable: bool) -> None:
    lib().tp_debug_inject_wait_fault(1 if enable else 0)


# ---------------------------------------------------------------- layers

def tp_gemm(A, B, C, M, N, K, a_trans, b_trans, dtype, stream=None):
    _check(lib().tp_gemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, int(bool(a_trans)),
                         int(bool(b_trans)), int(dtype), _stream(stream)))


def tp_col_linear(X, W, W_up, Y, Y_up, out, M, h, f, N, dtype, act, stream=None,
                  w_layout=WLayout.IN_OUT):
    _check(lib().tp_col_linear(_ptr(X), _ptr(W), _ptr(W_up), _ptr(Y), _ptr(Y_up), _ptr(out),
                               M, h, f, N, int(dtype), int(act), int(w_layout), _stream(stream)))


def tp_row_linear(Xs, W, residual, out, M, k, n, N, dtype, mode, ws, ws_bytes, stream=None,
                  w_layout=WLayout.IN_OUT):
    _check(lib().tp_row_linear(_ptr(Xs), _ptr(W), _ptr(residual), _ptr(out), M, k, n, N,
                               int(dtype), int(mode), _ptr(ws), int(ws_bytes), int(w_layout),
                               _stream(stream)))


def tp_shard_reduce(partials, residual, out, N, M, n, out_dtype, stream=None):
    _check(lib().tp_shard_reduce(_ptr(partials), _ptr(residual), _ptr(out), N, M, n,
                                 int(out_dtype), _stream(stream)))


def tp_shard_reduce_ln(partials, residual, gamma, beta, sum_out, y, mean, rstd, N, M, h, eps,
                       dtype, stream=None):
    _check(lib().tp_shard_reduce_ln(_ptr(partials), _ptr(residual), _ptr(gamma), _ptr(beta),
                                    _ptr(sum_out), _ptr(y), _ptr(mean), _ptr(rstd), N, M, h,
                                    float(eps), int(dtype), _stream(stream)))


def tp_row_linear_ln(Xs, W, residual, gamma, beta, sum_out, y, mean, rstd, M, k, n, N, eps,
                     dtype, mode, ws, ws_bytes, stream=None):
    _check(lib().tp_row_linear_ln(_ptr(Xs), _ptr(W), _ptr(residual), _ptr(gamma), _ptr(beta),
                                  _ptr(sum_out), _ptr(y), _ptr(mean), _ptr(rstd), M, k, n, N,
                                  float(eps), int(dtype), int(mode), _ptr(ws), int(ws_bytes),
                                  _stream(stream)))


def tp_mlp_fwd(X, W1, W1_up, W2, residual, Y, Y_up, H, Z, M, h, f, N, dtype, act, mode, ws,
               ws_bytes, stream=None, w_layout=WLayout.IN_OUT):
    _check(lib().tp_mlp_fwd(_ptr(X), _ptr(W1), _ptr(W1_up), _ptr(W2), _ptr(residual), _ptr(Y),
                            _ptr(Y_up), _ptr(H), _ptr(Z), M, h, f, N, int(dtype), int(act),
                            int(mode), _ptr(ws), int(ws_bytes), int(w_layout), _stream(stream)))


def tp_mlp_bwd(X, W1, W1_up, W2, Y, Y_up, H, dZ, dX, dW1, dW1_up, dW2, M, h, f, N, dtype, act,
               mode, ws, ws_bytes, stream=None, w_layout=WLayout.IN_OUT):
    _check(lib().tp_mlp_bwd(_ptr(X), _ptr(W1), _ptr(W1_up), _ptr(W2), _ptr(Y), _ptr(Y_up),
                            _ptr(H), _ptr(dZ), _ptr(dX), _ptr(dW1), _ptr(dW1_up), _ptr(dW2),
                            M, h, f, N, int(dtype), int(act), int(mode), _ptr(ws),
                            int(ws_bytes), int(w_layout), _stream(stream)))


def tp_gqa_qkv_cols(h, n_heads, n_kv_heads, N):
    return int(lib().tp_gqa_qkv_cols(h, n_heads, n_kv_heads, N))


def tp_gqa_workspace_size(fwd, M, h, n_heads, n_kv_heads, N, dtype, mode):
    return int(lib().tp_gqa_workspace_size(int(bool(fwd)), M, h, n_heads, n_kv_heads, N,
                                           int(dtype), int(mode)))


def tp_gqa_pack_qkv(Wq, Wk, Wv, Wqkv, h, n_heads, n_kv_heads, N, dtype, stream=None):
    _check(lib().tp_gqa_pack_qkv(_ptr(Wq), _ptr(Wk), _ptr(Wv), _ptr(Wqkv), h, n_heads,
                                 n_kv_heads, N, int(dtype), _stream(stream)))


def tp_gqa_attention_fwd(qkv, o, lse, b, s, h, n_heads, n_kv_heads, N, causal, dtype,
                         stream=None):
    _check(lib().tp_gqa_attention_fwd(_ptr(qkv), _ptr(o), _ptr(lse), b, s, h, n_heads,
                                      n_kv_heads, N, int(causal), int(dtype), _stream(stream)))


def tp_gqa_attention_bwd_workspace_size(b, s, n_heads):
    return lib().tp_gqa_attention_bwd_workspace_size(b, s, n_heads)


def tp_gqa_attention_bwd(qkv, o, lse, dO, dqkv, b, s, h, n_heads, n_kv_heads, N, causal, dtype,
                         ws=None, ws_bytes=0, stream=None):
    _check(lib().tp_gqa_attention_bwd(_ptr(qkv), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dqkv), b, s,
                                      h, n_heads, n_kv_heads, N, int(causal), int(dtype),
                                      _ptr(ws), ws_bytes, _stream(stream)))


def tp_gqa_attn_proj_fwd(x, gamma, beta, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, out, b, s, h,
                         n_heads, n_kv_heads, N, causal, dtype, mode, ws, ws_bytes, stream=None):
    _check(lib().tp_gqa_attn_proj_fwd(*[_ptr(t) for t in (x, gamma, beta, Wqkv, Wo, xn, mean,
                                                          rstd, qkv, o, lse, out)],
                                      b, s, h, n_heads, n_kv_heads, N, int(causal), int(dtype),
                                      int(mode), _ptr(ws), int(ws_bytes), _stream(stream)))


def tp_gqa_attn_proj_bwd(x, gamma, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, dout, dx, dgamma,
                         dbeta, dWqkv, dWo, b, s, h, n_heads, n_kv_heads, N, causal, dtype, mode,
                         ws, ws_bytes, stream=None):
    _check(lib().tp_gqa_attn_proj_bwd(*[_ptr(t) for t in (x, gamma, Wqkv, Wo, xn, mean, rstd,
                                                          qkv, o, lse, dout, dx, dgamma, dbeta,
                                                          dWqkv, dWo)],
                                      b, s, h, n_heads, n_kv_heads, N, int(causal), int(dtype),
                                      int(mode), _ptr(ws), int(ws_bytes), _stream(stream)))


def tp_sp_mlp_fwd(x, gamma, beta, W1, W1_up, W2, xn, mean, rstd, Y, Y_up, H, out, M, h, f, N,
                  dtype, act, mode, ws, ws_bytes, stream=None):
    _check(lib().tp_sp_mlp_fwd(*[_ptr(t) for t in (x, gamma, beta, W1, W1_up, W2, xn, mean, rstd,
                                                   Y, Y_up, H, out)],
                               M, h, f, N, int(dtype), int(act), int(mode), _ptr(ws),
                               int(ws_bytes), _stream(stream)))


def tp_sp_mlp_bwd(x, gamma, W1, W1_up, W2, xn, mean, rstd, Y, Y_up, H, dout, dx, dgamma, dbeta,
                  dgamma_ranks, dbeta_ranks, dW1, dW1_up, dW2, M, h, f, N, dtype, act, mode, ws,
                  ws_bytes, stream=None):
    _check(lib().tp_sp_mlp_bwd(*[_ptr(t) for t in (x, gamma, W1, W1_up, W2, xn, mean, rstd, Y,
                                                   Y_up, H, dout, dx, dgamma, dbeta, dgamma_ranks,
                                                   dbeta_ranks, dW1, dW1_up, dW2)],
                               M, h, f, N, int(dtype), int(act), int(mode), _ptr(ws),
                               int(ws_bytes), _stream(stream)))


def tp_vocab_embed_fwd(ids, E, x, M, vocab, h, N, dtype, stream=None):
    _check(lib().tp_vocab_embed_fwd(_ptr(ids), _ptr(E), _ptr(x), M, vocab, h, N, int(dtype),
                                    _stream(stream)))


def tp_vocab_embed_bwd(ids, dx, dE, M, vocab, h, N, accumulate, dtype, stream=None):
    _check(lib().tp_vocab_embed_bwd(_ptr(ids), _ptr(dx), _ptr(dE), M, vocab, h, N,
                                    int(bool(accumulate)), int(dtype), _stream(stream)))


def tp_vocab_ce_fwd(logits, targets, lse, row_loss, shard_loss, loss, M, vocab, N, dtype,
                    stream=None):
    _check(lib().tp_vocab_ce_fwd(_ptr(logits), _ptr(targets), _ptr(lse), _ptr(row_loss),
                                 _ptr(shard_loss), _ptr(loss), M, vocab, N, int(dtype),
                                 _stream(stream)))


def tp_vocab_ce_bwd(logits, targets, lse, dlogits, M, vocab, N, scale, dtype, stream=None):
    _check(lib().tp_vocab_ce_bwd(_ptr(logits), _ptr(targets), _ptr(lse), _ptr(dlogits), M, vocab,
                                 N, float(scale), int(dtype), _stream(stream)))


def tp_adamw_step(p, g, m, v, n, step, lr, beta1, beta2, eps, weight_decay, stream=None):
    _check(lib().tp_adamw_step(_ptr(p), _ptr(g), _ptr(m), _ptr(v), n, step, float(lr),
                               float(beta1), float(beta2), float(eps), float(weight_decay),
                               _stream(stream)))


def tp_train_step_advance(step, loss, loss_hist, hist_len, stream=None):
    _check(lib().tp_train_step_advance(_ptr(step), _ptr(loss), _ptr(loss_hist), int(hist_len),
                                       _stream(stream)))


def tp_adamw_step_device(p, g, m, v, n, step, lr, beta1, beta2, eps, weight_decay, stream=None):
    _check(lib().tp_adamw_step_device(_ptr(p), _ptr(g), _ptr(m), _ptr(v), n, _ptr(step),
                                      float(lr), float(beta1), float(beta2), float(eps),
                                      float(weight_decay), _stream(stream)))


def tp_gpt_workspace_size(cfg, dtype, mode):
    return int(lib().tp_gpt_workspace_size(ctypes.byref(cfg), int(dtype), int(mode)))


def tp_gpt_fwd_bwd(cfg, weights, grads, ids, targets, loss, dtype, mode, ws, ws_bytes, stream=None):
    _check(lib().tp_gpt_fwd_bwd(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(grads),
                                _ptr(ids), _ptr(targets), _ptr(loss), int(dtype), int(mode),
                                _ptr(ws), int(ws_bytes), _stream(stream)))


def tp_row_linear_noalloc(Xs, W, residual, out, M, k, n, N, dtype, stream=None):
    _check(lib().tp_row_linear_noalloc(_ptr(Xs), _ptr(W), _ptr(residual), _ptr(out), M, k, n, N,
                                       int(dtype), _stream(stream)))


# ---------------------------------------------------------------- attention block and layer

def tp_layernorm_fwd(x, gamma, beta, y, mean, rstd, M, h, eps, dtype, stream=None):
    _check(lib().tp_layernorm_fwd(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), _ptr(mean),
                                  _ptr(rstd), M, h, float(eps), int(dtype), _stream(stream)))


def tp_layernorm_bwd(x, gamma, mean, rstd, dy, dres, dx, dgamma, dbeta, M, h, dtype, ws, ws_bytes,
                     stream=None):
    _check(lib().tp_layernorm_bwd(_ptr(x), _ptr(gamma), _ptr(mean), _ptr(rstd), _ptr(dy),
                                  _ptr(dres), _ptr(dx), _ptr(dgamma), _ptr(dbeta), M, h,
                                  int(dtype), _ptr(ws), int(ws_bytes), _stream(stream)))


def tp_attn_proj_fwd(x, gamma, beta, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, out, b, s, h, n_heads,
                     N, causal, dtype, mode, ws, ws_bytes, stream=None):
    _check(lib().tp_attn_proj_fwd(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(Wqkv), _ptr(Wo), _ptr(xn),
                                  _ptr(mean), _ptr(rstd), _ptr(qkv), _ptr(o), _ptr(lse), _ptr(out),
                                  b, s, h, n_heads, N, int(causal), int(dtype), int(mode), _ptr(ws),
                                  int(ws_bytes), _stream(stream)))


def tp_attn_proj_bwd(x, gamma, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, dout, dx, dgamma, dbeta,
                     dWqkv, dWo, b, s, h, n_heads, N, causal, dtype, mode, ws, ws_bytes,
                     stream=None):
    _check(lib().tp_attn_proj_bwd(_ptr(x), _ptr(gamma), _ptr(Wqkv), _ptr(Wo), _ptr(xn), _ptr(mean),
                                  _ptr(rstd), _ptr(qkv), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dx),
                                  _ptr(dgamma), _ptr(dbeta), _ptr(dWqkv), _ptr(dWo), b, s, h,
                                  n_heads, N, int(causal), int(dtype), int(mode), _ptr(ws),
                                  int(ws_bytes), _stream(stream)))


def tp_layer_fwd(x, weights, saved, out, b, s, h, f, n_heads, N, causal, dtype, mode, ws, ws_bytes,
                 stream=None):
    _check(lib().tp_layer_fwd(_ptr(x), ctypes.byref(weights), ctypes.byref(saved), _ptr(out), b, s,
                              h, f, n_heads, N, int(causal), int(dtype), int(mode), _ptr(ws),
                              int(ws_bytes), _stream(stream)))


def tp_layer_bwd(x, weights, saved, dout, dx, grads, b, s, h, f, n_heads, N, causal, dtype, mode, ws,
                 ws_bytes, stream=None):
    _check(lib().tp_layer_bwd(_ptr(x), ctypes.byref(weights), ctypes.byref(saved), _ptr(dout),
                              _ptr(dx), ctypes.byref(grads), b, s, h, f, n_heads, N, int(causal),
                              int(dtype), int(mode), _ptr(ws), int(ws_bytes), _stream(stream)))

