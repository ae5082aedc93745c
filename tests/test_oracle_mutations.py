"""Plant plausible mistakes in the oracle (on the CPU, by monkeypatching) and
check that a pin catches each one: a dropped term, a wrong sign, a transposed
operand, a wrong shard index."""
import numpy as np

from oracle import tp_oracle as O
from tests import test_oracle_pins as pins


def test_dropped_term_in_gelu_prime_is_caught(monkeypatch):
    bad = lambda x: 0.5 * (1.0 + O._erf(np.asarray(x) / O.SQRT2))  # Phi only, x*phi dropped
    monkeypatch.setattr(O, "gelu_prime", bad)
    errs = pins.fd_errors_mlp_gelu(2)
    assert max(errs.values()) > 1e-3


def test_wrong_sign_in_swiglu_grad_is_caught(monkeypatch):
    def bad(dA, G, U):
        s = O.sigmoid(G)
        return dA * U * s * (1.0 - G * (1.0 - s)), dA * G * s
    monkeypatch.setattr(O, "_swiglu_grads", bad)
    errs = pins.fd_errors_mlp_swiglu(2)
    assert max(errs.values()) > 1e-3


def test_transposed_weight_grad_is_caught(monkeypatch):
    real = O.mlp_gelu_bwd

    def bad(X, W1, W2, dZ, N):
        g = real(X, W1, W2, dZ, N)
        # dW2 built as dZ^T H instead of H^T dZ, reshaped to fit
        H = O.gelu(X @ W1)
        g["dW2"] = (dZ.T @ H).reshape(g["dW2"].shape)
        return g
    monkeypatch.setattr(O, "mlp_gelu_bwd", bad)
    errs = pins.fd_errors_mlp_gelu(2)
    assert errs["dW2"] > 1e-3


def test_wrong_row_shard_is_caught(monkeypatch):
    real = O.row_shards

    def bad(W, N):
        s = real(W, N)
        return s[::-1]  # shard i paired with the wrong row block
    monkeypatch.setattr(O, "row_shards", bad)
    r = np.random.default_rng(0)
    X, W = r.normal(size=(3, 6)), r.normal(size=(6, 5))
    assert O.rel_err(O.row_linear(X, W, 2), X @ W) > 1e-3


def test_tanh_gelu_is_caught(monkeypatch):
    tanh_gelu = lambda x: 0.5 * np.asarray(x) * (1 + np.tanh(np.sqrt(2 / np.pi) * (x + 0.044715 * np.asarray(x) ** 3)))
    monkeypatch.setattr(O, "gelu", tanh_gelu)
    import pytest
    with pytest.raises(AssertionError):
        pins.test_gelu_phi_table()


def test_ln_before_sum_is_caught(monkeypatch):
    """LN applied to each shard's partial and the results summed: what the notes
    rule out (the statistics need the whole sum)."""
    def bad(partials, residual, gamma, beta, eps=O.LN_EPS):
        parts = [O.layernorm_fwd(P, gamma, beta, eps)[0] for P in partials]
        x = O.shard_reduce(partials, residual)
        _, mu, rs = O.layernorm_fwd(x, gamma, beta, eps)
        return x, O.shard_reduce(parts, residual), mu, rs
    monkeypatch.setattr(O, "shard_reduce_ln", bad)
    import pytest
    with pytest.raises(AssertionError):
        pins.test_shard_reduce_ln_bruteforce()


def test_residual_dropped_before_ln_is_caught(monkeypatch):
    def bad(partials, residual, gamma, beta, eps=O.LN_EPS):
        x = O.shard_reduce(partials, residual)
        y, mu, rs = O.layernorm_fwd(O.shard_reduce(partials), gamma, beta, eps)
        return x, y, mu, rs
    monkeypatch.setattr(O, "shard_reduce_ln", bad)
    import pytest
    with pytest.raises(AssertionError):
        pins.test_shard_reduce_ln_equals_ln_of_unsplit_row_gemm()


def test_sp_missing_residual_grad_is_caught(monkeypatch):
    """The block's input gradient without the residual's dout_r term."""
    real_sp = O.sp_mlp_block_bwd

    def bad(x, gamma, beta, W1, W2, N, dout, act="gelu", W1u=None, eps=O.LN_EPS):
        res = real_sp(x, gamma, beta, W1, W2, N, dout, act, W1u, eps)
        res["dx"] = res["dx"] - dout
        return res
    monkeypatch.setattr(O, "sp_mlp_block_bwd", bad)
    import pytest
    with pytest.raises(AssertionError):
        pins.test_sp_mlp_block_equals_unsplit_and_fd("gelu", 2)


def test_sp_rank_gradient_not_summed_is_caught(monkeypatch):
    """Taking rank 0's LN gradient as if it were replicated (no sum over ranks)."""
    real_sp = O.sp_mlp_block_bwd

    def bad(x, gamma, beta, W1, W2, N, dout, act="gelu", W1u=None, eps=O.LN_EPS):
        res = real_sp(x, gamma, beta, W1, W2, N, dout, act, W1u, eps)
        res["dgamma"] = res["dgamma_ranks"][0]
        return res
    monkeypatch.setattr(O, "sp_mlp_block_bwd", bad)
    import pytest
    with pytest.raises(AssertionError):
        pins.test_sp_mlp_block_equals_unsplit_and_fd("gelu", 2)


def test_sp_rank_rows_swapped_is_caught(monkeypatch):
    """Reduce-scatter handing rank r the rows of rank r+1."""
    real = O.seq_slices

    def bad(M, N):
        s = real(M, N)
        return s[1:] + s[:1]
    monkeypatch.setattr(O, "seq_slices", bad)
    import pytest
    with pytest.raises(AssertionError):
        pins.test_sp_mlp_block_equals_unsplit_and_fd("gelu", 2)


def test_tied_embedding_missing_input_grad_is_caught(monkeypatch):
    """grad_total = grad_out only (the input layer's gradient dropped)."""
    from oracle import gpt_oracle as G
    from tests import test_oracle_gpt_pins as gp
    monkeypatch.setattr(G, "vocab_embed_bwd", lambda ids, dx, v, N: np.zeros((v, dx.shape[1])))
    import pytest
    with pytest.raises(AssertionError):
        gp.test_gpt_backward_fd()


def test_ce_grad_without_onehot_is_caught(monkeypatch):
    from oracle import gpt_oracle as G
    from tests import test_oracle_gpt_pins as gp

    def bad(logits, targets, lse, N, scale):
        return np.exp(logits - lse[:, None]) * scale
    monkeypatch.setattr(G, "vocab_ce_bwd", bad)
    import pytest
    with pytest.raises(AssertionError):
        gp.test_vocab_ce_bwd_fd(2)


def test_adamw_without_bias_correction_is_caught(monkeypatch):
    from oracle import gpt_oracle as G
    from tests import test_oracle_gpt_pins as gp

    def bad(p, g, m, v, t, lr, beta1, beta2, eps, weight_decay):
        p = p * (1.0 - lr * weight_decay)
        m = beta1 * m + (1.0 - beta1) * g
        v = beta2 * v + (1.0 - beta2) * g * g
        return p - lr * m / (np.sqrt(v) + eps), m, v
    monkeypatch.setattr(G, "adamw_step", bad)
    import pytest
    with pytest.raises(AssertionError):
        gp.test_adamw_first_steps_closed_form()


def test_gqa_replicas_not_synchronised_is_caught(monkeypatch):
    """Replicated key/value heads whose weight gradients are not all-reduced: each
    replica keeps only its own query heads' share."""
    from oracle import gqa_oracle as Q
    from tests import test_oracle_gqa_pins as qp
    monkeypatch.setattr(Q, "gqa_split", lambda H, Hkv, N: (H // N, 1, 1) if N > Hkv else
                        (H // N, Hkv // N, 1))
    import pytest
    with pytest.raises((AssertionError, IndexError, ValueError)):
        qp.test_gqa_bwd_fd(4, 2, 4)


def test_gqa_wrong_group_is_caught(monkeypatch):
    """Query head t paired with key/value head t % Hkv instead of t // (H / Hkv)."""
    from oracle import gqa_oracle as Q
    from oracle import tp_oracle as T0
    from tests import test_oracle_gqa_pins as qp

    def bad(xn, Wq, Wk, Wv, b, s, H, Hkv, causal=False):
        d = Wq.shape[1] // H
        Qm, K, V = xn @ Wq, xn @ Wk, xn @ Wv
        O = np.zeros((xn.shape[0], H * d))
        for t in range(H):
            j = t % Hkv
            for bb in range(b):
                r = slice(bb * s, (bb + 1) * s)
                O[r, t * d:(t + 1) * d] = T0.attention_head_fwd(
                    Qm[r, t * d:(t + 1) * d], K[r, j * d:(j + 1) * d], V[r, j * d:(j + 1) * d],
                    causal)[0]
        return O
    monkeypatch.setattr(Q, "gqa_attention_unsplit", bad)
    import pytest
    with pytest.raises(AssertionError):
        qp.test_gqa_grouping_head_by_head()


def test_gqa_core_kv_grad_not_summed_over_group_is_caught(monkeypatch):
    """The attention core's key/value gradient overwritten by each query head of its
    group instead of summed over them."""
    from oracle import gqa_oracle as Q
    from oracle import tp_oracle as T0
    from tests import test_oracle_gqa_pins as qp

    def bad(QKV, dO, b, s, H, Hkv, N, causal=False):
        d = dO.shape[1] // H
        hq, hkv, Ws = Q._shard_views(H, Hkv, N, d)
        g = hq // hkv
        dQKV = np.zeros_like(QKV)
        for i in range(N):
            Qi, dQi = QKV[:, i * Ws:(i + 1) * Ws], dQKV[:, i * Ws:(i + 1) * Ws]
            dOi = dO[:, i * hq * d:(i + 1) * hq * d]
            for tl in range(hq):
                kl = tl // g
                qc = slice(tl * d, (tl + 1) * d)
                kc = slice((hq + kl) * d, (hq + kl + 1) * d)
                vc = slice((hq + hkv + kl) * d, (hq + hkv + kl + 1) * d)
                for bb in range(b):
                    rr = slice(bb * s, (bb + 1) * s)
                    dq, dk, dv = T0.attention_head_bwd(Qi[rr, qc], Qi[rr, kc], Qi[rr, vc],
                                                       dOi[rr, qc], causal)
                    dQi[rr, qc] += dq
                    dQi[rr, kc] = dk   # the mistake: the group's heads overwrite each other
                    dQi[rr, vc] = dv
        return dQKV
    monkeypatch.setattr(Q, "gqa_attention_bwd", bad)
    import pytest
    with pytest.raises(AssertionError):
        qp.test_gqa_core_bwd_fd(4, 2, 2, False)


def test_gqa_core_wrong_local_kv_head_is_caught(monkeypatch):
    """Inside a shard, local query head tl paired with local key/value head tl % hkv
    instead of tl // g."""
    from oracle import gqa_oracle as Q
    from oracle import tp_oracle as T0
    from tests import test_oracle_gqa_pins as qp

    def bad(QKV, b, s, H, Hkv, N, causal=False):
        hq, hkv, _ = Q.gqa_split(H, Hkv, N)
        d = QKV.shape[1] // (N * (hq + 2 * hkv))
        Ws = (hq + 2 * hkv) * d
        O = np.zeros((QKV.shape[0], H * d))
        for i in range(N):
            Qi = QKV[:, i * Ws:(i + 1) * Ws]
            for tl in range(hq):
                kl = tl % hkv  # the mistake
                for bb in range(b):
                    r = slice(bb * s, (bb + 1) * s)
                    O[r, (i * hq + tl) * d:(i * hq + tl + 1) * d] = T0.attention_head_fwd(
                        Qi[r, tl * d:(tl + 1) * d], Qi[r, (hq + kl) * d:(hq + kl + 1) * d],
                        Qi[r, (hq + hkv + kl) * d:(hq + hkv + kl + 1) * d], causal)[0]
        return O
    monkeypatch.setattr(Q, "gqa_attention_fwd", bad)
    import pytest
    with pytest.raises(AssertionError):
        qp.test_gqa_sharded_equals_unsplit(8, 2, 1, False)   # hq = 8, hkv = 2: g = 4
