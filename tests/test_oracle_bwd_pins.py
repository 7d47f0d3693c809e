"""CPU pins of the backward oracle: finite differences of the forward oracle,
torch float64 autograd, the softmax-Jacobian identities, sampled = full."""

import numpy as np
import pytest
import torch

from oracle import attention_bwd_head, attention_bwd_ref, attention_bwd_sampled, attention_ref


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).normal(size=shape) * std


def _loss(q, k, v, dout, scale, causal, kv):
    o, _ = attention_ref(q, k, v, scale, causal=causal, kv_lens=kv)
    return float(np.sum(o * dout))


@pytest.mark.parametrize("causal,kv", [(False, None), (True, None), (False, [3, 0]), (True, [4, 2])])
def test_gradients_match_central_differences(causal, kv):
    B, H, Sq, Sk, D = 2, 1, 4, 5, 3
    q, k, v = _rand((B, H, Sq, D), 1), _rand((B, H, Sk, D), 2), _rand((B, H, Sk, D), 3)
    dout = _rand((B, H, Sq, D), 4)
    scale = 0.7
    dq, dk, dv = attention_bwd_ref(q, k, v, dout, scale, causal=causal, kv_lens=kv)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], dout, scale, causal, kv)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], dout, scale, causal, kv)
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_torch_autograd(causal):
    B, H, Sq, Sk, D = 2, 3, 17, 23, 8
    kv = [23, 9]
    q, k, v = _rand((B, H, Sq, D), 5), _rand((B, H, Sk, D), 6), _rand((B, H, Sk, D), 7)
    dout = _rand((B, H, Sq, D), 8)
    scale = 0.4
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = torch.einsum("bhid,bhjd->bhij", tq, tk) * scale
    cols = torch.arange(Sk)
    valid = cols[None, None, None, :] < torch.tensor(kv)[:, None, None, None]
    if causal:
        valid = valid & (cols[None, None, None, :] <= torch.arange(Sq)[None, None, :, None])
    p = torch.softmax(s.masked_fill(~valid, float("-inf")), dim=-1)
    o = p @ tv
    (o * torch.tensor(dout)).sum().backward()
    dq, dk, dv = attention_bwd_ref(q, k, v, dout, scale, causal=causal, kv_lens=kv)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_identities_and_masked_rows():
    Sq, Sk, D = 9, 11, 4
    q, k, v, dout = _rand((Sq, D), 9), _rand((Sk, D), 10), _rand((Sk, D), 11), _rand((Sq, D), 12)
    scale = 0.5
    dq, dk, dv = attention_bwd_head(q, k, v, dout, scale, causal=True, kv_len=7)
    # dV: each valid row's probabilities sum to 1, so sum_j dV_j = sum of dO over rows with a key
    np.testing.assert_allclose(dv.sum(axis=0), dout.sum(axis=0), rtol=1e-12, atol=1e-12)
    # keys past kv_len get no gradient
    assert np.all(dk[7:] == 0) and np.all(dv[7:] == 0)
    # the softmax Jacobian has zero row sums: sum_i dQ_i-weighted... dK sums to scale * sum_i (sum_j dS_ij) q_i = 0
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    # Delta_i = sum_j P_ij dP_ij equals <dO_i, O_i>
    o, _ = attention_ref(q[None, None], k[None, None], v[None, None], scale, causal=True, kv_lens=[7])
    from oracle.backward import _probs
    p = _probs(q, np.arange(Sq), k, scale, True, 7)
    np.testing.assert_allclose(np.sum(p * (dout @ v.T), axis=1), np.sum(dout * o[0, 0], axis=1), rtol=1e-12)
    # no valid key anywhere: all gradients vanish
    z = attention_bwd_head(q, k, v, dout, scale, kv_len=0)
    assert all(np.all(g == 0) for g in z)


def test_sampled_equals_full():
    Sq, Sk, D = 40, 37, 6
    q, k, v, dout = _rand((Sq, D), 13), _rand((Sk, D), 14), _rand((Sk, D), 15), _rand((Sq, D), 16)
    for causal in (False, True):
        dq, dk, dv = attention_bwd_head(q, k, v, dout, 0.3, causal=causal, kv_len=30, block=7)
        qr, kr = [0, 5, 39], [0, 12, 29, 36]
        sq, sk, sv = attention_bwd_sampled(q, k, v, dout, 0.3, qr, kr, causal=causal, kv_len=30, block=9)
        np.testing.assert_allclose(sq, dq[qr], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(sk, dk[kr], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(sv, dv[kr], rtol=1e-12, atol=1e-13)


BWD_MUTATIONS = {
    "delta_sign": ("ds = p * (dp - delta[:, None])", "ds = p * (dp + delta[:, None])"),
    "dq_scale_dropped": ("dq[rows] = np.float64(scale) * (ds @ k)", "dq[rows] = (ds @ k)"),
    "dv_wrong_rows": ("dv += p.T @ dout[rows]", "dv += p.T @ dout[rows][::-1]"),
    "dk_uses_dout": ("dk += np.float64(scale) * (ds.T @ q[rows])", "dk += np.float64(scale) * (ds.T @ dout[rows])"),
    "causal_diag": ("lim = np.minimum(lim, row_index.astype(np.int64) + 1)",
                    "lim = np.minimum(lim, row_index.astype(np.int64))"),
}


def _torch_grads(q, k, v, dout, scale, causal):
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = torch.einsum("bhid,bhjd->bhij", tq, tk) * scale
    Sq, Sk = q.shape[2], k.shape[2]
    if causal:
        s = s.masked_fill(torch.arange(Sk)[None, :] > torch.arange(Sq)[:, None], float("-inf"))
    (torch.softmax(s, dim=-1) @ tv * torch.tensor(dout)).sum().backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("name", sorted(BWD_MUTATIONS))
def test_bwd_pins_catch_planted_mistake(name):
    """Each planted mistake makes the oracle disagree with torch's float64
    autograd (the independent pin above)."""
    import types

    import oracle.backward as real
    src = open(real.__file__).read().replace("from .attention import _as_f64", "from oracle.attention import _as_f64")
    old, new = BWD_MUTATIONS[name]
    assert src.count(old) == 1, name
    mod = types.ModuleType("oracle_bwd_mutant_" + name)
    exec(compile(src.replace(old, new), "<bwd mutant>", "exec"), mod.__dict__)
    B, H, Sq, Sk, D = 1, 2, 6, 6, 4
    q, k, v = _rand((B, H, Sq, D), 17), _rand((B, H, Sk, D), 18), _rand((B, H, Sk, D), 19)
    dout = _rand((B, H, Sq, D), 20)
    want = _torch_grads(q, k, v, dout, 0.6, True)
    assert all(np.allclose(a, b, rtol=1e-10, atol=1e-12)
               for a, b in zip(attention_bwd_ref(q, k, v, dout, 0.6, causal=True), want))
    got = mod.attention_bwd_ref(q, k, v, dout, 0.6, causal=True)
    assert any(not np.allclose(a, b, rtol=1e-9, atol=1e-12) for a, b in zip(got, want)), name
