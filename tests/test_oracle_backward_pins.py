"""Pins for the oracle's backward (the training form of the MoE block and of
the FarSkip stack).  The pages give no gradient formulas, so the backward is
fixed by what the forward fixes:

  finite differences -- central differences of the pinned forward oracle (fp64,
                        exact storage) for the input and every weight tensor,
                        every gate rule and every MoE wiring (a dropped term, a
                        wrong sign, a transposed or swapped operand, a wiring
                        gradient sent to the wrong residual all fail here)
  library autodiff   -- torch.autograd through a float64 dense evaluation of
                        one block (all experts, masked by the oracle's routing)
  identities         -- do_prev = dO + dOs; gradients are linear in (dO, dOs);
                        bf16 storage changes the gradients only by rounding
"""

import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import W, cfg_of, rand_weights

WIRINGS = ["partial", "outdated", "disabled"]
GATES = ["softmax", "softmax_renorm", "sigmoid", "sigmoid_norm"]


def _problem(seed, L=2, T=6, d=12, E=5, k=2, c=8, ns=2, cs=4, gate="sigmoid_norm"):
    r = np.random.default_rng(seed)
    ws = [rand_weights(r, d, E, c, ns, cs, bias=True) for _ in range(L)]
    x = r.standard_normal((T, d))
    G = r.standard_normal((T, d))
    Gs = r.standard_normal((T, d))
    return cfg_of(d, E, k, c, ns, cs, gate), ws, x, G, Gs, r


def _loss(cfg, ws, wiring, x, G, Gs):
    o = oracle.stack(cfg, [W(v) for v in ws], wiring, x, want_logits=False)
    return float((o["o"] * G).sum() + (o["o_star"] * Gs).sum())


def _fd_check(cfg, ws, wiring, x, G, Gs, r, n_w=4, eps=1e-6, tol=1e-6):
    b = oracle.stack_backward(cfg, [W(v) for v in ws], wiring, x, G, Gs)
    fd = np.zeros_like(x)
    for t in range(x.shape[0]):
        for i in range(x.shape[1]):
            xp, xm = x.copy(), x.copy()
            xp[t, i] += eps
            xm[t, i] -= eps
            fd[t, i] = (_loss(cfg, ws, wiring, xp, G, Gs) - _loss(cfg, ws, wiring, xm, G, Gs)) / (2 * eps)
    assert np.linalg.norm(fd - b["dx"]) <= tol * max(1.0, np.linalg.norm(fd)), "dx"
    keys = [("w_r", "dW_R"), ("w1", "dW1"), ("w2", "dW2"), ("w3", "dW3")]
    if cfg.n_shared:
        keys += [("w1s", "dW1s"), ("w2s", "dW2s"), ("w3s", "dW3s")]
    for blk in range(len(ws)):
        for name, key in keys:
            W0 = ws[blk][name]
            for _ in range(n_w):
                ix = tuple(int(r.integers(0, s)) for s in W0.shape)
                wp = [dict(v) for v in ws]
                wm = [dict(v) for v in ws]
                wp[blk][name] = W0.copy()
                wm[blk][name] = W0.copy()
                wp[blk][name][ix] += eps
                wm[blk][name][ix] -= eps
                f = (_loss(cfg, wp, wiring, x, G, Gs) - _loss(cfg, wm, wiring, x, G, Gs)) / (2 * eps)
                assert abs(f - b[key][blk][ix]) <= tol * max(1.0, abs(f)), (blk, key, ix, f, b[key][blk][ix])
    return b


@pytest.mark.parametrize("wiring", WIRINGS)
def test_stack_backward_finite_differences_wirings(wiring):
    cfg, ws, x, G, Gs, r = _problem(31, L=3)
    _fd_check(cfg, ws, wiring, x, G, Gs, r)


@pytest.mark.parametrize("gate", GATES)
def test_stack_backward_finite_differences_gates(gate):
    cfg, ws, x, G, Gs, r = _problem(32, L=2, gate=gate, E=6, k=3)
    _fd_check(cfg, ws, "partial", x, G, Gs, r)


def test_stack_backward_finite_differences_no_shared_top1():
    cfg, ws, x, G, Gs, r = _problem(33, L=2, ns=0, cs=0, k=1, gate="sigmoid")
    _fd_check(cfg, ws, "outdated", x, G, Gs, r)


def _torch_block(cfg, w, u):
    """Float64 dense evaluation of one block (every expert on every token,
    combined with the oracle's routing as a constant mask) for autograd."""
    T = u.shape[0]
    z = u @ w["w_r"].T + w["bias"]
    logits, idx, _ = oracle.router(cfg, u.detach().numpy(), w["w_r"].detach().numpy(), w["bias"].detach().numpy())
    mask = torch.zeros(T, cfg.E, dtype=torch.float64)
    mask[torch.arange(T)[:, None], torch.from_numpy(idx).long()] = 1.0
    if cfg.gate == oracle.GATES["softmax"]:
        wt = torch.softmax(z, dim=1) * mask
    elif cfg.gate == oracle.GATES["softmax_renorm"]:
        e = torch.exp(z - z.max(dim=1, keepdim=True).values) * mask
        wt = e / e.sum(dim=1, keepdim=True)
    elif cfg.gate == oracle.GATES["sigmoid"]:
        wt = torch.sigmoid(z) * mask
    else:
        sg = torch.sigmoid(z) * mask
        wt = sg / sg.sum(dim=1, keepdim=True)
    R = torch.zeros_like(u)
    for e in range(cfg.E):
        y = (torch.nn.functional.silu(u @ w["w2"][e].T) * (u @ w["w1"][e].T)) @ w["w3"][e].T
        R = R + wt[:, e:e + 1] * y
    S = torch.zeros_like(u)
    for s in range(cfg.n_shared):
        S = S + (torch.nn.functional.silu(u @ w["w2s"][s].T) * (u @ w["w1s"][s].T)) @ w["w3s"][s].T
    return R, S


@pytest.mark.parametrize("gate", GATES)
def test_block_backward_matches_autograd(gate):
    cfg, ws, x, G, Gs, r = _problem(34, L=1, gate=gate, E=6, k=3)
    w = {k_: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k_, v in ws[0].items()}
    u = torch.tensor(x, requires_grad=True)
    o_prev = torch.tensor(r.standard_normal(x.shape))
    R, S = _torch_block(cfg, w, u)
    o_star = o_prev + S
    o = o_star + R
    loss = (o * torch.from_numpy(G)).sum() + (o_star * torch.from_numpy(Gs)).sum()
    loss.backward()
    b = oracle.block_backward(cfg, W(ws[0]), x, G, Gs)
    np.testing.assert_allclose(b["du"], u.grad.numpy(), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(b["do_prev"], G + Gs, rtol=0, atol=0)
    for name, key in (("w_r", "dW_R"), ("w1", "dW1"), ("w2", "dW2"), ("w3", "dW3"), ("w1s", "dW1s"),
                      ("w2s", "dW2s"), ("w3s", "dW3s")):
        np.testing.assert_allclose(b[key], w[name].grad.numpy(), rtol=1e-10, atol=1e-10, err_msg=key)


def test_backward_is_linear_in_the_output_gradients():
    cfg, ws, x, G, Gs, r = _problem(35, L=1)
    b1 = oracle.block_backward(cfg, W(ws[0]), x, G, Gs)
    b2 = oracle.block_backward(cfg, W(ws[0]), x, 2.0 * G, 2.0 * Gs)
    b3 = oracle.block_backward(cfg, W(ws[0]), x, G, None)
    b4 = oracle.block_backward(cfg, W(ws[0]), x, np.zeros_like(G), Gs)
    for key in ("du", "dW_R", "dW1", "dW2", "dW3", "dW1s", "dW2s", "dW3s"):
        np.testing.assert_allclose(b2[key], 2.0 * b1[key], rtol=1e-12, atol=1e-13, err_msg=key)
        np.testing.assert_allclose(b3[key] + b4[key], b1[key], rtol=1e-10, atol=1e-12, err_msg=key)
    # dOs reaches only the shared experts and o_prev: no routed or router gradient
    for key in ("dW_R", "dW1", "dW2", "dW3"):
        assert not b4[key].any(), key


def test_bf16_storage_backward_differs_only_by_rounding():
    cfg, ws, x, G, Gs, r = _problem(36, L=2)
    ex = oracle.stack_backward(cfg, [W(v) for v in ws], "partial", x, G, Gs)
    cb = cfg_of(cfg.d, cfg.E, cfg.k, cfg.c, cfg.n_shared, cfg.c_shared, "sigmoid_norm", storage=oracle.STORE_BF16)
    bf = oracle.stack_backward(cb, [W(v) for v in ws], "partial", x, G, Gs)
    for key in ("dx", "dW1", "dW3", "dW_R", "dW3s"):
        rel = np.linalg.norm(bf[key] - ex[key]) / np.linalg.norm(ex[key])
        assert 0 < rel < 3e-2, (key, rel)
