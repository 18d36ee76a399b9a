"""Pins of the per-layer predictor's firing rule and of the float32 error bound
that decides when a GPU argmax or firing decision may differ from the fp64
oracle.  CPU only.

* Firing rule (LLM in a flash, section 3.1 "Reducing Data Transfer": a
  neuron is predicted active where the predictor's sigmoid output exceeds
  0.5, i.e. where its logit, bias included, is strictly positive): a
  hand-worked decode through the oracle's own step function.
* Error bound (oracle.fp32_dot_bound / argmax_tolerance): it must hold for
  real float32 evaluations (torch's float32 matmul, a sequential float32 loop
  with separate multiply and add, a blocked tree of the stated height, a
  perturbed input), and it must be tight enough at the full predictor shapes
  that it cannot accept a plainly wrong decision.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from oracle import OracleDecoder
from tests.parity import (X_REL, _fire_accept, _ids_accept, predictor_bound_args,
                          rowdot_depth)
from workloads import LLAMA7B, OPT67B, SMALL_OPT, make_workload
from workloads.synth import Workload


# ---------------------------------------------------------------------------
# Firing rule, worked by hand
# ---------------------------------------------------------------------------
def _hand_opt_workload():
    """One sparse layer, D = 2, H = 2, F = 5, float32, token input [2, -2].

    x_hat = [2, -2] / sqrt(4 + 1e-6) = [s, -s], s just below 1
    z = relu(W1 x_hat) with W1 = I: [s, 0]
    neuron | W2 row  | b2    | logit                   | fires
    0      | [1, 0]  |  0    | s                       | yes
    1      | [1, 0]  | -2    | s - 2 < 0 (bias flips)  | no
    2      | [0, 5]  |  0    | 5 * 0 = 0 exactly       | no (strict)
    3      | [0, 3]  |  0.5  | 0.5 (ReLU zeroed z_1)   | yes
    4      | [0, 0]  |  0.25 | 0.25 (bias alone)       | yes
    """
    cfg = SMALL_OPT.replace(name="hand-opt", n_layers=1, d_model=2, d_ff=5, k_max=5, pred_hidden=2,
                            dtype="f32", n_decode=1, window=5)
    w1 = torch.eye(2, dtype=torch.float32).reshape(1, 2, 2)
    w2 = torch.tensor([[[1.0, 0.0], [1.0, 0.0], [0.0, 5.0], [0.0, 3.0], [0.0, 0.0]]])
    b2 = torch.tensor([[0.0, -2.0, 0.0, 0.5, 0.25]])
    store = torch.arange(5 * 2 * 2, dtype=torch.float32).reshape(1, 5, 2, 2)
    x = torch.tensor([[[2.0, -2.0]]])
    return Workload(cfg=cfg, dense_w=None, store=store, centroids=None, pred_w1=w1, pred_w2=w2,
                    pred_b2=b2, x=x)


def test_perlayer_firing_rule_hand_worked():
    wl = _hand_opt_workload()
    rec = OracleDecoder(wl).step(wl.x[0].numpy())
    s = 2.0 / np.sqrt(4.0 + 1e-6)
    lg = rec.pred_logits_layer[0]
    assert np.allclose(lg, [s, s - 2.0, 0.0, 0.5, 0.25], rtol=0, atol=1e-15)
    assert lg[2] == 0.0                      # exactly zero: the boundary case
    assert rec.active[0] == [0, 3, 4]        # strict > 0, bias included, ReLU on z
    # the same decisions as sigmoid(logit) > 0.5 (the pages' statement)
    assert (np.flatnonzero(expit(lg) > 0.5) == [0, 3, 4]).all()
    assert expit(0.0) == 0.5
    # cold start: every active neuron is incoming, slots in ascending order
    assert rec.d_in[0] == [(0, 0), (3, 1), (4, 2)]


# ---------------------------------------------------------------------------
# float32 evaluations the bound must cover
# ---------------------------------------------------------------------------
def _rand(shape, dtype, seed, std=0.02):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float64) * std).to(dtype)


def _sequential_fp32(w32: np.ndarray, v32: np.ndarray) -> np.ndarray:
    """Row dot products in float32, one term at a time, multiply and add
    rounded separately (the longest chain of roundings: depth k)."""
    acc = np.zeros(w32.shape[0], dtype=np.float32)
    for j in range(w32.shape[1]):
        acc = (acc + (w32[:, j] * v32[j]).astype(np.float32)).astype(np.float32)
    return acc


def _tree_fp32(w32: np.ndarray, v32: np.ndarray, elem_bytes: int) -> np.ndarray:
    """Row dot products in float32 in a tree of the batch-1 predictor's
    shape: 256 threads each chain fused multiply-adds over their 16-byte
    chunks into two sums (even and odd elements of every chunk), add the two,
    then a 5-level butterfly inside each warp of 32, then the 8 warp sums in
    order.  A fused multiply-add is emulated as one rounding to float32 of the
    (exact in float64) product plus the accumulator."""
    rows, k = w32.shape
    e = 16 // elem_bytes
    nc = k // e
    chunks = -(-nc // 256)
    prod = w32.astype(np.float64) * v32.astype(np.float64)          # exact
    pad = np.zeros((rows, chunks * 256 * e))
    pad[:, :k] = prod
    p = pad.reshape(rows, chunks, 256, e)
    even = np.zeros((rows, 256), dtype=np.float32)
    odd = np.zeros((rows, 256), dtype=np.float32)
    for c in range(chunks):
        for i in range(0, e, 2):
            even = (even.astype(np.float64) + p[:, c, :, i]).astype(np.float32)
            odd = (odd.astype(np.float64) + p[:, c, :, i + 1]).astype(np.float32)
    acc = (even + odd).astype(np.float32)
    lanes = acc.reshape(rows, 8, 32)
    idx = np.arange(32)
    for off in (16, 8, 4, 2, 1):
        lanes = (lanes + lanes[:, :, idx ^ off]).astype(np.float32)
    dot = np.zeros(rows, dtype=np.float32)
    for wv in range(8):
        dot = (dot + lanes[:, wv, 0]).astype(np.float32)
    return dot


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_dot_bound_holds_for_any_order_evaluations(dtype):
    rows, k = 192, 4096
    w = _rand((rows, k), dtype, 1)
    v = oracle.rmsnorm(np.random.default_rng(2).standard_normal(k)).astype(np.float32)
    exact = oracle.f64(w) @ v.astype(np.float64)
    bound = oracle.fp32_dot_bound(oracle.f64(w), v.astype(np.float64), 0.0)
    w32 = w.float().numpy()
    for got in (_sequential_fp32(w32, v), (w.float() @ torch.from_numpy(v)).numpy()):
        err = np.abs(got.astype(np.float64) - exact)
        assert np.all(err <= bound)
        assert err.max() > 0.0               # the evaluations really round
    # the bound is the any-order one: it exceeds the observed error by far
    assert bound.min() > 10 * np.abs(_sequential_fp32(w32, v) - exact).max()


@pytest.mark.parametrize("dtype,k", [(torch.float16, 4096), (torch.bfloat16, 2816), (torch.float32, 512)])
def test_dot_bound_holds_for_tree_of_stated_height(dtype, k):
    eb = torch.tensor([], dtype=dtype).element_size()
    rows = 256
    w = _rand((rows, k), dtype, 3, std=0.05)
    v = np.random.default_rng(4).standard_normal(k).astype(np.float32)
    exact = oracle.f64(w) @ v.astype(np.float64)
    depth = rowdot_depth(k, eb)
    got = _tree_fp32(w.float().numpy(), v, eb)
    err = np.abs(got.astype(np.float64) - exact)
    bound = oracle.fp32_dot_bound(oracle.f64(w), v.astype(np.float64), 0.0, depth=depth)
    assert np.all(err <= bound)
    # the height-bounded form is much tighter than the any-order one
    assert np.all(bound < oracle.fp32_dot_bound(oracle.f64(w), v.astype(np.float64), 0.0) / 20)


def test_dot_bound_input_error_term():
    # an input off by a relative 2-norm r moves each dot by at most
    # ||w_row|| * r * ||v|| (Cauchy-Schwarz), evaluated here exactly; along
    # a row's own direction that much is attained
    rows, k, r = 300, 2048, 3e-6
    w = oracle.f64(_rand((rows, k), torch.float16, 5))
    rng = np.random.default_rng(6)
    v = rng.standard_normal(k)
    bound = oracle.fp32_dot_bound(w, v, r, depth=0)
    for trial in range(5):
        d = rng.standard_normal(k) if trial else w[0].copy()
        d *= r * np.linalg.norm(v) / np.linalg.norm(d)
        moved = np.abs(w @ (v + d) - w @ v)
        assert np.all(moved <= bound)
        if trial == 0:
            assert moved[0] >= (1 - 1e-6) * np.linalg.norm(w[0]) * r * np.linalg.norm(v)


@pytest.mark.parametrize("bias", [False, True])
def test_argmax_tolerance_covers_float32_predictor(bias):
    # logits = W2 relu(W1 x) (+ b2), evaluated in float32 on an input that
    # differs from x by a relative 2e-6, in the tree order of stated height
    # and in torch's float32 matmul, against the fp64 logits of x
    D, H, F, r = 1024, 512, 1024, 2e-6
    w1 = _rand((H, D), torch.float16, 7)
    w2 = _rand((F, H), torch.float16, 8)
    b2 = _rand((F,), torch.float16, 9, std=0.3) if bias else None
    rng = np.random.default_rng(10)
    x = oracle.rmsnorm(rng.standard_normal(D))
    d = rng.standard_normal(D)
    x_gpu = (x + d * r * np.linalg.norm(x) / np.linalg.norm(d)).astype(np.float32)
    exact = oracle.predictor_logits(oracle.f64(w1), oracle.f64(w2), None if b2 is None else oracle.f64(b2), x)
    d1, d2 = rowdot_depth(D, 2), rowdot_depth(H, 2, bias)
    eps = oracle.argmax_tolerance(oracle.f64(w1), oracle.f64(w2), x, r, d1, d2,
                                  b2=None if b2 is None else oracle.f64(b2))
    z = np.maximum(_tree_fp32(w1.float().numpy(), x_gpu, 2), np.float32(0))
    lg_tree = _tree_fp32(w2.float().numpy(), z, 2)
    zt = torch.relu(w1.float() @ torch.from_numpy(x_gpu))
    lg_torch = (w2.float() @ zt).numpy()
    if b2 is not None:
        lg_tree = (lg_tree + b2.float().numpy()).astype(np.float32)
        lg_torch = (lg_torch + b2.float().numpy()).astype(np.float32)
    assert np.all(np.abs(lg_tree - exact) <= eps)
    # torch's order is not the stated tree: give it the any-order bound
    eps_any = oracle.argmax_tolerance(oracle.f64(w1), oracle.f64(w2), x, r,
                                      b2=None if b2 is None else oracle.f64(b2))
    assert np.all(np.abs(lg_torch - exact) <= eps_any)


# ---------------------------------------------------------------------------
# Tightness at the full predictor shapes
# ---------------------------------------------------------------------------
def test_bound_tight_at_shared_predictor_7b_shape():
    # Llama-2-7B shape: 4096 -> 2816 -> heads of 1024 centroids, planted
    cfg = LLAMA7B.replace(n_layers=2, d_ff=64, k_max=64, n_decode=3)
    wl = make_workload(cfg)
    w1, w2 = oracle.f64(wl.pred_w1), oracle.f64(wl.pred_w2)
    args = predictor_bound_args(cfg)
    assert args["x_rel_err"] == X_REL and args["depth1"] == 22 and args["depth2"] == 22
    for t in range(cfg.n_tokens):
        x = oracle.rmsnorm(wl.x[t, 0].numpy())
        lg = oracle.predictor_logits(w1, w2, None, x).reshape(cfg.n_heads, cfg.n_centroids)
        eps = oracle.argmax_tolerance(w1, w2, x, **args).reshape(cfg.n_heads, cfg.n_centroids)
        spread = lg.std(axis=1)
        assert np.all(eps.max(axis=1) <= 1e-2 * spread)
        top2 = np.sort(lg, axis=1)[:, -2:]
        assert np.all(top2[:, 1] - top2[:, 0] > 100 * eps.max(axis=1))   # planted margins


def test_bound_tight_at_perlayer_predictor_opt_shape():
    # OPT-6.7B style per-layer predictor: 4096 -> 1024 -> d_ff, with bias
    cfg = OPT67B.replace(n_layers=1, d_ff=4096, k_max=1024, n_decode=2)
    wl = make_workload(cfg)
    w1, w2, b2 = (oracle.f64(t[0]) for t in (wl.pred_w1, wl.pred_w2, wl.pred_b2))
    args = predictor_bound_args(cfg)
    assert args["depth1"] == 22 and args["depth2"] == 19
    for t in range(cfg.n_tokens):
        x = oracle.rmsnorm(wl.x[t, 0].numpy())
        lg = oracle.predictor_logits(w1, w2, b2, x)
        eps = oracle.argmax_tolerance(w1, w2, x, b2=b2, **args)
        assert eps.max() <= 2e-2 * (lg - b2).std()
        # decisions the bound leaves open: a few in ten thousand
        assert np.mean(np.abs(lg) <= eps) <= 5e-3


# ---------------------------------------------------------------------------
# The checker accepts a genuine near tie and rejects a planted wrong decision
# ---------------------------------------------------------------------------
class _Rec:
    pass


def test_checker_rejects_wrong_id_accepts_near_tie():
    cfg = LLAMA7B.replace(n_layers=2, d_ff=64, k_max=64, n_decode=2)
    wl = make_workload(cfg)
    w1, w2 = oracle.f64(wl.pred_w1), oracle.f64(wl.pred_w2)
    x = oracle.rmsnorm(wl.x[0, 0].numpy())
    lg = oracle.predictor_logits(w1, w2, None, x)
    rec = _Rec()
    rec.logits, rec.pred_xhat = [lg], [x]
    own = lg.reshape(cfg.n_heads, -1).argmax(axis=1)
    assert _ids_accept(rec, own[None, :], cfg, w1, w2) == 0
    wrong = own.copy()
    wrong[1] = np.argsort(lg.reshape(cfg.n_heads, -1)[1])[-2]          # runner-up, far behind
    with pytest.raises(AssertionError):
        _ids_accept(rec, wrong[None, :], cfg, w1, w2)
    # make the runner-up a genuine near tie: within the bound, accepted
    eps = oracle.argmax_tolerance(w1, w2, x, **predictor_bound_args(cfg))
    lg2 = lg.copy().reshape(cfg.n_heads, -1)
    lg2[1, wrong[1]] = lg2[1, own[1]] - 0.5 * eps.reshape(cfg.n_heads, -1)[1, wrong[1]]
    rec.logits = [lg2.reshape(-1)]
    assert _ids_accept(rec, wrong[None, :], cfg, w1, w2) == 1


def test_checker_rejects_wrong_firing_accepts_near_zero():
    cfg = OPT67B.replace(n_layers=1, d_ff=2048, k_max=1024, n_decode=1)
    wl = make_workload(cfg)
    w1, w2, b2 = (oracle.f64(t[0]) for t in (wl.pred_w1, wl.pred_w2, wl.pred_b2))
    x = oracle.rmsnorm(wl.x[0, 0].numpy())
    lg = oracle.predictor_logits(w1, w2, b2, x)
    rec = _Rec()
    rec.pred_logits_layer, rec.pred_xhat = [lg], [x]
    fire = lg > 0
    assert _fire_accept(rec, fire, 0, w1, w2, b2, cfg) == 0
    eps = oracle.argmax_tolerance(w1, w2, x, b2=b2, **predictor_bound_args(cfg))
    n_far = int(np.flatnonzero(np.abs(lg) > 10 * eps)[0])
    bad = fire.copy()
    bad[n_far] = not bad[n_far]
    with pytest.raises(AssertionError):
        _fire_accept(rec, bad, 0, w1, w2, b2, cfg)
    lg2 = lg.copy()
    lg2[n_far] = 0.5 * eps[n_far]            # a logit inside the bound: either decision
    rec.pred_logits_layer = [lg2]
    assert _fire_accept(rec, bad, 0, w1, w2, b2, cfg) == (1 if bad[n_far] != (lg2[n_far] > 0) else 0)
