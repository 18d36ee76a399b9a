"""The allocation-free FFN entry point (np_ffn_rows_noalloc) against the
model-owned one (np_sparse_mlp) and against the fp64 oracle, and its error
check (np_ffn_rows_noalloc_check).

Callers that cannot allocate device memory (a serving loop whose allocator
owns a fixed budget, or a latency-critical path where cudaMalloc would
synchronize the device) use the allocation-free variant; its scratch is a
fixed device array shared by all calls, so two calls in a row must give the
same answer, and an error one call records must reach the next check.  This
file is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import FFN_TOL, build_decoder
from workloads import SMALL_F16, make_workload

pytestmark = pytest.mark.gpu

_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_activation_decode_gb300.build import build
    build()


def test_noalloc_ffn_matches_model_entry_point_twice():
    from sparse_activation_decode_gb300 import ffn_rows_noalloc, ffn_rows_noalloc_check
    cfg = SMALL_F16
    wl = make_workload(cfg)
    dec = build_decoder(wl)
    for t in range(3):
        dec.decode_token(wl.x[t].cuda().clone())
    s = 1
    layer = cfg.n_dense + s
    view = dec.last_delta()
    n = int(view["counts"][s, 0].item())
    assert n > 0
    rows = view["active_slot"][s, :n].contiguous()
    g, u, d = (dec.resident_rows(layer, p) for p in range(3))
    h = torch.from_numpy(np.random.default_rng(5).standard_normal(cfg.d_model).astype(np.float32)).cuda()
    y_ref = dec.sparse_mlp(layer, h).cpu().numpy()
    for _ in range(2):
        y = ffn_rows_noalloc(h, g, u, d, rows, n)
        torch.cuda.synchronize()
        assert oracle.rel_l2(y.cpu().numpy(), y_ref) <= FFN_TOL
    ffn_rows_noalloc_check()
    dec.close()


def _case(dtype, gated, n_rows_total=300, d_model=512, seed=0):
    g = torch.Generator().manual_seed(seed)
    tdt = _DT[dtype]
    mk = lambda: (torch.randn((n_rows_total, d_model), generator=g) * 0.05).to(tdt).cuda()
    w_gate = mk() if gated else None
    w_up, w_down = mk(), mk()
    h = torch.randn(d_model, generator=g).cuda()
    return w_gate, w_up, w_down, h


def _oracle_y(w_gate, w_up, w_down, h, rows):
    idx = rows.tolist()
    xhat = oracle.rmsnorm(oracle.f64(h))
    gate = None if w_gate is None else oracle.f64(w_gate)[idx]
    y, _ = oracle.ffn_rows(gate, oracle.f64(w_up)[idx], oracle.f64(w_down)[idx], xhat)
    return y


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("gated", [True, False], ids=["gated", "ungated"])
@pytest.mark.parametrize("listed", [True, False], ids=["row-list", "first-rows"])
def test_noalloc_ffn_matches_oracle_twice(dtype, gated, listed):
    from sparse_activation_decode_gb300 import ffn_rows_noalloc, ffn_rows_noalloc_check
    w_gate, w_up, w_down, h = _case(dtype, gated, seed=4 * ["f32", "f16", "bf16"].index(dtype) + 2 * gated + listed)
    if listed:
        # unsorted, ragged count spanning several CTAs' shares of rows
        rows_np = np.random.default_rng(3).permutation(300)[:237].astype(np.int32)
        rows = torch.from_numpy(rows_np).cuda()
        n = len(rows_np)
    else:
        rows, n = None, 211
        rows_np = np.arange(n, dtype=np.int32)
    ref = _oracle_y(w_gate, w_up, w_down, h, rows_np)
    ys = []
    for _ in range(2):
        y = ffn_rows_noalloc(h, w_gate, w_up, w_down, rows, n)
        torch.cuda.synchronize()
        ys.append(y.cpu().numpy())
        assert oracle.rel_l2(ys[-1], ref) <= FFN_TOL
    assert oracle.rel_l2(ys[0], ys[1]) <= 1e-6
    ffn_rows_noalloc_check()


def test_noalloc_ffn_no_rows_gives_zero():
    from sparse_activation_decode_gb300 import ffn_rows_noalloc, ffn_rows_noalloc_check
    w_gate, w_up, w_down, h = _case("f16", True)
    y = torch.full_like(h, 7.0)
    for rows in (None, torch.zeros(4, dtype=torch.int32, device="cuda")):
        ffn_rows_noalloc(h, w_gate, w_up, w_down, rows, 0, y=y)
        torch.cuda.synchronize()
        assert torch.count_nonzero(y).item() == 0
    ffn_rows_noalloc_check()


def test_noalloc_out_of_range_row_is_reported():
    from sparse_activation_decode_gb300 import NpError, ffn_rows_noalloc, ffn_rows_noalloc_check
    w_gate, w_up, w_down, h = _case("f16", True)
    ffn_rows_noalloc_check()                       # start from a clear error word
    rows = torch.tensor([5, 17, 300, 2], dtype=torch.int32, device="cuda")   # 300 = row_limit
    ffn_rows_noalloc(h, w_gate, w_up, w_down, rows, 4)
    with pytest.raises(NpError) as e:
        ffn_rows_noalloc_check()
    assert e.value.status == -6
    ffn_rows_noalloc_check()                       # the check cleared it
    # a later good call on the shared array still gives the right answer
    good = torch.tensor([5, 17, 299, 2], dtype=torch.int32, device="cuda")
    y = ffn_rows_noalloc(h, w_gate, w_up, w_down, good, 4)
    torch.cuda.synchronize()
    assert oracle.rel_l2(y.cpu().numpy(), _oracle_y(w_gate, w_up, w_down, h, good.cpu().numpy())) <= FFN_TOL
    ffn_rows_noalloc_check()


def test_noalloc_wrapper_rejects_misuse():
    from sparse_activation_decode_gb300 import ffn_rows_noalloc
    w_gate, w_up, w_down, h = _case("f16", True)
    rows = torch.arange(10, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):      # y aliases h
        ffn_rows_noalloc(h, w_gate, w_up, w_down, rows, 10, y=h)
    with pytest.raises(ValueError):      # int64 row indices
        ffn_rows_noalloc(h, w_gate, w_up, w_down, rows.long(), 10)
    with pytest.raises(ValueError):      # a shorter down projection
        ffn_rows_noalloc(h, w_gate, w_up, w_down[:100].contiguous(), rows, 10)
    with pytest.raises(ValueError):      # mixed weight dtypes
        ffn_rows_noalloc(h, w_gate.float(), w_up, w_down, rows, 10)
    with pytest.raises(ValueError):      # h of the wrong length
        ffn_rows_noalloc(h[:256].contiguous(), w_gate, w_up, w_down, rows, 10)
