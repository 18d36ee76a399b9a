"""The allocation-free FFN entry point (np_ffn_rows_noalloc) against the
model-owned one (np_sparse_mlp) on the same rows, weights and input.

Callers that cannot allocate device memory (a serving loop whose allocator
owns a fixed budget, or a latency-critical path where cudaMalloc would
synchronize the device) use the allocation-free variant; its scratch is a
fixed device array shared by all calls, so two calls in a row must give the
same answer.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import FFN_TOL, build_decoder
from workloads import SMALL_F16, make_workload

pytestmark = pytest.mark.gpu


def test_noalloc_ffn_matches_model_entry_point_twice():
    from sparse_activation_decode_gb300 import ffn_rows_noalloc
    from sparse_activation_decode_gb300.build import build
    build()
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
    dec.close()
