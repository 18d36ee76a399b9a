"""A bounded device wait that runs out, on the GPU, without a fault.

The per-token pipeline is one cooperative launch: reader warps copy each
sparse layer's incoming records from the host store and count themselves on
a per-layer counter, and each CTA's producer waits for that count before it
streams the layer's rows.  The test hook NP_TEST_WITHHOLD_ARRIVAL=l makes
CTA 0's readers skip their arrival for layer l, so the count never completes
(a flag that nothing sets).  Every wait behind it gives up after its limit:
the producers' waits on the count, the consumers' waits on copies that were
never issued, the reducers' waits on the partial sums of CTAs that stopped.
The kernel then drains its own copies in flight and returns, the error word
holds the timeout, and np_check_error reports NP_ERR_TIMEOUT.  The same
process then decodes with a fresh model and matches the oracle, so the
context stayed usable."""
import time

import pytest
import torch

from tests.parity import FFN_TOL, build_decoder, run_and_compare
from workloads import SMALL_F16, make_workload

pytestmark = pytest.mark.gpu

NP_ERR_TIMEOUT = -5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_activation_decode_gb300.build import build
    build()


def test_withheld_arrival_times_out_and_context_stays_usable(monkeypatch):
    from sparse_activation_decode_gb300 import NpError
    cfg = SMALL_F16
    wl = make_workload(cfg)
    monkeypatch.setenv("NP_TUNE_TOKEN_CHAIN", "1")
    monkeypatch.setenv("NP_TUNE_GRAPH", "0")
    # the second sparse layer: the first one's rows stream normally, so the
    # timeout is met in the middle of the launch, with copies already issued
    monkeypatch.setenv("NP_TEST_WITHHOLD_ARRIVAL", str(cfg.n_dense + 1))
    dec = build_decoder(wl, h2d_mode="fused")
    h = wl.x[0].cuda().clone()
    t0 = time.monotonic()
    dec.decode_token(h)
    with pytest.raises(NpError) as e:
        dec.check_error()
    waited = time.monotonic() - t0
    assert e.value.status == NP_ERR_TIMEOUT
    # one limit for the producers, at most one per row of a consumer group
    # for the consumers: seconds, not a hang
    assert waited < 30.0
    dec.check_error()                      # reading the error cleared it
    dec.close()

    monkeypatch.delenv("NP_TEST_WITHHOLD_ARRIVAL")
    summ = run_and_compare(make_workload(cfg, device="cuda"), 3, h2d_mode="fused")
    assert summ["tokens"] == 3
    assert summ["max_h_rel"] < FFN_TOL
    torch.cuda.synchronize()
