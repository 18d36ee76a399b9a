"""Parity of the CUDA path (through the C ABI) with the fp64 oracle."""
import ctypes
import re

import numpy as np
import pytest
import torch

import oracle
from oracle import OracleDecoder
from tests.parity import FFN_TOL, build_decoder, run_and_compare
from workloads import (BATCHED7B, LLAMA7B, LLAMA13B, OPT67B, SMALL_BATCHED, SMALL_BF16, SMALL_F16, SMALL_OPT,
                       TINY, make_workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_activation_decode_gb300.build import build
    build()
    torch.cuda.init()


SMALL_CASES = {
    "tiny": (TINY, {}),
    "tiny-intersect": (TINY.replace(combine="intersect"), {}),
    "small-f16": (SMALL_F16, {}),
    "small-bf16": (SMALL_BF16, {}),
    "small-opt-window": (SMALL_OPT, {}),
    "small-f16-fused": (SMALL_F16, {"h2d_mode": "fused"}),
    "small-f16-staging3": (SMALL_F16, {"staging_rows": 3}),
    "small-bf16-staging7": (SMALL_BF16, {"staging_rows": 7}),
    "small-opt-capped": (SMALL_OPT.replace(k_max=150), {}),
    # batched decoding on the tensor cores (union of the sequences' sets)
    "small-batched": (SMALL_BATCHED, {}),
    "small-batched-fused": (SMALL_BATCHED, {"h2d_mode": "fused"}),
    "small-batched-b3-f16": (SMALL_BATCHED.replace(batch=3, dtype="f16", k_max=700), {}),
    "small-batched-nogate": (SMALL_BATCHED.replace(has_gate=False), {}),
    # SwiGLU activation (silu gate) on the CUDA-core and tensor-core FFNs
    "small-f16-swiglu": (SMALL_F16.replace(activation="swiglu"), {}),
    "small-batched-swiglu": (SMALL_BATCHED.replace(activation="swiglu"), {}),
    # compact placement (swap-with-last + append): moves, appends and the FFN
    # over the occupied region, with and without windowing
    "small-f16-compact": (SMALL_F16.replace(slots="compact"), {}),
    "small-f16-compact-fused": (SMALL_F16.replace(slots="compact"), {"h2d_mode": "fused"}),
    "small-bf16-compact-staging7": (SMALL_BF16.replace(slots="compact"), {"staging_rows": 7}),
    "small-opt-window-compact": (SMALL_OPT.replace(slots="compact"), {}),
    "small-batched-compact": (SMALL_BATCHED.replace(slots="compact"), {}),
    "small-batched-window-compact": (SMALL_BATCHED.replace(residency="window", window=3, slots="compact"), {}),
    # cross-layer lookahead of the per-layer predictor and frequency-weighted
    # residency (evictions once the cache is full)
    "small-opt-lookahead1": (SMALL_OPT.replace(lookahead=1), {}),
    "small-opt-lookahead2-compact": (SMALL_OPT.replace(lookahead=2, slots="compact"), {}),
    "small-opt-lookahead3-frequency": (SMALL_OPT.replace(lookahead=3, residency="frequency", k_max=150), {}),
    "small-opt-frequency": (SMALL_OPT.replace(residency="frequency", k_max=150), {}),
    "small-f16-frequency": (SMALL_F16.replace(residency="frequency", k_max=300), {}),
    "small-batched-frequency-compact": (SMALL_BATCHED.replace(residency="frequency", slots="compact"), {}),
    # degenerate sets: intersections of two 2% masks are mostly empty (FFN over
    # no rows, empty deltas); a K_max of one row
    "tiny-intersect-sparse": (TINY.replace(combine="intersect", density=0.02), {}),
    "tiny-kmax1": (TINY.replace(k_max=1), {}),
}


@pytest.mark.parametrize("name", list(SMALL_CASES))
def test_decode_parity_small(name):
    cfg, kw = SMALL_CASES[name]
    if name == "small-opt-capped":
        # the window cap binds; per-layer parity needs |A| <= K so shrink nothing else
        pass
    wl = make_workload(cfg)
    summ = run_and_compare(wl, **kw)
    assert summ["tokens"] == cfg.n_tokens
    assert summ["max_h_rel"] < FFN_TOL


def test_batched_multi_tile(monkeypatch):
    # one cluster per launch: every product runs several 128-row tiles through
    # the same cluster (exchange buffers and accumulators reused across tiles)
    monkeypatch.setenv("NP_TUNE_MMA_CLUSTERS", "1")
    wl = make_workload(SMALL_BATCHED)
    summ = run_and_compare(wl, 4)
    assert summ["max_h_rel"] < FFN_TOL


def test_chunked_equals_unchunked_bytes():
    cfg = SMALL_F16
    wl = make_workload(cfg)
    outs = []
    for rows in (0, 1, 5):
        dec = build_decoder(wl, staging_rows=rows)
        for t in range(5):
            h = wl.x[t].cuda().clone()
            dec.decode_token(h)
        bufs = [dec.resident_rows(cfg.n_dense + s, p).cpu().view(torch.int16)
                for s in range(cfg.n_sparse) for p in range(3)]
        outs.append((h.cpu(), bufs))
        dec.close()
    for h, bufs in outs[1:]:
        # buffer bytes are identical; h only up to the order of the FFN's
        # fp32 split-K additions
        assert oracle.rel_l2(h.numpy(), outs[0][0].numpy()) < 1e-5
        assert all(torch.equal(a, b) for a, b in zip(bufs, outs[0][1]))


def test_repeated_token_has_empty_delta():
    wl = make_workload(SMALL_F16)
    dec = build_decoder(wl)
    x = wl.x[2].cuda()
    dec.decode_token(x.clone())
    st = dec.decode_token(x.clone(), stats=True)
    assert st["din_rows"] == 0 and st["dout_rows"] == 0
    dec.close()


@pytest.mark.parametrize("slots,residency", [("reuse", "slotmap"), ("compact", "slotmap"), ("reuse", "frequency")])
def test_reset_sequence_is_cold_start(slots, residency):
    cfg = SMALL_F16.replace(slots=slots, residency=residency, k_max=300 if residency == "frequency" else 192)
    wl = make_workload(cfg)
    dec = build_decoder(wl)
    orc = OracleDecoder(wl)
    run_and_compare(wl, 4, dec=dec, orc=orc)
    dec.reset_sequence()
    orc.reset()
    orc.bufs = None  # buffers keep their bytes across a reset; compare sets only
    orc.materialize = False
    summ = run_and_compare(wl, 3, dec=dec, orc=orc, start=4, check_buffers=False)
    counts_first = summ["din_rows"]
    assert counts_first > 0
    dec.close()


@pytest.mark.parametrize("slots", ["reuse", "compact"])
def test_piecewise_entry_points_match_decode(slots):
    cfg = SMALL_BF16.replace(slots=slots)
    wl = make_workload(cfg)
    dec = build_decoder(wl)
    orc = OracleDecoder(wl)
    for t in range(4):
        x = wl.x[t].cuda().reshape(-1).clone()
        rec = orc.step(wl.x[t].numpy())
        h = x.clone()
        for l in range(cfg.n_dense):
            y = dec.dense_mlp(l, h)
            if l == 0:
                ids = dec.predict(h + y)
                assert ids.cpu().numpy().astype(np.int64)[0].tolist() == rec.ids[0].tolist()
            h = h + y
        view = dec.delta(ids, -1)
        dec.scatter(-1)
        counts = view["counts"].cpu().numpy()
        for s in range(cfg.n_sparse):
            assert view["active"][s, :counts[s, 0]].cpu().tolist() == rec.active[s]
            y = dec.sparse_mlp(cfg.n_dense + s, h)
            assert oracle.rel_l2(y.cpu().numpy(), rec.y[s][0]) < FFN_TOL
            h = h + y
        assert oracle.rel_l2(h.cpu().numpy(), rec.h[0]) < FFN_TOL
    dec.close()


def test_state_machine_errors():
    from sparse_activation_decode_gb300 import NpError
    wl = make_workload(SMALL_F16)
    dec = build_decoder(wl)
    with pytest.raises(NpError) as e:
        dec.scatter(-1)          # nothing pending
    assert e.value.status == -6
    h = wl.x[0].cuda().reshape(-1).clone()
    ids = dec.predict(h)
    dec.delta(ids, -1)
    with pytest.raises(NpError) as e:
        dec.delta(ids, -1)       # already pending
    assert e.value.status == -6
    with pytest.raises(NpError) as e:
        dec.decode_token(h)      # pending delta blocks a new token
    assert e.value.status == -6
    dec.scatter(-1)
    with pytest.raises(NpError) as e:
        dec.sparse_mlp(0, h)     # layer 0 is dense
    assert e.value.status == -1
    dec.close()


@pytest.mark.parametrize("bad", [{"k_max": 5000}, {"d_model": 12}, {"n_dense": 0},
                                 {"activation": "swiglu", "has_gate": False},
                                 {"batch": 2, "pred_hidden": 128, "residency": "window", "window": 3},
                                 {"batch": 2, "pred_hidden": 128, "residency": "frequency"},
                                 {"lookahead": 1}])
def test_invalid_config_rejected(bad):
    from sparse_activation_decode_gb300 import NpError
    cfg = SMALL_F16
    wl = make_workload(cfg)
    kw = dict(n_layers=cfg.n_layers, n_dense=cfg.n_dense, d_model=cfg.d_model, d_ff=cfg.d_ff,
              k_max=cfg.k_max, n_centroids=cfg.n_centroids, dtype=cfg.torch_dtype, host_store=wl.store,
              pred_w1=wl.pred_w1.cuda(), pred_w2=wl.pred_w2.cuda(), dense_w=wl.dense_w.cuda(),
              centroids=torch.from_numpy(wl.centroids.view("int32")).cuda(), pred_hidden=cfg.pred_hidden)
    kw.update(bad)
    from sparse_activation_decode_gb300 import SparseDecoder
    with pytest.raises(NpError) as e:
        SparseDecoder(**kw)
    assert e.value.status == -1


@pytest.mark.parametrize("cfg", [SMALL_F16, SMALL_F16.replace(slots="compact"),
                                 SMALL_OPT.replace(lookahead=2, residency="frequency", k_max=150)],
                         ids=["reuse", "compact", "opt-lookahead2-frequency"])
def test_read_failure_restores_committed_state(cfg):
    wl = make_workload(cfg)
    fail_layer = {"layer": -1}

    def hook(ctx, layer, token):
        return 1 if layer == fail_layer["layer"] else 0

    dec = build_decoder(wl, read_hook=hook)
    for t in range(3):
        dec.decode_token(wl.x[t].cuda().clone())
    before = [dec.get_state(cfg.n_dense + s) for s in range(cfg.n_sparse)]
    bufs = [dec.resident_rows(cfg.n_dense + s, p).cpu().view(torch.int16).clone()
            for s in range(cfg.n_sparse) for p in range(cfg.n_proj)]
    from sparse_activation_decode_gb300 import NpError
    fail_layer["layer"] = cfg.n_dense + 2     # third sparse layer fails to read
    with pytest.raises(NpError) as e:
        dec.decode_token(wl.x[3].cuda().clone())
    assert e.value.status == -4
    dec.check_error()
    after = [dec.get_state(cfg.n_dense + s) for s in range(cfg.n_sparse)]
    assert after == before
    bufs2 = [dec.resident_rows(cfg.n_dense + s, p).cpu().view(torch.int16)
             for s in range(cfg.n_sparse) for p in range(cfg.n_proj)]
    assert all(torch.equal(a, b) for a, b in zip(bufs, bufs2))
    # the token can be decoded once the read succeeds, matching an oracle that
    # never saw the failure
    fail_layer["layer"] = -1
    orc = OracleDecoder(wl)
    for t in range(3):
        orc.step(wl.x[t].numpy())
    run_and_compare(wl, 2, dec=dec, orc=orc, start=3)
    dec.close()


# ---------------------------------------------------------------------------
# Full-size shapes: every integer output compared in full, buffer bytes on
# sampled slots, FFN outputs per layer.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg,tokens", [(LLAMA7B, 3), (LLAMA13B, 2), (OPT67B, 2), (BATCHED7B, 2),
                                        (LLAMA7B.replace(slots="compact"), 3),
                                        (BATCHED7B.replace(slots="compact"), 2),
                                        (OPT67B.replace(lookahead=2, residency="frequency"), 3)],
                         ids=["llama2-7b", "llama2-13b", "opt-6.7b", "llama2-7b-batch8", "llama2-7b-compact",
                              "llama2-7b-batch8-compact", "opt-6.7b-lookahead2-frequency"])
def test_full_size_sampled(cfg, tokens):
    wl = make_workload(cfg.replace(n_warm=0, n_decode=tokens), device="cuda")
    summ = run_and_compare(wl, tokens, check_buffers=False, sample_slots=64, check_layer_y=True)
    assert summ["near_ties"] == 0 or cfg.pred_kind == "perlayer_sigmoid"
    assert summ["max_h_rel"] < FFN_TOL


@pytest.mark.parametrize("cfg,tokens", [(LLAMA7B, 3), (OPT67B.replace(lookahead=2), 3), (BATCHED7B, 2)],
                         ids=["llama2-7b", "opt-6.7b-lookahead2", "llama2-7b-batch8"])
def test_full_size_fused(cfg, tokens):
    # the host-link mode the benchmark times: records read from host memory
    # straight into their slots, at the full shapes
    wl = make_workload(cfg.replace(n_warm=0, n_decode=tokens), device="cuda")
    summ = run_and_compare(wl, tokens, h2d_mode="fused", check_buffers=False, sample_slots=64,
                           check_layer_y=True)
    assert summ["tokens"] == tokens
    assert summ["max_h_rel"] < FFN_TOL


def test_llama7b_warm_state_fused_every_buffer_byte():
    # the state the benchmark decodes from: 26 tokens of slot churn after the
    # cold start (freed slots reused all over the K_max range), fused host-link
    # mode, every token's integer state compared in full; then every byte of
    # all 31 layers' three resident buffers against the oracle's buffers, and
    # each layer's FFN output on the last token
    T = 26
    cfg = LLAMA7B.replace(n_warm=0, n_decode=T)
    wl = make_workload(cfg, device="cuda")
    dec = build_decoder(wl, h2d_mode="fused")
    orc = OracleDecoder(wl, materialize_buffers=True)
    try:
        summ = run_and_compare(wl, T - 1, dec=dec, orc=orc, check_buffers=False, check_layer_y=False)
        assert summ["near_ties"] == 0
        # the slots in use are spread over the whole buffer by now
        inv = orc.inv
        assert (inv >= 0).sum(axis=1).min() > 0.9 * cfg.k_max
        last = run_and_compare(wl, 1, dec=dec, orc=orc, start=T - 1, check_buffers=True, check_layer_y=True)
        assert last["max_h_rel"] < FFN_TOL and last["max_y_rel"] < FFN_TOL
    finally:
        dec.close()


@pytest.mark.parametrize("cfg,tokens,kw", [(SMALL_BATCHED.replace(slots="compact"), 6, {}),
                                           (SMALL_OPT.replace(lookahead=2), 6, {"h2d_mode": "fused"}),
                                           (BATCHED7B.replace(slots="compact"), 3,
                                            {"check_buffers": False, "sample_slots": 64})],
                         ids=["small-batched-compact", "small-opt-lookahead2-fused", "llama2-7b-batch8-compact"])
def test_programmatic_launch_on_every_kernel(cfg, tokens, kw, monkeypatch):
    # every kernel kind that supports programmatic dependent launch asks for
    # it (predictor, set kernel, tensor-core kernels; the FFN always does);
    # the library grants it only between two kernels of one call back to
    # back on one stream, so the results must agree with the oracle as they
    # do without it.  The full-size 8-sequence compact case changed h
    # (rel-L2 3e-3) when a captured dependency on another stream's kernel
    # was relaxed.
    monkeypatch.setenv("NP_TUNE_PDL", "7")
    wl = make_workload(cfg.replace(n_warm=0, n_decode=tokens), device="cuda")
    summ = run_and_compare(wl, tokens, **kw)
    assert summ["tokens"] == tokens
    assert summ["max_h_rel"] < FFN_TOL


@pytest.mark.parametrize("cfg", [SMALL_F16, SMALL_BATCHED, SMALL_F16.replace(activation="swiglu"),
                                 SMALL_F16.replace(slots="compact"), SMALL_OPT.replace(slots="compact"),
                                 SMALL_BF16.replace(name="wide-bf16", d_model=5120, d_ff=1024, k_max=256,
                                                    n_layers=4, n_dense=1)],
                         ids=["small-f16", "small-batched", "small-f16-swiglu", "small-f16-compact",
                              "small-opt-window-compact", "wide-rows-bf16"])
def test_ffn_layers_equals_layer_by_layer(cfg):
    # the chained FFN entry point equals h += FFN_l(h) applied layer by layer
    # through the standalone entry points, over dense and sparse layers
    wl = make_workload(cfg)
    dec = build_decoder(wl)
    for t in range(3):
        dec.decode_token(wl.x[t].cuda().clone())
    h0 = wl.x[3].cuda().reshape(-1).clone()
    ref = h0.clone()
    for l in range(cfg.n_layers):
        y = dec.dense_mlp(l, ref) if l < cfg.n_dense else dec.sparse_mlp(l, ref)
        ref = ref + y
    got = dec.ffn_layers(0, cfg.n_layers, h0.clone())
    torch.cuda.synchronize()
    for b in range(cfg.batch):
        g = got.reshape(cfg.batch, -1)[b].cpu().numpy()
        r = ref.reshape(cfg.batch, -1)[b].cpu().numpy()
        assert oracle.rel_l2(g, r) < 1e-5
    # the sparse suffix alone against its layer-by-layer application
    part = dec.ffn_layers(cfg.n_dense, cfg.n_sparse, h0.clone())
    ref_s = h0.clone()
    for l in range(cfg.n_dense, cfg.n_layers):
        ref_s = ref_s + dec.sparse_mlp(l, ref_s)
    torch.cuda.synchronize()
    for b in range(cfg.batch):
        g = part.reshape(cfg.batch, -1)[b].cpu().numpy()
        r = ref_s.reshape(cfg.batch, -1)[b].cpu().numpy()
        assert oracle.rel_l2(g, r) < 1e-5
    from sparse_activation_decode_gb300 import NpError
    with pytest.raises(NpError):
        dec.ffn_layers(0, cfg.n_layers + 1, h0.clone())
    dec.close()


@pytest.mark.parametrize("cfg", [SMALL_F16, SMALL_OPT.replace(lookahead=2), SMALL_BATCHED],
                         ids=["small-f16", "small-opt-lookahead2", "small-batched"])
def test_graph_replay_matches_eager(cfg, monkeypatch):
    # tokens after the first are replayed from a captured graph; with graphs
    # switched off every launch is issued one by one: the integer state must
    # agree bit for bit and h up to the order of the FFN's split-K additions
    wl = make_workload(cfg)
    outs = []
    for graph in ("1", "0"):
        monkeypatch.setenv("NP_TUNE_GRAPH", graph)
        dec = build_decoder(wl)
        hs, states = [], []
        for t in range(6):
            h = wl.x[t].cuda().clone()
            dec.decode_token(h)
            hs.append(h.cpu())
            states.append([dec.get_state(cfg.n_dense + s) for s in range(cfg.n_sparse)])
        dec.check_error()
        outs.append((hs, states))
        dec.close()
    (h1, s1), (h0, s0) = outs
    assert s1 == s0
    for a, b in zip(h1, h0):
        assert oracle.rel_l2(a.numpy().ravel(), b.numpy().ravel()) < 1e-5


@pytest.mark.parametrize("cfg,tokens,kw", [
    (SMALL_F16, 6, {"h2d_mode": "fused"}),
    (SMALL_BF16, 6, {}),                      # dense layer 1 -> the first sparse layer as well
    (SMALL_BATCHED, 6, {}),
    (SMALL_OPT.replace(lookahead=2), 6, {"h2d_mode": "fused"}),
    (BATCHED7B, 4, {"check_buffers": False, "sample_slots": 64}),
], ids=["small-f16-fused", "small-bf16", "small-batched", "small-opt-lookahead2-fused", "llama2-7b-batch8"])
def test_graph_programmatic_ffn_edges(cfg, tokens, kw, monkeypatch, capfd):
    # in the captured token each layer's FFN takes a programmatic edge from
    # the previous layer's FFN, while the edges from its rows' reads (and
    # from predictions that read its input buffers) stay full; the replayed
    # tokens must agree with the oracle as the eager first token does
    monkeypatch.setenv("NP_TUNE_VERBOSE", "1")
    wl = make_workload(cfg.replace(n_warm=0, n_decode=tokens), device="cuda")
    summ = run_and_compare(wl, tokens, **kw)
    err = capfd.readouterr().err
    cap = re.search(r"token captured \((\d+) kernels, (\d+) programmatic FFN edges\)", err)
    assert cap, err[-2000:]
    assert int(cap.group(2)) >= 1
    assert summ["tokens"] == tokens
    assert summ["max_h_rel"] < FFN_TOL


@pytest.mark.parametrize("residency", ["window", "frequency"])
@pytest.mark.parametrize("graph", ["1", "0"], ids=["replay", "eager"])
def test_set_stream_matches_single_stream(residency, graph, monkeypatch):
    # with a lookahead the set kernels run on a stream of their own, with two
    # firing-mask buffers alternating by layer; that changes only the
    # schedule, so the slot state must equal the single-stream run bit for bit
    # and h must agree up to the FFN's split-K addition order
    monkeypatch.setenv("NP_TUNE_GRAPH", graph)
    cfg = SMALL_OPT.replace(lookahead=2, residency=residency)
    wl = make_workload(cfg)
    outs = []
    for ss in ("1", "0"):
        monkeypatch.setenv("NP_TUNE_SET_STREAM", ss)
        dec = build_decoder(wl, h2d_mode="fused")
        hs, states = [], []
        for t in range(8):
            h = wl.x[t].cuda().clone()
            dec.decode_token(h)
            hs.append(h.cpu())
            states.append([dec.get_state(cfg.n_dense + s) for s in range(cfg.n_sparse)])
        dec.check_error()
        outs.append((hs, states))
        dec.close()
    (h1, s1), (h0, s0) = outs
    assert s1 == s0
    for a, b in zip(h1, h0):
        assert oracle.rel_l2(a.numpy().ravel(), b.numpy().ravel()) < 1e-5


def test_max_sizes():
    # the largest shapes the ABI accepts: d_model 8192 (fp16 rows of 16 KiB,
    # four chunks per FFN thread), d_ff 16384 (512 mask words, one per set
    # thread) and K_max 8192, with the cap binding (union of two 30% masks)
    from workloads.synth import Config
    cfg = Config(name="max-shape", n_layers=3, n_dense=1, d_model=8192, d_ff=16384, k_max=8192,
                 n_centroids=32, dtype="f16", density=0.30, persistence=0.83, pred_hidden=256,
                 planted_scale=60.0, n_warm=0, n_decode=3, seed=2011)
    wl = make_workload(cfg, device="cuda")
    summ = run_and_compare(wl, 3, check_buffers=False, sample_slots=64, check_layer_y=True)
    assert summ["max_h_rel"] < FFN_TOL


# ---------------------------------------------------------------------------
# Per-token pipeline (NP_TUNE_TOKEN_CHAIN=1): after layer 0, the predictor and
# one set kernel, a single persistent launch reads every sparse layer's
# incoming records into their slots and runs layers 1..L-1, each layer's FFN
# waiting inside the kernel for its rows.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg,tokens,kw", [
    (TINY, 6, {}),
    (SMALL_F16, 8, {}),
    (SMALL_BF16, 6, {}),
    (SMALL_F16.replace(activation="swiglu"), 5, {}),
    (LLAMA7B.replace(n_warm=0, n_decode=3), 3, {"check_buffers": False, "sample_slots": 64}),
    (LLAMA13B.replace(n_warm=0, n_decode=2), 2, {"check_buffers": False, "sample_slots": 64}),
], ids=["tiny", "small-f16", "small-bf16", "small-f16-swiglu", "llama2-7b", "llama2-13b"])
def test_token_pipeline_matches_oracle(cfg, tokens, kw, monkeypatch):
    monkeypatch.setenv("NP_TUNE_TOKEN_CHAIN", "1")
    wl = make_workload(cfg, device="cuda")
    summ = run_and_compare(wl, tokens, h2d_mode="fused", **kw)
    assert summ["tokens"] == tokens
    assert summ["max_h_rel"] < FFN_TOL


def test_token_pipeline_replay_matches_eager(monkeypatch):
    # the captured token (cooperative launches inside the graph) against the
    # launches issued one by one: every FFN of this pipeline adds its split-K
    # partials in a fixed order, so integer state and h agree bit for bit
    monkeypatch.setenv("NP_TUNE_TOKEN_CHAIN", "1")
    cfg = SMALL_F16
    wl = make_workload(cfg)
    outs = []
    for graph in ("1", "0"):
        monkeypatch.setenv("NP_TUNE_GRAPH", graph)
        dec = build_decoder(wl, h2d_mode="fused")
        hs, states = [], []
        for t in range(6):
            h = wl.x[t].cuda().clone()
            dec.decode_token(h)
            hs.append(h.cpu())
            states.append([dec.get_state(cfg.n_dense + s) for s in range(cfg.n_sparse)])
        dec.check_error()
        outs.append((hs, states))
        dec.close()
    (h1, s1), (h0, s0) = outs
    assert s1 == s0
    for a, b in zip(h1, h0):
        assert torch.equal(a, b)


@pytest.mark.parametrize("cfg", [BATCHED7B.replace(n_warm=0, n_decode=3),
                                 BATCHED7B.replace(n_warm=0, n_decode=3, slots="compact")],
                         ids=["llama2-7b-batch8", "llama2-7b-batch8-compact"])
def test_batched_sparse_chain_full_size(cfg):
    # np_ffn_layers over the 31 sparse layers of 8 sequences (the residual
    # chained on the device) against the layers applied one call at a time,
    # after two decoded tokens of slot churn
    wl = make_workload(cfg, device="cuda")
    dec = build_decoder(wl)
    for t in range(2):
        dec.decode_token(wl.x[t].cuda().clone())
    h0 = wl.x[2].cuda().reshape(-1).clone()
    got = dec.ffn_layers(cfg.n_dense, cfg.n_sparse, h0.clone())
    ref = h0.clone()
    for l in range(cfg.n_dense, cfg.n_layers):
        ref = ref + dec.sparse_mlp(l, ref)
    torch.cuda.synchronize()
    # both add their CTAs' partial y with fp32 atomics in arrival order, and
    # the 16+16-bit operand split passes such differences on to later layers;
    # the bound stays well inside FFN_TOL
    for b in range(cfg.batch):
        assert oracle.rel_l2(got.reshape(cfg.batch, -1)[b].cpu().numpy(),
                             ref.reshape(cfg.batch, -1)[b].cpu().numpy()) < 1e-4
    dec.check_error()
    dec.close()
