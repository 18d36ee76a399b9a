"""Run the CUDA decode path and the fp64 oracle on the same seeded inputs and
compare them: bit-exact for predictor IDs (after the fp32 near-tie rule),
active sets, deltas, slot maps and buffer bytes; relative L2 for FFN outputs.

Near ties: an fp32 evaluation may legitimately pick another argmax (or firing
decision) than the fp64 oracle when the two candidates are closer than the
fp32 error bound.  The GPU's choice is accepted only inside that bound, and
the oracle then continues with the GPU's choice so that every later stage is
compared bit-exactly on the same decisions.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import OracleDecoder

FFN_TOL = 1e-3   # relative L2 of FFN outputs and of the residual stream


def build_decoder(wl, **kw):
    from sparse_activation_decode_gb300 import decoder_for
    return decoder_for(wl, **kw)


def _ids_accept(rec, ids_gpu, cfg, w1, w2):
    """Per sequence and head, GPU id must be within the fp32 bound of the max."""
    near = 0
    for b in range(cfg.batch):
        lg = rec.logits[b].reshape(cfg.n_heads, cfg.n_centroids)
        own = lg.argmax(axis=1)
        if np.array_equal(own, ids_gpu[b]):
            continue
        eps = oracle.argmax_tolerance(w1, w2, rec.pred_xhat[b]).reshape(cfg.n_heads, cfg.n_centroids)
        for h in np.flatnonzero(own != ids_gpu[b]):
            g = int(ids_gpu[b][h])
            assert 0 <= g < cfg.n_centroids
            bound = eps[h, g] + eps[h, own[h]]
            assert lg[h, g] >= lg[h, own[h]] - bound, (
                f"head {h}: GPU id {g} logit {lg[h, g]} vs max {lg[h, own[h]]} (bound {bound})")
            near += 1
    return near


def _fire_accept(rec, fire_gpu, s, w1, w2):
    lg = rec.pred_logits_layer[s]
    ref = lg > 0.0
    diff = np.flatnonzero(ref != fire_gpu)
    if diff.size:
        eps = oracle.argmax_tolerance(w1, w2, rec.pred_xhat[s])
        for n in diff:
            assert abs(lg[n]) <= eps[n], f"neuron {n}: logit {lg[n]} bound {eps[n]}"
    return int(diff.size)


def run_and_compare(wl, n_tokens=None, *, h2d_mode="staged", staging_rows=None, check_buffers=True,
                    check_layer_y=True, sample_slots=None, dec=None, orc=None, start=0, inputs=None,
                    rng_seed=0):
    """Decode n_tokens tokens on the GPU and in the oracle; assert parity.
    Returns a summary dict (max errors, near-tie counts, rows moved)."""
    cfg = wl.cfg
    T = cfg.n_tokens if n_tokens is None else n_tokens
    own_dec = dec is None
    if dec is None:
        dec = build_decoder(wl, h2d_mode=h2d_mode, staging_rows=staging_rows)
    if orc is None:
        orc = OracleDecoder(wl, materialize_buffers=check_buffers)
    shared = cfg.pred_kind == "shared_argmax"
    if shared:
        w1, w2 = oracle.f64(wl.pred_w1), oracle.f64(wl.pred_w2)
    rng = np.random.default_rng(rng_seed)
    summary = {"max_h_rel": 0.0, "max_y_rel": 0.0, "near_ties": 0, "din_rows": 0, "tokens": 0}
    try:
        for t in range(start, start + T):
            x = (wl.x[t] if inputs is None else inputs[t - start])
            h = x.to("cuda", torch.float32).contiguous().clone()
            st = dec.decode_token(h, stats=True)
            view = dec.last_delta()
            counts = view["counts"].cpu().numpy()
            active = view["active"].cpu().numpy()
            din_n = view["din_neuron"].cpu().numpy()
            din_s = view["din_slot"].cpu().numpy()
            dout = view["dout_neuron"].cpu().numpy()
            x_np = x.cpu().numpy().reshape(cfg.batch, cfg.d_model)
            if shared:
                ids_gpu = view["ids"].cpu().numpy().astype(np.int64)
                rec = orc.step(x_np, ids_override=ids_gpu)
                summary["near_ties"] += _ids_accept(rec, ids_gpu, cfg, w1, w2)
            else:
                fire = []
                for s in range(cfg.n_sparse):
                    f = np.zeros(cfg.d_ff, dtype=bool)
                    f[active[s, :counts[s, 0]]] = True
                    assert counts[s, 3] == 0, "per-layer parity assumes no K_max overflow"
                    fire.append(f)
                rec = orc.step(x_np, fire_override=fire)
                for s in range(cfg.n_sparse):
                    layer = cfg.n_dense + s
                    summary["near_ties"] += _fire_accept(rec, fire[s], s, oracle.f64(wl.pred_w1[layer]),
                                                         oracle.f64(wl.pred_w2[layer]))
            # ---- bit-exact integer state
            for s in range(cfg.n_sparse):
                a_ref = rec.active[s]
                assert counts[s, 0] == len(a_ref), f"token {t} layer {s}: |A| {counts[s, 0]} vs {len(a_ref)}"
                assert active[s, :counts[s, 0]].tolist() == a_ref
                assert counts[s, 3] == rec.overflow[s]
                pairs = rec.d_in[s]
                assert counts[s, 1] == len(pairs)
                assert din_n[s, :counts[s, 1]].tolist() == [p[0] for p in pairs]
                assert din_s[s, :counts[s, 1]].tolist() == [p[1] for p in pairs]
                assert counts[s, 2] == len(rec.d_out[s])
                assert dout[s, :counts[s, 2]].tolist() == rec.d_out[s]
                sm, inv = dec.get_state(cfg.n_dense + s)
                assert np.array_equal(np.asarray(sm), orc.slotmap[s]), f"slot map differs, layer {s}"
                assert np.array_equal(np.asarray(inv), orc.inv[s]), f"inverse map differs, layer {s}"
            # ---- row moves of the compact placement (none under slot reuse)
            mvc = view["move_count"].cpu().numpy()
            msrc = view["move_src"].cpu().numpy() if view["move_src"] is not None else None
            mdst = view["move_dst"].cpu().numpy() if view["move_dst"] is not None else None
            for s in range(cfg.n_sparse):
                assert mvc[s] == len(rec.moves[s]), f"token {t} layer {s}: {mvc[s]} moves vs {len(rec.moves[s])}"
                if mvc[s]:
                    got = list(zip(msrc[s, :mvc[s]].tolist(), mdst[s, :mvc[s]].tolist()))
                    assert got == [tuple(m) for m in rec.moves[s]], f"token {t} layer {s}: moves differ"
            assert st["moved_rows"] == int(mvc.sum())
            summary["moved_rows"] = summary.get("moved_rows", 0) + int(mvc.sum())
            summary["din_rows"] += int(counts[:, 1].sum())
            assert st["din_rows"] == int(counts[:, 1].sum())
            # ---- residual stream after all layers
            hg = h.cpu().numpy().reshape(cfg.batch, -1)
            rel = max(oracle.rel_l2(hg[b], rec.h[b]) for b in range(cfg.batch))
            summary["max_h_rel"] = max(summary["max_h_rel"], rel)
            assert rel <= FFN_TOL, f"token {t}: h rel-L2 {rel}"
            # ---- per-layer FFN outputs through the standalone entry points
            if check_layer_y:
                for l in range(cfg.n_dense):
                    hin = torch.from_numpy(rec.h_in_dense[l].astype(np.float32)).cuda().reshape(-1)
                    y = dec.dense_mlp(l, hin).cpu().numpy().reshape(cfg.batch, -1)
                    r = max(oracle.rel_l2(y[b], rec.y_dense[l][b]) for b in range(cfg.batch))
                    summary["max_y_rel"] = max(summary["max_y_rel"], r)
                    assert r <= FFN_TOL, f"token {t} dense layer {l}: rel-L2 {r}"
                for s in range(cfg.n_sparse):
                    hin = torch.from_numpy(rec.h_in[s].astype(np.float32)).cuda().reshape(-1)
                    y = dec.sparse_mlp(cfg.n_dense + s, hin).cpu().numpy().reshape(cfg.batch, -1)
                    for b in range(cfg.batch):
                        ref = rec.y[s][b]
                        if np.linalg.norm(ref) == 0.0:
                            assert np.all(y[b] == 0.0)
                        else:
                            r = oracle.rel_l2(y[b], ref)
                            summary["max_y_rel"] = max(summary["max_y_rel"], r)
                            assert r <= FFN_TOL, f"token {t} sparse layer {s} sequence {b}: rel-L2 {r}"
            # ---- resident buffer bytes
            if check_buffers or sample_slots:
                compare_buffers(dec, orc, wl, sample_slots, rng)
            summary["tokens"] += 1
        dec.check_error()
    finally:
        if own_dec:
            dec.close()
    return summary


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def compare_buffers(dec, orc, wl, sample_slots, rng):
    cfg = wl.cfg
    for s in range(cfg.n_sparse):
        layer = cfg.n_dense + s
        if orc.materialize:
            for p in range(cfg.n_proj):
                got = dec.resident_rows(layer, p).cpu()
                assert torch.equal(_bits(got), _bits(orc.bufs[s, p])), f"buffer bytes differ: layer {s} proj {p}"
        else:
            k = min(sample_slots, cfg.k_max)
            slots = np.sort(rng.choice(cfg.k_max, size=k, replace=False))
            inv = orc.inv[s]
            for p in range(cfg.n_proj):
                rows = dec.resident_rows(layer, p)[torch.from_numpy(slots).cuda()].cpu()
                for i, slot in enumerate(slots):
                    n = int(inv[slot])
                    if n >= 0:
                        assert torch.equal(_bits(rows[i]), _bits(wl.store[s, n, p])), \
                            f"layer {s} slot {slot} proj {p} != record {n}"
