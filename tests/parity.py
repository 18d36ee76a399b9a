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

# Near-tie acceptance (see oracle.argmax_tolerance).  The GPU's predictor
# input is its own float32 residual stream, which differs from the oracle's by
# accumulated rounding; X_REL bounds that difference (relative 2-norm) on the
# CUDA-core path, X_REL_TC adds the 16+16-bit operand split of the tensor-core
# path (hi + lo keeps about 17 significant bits: relative error <= 2^-17).
# Whenever a near tie is accepted, the token's final residual stream must
# itself be within X_REL of the oracle's, which checks the assumption.
X_REL = 4e-6
X_REL_TC = 1e-5


def rowdot_depth(length: int, elem_bytes: int, bias: bool = False) -> int:
    """Rounded additions on any product's path in the batch-1 predictor
    kernel: a thread's chunks of 16 bytes (E elements each) go into two
    interleaved fp32 sums by fused multiply-adds (even and odd elements, E/2
    per chunk each), which are then added; a 5-level warp tree; 8 warp
    partials added in order; and the bias of the per-layer predictor."""
    e = 16 // elem_bytes
    chunks = -(-(length // e) // 256)
    return (e // 2) * chunks + 1 + 5 + 8 + (1 if bias else 0)


def predictor_bound_args(cfg) -> dict:
    """x_rel_err and accumulation depths of the predictor's two products on
    the GPU path that decodes `cfg`.  The tensor-core path (batch > 1) is
    given the any-order bound with twice the roundings (its accumulator's
    rounding is not specified as round-to-nearest)."""
    bias = cfg.pred_kind != "shared_argmax"
    if cfg.batch > 1:
        return {"x_rel_err": X_REL_TC, "depth1": 2 * (cfg.d_model + 1),
                "depth2": 2 * (cfg.pred_hidden + 1)}
    return {"x_rel_err": X_REL, "depth1": rowdot_depth(cfg.d_model, cfg.elem_bytes),
            "depth2": rowdot_depth(cfg.pred_hidden, cfg.elem_bytes, bias)}


def build_decoder(wl, **kw):
    from sparse_activation_decode_gb300 import decoder_for
    return decoder_for(wl, **kw)


def _ids_accept(rec, ids_gpu, cfg, w1, w2):
    """Per sequence and head, GPU id must be within the fp32 bound of the max."""
    near = 0
    args = predictor_bound_args(cfg)
    for b in range(cfg.batch):
        lg = rec.logits[b].reshape(cfg.n_heads, cfg.n_centroids)
        own = lg.argmax(axis=1)
        if np.array_equal(own, ids_gpu[b]):
            continue
        eps = oracle.argmax_tolerance(w1, w2, rec.pred_xhat[b], **args).reshape(cfg.n_heads, cfg.n_centroids)
        for h in np.flatnonzero(own != ids_gpu[b]):
            g = int(ids_gpu[b][h])
            assert 0 <= g < cfg.n_centroids
            bound = eps[h, g] + eps[h, own[h]]
            assert lg[h, g] >= lg[h, own[h]] - bound, (
                f"head {h}: GPU id {g} logit {lg[h, g]} vs max {lg[h, own[h]]} (bound {bound})")
            near += 1
    return near


def _fire_accept(rec, fire_gpu, s, w1, w2, b2, cfg):
    """Firing decisions: where the GPU disagrees with logit > 0, the oracle's
    logit must be within the fp32 bound of zero."""
    lg = rec.pred_logits_layer[s]
    ref = lg > 0.0
    diff = np.flatnonzero(ref != fire_gpu)
    if diff.size:
        eps = oracle.argmax_tolerance(w1, w2, rec.pred_xhat[s], b2=b2, **predictor_bound_args(cfg))
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
            near_before = summary["near_ties"]
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
                                                         oracle.f64(wl.pred_w2[layer]),
                                                         oracle.f64(wl.pred_b2[layer]), cfg)
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
            if summary["near_ties"] > near_before:
                # the acceptance bound assumed the GPU's input error stays
                # within x_rel_err: check it on this token's residual stream
                x_rel = predictor_bound_args(cfg)["x_rel_err"]
                assert rel <= x_rel, f"token {t}: near tie accepted but h rel-L2 {rel} > {x_rel}"
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
