"""CPU oracle of the per-token sparse-MLP decode path, in float64.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
benchmark's CPU-baseline / reference leg may import this module; the product
path (the C-ABI library and its Python binding) never calls it and shares no
code with it.  Inputs come from the seeded generators in `workloads`.

Every step is written out plainly, in the order the pages give:

* dense prefix, predictor after layer 0, active set from centroid masks, set
  difference against the resident rows, slot map update, staged records copied
  into the three projection buffers, sparse FFN over the resident active rows
  (NeuroPrefetcher: Storage-Aware Sparse LLM Inference via Delta Prefetching,
  sections "System Overview", "Shared Activation Predictor", "Predictive Delta
  Prefetching", "I/O Path"; full-text HTML: Figure 2 execution flow, delta
  runtime, slot map, neuron-centric layout, launch_deinterleave_scatter);
* the window residency and up|down bundling variant (LLM in a flash: Efficient
  Large Language Model Inference with Limited Memory, sections 3.1 "Reducing
  Data Transfer" and 3.2 "Increasing Transfer Throughput").

Readings where the pages are silent or disagree (each also listed in the
design notes):

* the combine operator is a parameter: the pages intersect gate and up masks,
  the measured configuration takes their union;
* K_max is a cap: when the combined set is larger, the K_max lowest neuron IDs
  are kept;
* the lost set-difference formula is D_in = A_t minus R_{t-1} and
  D_out = R_{t-1} minus R_t (R = resident set);
* freed slots are handed out in ascending slot order to incoming neurons in
  ascending ID order;
* activation h_n = relu(g_n . x) * (u_n . x) (ReLU-fied Llama), or
  relu(u_n . x) without a gate (OPT); optionally silu(g_n . x) * (u_n . x)
  (SwiGLU) over the same predicted rows;
* the rest of the transformer block is replaced by a residual stream
  h <- h + y with a weightless RMSNorm (eps 1e-6) in front of every FFN and of
  the predictor;
* argmax ties go to the lowest centroid index; the per-layer predictor fires
  when its logit is strictly positive (sigmoid > 0.5);
* batched decoding takes the union of the sequences' active sets; every
  sequence's FFN runs over that union, on the same (unrounded) normalised
  input as a single sequence.

Functions without an external pin say so in their docstring ("parity
unpinned"); all others are pinned by the CPU tests against closed forms, brute
force and the pages' printed numbers.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

RMS_EPS = 1e-6


# ---------------------------------------------------------------------------
# Elementary steps
# ---------------------------------------------------------------------------
def f64(a) -> np.ndarray:
    """Widen a torch tensor / numpy array exactly to float64 on the CPU."""
    if isinstance(a, torch.Tensor):
        return a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def rmsnorm(h: np.ndarray) -> np.ndarray:
    """x_hat = h / sqrt(mean(h^2) + eps).  Stand-in for the norm in front of
    each MLP; the pages keep normalisation parameters resident but give no
    formula (reading)."""
    h = np.asarray(h, dtype=np.float64)
    return h / np.sqrt(np.mean(h * h) + RMS_EPS)


def silu(a: np.ndarray) -> np.ndarray:
    """silu(a) = a * sigmoid(a) = a / (1 + exp(-a)) (the SwiGLU gate)."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def ffn_rows(gate: np.ndarray | None, up: np.ndarray, down_t: np.ndarray,
             xhat: np.ndarray, activation: str = "relu") -> tuple[np.ndarray, np.ndarray]:
    """FFN over an explicit list of neurons.

    gate, up, down_t: [n, D] rows (row n of the gate, up and down^T
    projections of neuron n: NeuroPrefetcher full text, delta runtime, where
    each active neuron's output comes from its own three rows).  Returns
    (y[D], h[n]) with
        h_n = relu(gate_n . x) * (up_n . x)   (ReLU-fied Llama)
        h_n = silu(gate_n . x) * (up_n . x)   (activation "swiglu": the
                                               SwiGLU MLP of the pages'
                                               models, NeuroPrefetcher
                                               "Predictive Delta Prefetching")
        h_n = relu(up_n . x)                   (no gate: OPT)
        y   = sum_n h_n * down_t_n.
    """
    b = up @ xhat
    if gate is None:
        hn = np.maximum(b, 0.0)
    else:
        a = gate @ xhat
        g = silu(a) if activation == "swiglu" else np.where(a > 0.0, a, 0.0)
        hn = g * b
    y = down_t.T @ hn
    return y, hn


def predictor_logits(w1: np.ndarray, w2: np.ndarray, b2: np.ndarray | None,
                     xhat: np.ndarray) -> np.ndarray:
    """z = relu(W1 x); logits = W2 z (+ b2).  The pages' predictor (feature
    projection, residual trunk, 2x31 linear heads: NeuroPrefetcher "Shared
    Activation Predictor") is reduced to one hidden layer; the per-layer
    low-rank predictor of LLM in a flash ("Reducing Data Transfer") has the
    same form plus an output bias."""
    z = np.maximum(w1 @ xhat, 0.0)
    out = w2 @ z
    if b2 is not None:
        out = out + b2
    return out


def head_argmax(logits: np.ndarray, n_heads: int, n_centroids: int) -> np.ndarray:
    """Per head, the centroid with the highest logit; ties go to the lowest
    index (NeuroPrefetcher "Shared Activation Predictor": each head picks its
    most probable centroid)."""
    return np.argmax(logits.reshape(n_heads, n_centroids), axis=1).astype(np.int64)


def head_index(layer: int, proj: int) -> int:
    """Head of absolute layer `layer` >= 1; proj 0 = gate, 1 = up.  The
    predictor emits 2 x (L-1) IDs: one gate and one up centroid for each of
    layers 1..L-1 (NeuroPrefetcher full text: 2 x 31 = 62 for 32 layers)."""
    return 2 * (layer - 1) + proj


def mask_ids(words: np.ndarray, d_ff: int) -> list[int]:
    """Neuron IDs set in a packed mask (bit n lives in word n//32, bit n%32)."""
    bits = np.unpackbits(np.asarray(words, dtype="<u4").view(np.uint8),
                         bitorder="little")[:d_ff]
    return [int(n) for n in np.flatnonzero(bits)]


def combine_sets(gate_ids: list[int], up_ids: list[int], mode: str) -> list[int]:
    """A = gate mask (intersect | union) up mask, sorted ascending
    (NeuroPrefetcher "Predictive Delta Prefetching": gate and up centroid masks
    are intersected; the measured configuration uses the union)."""
    g, u = set(gate_ids), set(up_ids)
    if mode == "intersect":
        return sorted(g & u)
    if mode == "union":
        return sorted(g | u)
    raise ValueError(mode)


def cap_set(active: list[int], k_max: int) -> tuple[list[int], int]:
    """Keep the k_max lowest IDs (NeuroPrefetcher full text, evaluation
    budgets: K_max bounds how many active neurons a sparse layer keeps).
    Returns (kept, number dropped)."""
    active = sorted(active)
    if len(active) <= k_max:
        return active, 0
    return active[:k_max], len(active) - k_max


def set_delta(active: list[int], resident_prev: list[int],
              resident_next: list[int]) -> tuple[list[int], list[int]]:
    """D_in = A_t minus R_{t-1}; D_out = R_{t-1} minus R_t (the set difference
    of NeuroPrefetcher's delta runtime; with the slot-map policy R_t = A_t)."""
    a, rp, rn = set(active), set(resident_prev), set(resident_next)
    return sorted(a - rp), sorted(rp - rn)


def assign_slots(slotmap: np.ndarray, inv: np.ndarray, d_in: list[int],
                 d_out: list[int], k_max: int) -> list[tuple[int, int]]:
    """Release the slots of D_out and give free slots to D_in, in place.

    Per-layer slot map S[n] = slot of neuron n or -1 (NeuroPrefetcher full
    text, delta runtime: outgoing neurons give up their slots, which the
    incoming ones then receive).  Reading: the i-th incoming neuron in
    ascending ID order takes the i-th free slot in ascending slot order.
    Returns the (neuron, slot) pairs of D_in."""
    for n in d_out:
        s = int(slotmap[n])
        assert s >= 0
        slotmap[n] = -1
        inv[s] = -1
    free = [s for s in range(k_max) if inv[s] < 0]
    assert len(free) >= len(d_in), "resident set larger than K_max"
    pairs = list(zip(d_in, free[:len(d_in)]))
    for n, s in pairs:
        slotmap[n] = s
        inv[s] = n
    return pairs


def assign_slots_compact(slotmap: np.ndarray, inv: np.ndarray, d_in: list[int],
                         d_out: list[int], n_rows: int) -> tuple[list[tuple[int, int]], list[tuple[int, int]], int]:
    """Compact placement, in place (LLM in a flash, 3.3 "Optimized Data
    Management in DRAM": the hole a removed neuron leaves is filled by one of
    the last occupied rows, new rows go after the occupied ones, and the
    occupied rows stay [0, num_rows)).

    Reading: with n_new = num_rows - |D_out|, every removed neuron whose slot
    lies below n_new is replaced by a surviving row from the end region
    [n_new, num_rows), the i-th such slot in ascending order by the i-th
    surviving end row in ascending order (one copy per slot to refill, the
    fewest possible); removed rows in the end region just fall away.  The
    incoming neurons, in ascending ID order, then take n_new, n_new + 1, ...
    Returns (the (neuron, slot) pairs of D_in, the (from_slot, to_slot) row
    moves, the new num_rows)."""
    out_slots = set()
    for n in d_out:
        sl = int(slotmap[n])
        assert 0 <= sl < n_rows
        out_slots.add(sl)
    n_new = n_rows - len(d_out)
    holes = sorted(sl for sl in out_slots if sl < n_new)
    movers = sorted(sl for sl in range(n_new, n_rows) if sl not in out_slots)
    assert len(holes) == len(movers)
    for n in d_out:
        sl = int(slotmap[n])
        slotmap[n] = -1
        inv[sl] = -1
    moves = list(zip(movers, holes))
    for src, dst in moves:
        n = int(inv[src])
        slotmap[n] = dst
        inv[dst] = n
        inv[src] = -1
    pairs = []
    for i, n in enumerate(d_in):
        sl = n_new + i
        assert sl < len(inv), "resident set larger than K_max"
        slotmap[n] = sl
        inv[sl] = n
        pairs.append((n, sl))
    return pairs, moves, n_new + len(d_in)


def window_resident(resident_prev: list[int], active: list[int], last_seen: dict,
                    t: int, window: int, k_max: int) -> list[int]:
    """Resident set after token t under windowing: the neurons active in the
    last `window` tokens (this one included) that were resident or are active
    now (LLM in a flash, 3.1 "Windowing": the rows predicted active for the
    recent tokens stay in memory).  If more than k_max remain, the ones whose last use is
    oldest go first, ties by ascending ID; neurons active now never go
    (reading: the pages give no cap rule).  `last_seen` must already hold t
    for the active neurons."""
    cand = (set(resident_prev) | set(active))
    cand = {n for n in cand if t - last_seen[n] < window}
    if len(cand) > k_max:
        act = set(active)
        order = sorted((n for n in cand if n not in act), key=lambda n: (last_seen[n], n))
        for n in order[:len(cand) - k_max]:
            cand.discard(n)
    return sorted(cand)


def frequency_resident(resident_prev: list[int], active: list[int], count, k_max: int) -> list[int]:
    """Resident set after a token under frequency-weighted caching
    (DynamicInfer, "hierarchical neuron cache": importance v = a + lambda f,
    a = predicted active now, f = the neuron's activation frequency so far in
    the sequence; the cache keeps the highest importance up to its budget).

    Reading: every active neuron must be resident (there is no CPU-side FFN
    here), so lambda f < 1 orders the rest: R = A plus the previously resident
    neurons, and while more than k_max remain the least frequently active of
    the non-active ones go first, ties by ascending ID.  `count[n]` = tokens of
    this sequence in which n was active, this one included."""
    cand = set(resident_prev) | set(active)
    if len(cand) > k_max:
        act = set(active)
        order = sorted((n for n in cand if n not in act), key=lambda n: (count[n], n))
        for n in order[:len(cand) - k_max]:
            cand.discard(n)
    return sorted(cand)


def predictor_source_layer(layer: int, lookahead: int) -> int:
    """Layer whose input feeds the per-layer predictor of `layer`: with a
    lookahead of k layers (DynamicInfer, "cross-layer sparse prediction": the
    predictor of layer i+k takes the hidden state of layer i) it is layer
    layer - k, and the token's input to layer 0 for the first layers."""
    return max(layer - lookahead, 0)


# ---------------------------------------------------------------------------
# Whole-token decode
# ---------------------------------------------------------------------------
@dataclass
class TokenRecord:
    """Everything the oracle computed for one token (per sparse layer lists are
    indexed by s = layer - n_dense)."""
    logits: list = field(default_factory=list)      # per sequence: fp64 logits
    ids: list = field(default_factory=list)         # per sequence: int64[heads]
    active: list = field(default_factory=list)      # per layer: sorted IDs
    overflow: list = field(default_factory=list)    # per layer: dropped by the cap
    d_in: list = field(default_factory=list)        # per layer: [(neuron, slot)]
    d_out: list = field(default_factory=list)       # per layer: sorted IDs
    moves: list = field(default_factory=list)       # per layer: [(from_slot, to_slot)] (compact)
    y: list = field(default_factory=list)           # per layer: [B][D] fp64
    h_in: list = field(default_factory=list)        # per layer: [B][D] input
    y_dense: list = field(default_factory=list)     # per dense layer: [B][D]
    h_in_dense: list = field(default_factory=list)  # per dense layer: [B][D] input
    pred_logits_layer: list = field(default_factory=list)  # per-layer predictor
    pred_xhat: list = field(default_factory=list)   # predictor input per sequence / layer
    h: np.ndarray | None = None                     # [B][D] after the last layer


class OracleDecoder:
    """Decode state (slot maps, resident buffers) plus the per-token step."""

    def __init__(self, wl, materialize_buffers: bool = True):
        cfg = self.cfg = wl.cfg
        self.wl = wl
        S, F, K, D = cfg.n_sparse, cfg.d_ff, cfg.k_max, cfg.d_model
        self.slotmap = np.full((S, F), -1, dtype=np.int64)
        self.inv = np.full((S, K), -1, dtype=np.int64)
        self.n_rows = [0] * S          # occupied rows under compact placement
        self.resident = [[] for _ in range(S)]
        self.last_seen = [dict() for _ in range(S)]
        self.count = [np.zeros(F, dtype=np.int64) for _ in range(S)]   # frequency residency
        self.t = 0
        self.materialize = materialize_buffers
        # Projection buffers start zeroed; storage dtype kept (exact copies).
        self.bufs = (torch.zeros((S, cfg.n_proj, K, D), dtype=wl.store.dtype)
                     if materialize_buffers else None)
        self._w1 = self._w2 = self._b2 = None

    # -- weights, widened on demand --------------------------------------
    def _pred(self, layer: int | None = None):
        wl = self.wl
        if layer is None:
            if self._w1 is None:
                self._w1, self._w2 = f64(wl.pred_w1), f64(wl.pred_w2)
            return self._w1, self._w2, None
        return f64(wl.pred_w1[layer]), f64(wl.pred_w2[layer]), f64(wl.pred_b2[layer])

    def _dense_rows(self, layer: int):
        """Gate, up and down^T rows of a dense layer (no gate rows when the
        model has none, as in its sparse records)."""
        w = f64(self.wl.dense_w[layer])
        if self.cfg.has_gate:
            return w[0], w[1], w[2]
        return None, w[0], w[1]

    def _sparse_rows(self, s: int, ids: list[int]):
        """Rows of the active neurons, read through the slot map from the
        resident buffers (or from the store when buffers are not kept)."""
        cfg = self.cfg
        if self.materialize:
            slots = [int(self.slotmap[s][n]) for n in ids]
            assert all(x >= 0 for x in slots), "active neuron not resident"
            rec = f64(self.bufs[s][:, slots, :])          # [n_proj][n][D]
        else:
            rec = f64(self.wl.store[s][ids]).transpose(1, 0, 2)
        if cfg.has_gate:
            return rec[0], rec[1], rec[2]
        return None, rec[0], rec[1]

    def reset(self):
        """Cold start: the next token loads its full predicted set."""
        self.__init__(self.wl, self.materialize)

    # -- the step ----------------------------------------------------------
    def step(self, x: np.ndarray, ids_override=None, fire_override=None) -> TokenRecord:
        """Decode one token (all sequences of the batch).

        x: [B][D] token inputs (the residual stream entering layer 0).
        ids_override: per sequence int[heads] to use instead of the oracle's
            own argmax (staged parity near fp32 ties).
        fire_override: per sparse layer, bool[F] firing decisions to use
            instead of logit > 0 (per-layer predictor, staged parity)."""
        cfg, wl = self.cfg, self.wl
        B = cfg.batch
        h = f64(x).reshape(B, cfg.d_model).copy()
        rec = TokenRecord()
        layer_in = []   # the residual stream entering each layer
        # Dense prefix (NeuroPrefetcher "System Overview": the first d layers
        # keep their MLP fully resident).
        for layer in range(cfg.n_dense):
            g, u, dt = self._dense_rows(layer)
            rec.h_in_dense.append(h.copy())
            layer_in.append(h.copy())
            yd = np.zeros((B, cfg.d_model))
            for b in range(B):
                yd[b], _ = ffn_rows(g, u, dt, rmsnorm(h[b]), cfg.activation)
                h[b] += yd[b]
            rec.y_dense.append(yd)
            if layer == 0:
                self._predict_shared(h, rec, ids_override)
        if cfg.n_dense == 0 and cfg.pred_kind == "shared_argmax":
            self._predict_shared(h, rec, ids_override)
        # Sparse suffix.
        for s in range(cfg.n_sparse):
            layer = cfg.n_dense + s
            layer_in.append(h.copy())
            if cfg.pred_kind == "shared_argmax":
                active = self._active_from_ids(s, layer, rec.ids)
            else:
                w1, w2, b2 = self._pred(layer)
                xs = rmsnorm(layer_in[predictor_source_layer(layer, cfg.lookahead)][0])
                lg = predictor_logits(w1, w2, b2, xs)
                rec.pred_xhat.append(xs)
                rec.pred_logits_layer.append(lg)
                fire = (lg > 0.0) if fire_override is None else np.asarray(fire_override[s])
                active = [int(n) for n in np.flatnonzero(fire)]
            active, dropped = cap_set(active, cfg.k_max)
            rec.active.append(active)
            rec.overflow.append(dropped)
            # Residency and delta.
            prev = self.resident[s]
            if cfg.residency == "window":
                for n in active:
                    self.last_seen[s][n] = self.t
                nxt = window_resident(prev, active, self.last_seen[s], self.t,
                                      cfg.window, cfg.k_max)
            elif cfg.residency == "frequency":
                self.count[s][active] += 1
                nxt = frequency_resident(prev, active, self.count[s], cfg.k_max)
            else:
                nxt = active
            d_in, d_out = set_delta(active, prev, nxt)
            moves = []
            if cfg.slots == "compact":
                pairs, moves, self.n_rows[s] = assign_slots_compact(
                    self.slotmap[s], self.inv[s], d_in, d_out, self.n_rows[s])
            else:
                pairs = assign_slots(self.slotmap[s], self.inv[s], d_in, d_out, cfg.k_max)
            self.resident[s] = nxt
            rec.d_in.append(pairs)
            rec.d_out.append(d_out)
            rec.moves.append(moves)
            # Compact placement first moves the kept rows into the freed
            # slots, then the incoming rows are written.  Scatter: each staged
            # record's rows go to the slot the delta runtime assigned
            # (NeuroPrefetcher "I/O Path", launch_deinterleave_scatter).
            if self.materialize:
                for src, dst in moves:
                    self.bufs[s, :, dst] = self.bufs[s, :, src]
                for n, slot in pairs:
                    for p in range(cfg.n_proj):
                        self.bufs[s, p, slot] = wl.store[s, n, p]
            # Sparse FFN over the resident active rows; the compact placement
            # computes over its whole occupied region (LLM in a flash 3.3: the
            # inference views are the first num_rows rows), which is the
            # active set unless windowing keeps recently used rows as well.
            g, u, dt = self._sparse_rows(s, nxt if cfg.slots == "compact" else active)
            rec.h_in.append(h.copy())
            ys = np.zeros((B, cfg.d_model))
            for b in range(B):
                ys[b], _ = ffn_rows(g, u, dt, rmsnorm(h[b]), cfg.activation)
                h[b] += ys[b]
            rec.y.append(ys)
        rec.h = h
        self.t += 1
        return rec

    def _predict_shared(self, h, rec, ids_override):
        cfg = self.cfg
        w1, w2, _ = self._pred()
        for b in range(cfg.batch):
            xs = rmsnorm(h[b])
            lg = predictor_logits(w1, w2, None, xs)
            rec.pred_xhat.append(xs)
            rec.logits.append(lg)
            ids = head_argmax(lg, cfg.n_heads, cfg.n_centroids)
            if ids_override is not None:
                ids = np.asarray(ids_override[b], dtype=np.int64)
            rec.ids.append(ids)

    def _active_from_ids(self, s: int, layer: int, ids_per_seq) -> list[int]:
        cfg, wl = self.cfg, self.wl
        out: set[int] = set()
        for ids in ids_per_seq:
            g = mask_ids(wl.centroids[s, 0, ids[head_index(layer, 0)]], cfg.d_ff)
            u = mask_ids(wl.centroids[s, 1, ids[head_index(layer, 1)]], cfg.d_ff)
            out |= set(combine_sets(g, u, cfg.combine))
        return sorted(out)


# ---------------------------------------------------------------------------
# Accounting (bytes the method must move)
# ---------------------------------------------------------------------------
def record_bytes(d_model: int, elem_bytes: int, n_proj: int = 3) -> int:
    """One neuron-centric record: gate | up | down^T rows of d_model elements
    (NeuroPrefetcher "I/O Path"), or up | down^T with row-column bundling
    (LLM in a flash 3.2: 2 d_model num_bytes)."""
    return n_proj * d_model * elem_bytes


def h2d_bytes(rec: TokenRecord, d_model: int, elem_bytes: int, n_proj: int) -> int:
    """Bytes read from the storage tier for one token: |D_in| records."""
    return sum(len(p) for p in rec.d_in) * record_bytes(d_model, elem_bytes, n_proj)


def rel_l2(got, ref) -> float:
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    return float(num / den) if den > 0 else float(num)


U32 = 2.0 ** -24   # unit roundoff of float32 (round to nearest)


def gamma(n: int) -> float:
    """gamma_n = n u / (1 - n u), u the float32 unit roundoff: the relative
    error factor of n successive roundings (Higham, Accuracy and Stability of
    Numerical Algorithms, Lemma 3.1)."""
    return n * U32 / (1.0 - n * U32)


def fp32_dot_bound(w: np.ndarray, v: np.ndarray, v_rel_err: float, depth: int | None = None) -> np.ndarray:
    """Bound on |computed - exact| for each row of w . v evaluated in float32,
    where the float32 inputs are exact copies of w and of a vector v' with
    ||v' - v||_2 <= v_rel_err ||v||_2.

    Rounding: any summation tree in which every product passes through at
    most `depth` rounded additions (one rounding per fused multiply-add, two
    for a multiply then an add) has |error| <= gamma_{depth+1} sum_i |w_i v'_i|
    (Higham, Lemma 3.1 and the tree-height form of Section 4.2).  depth=None
    takes the worst tree, a sequential sum over all k terms (depth k), so the
    bound holds for every evaluation order.  Input: |w . (v' - v)| <=
    ||w||_2 ||v' - v||_2 (Cauchy-Schwarz).  sum |w_i v'_i| is bounded by
    sum |w_i| |v_i| + ||w||_2 ||v' - v||_2."""
    k = w.shape[-1]
    h = k if depth is None else int(depth)
    wn = np.sqrt(np.sum(w * w, axis=-1))
    din = wn * (v_rel_err * float(np.linalg.norm(v)))
    mag = np.abs(w) @ np.abs(v) + din
    return gamma(h + 1) * mag + din


def argmax_tolerance(w1, w2, xhat, x_rel_err: float = 1e-5, depth1: int | None = None,
                     depth2: int | None = None, b2=None) -> np.ndarray:
    """Per-logit error bound of a float32 evaluation of logits = W2 relu(W1 x)
    (+ b2) whose input differs from x by at most x_rel_err (relative, 2-norm)
    and whose two products accumulate in trees of height depth1 and depth2
    (None: any order; with a bias, depth2 counts its addition as well).  relu
    is 1-Lipschitz, so each hidden unit carries the bound of its
    pre-activation, which W2 then propagates through |W2|.  The bias is a
    term of the second sum with an exact factor 1."""
    z = np.maximum(w1 @ xhat, 0.0)
    z_err = fp32_dot_bound(w1, xhat, x_rel_err, depth1)
    k2 = w2.shape[-1] + (0 if b2 is None else 1)
    h2 = k2 if depth2 is None else int(depth2)
    mag = np.abs(w2) @ (z + z_err)
    if b2 is not None:
        mag = mag + np.abs(np.asarray(b2, dtype=np.float64))
    return gamma(h2 + 1) * mag + np.abs(w2) @ z_err
