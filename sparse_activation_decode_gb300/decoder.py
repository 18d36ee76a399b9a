"""Python face of the C ABI: one decode model on the current CUDA device.

Argument marshalling only: every step of the decode path runs in the CUDA
library (libnp.so); this module passes pointers, sizes and streams.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib as L

_DTYPES = {torch.float32: L.NP_F32, torch.float16: L.NP_F16, torch.bfloat16: L.NP_BF16}


class _DevArray:
    """Zero-copy torch view of library-owned device memory."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def _wrap(ptr: int, shape, dtype: torch.dtype) -> torch.Tensor:
    typestr = {torch.int32: "<i4", torch.float32: "<f4", torch.float16: "<f2", torch.bfloat16: "<i2",
               torch.uint32: "<u4"}[dtype]
    t = torch.as_tensor(_DevArray(ptr, shape, typestr), device="cuda")
    return t.view(torch.bfloat16) if dtype == torch.bfloat16 else t


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


class SparseDecoder:
    """Wraps np_init_model ... np_free_model.  Tensors passed in are kept
    alive by this object.  Device tensors must be contiguous and on the
    current CUDA device; `host_store` is a contiguous CPU tensor."""

    def __init__(self, *, n_layers: int, n_dense: int, d_model: int, d_ff: int, k_max: int,
                 n_centroids: int, dtype: torch.dtype, host_store: torch.Tensor,
                 pred_w1: torch.Tensor, pred_w2: torch.Tensor, pred_b2: torch.Tensor | None = None,
                 dense_w: torch.Tensor | None = None, centroids: torch.Tensor | None = None,
                 pred_hidden: int, pred_kind: str = "shared_argmax", has_gate: bool = True,
                 combine: str = "union", residency: str = "slotmap", window: int = 1, batch: int = 1,
                 staging_rows: int = 0, h2d_mode: str = "fused", activation: str = "relu",
                 slots: str = "reuse", lookahead: int = 0,
                 main_stream: torch.cuda.Stream | None = None, side_stream: torch.cuda.Stream | None = None,
                 read_hook=None):
        self.lib = L.load()
        self.model = ctypes.c_void_p()
        self._keep = [host_store, pred_w1, pred_w2, pred_b2, dense_w, centroids]
        for t in (pred_w1, pred_w2, pred_b2, dense_w, centroids):
            if t is not None and (not t.is_cuda or not t.is_contiguous()):
                raise ValueError("device tensors must be contiguous CUDA tensors")
        if not host_store.is_contiguous() or host_store.is_cuda:
            raise ValueError("host_store must be a contiguous CPU tensor")
        self.main_stream = main_stream or torch.cuda.current_stream()
        self.side_stream = side_stream or torch.cuda.Stream(priority=-1)
        self._registered = None
        if not host_store.is_pinned():
            L.check(self.lib.np_host_register(host_store.data_ptr(),
                                              host_store.numel() * host_store.element_size()),
                    "np_host_register")
            self._registered = host_store.data_ptr()
        self._hook = L.READ_HOOK(read_hook) if read_hook is not None else L.READ_HOOK()
        d = L.ModelDesc()
        d.n_layers, d.n_dense, d.d_model, d.d_ff = n_layers, n_dense, d_model, d_ff
        d.k_max, d.n_centroids, d.dtype = k_max, n_centroids, _DTYPES[dtype]
        d.has_gate = int(has_gate)
        d.combine = {"intersect": L.NP_COMBINE_INTERSECT, "union": L.NP_COMBINE_UNION}[combine]
        d.residency = {"slotmap": L.NP_RES_SLOTMAP, "window": L.NP_RES_WINDOW,
                       "frequency": L.NP_RES_FREQUENCY}[residency]
        d.lookahead = lookahead
        d.window, d.batch, d.staging_rows, d.pred_hidden = window, batch, staging_rows, pred_hidden
        d.activation = {"relu": 0, "swiglu": 1}[activation]
        d.slots = {"reuse": L.NP_SLOTS_REUSE, "compact": L.NP_SLOTS_COMPACT}[slots]
        self.compact = slots == "compact"
        d.pred_kind = {"shared_argmax": L.NP_PRED_SHARED_ARGMAX,
                       "perlayer_sigmoid": L.NP_PRED_PERLAYER_SIGMOID}[pred_kind]
        d.h2d_mode = {"staged": L.NP_H2D_STAGED, "fused": L.NP_H2D_FUSED}[h2d_mode]
        d.host_store = host_store.data_ptr()
        d.dense_w = _ptr(dense_w)
        d.pred_w1, d.pred_w2, d.pred_b2 = _ptr(pred_w1), _ptr(pred_w2), _ptr(pred_b2)
        d.centroids = _ptr(centroids)
        d.main_stream = self.main_stream.cuda_stream
        d.side_stream = self.side_stream.cuda_stream
        d.read_hook = self._hook
        d.read_ctx = None
        self.desc = d
        try:
            L.check(self.lib.np_init_model(ctypes.byref(d), ctypes.byref(self.model)), "np_init_model")
        except Exception:
            self._unregister()
            raise
        self.n_layers, self.n_dense, self.d_model, self.d_ff, self.k_max = n_layers, n_dense, d_model, d_ff, k_max
        self.batch, self.dtype, self.pred_kind = batch, dtype, pred_kind
        self.n_sparse = n_layers - n_dense
        self.n_heads = 2 * (n_layers - 1) if pred_kind == "shared_argmax" else 0
        self.words = (d_ff + 31) // 32
        self.n_proj = 3 if has_gate else 2

    # -- lifetime ----------------------------------------------------------
    def _unregister(self):
        if self._registered is not None:
            self.lib.np_host_unregister(self._registered)
            self._registered = None

    def close(self):
        if self.model:
            L.check(self.lib.np_free_model(self.model), "np_free_model")
            self.model = ctypes.c_void_p()
        self._unregister()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- the path -----------------------------------------------------------
    def _on_main(self, *tensors):
        """Make the main stream wait for work the caller queued on torch's
        current stream for these tensors."""
        cur = torch.cuda.current_stream()
        if cur != self.main_stream:
            self.main_stream.wait_stream(cur)

    def _back(self):
        cur = torch.cuda.current_stream()
        if cur != self.main_stream:
            cur.wait_stream(self.main_stream)

    def decode_token(self, h: torch.Tensor, stats: bool = False):
        self._on_main(h)
        st = L.Stats() if stats else None
        L.check(self.lib.np_decode_token(self.model, h.data_ptr(), ctypes.byref(st) if st else None),
                "np_decode_token")
        self._back()
        if st is None:
            return None
        return {k: getattr(st, k) for k, _ in L.Stats._fields_}

    def predict(self, h: torch.Tensor, layer: int = 0) -> torch.Tensor:
        self._on_main(h)
        if self.pred_kind == "shared_argmax":
            out = torch.empty((self.batch, self.n_heads), dtype=torch.int32, device=h.device)
        else:
            out = torch.zeros((self.words,), dtype=torch.int32, device=h.device)
        L.check(self.lib.np_predict(self.model, layer, h.data_ptr(), out.data_ptr()), "np_predict")
        self._back()
        return out

    def delta(self, pred: torch.Tensor, layer: int = -1) -> dict:
        self._on_main(pred)
        v = L.DeltaView()
        L.check(self.lib.np_delta(self.model, layer, pred.data_ptr(), ctypes.byref(v)), "np_delta")
        self._back()
        return self._view(v)

    def last_delta(self) -> dict:
        """Device views of the last token's predictor output and delta."""
        v = L.DeltaView()
        L.check(self.lib.np_last_delta(self.model, ctypes.byref(v)), "np_last_delta")
        return self._view(v)

    def _view(self, v) -> dict:
        S, K = v.n_sparse, v.k_max
        ids = (_wrap(v.ids, (self.batch, self.n_heads), torch.int32)
               if v.ids and self.n_heads else None)
        return {"ids": ids, "counts": _wrap(v.counts, (S, 4), torch.int32),
                "active": _wrap(v.active, (S, K), torch.int32),
                "active_slot": _wrap(v.active_slot, (S, K), torch.int32),
                "din_neuron": _wrap(v.din_neuron, (S, K), torch.int32),
                "din_slot": _wrap(v.din_slot, (S, K), torch.int32),
                "dout_neuron": _wrap(v.dout_neuron, (S, K), torch.int32),
                "move_count": _wrap(v.move_count, (S,), torch.int32),
                "move_src": _wrap(v.move_src, (S, K), torch.int32) if v.move_src else None,
                "move_dst": _wrap(v.move_dst, (S, K), torch.int32) if v.move_dst else None}

    def scatter(self, layer: int = -1) -> None:
        L.check(self.lib.np_scatter(self.model, layer), "np_scatter")
        self._back()

    def sparse_mlp(self, layer: int, h: torch.Tensor) -> torch.Tensor:
        self._on_main(h)
        y = torch.empty_like(h)
        L.check(self.lib.np_sparse_mlp(self.model, layer, h.data_ptr(), y.data_ptr()), "np_sparse_mlp")
        self._back()
        return y

    def dense_mlp(self, layer: int, h: torch.Tensor) -> torch.Tensor:
        self._on_main(h)
        y = torch.empty_like(h)
        L.check(self.lib.np_dense_mlp(self.model, layer, h.data_ptr(), y.data_ptr()), "np_dense_mlp")
        self._back()
        return y

    def ffn_layers(self, first: int, count: int, h: torch.Tensor) -> torch.Tensor:
        """FFNs of layers first..first+count-1 on the resident rows, h updated
        in place ([batch][D] float32 on the device)."""
        self._on_main(h)
        L.check(self.lib.np_ffn_layers(self.model, first, count, h.data_ptr()), "np_ffn_layers")
        self._back()
        return h

    def reset_sequence(self) -> None:
        L.check(self.lib.np_reset_sequence(self.model), "np_reset_sequence")

    # -- inspection ---------------------------------------------------------
    def get_state(self, layer: int):
        sm = (ctypes.c_int32 * self.d_ff)()
        inv = (ctypes.c_int32 * self.k_max)()
        L.check(self.lib.np_get_state(self.model, layer, sm, inv), "np_get_state")
        return list(sm), list(inv)

    def counts(self):
        c = (ctypes.c_int32 * (4 * max(self.n_sparse, 1)))()
        L.check(self.lib.np_get_counts(self.model, c), "np_get_counts")
        return [list(c[4 * s:4 * s + 4]) for s in range(self.n_sparse)]

    def resident_rows(self, layer: int, proj: int) -> torch.Tensor:
        p = ctypes.c_void_p()
        L.check(self.lib.np_resident_rows(self.model, layer, proj, ctypes.byref(p)), "np_resident_rows")
        return _wrap(p.value, (self.k_max, self.d_model), self.dtype)

    def check_error(self) -> None:
        L.check(self.lib.np_check_error(self.model), "np_check_error")

    def set_profiling(self, on: bool, exact: bool = False) -> None:
        """Per-launch event timing; exact=True orders each start event after
        the launch's cross-stream waits (one extra empty launch per kernel)."""
        L.check(self.lib.np_set_profiling(self.model, (2 if exact else 1) if on else 0), "np_set_profiling")

    def profile(self) -> dict:
        ms = (ctypes.c_double * L.NP_N_KINDS)()
        n = (ctypes.c_int64 * L.NP_N_KINDS)()
        b = (ctypes.c_int64 * L.NP_N_KINDS)()
        L.check(self.lib.np_get_profile(self.model, ms, n, b), "np_get_profile")
        return {k: {"ms": ms[i], "launches": n[i], "bytes": b[i]} for i, k in enumerate(L.KIND_NAMES)}

    def timeline(self, max_entries: int = 65536):
        """[(kind, start_ms, end_ms)] of the launches timed since the last
        profile() call, in issue order.  The library keeps at most the most
        recent 16384 launches (older ones only enter the profile() sums)."""
        kinds = (ctypes.c_int32 * max_entries)()
        a = (ctypes.c_float * max_entries)()
        b = (ctypes.c_float * max_entries)()
        n = ctypes.c_int32()
        L.check(self.lib.np_get_timeline(self.model, kinds, a, b, max_entries, ctypes.byref(n)), "np_get_timeline")
        return [(L.KIND_NAMES[kinds[i]], a[i], b[i]) for i in range(n.value)]

    def launch_count(self) -> int:
        return int(self.lib.np_launch_count(self.model))


def decoder_for(wl, *, h2d_mode: str = "fused", staging_rows: int | None = None, read_hook=None,
                centroids_dev: torch.Tensor | None = None, **kw) -> SparseDecoder:
    """Build a SparseDecoder from an object carrying a `cfg` (shapes) and the
    weight tensors (dense_w, store, pred_w1, pred_w2, pred_b2, centroids)."""
    cfg = wl.cfg
    dev = torch.device("cuda", torch.cuda.current_device())
    cent = centroids_dev
    if cent is None and wl.centroids is not None:
        cent = torch.from_numpy(wl.centroids.view("int32")).to(dev).contiguous()

    def on_dev(t):
        return None if t is None else t.to(dev).contiguous()

    return SparseDecoder(
        n_layers=cfg.n_layers, n_dense=cfg.n_dense, d_model=cfg.d_model, d_ff=cfg.d_ff, k_max=cfg.k_max,
        n_centroids=cfg.n_centroids, dtype=cfg.torch_dtype, host_store=wl.store,
        pred_w1=on_dev(wl.pred_w1), pred_w2=on_dev(wl.pred_w2), pred_b2=on_dev(wl.pred_b2),
        dense_w=on_dev(wl.dense_w), centroids=cent, pred_hidden=cfg.pred_hidden,
        pred_kind=cfg.pred_kind, has_gate=cfg.has_gate, combine=cfg.combine, residency=cfg.residency,
        window=cfg.window if cfg.residency == "window" else 1, batch=cfg.batch,
        staging_rows=cfg.staging_rows if staging_rows is None else staging_rows, h2d_mode=h2d_mode,
        activation=cfg.activation, slots=cfg.slots, lookahead=cfg.lookahead,
        read_hook=read_hook, **kw)


def _shares_storage(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Two device tensors' byte ranges overlap."""
    a0, b0 = a.data_ptr(), b.data_ptr()
    return a0 < b0 + b.numel() * b.element_size() and b0 < a0 + a.numel() * a.element_size()


def ffn_rows_noalloc(h: torch.Tensor, w_gate: torch.Tensor | None, w_up: torch.Tensor, w_down: torch.Tensor,
                     rows: torch.Tensor | None, n_rows: int, y: torch.Tensor | None = None) -> torch.Tensor:
    """np_ffn_rows_noalloc: the FFN over listed rows without any device
    allocation by the library (its scratch is a fixed device array); for
    callers that cannot allocate.  Enqueued on torch's current stream.
    h: float32 [d_model]; weights [row_limit][d_model], one dtype, all the
    same shape; rows: int32 row indices or None for rows 0..n_rows-1.
    Raises ValueError for inputs the C entry point would misread."""
    lib = L.load()
    ws = [w for w in (w_gate, w_up, w_down) if w is not None]
    for w in ws:
        if not w.is_cuda or not w.is_contiguous() or w.dim() != 2:
            raise ValueError("weights must be contiguous 2-D CUDA tensors")
        if w.shape != w_up.shape or w.dtype != w_up.dtype:
            raise ValueError("gate, up and down weights must share one shape and dtype")
    if w_up.dtype not in _DTYPES:
        raise ValueError(f"unsupported weight dtype {w_up.dtype}")
    d_model = int(w_up.shape[1])
    if h.dtype != torch.float32 or not h.is_cuda or not h.is_contiguous() or h.numel() != d_model:
        raise ValueError("h must be a contiguous float32 CUDA tensor of d_model elements")
    if rows is not None:
        if rows.dtype != torch.int32 or not rows.is_cuda or not rows.is_contiguous() or rows.numel() < n_rows:
            raise ValueError("rows must be a contiguous int32 CUDA tensor holding at least n_rows indices")
    elif n_rows > w_up.shape[0]:
        raise ValueError("n_rows exceeds the weights' rows")
    if y is None:
        y = torch.empty_like(h)
    elif y.dtype != torch.float32 or not y.is_cuda or not y.is_contiguous() or y.numel() != d_model:
        raise ValueError("y must be a contiguous float32 CUDA tensor of d_model elements")
    for t in ws + [h] + ([rows] if rows is not None else []):
        if _shares_storage(y, t):
            raise ValueError("y may not share memory with h, the weights or the row list")
    L.check(lib.np_ffn_rows_noalloc(h.data_ptr(), None if w_gate is None else w_gate.data_ptr(), w_up.data_ptr(),
                                    w_down.data_ptr(), None if rows is None else rows.data_ptr(), int(n_rows),
                                    int(w_up.shape[0]), d_model, _DTYPES[w_up.dtype],
                                    int(w_gate is not None), y.data_ptr(), torch.cuda.current_stream().cuda_stream),
            "np_ffn_rows_noalloc")
    return y


def ffn_rows_noalloc_check() -> None:
    """np_ffn_rows_noalloc_check on torch's current stream: synchronise it,
    then raise NpError if any np_ffn_rows_noalloc call since the last check
    recorded a row index out of range (status -6) or an expired wait (-5)."""
    lib = L.load()
    L.check(lib.np_ffn_rows_noalloc_check(torch.cuda.current_stream().cuda_stream), "np_ffn_rows_noalloc_check")
