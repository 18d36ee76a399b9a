"""Seeded synthetic inputs for the per-token sparse-MLP decode path.

This module draws random numbers and lays them out; it performs no step of the
decode method (no normalisation, no dot product, no set operation, no slot
assignment).  Both the CUDA path and the CPU oracle consume exactly the arrays
it returns, so neither side ever produces the other's inputs.

What stands in for what (the pages measure trained Mistral / Llama / OPT models
on WikiText-2, HellaSwag, C4 and Alpaca, none of which exist here):

* FFN weights: i.i.d. normal, rounded once to the storage dtype.
* Centroid vocabulary (NeuroPrefetcher, "Offline Sparse Centroid Preparation"):
  per (sparse layer, projection) a chain of C binary masks.  Mask 0 holds
  exactly round(rho*F) random bits; mask c+1 keeps every set bit of mask c with
  probability p and refills the dropped count with bits that were unset in
  mask c, so the popcount stays exact and the overlap of consecutive masks is
  Binomial(n, p).
* Planted predictor: token t carries phase phi_t = phi0 + t (plus 2*s for the
  s-th sequence of a batch).  Its input x_t = N(0,1)^D + scale * v_{phi_t};
  rows j < C of the first predictor matrix are the unit vectors v_j and head h
  of the second matrix holds a spike of height `spike` at column
  (c - off_h) mod C for centroid c.  Consecutive tokens therefore select
  consecutive chain links, which realises the token-to-token persistence p
  (NeuroPrefetcher reports 82-85% row reuse, "I/O Reduction via Delta Reuse").
* OPT-style per-layer predictor (LLM in a flash, "Reducing Data Transfer"):
  random low-rank MLP whose output biases give neuron n a firing rate r_n drawn
  from Beta(a, b) with mean `active_rate`, so that a few hot neurons recur.

All structure is drawn with numpy's PCG64 (platform independent).  The bulk FFN
weights are drawn with torch's generator on the requested device (fast on a
GPU); whichever device draws them, the same tensors feed both sides.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np
import torch

_TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
_ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclass(frozen=True)
class Config:
    """Shapes and distribution parameters of one synthetic decode workload."""

    name: str
    n_layers: int            # L
    n_dense: int             # d: layers 0..d-1 keep their full FFN resident
    d_model: int             # D
    d_ff: int                # F
    k_max: int               # K: resident rows per sparse layer
    n_centroids: int         # C per (layer, projection); 0 for the per-layer predictor
    dtype: str               # 'f32' | 'f16' | 'bf16'
    density: float = 0.10    # rho: set bits per centroid mask / F
    persistence: float = 0.83  # p: chain persistence
    pred_hidden: int = 512   # predictor hidden width
    pred_kind: str = "shared_argmax"  # or 'perlayer_sigmoid'
    has_gate: bool = True    # False: OPT-style records (up | down^T)
    activation: str = "relu"  # gated FFN: 'relu' (ReLU-fied) or 'swiglu' (silu gate)
    combine: str = "union"   # 'union' | 'intersect' of the gate and up masks
    residency: str = "slotmap"  # 'slotmap' | 'window' | 'frequency'
    window: int = 5          # W tokens (window residency)
    lookahead: int = 0       # per-layer predictor of layer l reads the input of layer max(l - k, 0)
    slots: str = "reuse"     # 'reuse' free slots, or 'compact' (swap-with-last + append)
    batch: int = 1           # sequences decoded together
    weight_std: float = 0.02
    pred_std: float = 0.02
    planted: bool = True
    planted_scale: float = 200.0
    spike: float = 1.0
    active_rate: float = 0.05   # per-layer predictor: mean firing rate
    rate_beta: tuple = (0.25, 4.75)
    phase_step: int = 2      # batched: phase offset between sequences
    n_warm: int = 0          # tokens decoded before timing starts (prompt warm fill)
    n_decode: int = 16
    staging_rows: int = 0    # staging capacity in records (0: k_max)
    seed: int = 1000

    # ---- derived sizes -------------------------------------------------
    @property
    def n_sparse(self) -> int:
        return self.n_layers - self.n_dense

    @property
    def n_heads(self) -> int:
        """One gate head and one up head for every layer after layer 0."""
        return 2 * (self.n_layers - 1) if self.pred_kind == "shared_argmax" else 0

    @property
    def words(self) -> int:
        return (self.d_ff + 31) // 32

    @property
    def n_proj(self) -> int:
        return 3 if self.has_gate else 2

    @property
    def elem_bytes(self) -> int:
        return _ELEM_BYTES[self.dtype]

    @property
    def torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPES[self.dtype]

    @property
    def record_bytes(self) -> int:
        return self.n_proj * self.d_model * self.elem_bytes

    @property
    def n_tokens(self) -> int:
        return self.n_warm + self.n_decode

    @property
    def staging(self) -> int:
        return self.staging_rows if self.staging_rows > 0 else self.k_max

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


# ---------------------------------------------------------------------------
# The five workloads (shapes of the pages' models) and small parity cases.
# ---------------------------------------------------------------------------
TINY = Config(
    name="tiny", n_layers=4, n_dense=1, d_model=256, d_ff=1024, k_max=256,
    n_centroids=16, dtype="f32", density=0.10, persistence=0.83, pred_hidden=512,
    weight_std=1.0 / 16.0, pred_std=0.02, planted=False, n_warm=0, n_decode=16,
    seed=1000)

LLAMA7B = Config(
    name="llama2-7b-relu", n_layers=32, n_dense=1, d_model=4096, d_ff=11008,
    k_max=2048, n_centroids=1024, dtype="f16", density=0.10, persistence=0.83,
    pred_hidden=2816, n_warm=128, n_decode=256, seed=1001)

LLAMA13B = Config(
    name="llama2-13b-relu", n_layers=40, n_dense=4, d_model=5120, d_ff=13824,
    k_max=2048, n_centroids=1024, dtype="bf16", density=0.08, persistence=0.85,
    pred_hidden=3072, n_warm=128, n_decode=256, seed=1002)

OPT67B = Config(
    name="opt-6.7b-window", n_layers=32, n_dense=0, d_model=4096, d_ff=16384,
    k_max=4096, n_centroids=0, dtype="f16", pred_hidden=1024,
    pred_kind="perlayer_sigmoid", has_gate=False, residency="window", window=5,
    planted=False, n_warm=128, n_decode=256, seed=1003)

BATCHED7B = Config(
    name="llama2-7b-batch8", n_layers=32, n_dense=1, d_model=4096, d_ff=11008,
    k_max=4096, n_centroids=1024, dtype="bf16", density=0.055, persistence=0.83,
    pred_hidden=2816, batch=8, n_warm=128, n_decode=256, seed=1004)
# density 0.055 with sequences two chain links apart puts the union of the
# eight sequences' gate|up sets near 30% of d_ff at persistence 0.83 (48-52%
# at 0.5, 18% at 0.95; above K_max = 37% it is capped).

CONFIGS = {c.name: c for c in (TINY, LLAMA7B, LLAMA13B, OPT67B, BATCHED7B)}

# Small cases with the structure of the large ones: several CTA tiles of rows,
# d_ff not a multiple of 32 (ragged last mask word), planted predictor.
SMALL_F16 = Config(
    name="small-f16", n_layers=5, n_dense=1, d_model=512, d_ff=1000, k_max=192,
    n_centroids=64, dtype="f16", density=0.10, persistence=0.83, pred_hidden=160,
    planted_scale=60.0, n_warm=0, n_decode=12, seed=2001)

SMALL_BF16 = Config(
    name="small-bf16", n_layers=6, n_dense=2, d_model=640, d_ff=1400, k_max=224,
    n_centroids=48, dtype="bf16", density=0.08, persistence=0.85, pred_hidden=128,
    planted_scale=60.0, n_warm=0, n_decode=10, seed=2002)

SMALL_OPT = Config(
    name="small-opt", n_layers=3, n_dense=0, d_model=256, d_ff=2048, k_max=300,
    n_centroids=0, dtype="f16", pred_hidden=128, pred_kind="perlayer_sigmoid",
    has_gate=False, residency="window", window=5, planted=False, n_decode=14,
    seed=2003)

SMALL_BATCHED = Config(
    name="small-batched", n_layers=4, n_dense=1, d_model=512, d_ff=1000,
    k_max=512, n_centroids=64, dtype="bf16", density=0.10, persistence=0.83,
    pred_hidden=256, batch=8, planted_scale=60.0, n_decode=8, seed=2004)


# ---------------------------------------------------------------------------
# Random structure
# ---------------------------------------------------------------------------
def pack_bits(bits: np.ndarray) -> np.ndarray:
    """bool[..., F] -> uint32[..., ceil(F/32)], bit n at word n//32, bit n%32."""
    f = bits.shape[-1]
    w = (f + 31) // 32
    pad = np.zeros(bits.shape[:-1] + (w * 32,), dtype=np.uint8)
    pad[..., :f] = bits
    by = np.packbits(pad, axis=-1, bitorder="little")
    return by.view("<u4").reshape(bits.shape[:-1] + (w,)).astype(np.uint32)


def centroid_chain(rng: np.random.Generator, f: int, n_masks: int, density: float,
                   persistence: float) -> np.ndarray:
    """bool[n_masks, f]: one chain of masks with exact popcount round(density*f)."""
    n = int(round(density * f))
    out = np.zeros((n_masks, f), dtype=bool)
    cur = np.sort(rng.choice(f, size=n, replace=False))
    out[0, cur] = True
    for c in range(1, n_masks):
        keep = rng.random(n) < persistence
        kept = cur[keep]
        need = n - kept.size
        taken = out[c - 1].copy()          # refill only from bits unset in mask c-1
        new = []
        while need > 0:
            cand = rng.integers(0, f, size=2 * need + 8)
            cand = cand[~taken[cand]]
            _, first = np.unique(cand, return_index=True)
            pick = cand[np.sort(first)][:need]
            taken[pick] = True
            new.append(pick)
            need -= pick.size
        cur = np.sort(np.concatenate([kept] + new)) if new else kept
        out[c, cur] = True
    return out


def _torch_normal(shape, std, dtype, device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (t * std).to(dtype)


@dataclass
class Workload:
    """All inputs of one decode run.  Tensors live where `device` says, except
    the host weight store, which is always CPU memory (the storage tier)."""

    cfg: Config
    dense_w: torch.Tensor | None      # [d][n_proj][F][D]  (gate, up, down^T; no gate rows without a gate)
    store: torch.Tensor                # [S][F][n_proj][D]  record layout, CPU
    centroids: np.ndarray | None       # uint32 [S][2][C][words]
    pred_w1: torch.Tensor              # [H][D]       or [L][H][D]  (per layer)
    pred_w2: torch.Tensor              # [heads*C][H] or [L][F][H]
    pred_b2: torch.Tensor | None       # None         or [L][F]
    x: torch.Tensor                    # float32 [T][B][D] token inputs
    phases: np.ndarray | None = None   # int [T][B] planted phase per token
    offsets: np.ndarray | None = None  # int [heads] planted head offsets
    meta: dict = field(default_factory=dict)


def _batch_phase_offsets(cfg: Config) -> np.ndarray:
    return np.arange(cfg.batch, dtype=np.int64) * cfg.phase_step


def make_workload(cfg: Config, device: str | torch.device = "cpu",
                  store_out: torch.Tensor | None = None) -> Workload:
    """Draw every input of `cfg`.  `store_out`, if given, is a preallocated CPU
    tensor of the store's shape (for example page-locked memory) to fill."""
    rng = np.random.default_rng(cfg.seed)
    D, F, L, d, S = cfg.d_model, cfg.d_ff, cfg.n_layers, cfg.n_dense, cfg.n_sparse
    T, B = cfg.n_tokens, cfg.batch
    tdt = cfg.torch_dtype
    dev = torch.device(device)

    # ---- FFN weights: dense prefix on `device`, sparse layers into the store
    dense_w = None
    if d > 0:
        dense_w = torch.empty((d, cfg.n_proj, F, D), dtype=tdt, device=dev)
        for layer in range(d):
            dense_w[layer] = _torch_normal((cfg.n_proj, F, D), cfg.weight_std, tdt, dev,
                                           cfg.seed * 1000 + layer)
    if store_out is None:
        store = torch.empty((S, F, cfg.n_proj, D), dtype=tdt)
    else:
        assert tuple(store_out.shape) == (S, F, cfg.n_proj, D) and store_out.dtype == tdt
        store = store_out
    for s in range(S):
        layer = d + s
        w = _torch_normal((cfg.n_proj, F, D), cfg.weight_std, tdt, dev,
                          cfg.seed * 1000 + layer)
        store[s].copy_(w.permute(1, 0, 2))
        del w

    # ---- token inputs and predictor -----------------------------------
    phases = offsets = None
    centroids = None
    meta: dict = {}
    if cfg.pred_kind == "shared_argmax":
        C, H, NH = cfg.n_centroids, cfg.pred_hidden, cfg.n_heads
        chains = np.zeros((S, 2, C, cfg.words), dtype=np.uint32)
        for s in range(S):
            for p in range(2):
                chains[s, p] = pack_bits(centroid_chain(rng, F, C, cfg.density,
                                                        cfg.persistence))
        centroids = chains
        x = rng.standard_normal((T, B, D)).astype(np.float32)
        if cfg.planted:
            span = T + int(_batch_phase_offsets(cfg)[-1])
            assert span < C, "planted phases must not wrap"
            assert C <= H, "planted predictor needs one hidden unit per centroid"
            phi0 = int(rng.integers(0, C - span))
            phases = phi0 + np.arange(T)[:, None] + _batch_phase_offsets(cfg)[None, :]
            v = rng.standard_normal((C, D))
            v /= np.linalg.norm(v, axis=1, keepdims=True)
            x = (x + cfg.planted_scale * v[phases]).astype(np.float32)
            offsets = rng.integers(0, C, size=NH)
            w1 = torch.from_numpy(
                np.concatenate([v, rng.standard_normal((H - C, D)) * cfg.pred_std]))
            w2 = rng.standard_normal((NH, C, H)) * cfg.pred_std
            cc = np.arange(C)
            for hd in range(NH):
                w2[hd, cc, (cc - offsets[hd]) % C] += cfg.spike
            w2 = torch.from_numpy(w2.reshape(NH * C, H))
            meta["phi0"] = phi0
        else:
            w1 = torch.from_numpy(rng.standard_normal((H, D)) * cfg.pred_std)
            w2 = torch.from_numpy(rng.standard_normal((NH * C, H)) * cfg.pred_std)
        pred_w1 = w1.to(tdt).to(dev)
        pred_w2 = w2.to(tdt).to(dev)
        pred_b2 = None
    else:
        H = cfg.pred_hidden
        x = rng.standard_normal((T, B, D)).astype(np.float32)
        pred_w1 = torch.empty((L, H, D), dtype=tdt, device=dev)
        pred_w2 = torch.empty((L, F, H), dtype=tdt, device=dev)
        for layer in range(L):
            pred_w1[layer] = _torch_normal((H, D), cfg.pred_std, tdt, dev,
                                           cfg.seed * 1000 + 500 + layer)
            pred_w2[layer] = _torch_normal((F, H), cfg.pred_std, tdt, dev,
                                           cfg.seed * 1000 + 700 + layer)
        # Output bias: neuron n fires with probability ~ r_n ~ Beta(a, b).  The
        # pre-bias output has spread pred_std * sqrt(H * E[relu(g)^2]) with
        # g ~ N(0, pred_std^2 * D), E[relu(g)^2] = var(g) / 2.
        a, b = cfg.rate_beta
        sig = cfg.pred_std * math.sqrt(H * 0.5 * cfg.pred_std ** 2 * D)
        r = np.clip(rng.beta(a, b, size=(L, F)), 1e-6, 1 - 1e-6)
        from scipy.special import ndtri
        b2 = sig * ndtri(r)
        pred_b2 = torch.from_numpy(b2).to(tdt).to(dev)
    x_t = torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    return Workload(cfg=cfg, dense_w=dense_w, store=store, centroids=centroids,
                    pred_w1=pred_w1, pred_w2=pred_w2, pred_b2=pred_b2, x=x_t,
                    phases=phases, offsets=offsets, meta=meta)
