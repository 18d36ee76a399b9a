"""The seeded synthetic inputs keep the recipe they state: centroid chains
with an exact popcount and a per-link persistence, refills drawn from bits
unset in the previous mask, little-endian bit packing, a deterministic draw
per seed, and the bundled record layout of the host store."""
import numpy as np
import torch

from workloads import SMALL_OPT, TINY, make_workload
from workloads.synth import centroid_chain, pack_bits


def test_centroid_chain_popcount_and_persistence():
    rng = np.random.default_rng(5)
    f, n_masks, density, p = 4096, 60, 0.25, 0.83
    m = centroid_chain(rng, f, n_masks, density, p)
    n = int(round(density * f))
    assert m.shape == (n_masks, f) and m.dtype == bool
    assert (m.sum(axis=1) == n).all()
    shared = (m[1:] & m[:-1]).sum(axis=1) / n
    # each bit survives one link with probability p; refills come from bits
    # unset in the previous mask, so the overlap is exactly the survivors
    assert abs(shared.mean() - p) < 0.01
    assert shared.min() > p - 0.05 and shared.max() < p + 0.05


def test_centroid_chain_persistence_extremes():
    rng = np.random.default_rng(9)
    keep_all = centroid_chain(rng, 1000, 5, 0.1, 1.0)
    assert (keep_all == keep_all[0]).all()
    fresh = centroid_chain(rng, 1000, 5, 0.1, 0.0)
    assert not (fresh[1:] & fresh[:-1]).any()        # nothing survives, refills avoid old bits
    assert (fresh.sum(axis=1) == 100).all()


def test_pack_bits_is_little_endian_per_word():
    rng = np.random.default_rng(3)
    for f in (1, 31, 32, 33, 100, 1000):
        bits = rng.random((3, f)) < 0.3
        words = pack_bits(bits)
        assert words.dtype == np.uint32 and words.shape == (3, (f + 31) // 32)
        for r in range(3):
            for nbit in range(f):
                assert bool((int(words[r, nbit // 32]) >> (nbit % 32)) & 1) == bool(bits[r, nbit])
            if f % 32:  # the padding bits of the last word are zero
                assert int(words[r, -1]) >> (f % 32) == 0


def test_same_seed_same_inputs_other_seed_other_inputs():
    a, b = make_workload(TINY), make_workload(TINY)
    for name in ("x", "store", "pred_w1", "pred_w2", "dense_w"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert np.array_equal(a.centroids, b.centroids)
    c = make_workload(TINY.replace(seed=TINY.seed + 1))
    assert not torch.equal(a.x, c.x) and not np.array_equal(a.centroids, c.centroids)


def test_store_holds_bundled_records():
    wl = make_workload(TINY)
    cfg = wl.cfg
    assert tuple(wl.store.shape) == (cfg.n_sparse, cfg.d_ff, 3, cfg.d_model)
    assert wl.store.is_contiguous() and not wl.store.is_cuda
    # one record = gate | up | down^T rows of one neuron, contiguous
    assert wl.store[0, 5].numel() * wl.store.element_size() == cfg.record_bytes
    opt = make_workload(SMALL_OPT)
    assert opt.store.shape[2] == 2 and opt.pred_b2 is not None       # up | down^T, per-layer predictor


def test_full_size_workloads_start_from_a_prompt_warm_fill():
    # every full-size shape decodes a 128-token prompt (its first token is
    # the cold start) before the 256 generated tokens; the benchmark times
    # only generated tokens, after the transient that follows a cold start
    from workloads import CONFIGS
    full = [c for c in CONFIGS.values() if c.d_model >= 4096]
    assert {c.name for c in full} >= {"llama2-7b-relu", "llama2-13b-relu", "opt-6.7b-window",
                                      "llama2-7b-batch8"}
    for c in full:
        assert c.n_warm == 128, c.name
        assert c.n_decode == 256, c.name
