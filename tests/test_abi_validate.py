"""np_init_model checks its description before any CUDA call: every rule
that include/np.h states for np_model_desc turns a bad description into
NP_ERR_ARG with a message, on a machine without a GPU, and nothing is
created.  Pointers are placeholders: the checks only test them for null."""
import ctypes

import pytest
import torch

from sparse_activation_decode_gb300 import _lib as L

FAKE = 0x10000  # a non-null placeholder; never dereferenced by the checks


def valid_desc(**kw):
    d = L.ModelDesc()
    d.n_layers, d.n_dense, d.d_model, d.d_ff, d.k_max, d.n_centroids = 4, 1, 256, 1024, 256, 16
    d.dtype, d.has_gate, d.combine, d.residency, d.window, d.batch = L.NP_F16, 1, L.NP_COMBINE_UNION, \
        L.NP_RES_SLOTMAP, 1, 1
    d.staging_rows, d.pred_hidden, d.pred_kind = 0, 512, L.NP_PRED_SHARED_ARGMAX
    d.h2d_mode, d.activation, d.slots, d.lookahead = L.NP_H2D_FUSED, 0, L.NP_SLOTS_REUSE, 0
    d.host_store = d.dense_w = d.pred_w1 = d.pred_w2 = d.centroids = FAKE
    d.pred_b2 = None
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.fixture(scope="module")
def lib():
    from sparse_activation_decode_gb300.build import build
    build()
    return L.load()


BAD = {
    "no layers": dict(n_layers=0),
    "dense > layers": dict(n_dense=5),
    "65 sparse layers": dict(n_layers=66, n_dense=1),
    "bad dtype": dict(dtype=3),
    "d_model too small": dict(d_model=4),
    "row not 16-byte multiple": dict(d_model=260),
    "d_model too large": dict(d_model=16384),
    "d_ff zero": dict(d_ff=0),
    "d_ff too large": dict(d_ff=16385),
    "k_max above d_ff": dict(k_max=1025),
    "k_max zero": dict(k_max=0),
    "has_gate 2": dict(has_gate=2),
    "bad combine": dict(combine=7),
    "bad residency": dict(residency=9),
    "window 0": dict(residency=L.NP_RES_WINDOW, window=0),
    "window 33": dict(residency=L.NP_RES_WINDOW, window=33),
    "batch 0": dict(batch=0),
    "batch 9": dict(batch=9),
    "batched f32": dict(batch=2, dtype=L.NP_F32),
    "batched per-layer predictor": dict(batch=2, pred_kind=L.NP_PRED_PERLAYER_SIGMOID, pred_b2=FAKE),
    "batched d_model not /128": dict(batch=2, d_model=320),
    "batched hidden not /64": dict(batch=2, pred_hidden=96),
    "batched window reuse": dict(batch=2, residency=L.NP_RES_WINDOW, window=5),
    "batched frequency reuse": dict(batch=2, residency=L.NP_RES_FREQUENCY),
    "staging above k_max": dict(staging_rows=257),
    "bad h2d_mode": dict(h2d_mode=5),
    "bad activation": dict(activation=3),
    "swiglu without gate": dict(activation=1, has_gate=0),
    "bad slots": dict(slots=4),
    "lookahead with shared predictor": dict(lookahead=1),
    "negative lookahead": dict(lookahead=-1),
    "hidden zero": dict(pred_hidden=0),
    "dense_w null": dict(dense_w=None),
    "host_store null": dict(host_store=None),
    "predictor null": dict(pred_w2=None),
    "shared predictor without dense layer": dict(n_dense=0, dense_w=None),
    "no centroids": dict(centroids=None),
    "per-layer predictor without bias": dict(pred_kind=L.NP_PRED_PERLAYER_SIGMOID),
    "bad pred_kind": dict(pred_kind=2),
}


@pytest.mark.parametrize("name", list(BAD))
def test_bad_description_is_rejected_before_cuda(lib, name):
    out = ctypes.c_void_p()
    d = valid_desc(**BAD[name])
    assert lib.np_init_model(ctypes.byref(d), ctypes.byref(out)) == L.NP_ERR_ARG, name
    assert not out.value
    lib.np_last_error.restype = ctypes.c_char_p
    assert lib.np_last_error(), name


def test_null_out_is_rejected(lib):
    d = valid_desc()
    assert lib.np_init_model(ctypes.byref(d), None) == L.NP_ERR_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_valid_description_reaches_cuda_and_fails_cleanly_without_a_gpu(lib):
    # the description passes every check; the first CUDA call then fails and
    # the call returns NP_ERR_CUDA with no model
    out = ctypes.c_void_p()
    d = valid_desc()
    assert lib.np_init_model(ctypes.byref(d), ctypes.byref(out)) == L.NP_ERR_CUDA
    assert not out.value
    d = valid_desc(pred_kind=L.NP_PRED_PERLAYER_SIGMOID, n_dense=0, dense_w=None, pred_b2=FAKE,
                   residency=L.NP_RES_WINDOW, window=5, has_gate=0, lookahead=2, slots=L.NP_SLOTS_COMPACT)
    assert lib.np_init_model(ctypes.byref(d), ctypes.byref(out)) == L.NP_ERR_CUDA


_INTS = (ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint32)


@pytest.mark.parametrize("name", sorted(n for n, (res, args) in L.SIGNATURES.items()
                                        if args and res is ctypes.c_int32 and n != "np_status_str"))
def test_every_entry_point_rejects_null_arguments(lib, name):
    # a null model (and null buffers, zero sizes) is an argument error, not a
    # crash; freeing a null model is a no-op
    res, args = L.SIGNATURES[name]
    vals = [0 if a in _INTS else None for a in args]
    if name == "np_ffn_rows_noalloc_check":
        # its only argument is a stream, and NULL (the default stream) is a
        # valid one: without a GPU the call fails in CUDA, cleanly
        assert getattr(lib, name)(*vals) in (L.NP_OK, L.NP_ERR_CUDA)
        return
    expected = L.NP_OK if name == "np_free_model" else L.NP_ERR_ARG
    assert getattr(lib, name)(*vals) == expected


@pytest.mark.parametrize("case", ["y is h", "y inside h", "y inside down", "y over the row list",
                                  "unaligned y", "row_limit 0", "d_model 4"])
def test_noalloc_rejects_bad_arguments_before_cuda(lib, case):
    # np_ffn_rows_noalloc: y may share no byte with its inputs (it is cleared
    # on the stream before they are read), pointers are 16-byte aligned and
    # sizes in range; all checked on the host before any CUDA call.
    D = 256
    h, g, u, d, rows, y = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000
    n_rows, limit, dm = 10, 100, D
    if case == "y is h":
        y = h
    elif case == "y inside h":
        y = h + 512
    elif case == "y inside down":
        y = d + 100 * D * 2 - 16          # the last 16 bytes of a 100-row f16 block
    elif case == "y over the row list":
        y = rows - 16
    elif case == "unaligned y":
        y = 0x600008
    elif case == "row_limit 0":
        limit = 0
    elif case == "d_model 4":
        dm = 4
    st = lib.np_ffn_rows_noalloc(h, g, u, d, rows, n_rows, limit, dm, L.NP_F16, 1, y, None)
    assert st == L.NP_ERR_ARG
