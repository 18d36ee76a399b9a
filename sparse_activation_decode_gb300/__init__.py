"""GB300-native per-token sparse-MLP decode path (predictive delta prefetching).

The compute runs in the CUDA library built from csrc/ (see build.py); this
package only marshals arguments to its C ABI (include/np.h).
"""
from ._lib import NpError, load  # noqa: F401
from .decoder import SparseDecoder, decoder_for, ffn_rows_noalloc, ffn_rows_noalloc_check  # noqa: F401

__all__ = ["SparseDecoder", "decoder_for", "ffn_rows_noalloc", "ffn_rows_noalloc_check", "NpError", "load"]
