"""GB300-native entropy-bounded denoising step for block-diffusion language models.

The hot path (per-position softmax / entropy / argmax / Gumbel-max sample, entropy-bound
acceptance, renoise, convergence, and the self-conditioning feedback on tcgen05 tensor cores)
lives in ``libdg.so`` behind the C ABI in ``include/dg.h``; this package is its thin Python
binding (``_native``), the in-tree build (``build``) and the seeded input generator
(``synth``).
"""
from ._native import *  # noqa: F401,F403
from ._native import load, library_path, DGError, params_tensor, pack_params, unpack_params  # noqa: F401
from .build import build as build_library  # noqa: F401
