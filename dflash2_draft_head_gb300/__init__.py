"""DFlash2 draft-head hot path on GB300 (sm_103a).

The CUDA library (libdflash2.so, C ABI in include/dflash2.h) implements the
grouped dynamic depthwise causal convolution (also fused with the prediction
of its taps from its input), the top-K candidate extraction
that feeds the selector, and the candidate selector (projection,
codebook-gathered edge scores, per-predecessor argmax) and the greedy chain
readout with its p_min cut, of
ggml-org/llama.cpp PR #27342, "spec : add DFlash2 support (local convolution
+ candidate selector)".  This package is the thin Python binding over it.
"""
from .binding import (Dflash2Error, chain, dynconv, dynconv_predicted, edges, lib,  # noqa: F401
                      predict_delta, probe_gather, project, project_noalloc,
                      project_workspace_bytes, select, select_plan,
                      take_device_faults, topk, version)
from .build import build as build_library  # noqa: F401
