"""GB300 (sm_103a) hyper-connection low-rank mix block.

The block of ONNX Runtime PR #33384 "HyperConnectionLowRankMix", computed by
hand-written CUDA kernels behind the C ABI in include/hc_lowrank_mix.h.
``lowrank_mix`` is the Python entry point; the library is loaded on first use
and must have been built (``hyper_connection_rank_gb300.build.build()``).
"""
from ._binding import (HC_FLAG_FORCE_GENERAL, HC_FLAG_WEIGHTS_STATIC, HC_PATH_DECODE, HC_PATH_GENERAL,
                       HC_PATH_NONE, HC_PATH_PREFILL, PATH_NAMES, HcError, attrs_default, debug_sigmoid_exact,
                       debug_sigmoid_table, debug_sigmoid_table_f16, debug_wait_timeout, debug_wait_timeouts, engram_gate, inv_rms, load_library, lowrank_mix, path,
                       workspace_size)

__all__ = ["lowrank_mix", "inv_rms", "engram_gate", "path", "workspace_size", "attrs_default", "load_library", "debug_wait_timeouts",
           "debug_wait_timeout", "debug_sigmoid_exact", "debug_sigmoid_table_f16", "debug_sigmoid_table",
           "HcError", "HC_FLAG_WEIGHTS_STATIC", "HC_FLAG_FORCE_GENERAL", "HC_PATH_NONE", "HC_PATH_DECODE",
           "HC_PATH_PREFILL", "HC_PATH_GENERAL", "PATH_NAMES"]
