"""Tiled dense GEMM (C = A·B, fp16/bf16 in, fp32 accumulate) for NVIDIA GB300 (sm_103a).

The compute path is the CUDA library ``libdtgemm.so`` behind the C ABI in
``include/gemm.h``; :mod:`.native` binds it with ctypes.  PyTorch provides device
memory and streams only.
"""
from .native import (CONFIG_128x64, CONFIG_128x128, CONFIG_128x256, CONFIG_256x256, CONFIG_AUTO, Gemm, GemmError,
                     LAYOUT_NN, LAYOUT_TN, OPT_CONFIG, OPT_FAULT_INJECT, OPT_HOST_COL_CHUNKS, OPT_HOST_ROW_CHUNKS,
                     OPT_K_SNAKE, OPT_MAX_CTAS, OPT_RASTER_GROUP, OPT_SK_MIN_BLOCKS, OPT_SPLIT_MIN_BLOCKS,
                     OPT_STREAM_K, OPT_TIMEOUT_NS, empty_output, load, matmul)

__all__ = ["Gemm", "GemmError", "matmul", "load", "empty_output", "LAYOUT_NN", "LAYOUT_TN",
           "OPT_CONFIG", "OPT_TIMEOUT_NS", "OPT_MAX_CTAS", "OPT_RASTER_GROUP", "OPT_FAULT_INJECT", "OPT_STREAM_K",
           "OPT_HOST_ROW_CHUNKS", "OPT_HOST_COL_CHUNKS", "OPT_SK_MIN_BLOCKS", "OPT_SPLIT_MIN_BLOCKS", "OPT_K_SNAKE",
           "CONFIG_AUTO", "CONFIG_128x256", "CONFIG_128x128", "CONFIG_256x256", "CONFIG_128x64"]
