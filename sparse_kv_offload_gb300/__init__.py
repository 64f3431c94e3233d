"""GB300-native sparse-KV decode step: landmark scoring of real and speculative
queries, per-KV-head top-k, cross-query union and miss resolution, host-to-HBM
chunk gather into a layer-scoped ping-pong buffer, and split-K GQA attention
over the selected rows.  The compute runs in the CUDA library ``libdd`` (C ABI,
declared in ``include/dd.h``); ``sparse_kv_offload_gb300.dd`` is its thin
Python binding."""
