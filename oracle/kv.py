"""KV-cache compaction after acceptance (oracle; test infrastructure only).

"大模型推理 memory bandwidth bound (5) - Medusa", 二.7
update_inference_inputs(): the accepted path's rows (tree node indices
``nodes``, root first, ``acc + 1`` of them) sit at ``prefix + nodes`` in the
cache; they are gathered and written to rows prefix .. prefix+acc, and the
current length becomes prefix + acc + 1. The gather reads the cache as it
was before any write (index-gather semantics, as a tensor copy has).
"""
from __future__ import annotations

import numpy as np


def kv_compact(cache, prefix_len, nodes):
    """Return (new cache, new length) for cache [..., S, D] along axis -2."""
    nodes = np.asarray(nodes, dtype=np.int64)
    out = np.array(cache, copy=True)
    src = np.asarray(cache)[..., prefix_len + nodes, :]
    out[..., prefix_len: prefix_len + len(nodes), :] = src
    return out, prefix_len + len(nodes)
