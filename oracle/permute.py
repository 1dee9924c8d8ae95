"""Oracle re-layout (test infrastructure; see the package docstring).

"Window-Aligned Sequence Parallelism (SeedVR2)", §Motivation and §Plan A
redistribution: when every token stays on the same device (SP=1), a layout
boundary is a local permutation of rows.  Row q of the destination layout
holds canonical token ids_dst[q]; that token sits at row pos_src[id] of the
source layout, where pos_src is the inverse of ids_src.  Rows are copied
bit for bit.
"""
import numpy as np


def inverse(ids):
    """pos[ids[q]] = q."""
    pos = np.empty_like(ids)
    pos[ids] = np.arange(ids.size, dtype=ids.dtype)
    return pos


def permute_rows(src, ids_src, ids_dst):
    """dst[q] = src[pos_src[ids_dst[q]]] -- an exact row copy."""
    return src[inverse(ids_src)[ids_dst]].copy()
