"""Seeded draft-tree inputs shared by the oracle pins and the GPU tests.

A draft tree of R proposals is flattened parents-first: parents[r] < r, or -1
for a node that hangs directly off the cached context.  The op takes one mask
word per node with bit i set for every node i on the node's path (itself
included).  This module only builds those inputs; it computes nothing of the
op.
"""
import numpy as np


def path_of(parents, r):
    """Nodes from r up to the cached context, r first."""
    path = []
    while r >= 0:
        path.append(r)
        r = parents[r]
    return path


def mask_words(parents):
    """Tree-mask word of every node: bit i for each node on its path."""
    return np.array([sum(1 << i for i in path_of(parents, r)) for r in range(len(parents))],
                    dtype=np.uint32)


def random_parents(rng, R, forest=True):
    lo = -1 if forest else 0
    return [-1] + [int(rng.integers(lo, r)) for r in range(1, R)]


def chain(R):
    return list(range(-1, R - 1))
