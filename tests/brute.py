"""Brute-force attention with Python lists and math.exp (test helper).

An independent second route to the op's result, used only to pin the oracle
on tiny inputs.  It takes the K/V rows of one sequence already gathered into
contiguous lists (no page table) and plain Python floats, and writes out the
definition with explicit positions:

    row r of a call with R rows over a sequence of final length L sits at
    position L - R + r and sees keys 0 .. L - R + r (kern manifest v7,
    $defs.Fill `seq_len`); query head h reads KV head h // (H / Hkv).
    With a sliding window W > 0 (a RAD_KV_WINDOW group, Radiance architecture
    plugins, "Declare: buffers and KV groups") it sees only keys
    max(0, position - W + 1) .. position.

    Tree verify ("Adding a model", step 4: forward_tree): with parents given,
    the call's R rows are draft-tree nodes flattened parents-first (parents[r]
    < r, or -1 for a node hanging off the cached context), and row r sees the
    cached keys 0 .. L - R - 1 plus the keys of the nodes on its own path to
    the context, itself included.
"""
import math


def _path(parents, r):
    """Node r and its ancestors, walked up the parents list to the context."""
    nodes = []
    while r >= 0:
        nodes.append(r)
        r = parents[r]
    return nodes


def attend_sequence(q_rows, keys, values, scale, n_head_kv, window=0, parents=None):
    """q_rows: [R][H][D] floats; keys/values: [L][Hkv][D] floats.

    Returns out [R][H][D] as floats.
    """
    R = len(q_rows)
    H = len(q_rows[0])
    L = len(keys)
    group = H // n_head_kv
    out = []
    for r in range(R):
        position = L - R + r
        first = max(0, position - window + 1) if window > 0 else 0
        visible = range(first, position + 1)
        if parents is not None:
            visible = list(range(L - R)) + sorted(L - R + i for i in _path(parents, r))
        row_out = []
        for h in range(H):
            kvh = h // group
            logits = []
            for j in visible:
                acc = 0.0
                for a, b in zip(q_rows[r][h], keys[j][kvh]):
                    acc += a * b
                logits.append(scale * acc)
            top = max(logits)
            ex = [math.exp(x - top) for x in logits]
            total = sum(ex)
            D = len(values[0][kvh])
            vec = [0.0] * D
            for j, e in zip(visible, ex):
                wgt = e / total
                vj = values[j][kvh]
                for d in range(D):
                    vec[d] += wgt * vj[d]
            row_out.append(vec)
        out.append(row_out)
    return out
