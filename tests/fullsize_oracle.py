"""Oracle side of the full-size parity tests: one (layer, group, row, head) slice.

Runs in a worker process (spawned, so it never inherits a CUDA context).  The
slice's KV comes from synth.looped_kv_slice; the oracle compresses it into a
one-row, one-head cache whose region layout equals the device cache's (the
layout depends on loops, head width, group size and capacity only) and attends
over it for every loop of the group, the anchor loop's call also appending
the current token (as the benchmark's step does).
"""
from __future__ import annotations

import numpy as np

import oracle
import synth


def slice_job(args):
    (w, seed, layer, group, b, h, ntok, capacity, seq_len, chained, q, k_cur, v_cur, scale) = args
    _, kv = synth.looped_kv_slice(seed, w, ntok, layer, group, b, h)
    R = synth.rotation(w.head_dim).astype(np.float32).astype(np.float64)
    P = w.loops_per_group
    geom = oracle.Geometry(1, P, 1, 1, w.head_dim, w.group_size, 1, capacity)
    buf = np.zeros(geom.total_bytes, dtype=np.uint8)
    oracle.append(buf, geom, R, 0, 0, kv[:, :, None, None], np.zeros(1, dtype=np.int64), chained=chained)
    outs = []
    for loop in range(P - 1):
        o = oracle.decode_attention(buf, geom, R, 0, 0, loop, q[loop][None, None], k_cur[loop][None, None],
                                    v_cur[loop][None, None], [seq_len], scale, chained=chained)
        outs.append(o[0, 0])
    # the anchor loop's call also appends the current token of every loop at slot seq_len
    kv_cur = np.stack([k_cur, v_cur], axis=1)[:, :, None, None, :]        # [P, 2, 1, 1, d]
    o, ok = oracle.decode_attention_append(buf, geom, R, 0, 0, q[P - 1][None, None], kv_cur, [seq_len], scale,
                                           chained=chained)
    assert ok.all()
    outs.append(o[0, 0])
    return buf, np.stack(outs)
