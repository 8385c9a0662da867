"""Host processes that run the oracle on whole sequences of a decode workload.

Each worker regenerates one sequence from the seeded recipe (inputs.py) and
returns the oracle's fp64 decode for every KV head of it (a one-head oracle
cache per head, filled from the same bf16 values).  Started with the "spawn"
method, so they are safe to use from a process that has used the GPU.
Nothing here computes any of the method's arithmetic; the oracle does.
"""
import numpy as np

import oracle
from nvfp4_quantized_paged_quantize_gb300 import inputs


def oracle_sequence(args):
    """(workload index, sequence b, k global scale, v global scale) ->
    (b, out [Hkv, G, 128] float64)."""
    index, b, gk, gv = args
    wl = inputs.decode_config(index)
    k, v = wl.prompt_kv(b)
    if wl.append:
        nk, nv = wl.new_kv()
        k = np.concatenate([k, nk[b:b + 1]])
        v = np.concatenate([v, nv[b:b + 1]])
    q = wl.q()
    L = k.shape[0]
    npg = (L + 15) // 16
    G = wl.num_q_heads // wl.num_kv_heads
    outs = []
    for h in range(wl.num_kv_heads):
        c = oracle.Cache(max(npg, 1), 1, 128, 16, gk, gv)
        assert oracle.quantize_append(c, np.ascontiguousarray(k[:, h:h + 1]), np.ascontiguousarray(v[:, h:h + 1]),
                                      np.arange(L, dtype=np.int64)) == 0
        qh = np.ascontiguousarray(q[b:b + 1, h * G:(h + 1) * G])
        pt = np.arange(max(npg, 1), dtype=np.int32)[None, :]
        out, st = oracle.decode_attention(c, qh, pt, np.array([L], np.int32), wl.softmax_scale)
        assert st == 0
        outs.append(out[0])
    return b, np.stack(outs)


def oracle_workload(index, gk, gv, batches, processes):
    """Oracle decode of the given sequences of a workload, one spawned process
    per sequence at a time; returns {b: out [Hkv, G, 128]}."""
    import multiprocessing as mp

    with mp.get_context("spawn").Pool(processes) as pool:
        return dict(pool.map(oracle_sequence, [(index, b, gk, gv) for b in batches]))
