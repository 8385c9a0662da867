"""The pools a format variant's append writes, built from the oracle's block
functions row by row at each slot (the expected side of the variant tests).
Variant ids follow the library's: 1 stochastic rounding, 2 Hadamard, 3 MXFP4."""
import numpy as np

import oracle
from nvfp4_quantized_paged_quantize_gb300 import inputs

SR, HADAMARD, MXFP4 = 1, 2, 3


def oracle_variant_pools(variant, k, v, slots, pages, H, gk=1.0, gv=1.0, rk=None, rv=None):
    """{"k": (data [rows, 64], scales [rows, 8 or 4]), "v": ...} for bf16 bits k, v [n, H, 128]."""
    rows = pages * H * 16
    nsc = 4 if variant == MXFP4 else 8
    out = {t: (np.zeros((rows, 64), np.uint8), np.zeros((rows, nsc), np.uint8)) for t in "kv"}
    for t, slot in enumerate(slots):
        if slot < 0 or slot >= pages * 16:
            continue
        for h in range(H):
            row = ((slot // 16) * H + h) * 16 + slot % 16
            for name, bits, g, rnd in (("k", k, gk, rk), ("v", v, gv, rv)):
                x = inputs.bf16_bits_to_f32(bits[t, h])
                data, scale = out[name]
                if variant == MXFP4:
                    for j in range(4):
                        packed, sc = oracle.mxfp4_quantize_block(x[32 * j:32 * j + 32])
                        data[row, 16 * j:16 * j + 16] = packed
                        scale[row, j] = sc
                    continue
                if variant == HADAMARD:
                    x = oracle.hadamard(x)
                for j in range(8):
                    blk = x[16 * j:16 * j + 16]
                    if variant == SR:
                        packed, sc = oracle.quantize_block_sr(blk, g, rnd[t, h, 16 * j:16 * j + 16])
                    else:
                        packed, sc = oracle.quantize_block(blk, g)
                    data[row, 8 * j:8 * j + 8] = packed
                    scale[row, j] = sc
    return out
