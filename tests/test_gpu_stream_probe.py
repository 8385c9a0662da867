"""The streaming probe reads exactly the page-heads a decode reads.

The probe (a measurement aid: the decode's memory stream with no attention
math) XORs the first 128 bytes of every stage it consumes into a sink word.
With random pool bytes, that XOR is checked against the XOR of the page-heads
the batch covers, computed on the host: any page read twice, skipped or read
from the wrong place changes it.
"""
import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import dev, status_word

pytestmark = pytest.mark.gpu


def _xor_words(a):
    return int(np.bitwise_xor.reduce(np.ascontiguousarray(a).view(np.uint32).reshape(-1))) if a.size else 0


@pytest.mark.parametrize("lens,hkv", [([101, 258], 2), ([8193] * 3, 8), ([0, 1, 17, 5000, 33], 4),
                                      (list(np.random.default_rng(3).integers(0, 3000, 40)), 8)])
def test_probe_reads_each_page_head_once(cuda_lib, lens, hkv):
    wl = inputs.DecodeWorkload("custom", 1, np.array(lens, np.int64), False, hkv, hkv, inputs.KVDist(),
                               pool_factor=1.3)
    rng = np.random.default_rng(11)
    pool = rng.integers(0, 256, (wl.num_pages, hkv, kv.NVFP4KV_PAGE_HEAD_BYTES), dtype=np.uint8)
    cache = kv.Cache(dev(pool), wl.num_pages, hkv)
    pt, sl = dev(wl.page_table), dev(wl.seq_lens.astype(np.int32))
    first = pool[:, :, :128]
    pattern = 0                                          # every (sequence, KV head, page) page-head
    pages = 0                                            # every (sequence, page): the page's first 128 bytes
    for b, n in enumerate(wl.pages_per_seq):
        ids = wl.page_table[b, :n]
        pattern ^= _xor_words(first[ids])
        pages ^= _xor_words(pool[ids, 0, :128])
    for mode, want in ((kv.NVFP4KV_PROBE_DECODE_PATTERN, pattern), (kv.NVFP4KV_PROBE_WHOLE_PAGES, pages)):
        sink = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = status_word()
        kv.nvfp4kv_stream_probe(cache, pt, sl, sink, mode, device_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert (int(sink.item()) & 0xFFFFFFFF) == want, mode
