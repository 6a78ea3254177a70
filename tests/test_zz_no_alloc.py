"""dec_attend_noalloc: the attention entry point for callers that cannot
allocate device memory themselves (a plug-in inside a framework whose pooled
allocator owns the GPU, or a path where cudaMalloc may not be called).

Called through the C ABI with ctypes, twice in a row (the shared fixed
scratch keeps the first call's contents), and compared with the oracle's
brute-force attention and with dec_attend on a caller buffer, within the
attention tolerance of the other tests.  This file
sorts last so that a run stopping at its first failure has run everything else.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import attend_ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    return dec


def _call_noalloc(dec_mod, q, k, v, pos, sw, out, stream):
    max_seq, nkv, hd = k.shape
    kvd = dec_mod.DEC_F32 if k.dtype == torch.float32 else dec_mod.DEC_BF16
    return dec_mod.lib.dec_attend_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.shape[0], nkv, hd, max_seq,
                                          sw, kvd, pos, out.data_ptr(), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("kv_dtype", [torch.float32, torch.bfloat16])
def test_noalloc_matches_dec_attend_twice(dec_mod, kv_dtype):
    stream = torch.cuda.Stream()
    calls = [(32, 8, 128, 4096, 4096, 5000, 11), (9, 3, 64, 640, 0, 300, 12)]
    for nq, nkv, hd, max_seq, sw, pos, seed in calls:
        g = torch.Generator().manual_seed(seed)
        q = torch.randn(nq, hd, generator=g).cuda()
        k = torch.randn(max_seq, nkv, hd, generator=g).to(kv_dtype).cuda()
        v = torch.randn(max_seq, nkv, hd, generator=g).to(kv_dtype).cuda()
        ref = torch.empty(nq, hd, device="cuda")
        scratch = torch.empty(dec_mod.attend_scratch_bytes(nq, nkv, hd, max_seq), dtype=torch.uint8,
                              device="cuda")
        dec_mod.attend(q, k, v, pos, sw, ref, scratch, stream)
        m = min(pos + 1, max_seq) if sw > 0 else pos + 1
        brute = attend_ref(q.double().cpu().numpy(), k[:m].double().cpu().numpy(),
                           v[:m].double().cpu().numpy(), nq, nkv)
        for _ in range(2):   # two calls in a row on the shared scratch
            out = torch.full((nq, hd), float("nan"), device="cuda")
            st = _call_noalloc(dec_mod, q, k, v, pos, sw, out, stream)
            assert st == dec_mod.DEC_OK, dec_mod.lib.dec_last_error(None)
            stream.synchronize()
            np.testing.assert_allclose(out.cpu().numpy(), brute, atol=1e-5, rtol=1e-5)
            np.testing.assert_allclose(out.cpu().numpy(), ref.cpu().numpy(), atol=1e-5, rtol=1e-5)


def test_noalloc_rejects_sizes_beyond_its_scratch(dec_mod):
    q = torch.zeros(128, 128, device="cuda")
    k = torch.zeros(8192, 16, 128, device="cuda")
    out = torch.empty(128, 128, device="cuda")
    st = _call_noalloc(dec_mod, q, k, k, 10, 0, out, torch.cuda.current_stream())
    assert st == dec_mod.DEC_EINVAL
    assert b"1 MiB" in dec_mod.lib.dec_last_error(None)
