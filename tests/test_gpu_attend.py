"""GPU parity of the standalone attention entry point (dec_attend) against the
oracle's brute-force attention, over KV rings with and without a window, with
several split counts and ragged last splits."""

import numpy as np
import pytest
import torch

from oracle import attend_ref

pytestmark = pytest.mark.gpu

CASES = [
    # (n_heads, n_kv_heads, head_dim, max_seq, sliding_window, pos)
    (4, 2, 16, 40, 0, 0),
    (4, 2, 16, 40, 0, 39),
    (4, 2, 16, 300, 0, 299),      # 3 splits of 100
    (9, 3, 64, 640, 0, 5),
    (9, 3, 64, 640, 0, 639),      # 5 splits
    (14, 2, 64, 2304, 0, 1000),   # group of 7
    (32, 8, 128, 4096, 4096, 100),
    (32, 8, 128, 4096, 4096, 5000),   # wrapped ring: all 4096 slots readable
    (8, 8, 128, 257, 257, 1000),      # MHA, ragged split tail
    (8, 1, 64, 130, 0, 129),          # MQA
]


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    return dec


def _inputs(nq, nkv, hd, max_seq, kv_dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(nq, hd, generator=g)
    k = torch.randn(max_seq, nkv, hd, generator=g)
    v = torch.randn(max_seq, nkv, hd, generator=g)
    k, v = k.to(kv_dtype), v.to(kv_dtype)
    return q, k, v


@pytest.mark.parametrize("kv_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("case", CASES)
def test_attend_matches_oracle(dec_mod, case, kv_dtype):
    nq, nkv, hd, max_seq, sw, pos = case
    q, k, v = _inputs(nq, nkv, hd, max_seq, kv_dtype, seed=hash(case) & 0xFFFF)
    out = torch.empty(nq, hd, device="cuda")
    scratch = torch.empty(dec_mod.attend_scratch_bytes(nq, nkv, hd, max_seq), dtype=torch.uint8, device="cuda")
    dec_mod.attend(q.cuda(), k.cuda(), v.cuda(), pos, sw, out, scratch)
    torch.cuda.synchronize()
    m = min(pos + 1, max_seq) if sw > 0 else pos + 1
    ref = attend_ref(q.double().numpy(), k[:m].double().numpy(), v[:m].double().numpy(), nq, nkv)
    np.testing.assert_allclose(out.cpu().numpy(), ref, atol=1e-5, rtol=1e-5)


def test_attend_argument_errors(dec_mod):
    q = torch.zeros(4, 16, device="cuda")
    k = torch.zeros(8, 2, 16, device="cuda")
    out = torch.empty(4, 16, device="cuda")
    scratch = torch.empty(dec_mod.attend_scratch_bytes(4, 2, 16, 8), dtype=torch.uint8, device="cuda")
    with pytest.raises(dec_mod.DecError) as e:
        dec_mod.attend(q, k, k, 8, 0, out, scratch)      # pos beyond capacity, no window
    assert e.value.status == dec_mod.DEC_EINVAL
    with pytest.raises(dec_mod.DecError) as e:
        dec_mod.attend(q, k, k, 3, 0, out, scratch[:16])
    assert e.value.status == dec_mod.DEC_ENOMEM
    with pytest.raises(dec_mod.DecError) as e:
        # A 8-slot ring under a 16-position window cannot hold the window once it wraps.
        dec_mod.attend(q, k, k, 8, 16, out, scratch)
    assert e.value.status == dec_mod.DEC_EINVAL
    dec_mod.attend(q, k, k, 7, 16, out, scratch)          # still below max_seq: accepted
    torch.cuda.synchronize()
