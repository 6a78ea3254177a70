"""A bounded device wait that runs out reports DEC_ETIMEOUT and leaves the handle usable.

rml "The decoder", One forward pass: errors come back to the caller as a status.
Every spin-wait in the library's kernels gives up after a time limit instead of
hanging the GPU.  dec_selftest_wait_timeout enters the persistent step's own grid
barrier on a one-CTA grid that expects two arrivals, with a short limit: the wait
runs out, the kernel records the site and returns.  No fault, trap or endless loop
is involved."""

import numpy as np
import pytest
import torch

from decoder_only_forward_gb300 import synthetic
from tests.gpu_helpers import gpu_greedy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return dec


@pytest.mark.parametrize("mode", ["off", "grid"])
def test_wait_runs_out_then_handle_decodes_normally(dec_mod, mode):
    w = synthetic.workload("toy")
    prompt = synthetic.prompt_tokens(w, 12, seed=4)
    ref = dec_mod.Decoder(w)
    ref.set_fused(mode)
    rows_ref, taus_ref = gpu_greedy(ref, prompt, 6)

    d = dec_mod.Decoder(w, weights=ref.weights)
    d.set_fused(mode)
    lg = torch.empty(w["vocab"], device="cuda")
    d.prefill(prompt[:5], 0, lg)
    d.selftest_wait_timeout(2000)          # 2 ms, then the kernel gives up and returns
    with pytest.raises(dec_mod.DecError) as ei:
        d.check()
    assert ei.value.status == dec_mod.DEC_ETIMEOUT
    assert f"site {dec_mod.DEC_SITE_SELFTEST}" in str(ei.value)
    d.check()                              # the error was reported once and cleared
    # The same handle then runs a whole sequence, on the schedule whose barrier timed out.
    d.kv_reset()
    rows, taus = gpu_greedy(d, prompt, 6)
    assert taus == taus_ref
    np.testing.assert_array_equal(rows, rows_ref)


def test_limit_out_of_range_rejected_on_host(dec_mod):
    w = synthetic.workload("toy")
    d = dec_mod.Decoder(w)
    for bad in (0, -5, 100001):
        with pytest.raises(dec_mod.DecError) as ei:
            d.selftest_wait_timeout(bad)
        assert ei.value.status == dec_mod.DEC_EINVAL
    d.check()
