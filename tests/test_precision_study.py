"""The operand-precision study (oracle/precision_study.py) on a small model, CPU only:
the all-exact variant is the reference itself, (hi, lo) pairs carry ~16 bits so their
error is far below a single bf16's, and the rounding helper is the round-to-nearest-even
bf16 of the value."""

import numpy as np

from decoder_only_forward_gb300 import synthetic
from oracle import precision_study as ps


def test_bf16_round_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 3.0e-3, 0.0])
    r = ps.bf16_round(x)
    assert r[0] == 1.0
    assert r[1] == 1.0                      # halfway between 1 and 1 + 2^-7: to even (1)
    assert r[2] == 1.0 + 2 ** -7            # above halfway: up
    assert r[3] == -2.5 and r[5] == 0.0
    assert abs(r[4] - 3.0e-3) <= 3.0e-3 * 2 ** -8     # half a unit of the 7 stored bits
    hilo = ps.apply(np.array([np.pi]), "hilo")[0]
    assert abs(hilo - np.pi) < np.pi * 2 ** -16 < abs(ps.bf16_round(np.pi) - np.pi)


def test_study_orders_variants_on_a_toy():
    w = synthetic.workload("toy")
    src = synthetic.OracleWeightSource(w, device="cpu", cache=True)
    res = ps.study(w, src, P=12, rows=4, variants=ps.variants_default(), log=lambda m: None)
    assert res["exact"] == (0.0, 0.0)
    assert res["hilo_all"][0] < 1e-4
    for name in ("bf16_qkv", "bf16_o", "bf16_gateup", "bf16_down", "bf16_attn"):
        assert res[name][0] > 10 * res["hilo_all"][0], name
    assert res["bf16_all"][0] >= max(res[n][0] for n in ("bf16_qkv", "bf16_o")) * 0.5
