"""Oracle pins: dynamic loss scaling and the skip rule ("DeepSpeed ZeRO 优化"
§六 Loss Scaling, §九 Q6)."""
import pytest

import oracle
from tests._golden import rows


@pytest.mark.parametrize("row", rows("loss_scale_sequence.txt"))
def test_loss_scale_sequence(row):
    n, s0, flags, scales, steps = row
    sc = oracle.Scaler(float(s0), int(n))
    got_s, got_t = [], []
    for f in flags.split(","):
        sc.update(int(f))
        got_s.append(sc.scale)
        got_t.append(sc.step)
    assert got_s == [float(x) for x in scales.split(",")]
    assert got_t == [int(x) for x in steps.split(",")]
