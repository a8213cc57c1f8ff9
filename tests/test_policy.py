"""The verify-width controller on synthetic measurements (CPU)."""

import pytest

from block_speculative_decoding_dflash_gb300.policy import ThroughputController


def run(ctl, rate_of, windows):
    seen = []
    for _ in range(windows):
        w = ctl.next_width()
        seen.append(w)
        ctl.observe(w, tokens=int(rate_of[w] * 100), ms=100.0)
    return seen


def test_starts_at_depth_and_keeps_it_when_the_ceiling_does_not_pay():
    """Muse page: 16-row challenge windows measured lower tokens/ms and were
    not adopted."""
    ctl = ThroughputController(4, 16, window=32, challenge_every=3)
    seen = run(ctl, {4: 0.035, 16: 0.018}, 12)
    assert seen[0] == 4
    assert 16 in seen                   # the ceiling is challenged ...
    assert ctl.current == 4             # ... and not adopted
    assert seen.count(16) == 3


def test_widens_when_the_ceiling_pays():
    ctl = ThroughputController(4, 16, challenge_every=2)
    seen = run(ctl, {4: 0.030, 16: 0.045}, 8)
    assert seen[:3] == [4, 4, 16]
    assert ctl.current == 16 and seen[3] == 16
    # and the depth is re-challenged later
    assert seen.count(4) >= 3


def test_fixed_width_when_depth_equals_ceiling():
    ctl = ThroughputController(8, 8)
    assert run(ctl, {8: 1.0}, 5) == [8] * 5


def test_rejects_bad_parameters():
    with pytest.raises(ValueError):
        ThroughputController(1, 16)
    with pytest.raises(ValueError):
        ThroughputController(8, 4)


def test_probed_widths_cover_the_warm_up_depth_and_the_ceiling():
    assert ThroughputController(4, 16).probed_verify_widths() == (4, 16)
    assert ThroughputController(8, 8).probed_verify_widths() == (8,)
    c = ThroughputController(4, 16, window=2, challenge_every=1)
    # whatever the controller adopts stays inside the probed set
    for rate in (1.0, 2.0, 2.0, 3.0, 3.0, 1.0):
        w = c.next_width()
        c.observe(w, int(rate * 10), 10.0)
        assert w in c.probed_verify_widths() and c.current in c.probed_verify_widths()
