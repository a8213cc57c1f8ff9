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


# --- width resolution, the width ladder and the exactness gate ---------------------

from block_speculative_decoding_dflash_gb300.policy import ExactnessGate, resolve_widths


def test_resolve_widths_follows_the_round_loop_rule():
    """Muse page, "What changed": a depth below the requested width that the
    drafter does not insist on gives a controller between the two; no depth
    (Qwen 3.5 DFlash) or preferring the requested width (DSpark) keeps it."""
    assert resolve_widths(16, 4) == (4, 16)                 # Muse assistant
    assert resolve_widths(16, None) == (16, 16)             # Qwen 3.5 DFlash
    assert resolve_widths(10, 4, prefer_requested=True) == (10, 10)   # DSpark
    assert resolve_widths(4, 8) == (4, 4)                   # depth not below the request
    with pytest.raises(ValueError):
        resolve_widths(1)
    with pytest.raises(ValueError):
        resolve_widths(16, 1)


def test_ladder_challenges_every_width_and_adopts_the_fastest():
    ctl = ThroughputController(4, 16, challenge_every=1, widths=(4, 8, 16))
    assert ctl.probed_verify_widths() == (4, 8, 16)
    rates = {4: 0.030, 8: 0.036, 16: 0.050}
    seen = run(ctl, rates, 12)
    assert set(seen) == {4, 8, 16}
    assert ctl.current == 16                                # settles on the best width
    # a challenger that does not pay is never adopted
    ctl2 = ThroughputController(4, 16, challenge_every=1, widths=(4, 8, 16))
    run(ctl2, {4: 0.04, 8: 0.03, 16: 0.02}, 12)
    assert ctl2.current == 4
    assert all(not adopted for (_, _, _, adopted) in ctl2.history)
    with pytest.raises(ValueError):
        ThroughputController(4, 16, widths=(8, 16))          # must start at the depth
    with pytest.raises(ValueError):
        ctl2.observe(5, 1, 1.0)                              # not a probed width


def test_challenger_order_is_nearest_first():
    ctl = ThroughputController(4, 32, widths=(4, 8, 16, 32))
    assert ctl.challengers() == [8, 16, 32]
    ctl.current = 16
    assert ctl.challengers() == [8, 4, 32]


def test_exactness_gate_needs_every_probed_width_and_names_the_failure():
    """Muse page, "Pre-merge review round", first finding: the gate probed the
    ceiling only while the loop warms up at the depth; the probe declined at
    width 4 as well. Every probed width must pass and the decline names the
    width that failed."""
    results = {4: (False, "162404 of 404096 logit bytes differ"), 16: (True, "")}
    gate = ExactnessGate(probe=lambda w: results[w], model_key=("muse-a", 2048, 5))
    v = gate.allows_every_width((4, 16))
    assert not v.allowed and v.failed_width == 4
    assert "block_size=4" in v.message(16) and "requested 16" in v.message(16)
    assert gate.allows_every_width((16,)).allowed                # the ceiling alone would pass
    # cached per (model, width): no second probe of the same width ...
    calls = gate.calls
    gate.allows_every_width((4, 16))
    assert gate.calls == calls
    # ... but a second checkpoint of the same shape is probed on its own
    other = ExactnessGate(probe=lambda w: (True, ""), model_key=("muse-b", 2048, 5), cache=gate.cache)
    assert other.allows_every_width((4, 16)).allowed
