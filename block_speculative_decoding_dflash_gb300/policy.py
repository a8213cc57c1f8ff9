"""Verify-width policy of the round loop (host side, no kernel).

"Muse Glimmer DFlash assistant drafter on the round loop", "What changed"
(round loop bullet) and "Real-checkpoint validation" item 5: the Muse
assistant starts at its declared depth of 4 rows and widens to the requested
ceiling (16) only when a measurement window pays for it in tokens per
millisecond. This controller does that with two widths: it runs windows of
``window`` rounds at the current width, and every ``challenge_every`` windows
runs one window at the other width; the other width is adopted when its
tokens/ms beats the current width's last window.
"""

from __future__ import annotations


class ThroughputController:
    def __init__(self, depth: int = 4, ceiling: int = 16, window: int = 32,
                 challenge_every: int = 4):
        if depth < 2 or ceiling < depth or window < 1 or challenge_every < 1:
            raise ValueError("bad controller parameters")
        self.depth, self.ceiling = depth, ceiling
        self.window, self.challenge_every = window, challenge_every
        self.current = depth
        self.rate = {}
        self.since_challenge = 0
        self.history = []          # (width, tokens, ms, adopted)

    def probed_verify_widths(self) -> tuple:
        """Every width a run can settle on: the warm-up depth and the
        ceiling ("Pre-merge review round", the exactness-gate finding: a check
        made at one width says nothing about another, so anything that must
        hold at the widths the loop runs at has to be checked at all of
        these)."""
        return tuple(sorted({self.depth, self.ceiling}))

    def other(self) -> int:
        return self.ceiling if self.current == self.depth else self.depth

    def next_width(self) -> int:
        """Width of the next measurement window."""
        if self.depth == self.ceiling:
            return self.current
        if self.since_challenge >= self.challenge_every and self.current in self.rate:
            return self.other()
        return self.current

    def observe(self, width: int, tokens: int, ms: float) -> None:
        """Feed the emitted tokens and elapsed ms of one finished window."""
        rate = tokens / ms if ms > 0 else 0.0
        adopted = False
        if width == self.current:
            self.rate[width] = rate
            self.since_challenge += 1
        else:
            self.rate[width] = rate
            if rate > self.rate.get(self.current, float("inf")):
                self.current = width
                adopted = True
            self.since_challenge = 0
        self.history.append((width, tokens, ms, adopted))
