"""The speculation cost governor: a host policy over measured step times. TEST INFRASTRUCTURE.

[TS] "SpeculationCostGovernor": speculation must never make decoding slower, so
the governor measures speculative against plain steps at run time and parks
drafting while it is losing, re-probing with backoff. The paragraphs on the
shared governor fix its rules:
  * verdicts compare milliseconds per committed token of speculative steps
    against the plain baseline;
  * a probe is eight speculative steps; after a losing verdict a re-probe is
    three steps, and a winning verdict restores the full probe;
  * a loss parks drafting: the first park is 32 tokens, and consecutive losses
    back off (32, 64, 128, up to 256);
  * a win is not a blind hold: speculative steps keep being timed against the
    baseline, and the governor parks as soon as the last eight of them average
    a loss; the hold is re-measured every 64 steps with three plain steps;
  * a probe ends early, as a loss, once four measured speculative steps in a
    row accepted nothing;
  * a step whose drafter proposed nothing is a speculative sample of one token;
  * parked steps feed the plain baseline, except the first, which pays the
    transition;
  * a new request caps whatever park is left at the first interval (32) and
    forgets the backoff; one loss is remembered, so its re-probe is the short
    one;
  * the stats line reports plain and speculative ms per token, wins, losses
    and parked steps.

Readings where the page leaves a choice:
  * the first verdict needs a plain baseline: the governor starts with three
    plain calibration steps (the re-measure size);
  * the plain baseline is the mean ms per token over the last 64 plain samples
    (calibration, re-measure and parked steps);
  * a win needs the speculative ms per token strictly below the baseline;
  * a park counts committed tokens (one per plain step);
  * the hold window of eight and the 64-step re-measure count speculative
    steps taken since the win.
"""
from __future__ import annotations

from dataclasses import dataclass, field

CALIBRATE, PROBE, HOLD, REMEASURE, PARKED = "calibrate", "probe", "hold", "remeasure", "parked"


@dataclass
class GovernorConfig:
    probe_steps: int = 8
    reprobe_steps: int = 3
    first_park: int = 32
    max_park: int = 256
    hold_window: int = 8
    remeasure_every: int = 64
    remeasure_steps: int = 3
    zero_accept_end: int = 4
    baseline_samples: int = 64


@dataclass
class Governor:
    cfg: GovernorConfig = field(default_factory=GovernorConfig)

    def __post_init__(self):
        self.state = CALIBRATE
        self.plain = []                    # (ms, tokens) of recent plain samples
        self.left = self.cfg.remeasure_steps  # steps left in the calibration / re-measure / probe
        self.probe = []                    # (ms, tokens) of the current probe
        self.window = []                   # (ms, tokens) of the last hold steps
        self.zero_streak = 0
        self.next_probe = self.cfg.probe_steps
        self.park_len = self.cfg.first_park
        self.park_left = 0
        self.first_parked = False
        self.hold_steps = 0
        self.wins = self.losses = self.parked_steps = 0
        self.spec_ms = self.spec_tok = 0.0  # every speculative sample, for the stats

    # ------------------------------------------------------------------ the policy
    def speculate(self) -> bool:
        """Whether the next step drafts."""
        return self.state in (PROBE, HOLD)

    def baseline(self):
        """Plain ms per token, or None before any plain sample."""
        if not self.plain:
            return None
        return sum(m for m, _ in self.plain) / sum(t for _, t in self.plain)

    def _add_plain(self, ms, tokens):
        self.plain.append((ms, tokens))
        del self.plain[:-self.cfg.baseline_samples]

    def _start_probe(self):
        self.state, self.left, self.probe, self.zero_streak = PROBE, self.next_probe, [], 0

    def _loss(self):
        self.losses += 1
        self.state = PARKED
        self.park_left = self.park_len
        self.park_len = min(2 * self.park_len, self.cfg.max_park)
        self.first_parked = True
        self.next_probe = self.cfg.reprobe_steps

    def _win(self):
        self.wins += 1
        self.state, self.window, self.hold_steps = HOLD, [], 0
        self.park_len = self.cfg.first_park
        self.next_probe = self.cfg.probe_steps

    def record(self, speculative: bool, ms: float, committed: int, drafted: int, accepted: int) -> None:
        """One finished step: its device time, tokens committed, drafts proposed and accepted. A
        speculative step that proposed nothing is a speculative sample of one token."""
        if speculative:
            tokens = 1 if drafted == 0 else committed
            self.spec_ms += ms
            self.spec_tok += tokens
            if self.state == PROBE:
                self.probe.append((ms, tokens))
                self.zero_streak = self.zero_streak + 1 if accepted == 0 else 0
                self.left -= 1
                if self.zero_streak >= self.cfg.zero_accept_end:
                    self._loss()
                elif self.left == 0:
                    spec = sum(m for m, _ in self.probe) / sum(t for _, t in self.probe)
                    base = self.baseline()
                    self._win() if base is not None and spec < base else self._loss()
            elif self.state == HOLD:
                self.window.append((ms, tokens))
                del self.window[:-self.cfg.hold_window]
                self.hold_steps += 1
                spec = sum(m for m, _ in self.window) / sum(t for _, t in self.window)
                base = self.baseline()
                if len(self.window) == self.cfg.hold_window and base is not None and spec >= base:
                    self._loss()
                elif self.hold_steps >= self.cfg.remeasure_every:
                    self.state, self.left = REMEASURE, self.cfg.remeasure_steps
            return
        # plain step
        if self.state in (CALIBRATE, REMEASURE):
            self._add_plain(ms, committed)
            self.left -= 1
            if self.left == 0:
                if self.state == CALIBRATE:
                    self._start_probe()
                else:
                    self.state, self.hold_steps = HOLD, 0
        elif self.state == PARKED:
            if self.first_parked:
                self.first_parked = False      # the transition step: not a baseline sample
            else:
                self._add_plain(ms, committed)
            self.parked_steps += 1
            self.park_left -= committed
            if self.park_left <= 0:
                self._start_probe()

    def new_request(self) -> None:
        """A new request: cap the park left at the first interval and forget the backoff, keeping
        one loss (so the next re-probe is the short one)."""
        if self.state == PARKED:
            self.park_left = min(self.park_left, self.cfg.first_park)
        self.park_len = self.cfg.first_park

    def stats(self) -> dict:
        base = self.baseline()
        return {"plain_ms_per_tok": base, "spec_ms_per_tok": self.spec_ms / self.spec_tok if self.spec_tok else None,
                "wins": self.wins, "losses": self.losses, "parked": self.parked_steps, "state": self.state}
