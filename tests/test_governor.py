"""The speculation cost governor: hand-worked scenarios from [TS]'s governor
paragraphs pin the oracle (oracle/governor.py); the library's native governor
(sdv_governor_*, host code, no GPU work) must then make the oracle's decision at
every step of random traces.

Scenarios (plain steps 10 ms per token unless stated):
  A. [TS] "four matchless steps park an n-gram drafter ... it re-probes within 32
     steps": three calibration steps, a probe ended early by four speculative
     steps that proposed nothing, parks of 32, 64, 128, 256, 256 tokens, each
     followed by a short three-step re-probe that loses.
  B. [TS] "a win is not a blind hold": a probe at 5 ms per token wins; after 64
     held steps three plain steps re-measure the baseline; when drafts stop
     being accepted (20 ms per token) the window of the last eight steps
     crosses the baseline after six such steps and the governor parks for the
     first interval, 32.
  C. [TS] "a new request caps whatever park is left at the first interval and
     forgets the backoff (one loss is remembered, so the re-probe stays the
     short one)": mid-way through a 64-token park a new request leaves 32
     tokens of park, the re-probe is three steps, and its loss parks 32.
"""
import numpy as np
import pytest

from oracle.governor import Governor as OracleGovernor

PLAIN = (10.0, 1, 0, 0)                 # ms, committed, drafted, accepted
MATCHLESS = (15.0, 1, 0, 0)             # a speculative step whose lookup proposed nothing
GOOD = (20.0, 4, 7, 3)                  # 5 ms per token
BAD = (20.0, 1, 7, 0)                   # 20 ms per token


def _drive(gov, script, decide, record):
    """Run `script` (callables step -> step tuple by decision) and return the decisions."""
    out = []
    for pick in script:
        d = decide(gov)
        out.append(int(d))
        record(gov, d, *pick(d))
    return out


def _oracle_decide(g):
    return g.speculate()


def _oracle_record(g, d, ms, c, dr, ac):
    g.record(d, ms, c, dr, ac)


def _steps(n, spec_step, plain_step=PLAIN):
    return [lambda d, s=spec_step, p=plain_step: s if d else p] * n


def test_scenario_a_matchless_drafter_parks_with_backoff():
    g = OracleGovernor()
    dec = _drive(g, _steps(3 + 4 + 32 + 3 + 64 + 3 + 128 + 3 + 256 + 3 + 256, MATCHLESS), _oracle_decide,
                 _oracle_record)
    expect = ([0] * 3 + [1] * 4 + [0] * 32 + [1] * 3 + [0] * 64 + [1] * 3 + [0] * 128 + [1] * 3 + [0] * 256 +
              [1] * 3 + [0] * 256)
    assert dec == expect
    s = g.stats()
    assert s["losses"] == 5 and s["wins"] == 0 and s["parked"] == 32 + 64 + 128 + 256 + 256
    assert s["plain_ms_per_tok"] == pytest.approx(10.0) and s["spec_ms_per_tok"] == pytest.approx(15.0)


def test_scenario_b_win_hold_remeasure_then_park():
    g = OracleGovernor()
    script = _steps(3, GOOD) + _steps(8, GOOD) + _steps(64, GOOD) + _steps(3, GOOD) + _steps(10, GOOD)
    script += _steps(6, BAD) + _steps(32, BAD) + _steps(3, BAD)
    dec = _drive(g, script, _oracle_decide, _oracle_record)
    expect = [0] * 3 + [1] * 8 + [1] * 64 + [0] * 3 + [1] * 10 + [1] * 6 + [0] * 32 + [1] * 3
    assert dec == expect
    s = g.stats()
    assert s["wins"] == 1 and s["losses"] == 2 and s["state"] == "parked"


def test_scenario_c_new_request_caps_the_park():
    g = OracleGovernor()
    dec = _drive(g, _steps(3 + 4 + 32 + 3 + 10, MATCHLESS), _oracle_decide, _oracle_record)
    assert dec[-10:] == [0] * 10 and g.park_left == 54     # ten steps into the 64-token park
    g.new_request()
    dec = _drive(g, _steps(32 + 3 + 32 + 3, MATCHLESS), _oracle_decide, _oracle_record)
    assert dec == [0] * 32 + [1] * 3 + [0] * 32 + [1] * 3


def test_library_governor_matches_oracle_on_random_traces():
    """The native governor against the oracle, step by step, on random mixes of step costs,
    acceptance, empty proposals and new requests, under default and custom settings."""
    from speculative_decoding_verify_02_gb300 import Governor, GovernorCfg
    from oracle.governor import GovernorConfig
    cfgs = [None, (5, 2, 16, 64, 4, 20, 2, 3, 16)]
    for ci, cv in enumerate(cfgs):
        for seed in range(6):
            rng = np.random.default_rng(100 * ci + seed)
            lib = Governor(GovernorCfg(*cv) if cv else None)
            ora = OracleGovernor(GovernorConfig(*cv) if cv else GovernorConfig())
            plain_ms = rng.uniform(5, 15)
            for step in range(1500):
                if rng.random() < 0.01:
                    lib.new_request()
                    ora.new_request()
                d = lib.decide()
                assert d == ora.speculate(), (ci, seed, step)
                if d:
                    drafted = int(rng.integers(0, 8))
                    accepted = int(rng.integers(0, drafted + 1)) if rng.random() < 0.6 else 0
                    committed = accepted + 1
                    ms = float(rng.uniform(0.8, 2.5) * plain_ms)
                else:
                    drafted = accepted = 0
                    committed = 1
                    ms = float(rng.uniform(0.9, 1.1) * plain_ms)
                ms = float(np.float32(ms))                       # the library takes float32
                lib.record(d, ms, committed, drafted, accepted)
                ora.record(d, ms, committed, drafted, accepted)
            a, b = lib.stats(), ora.stats()
            assert (a["wins"], a["losses"], a["parked"], a["state"]) == (b["wins"], b["losses"], b["parked"],
                                                                          b["state"])
            assert a["plain_ms_per_tok"] == pytest.approx(b["plain_ms_per_tok"], rel=1e-5)
            lib.close()
