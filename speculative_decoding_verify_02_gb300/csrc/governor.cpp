// Speculation cost governor: a host-side policy that decides, step by step, whether the next
// verify step drafts, from the measured device time of past steps.
//
// [TS] SpeculationCostGovernor: speculation must never make decoding slower, so the governor
// times speculative against plain steps and parks drafting while it is losing, re-probing with
// backoff. The rules it keeps (the shared-governor paragraphs of that page):
//   - verdicts compare ms per committed token of speculative steps with the plain baseline;
//   - a probe is probe_steps (8) speculative steps; after a loss a re-probe is reprobe_steps (3);
//     a win restores the full probe;
//   - a loss parks drafting for first_park (32) tokens, doubling on each further loss up to
//     max_park (256);
//   - after a win the governor keeps timing speculative steps and parks as soon as the last
//     hold_window (8) of them average a loss; every remeasure_every (64) speculative steps it
//     takes remeasure_steps (3) plain steps to refresh the baseline;
//   - a probe ends early, as a loss, after zero_accept_end (4) speculative steps in a row that
//     accepted nothing;
//   - a speculative step that proposed nothing counts as a speculative sample of one token;
//   - parked steps feed the plain baseline, except the first (it pays the transition);
//   - a new request caps the park left at first_park and forgets the backoff, keeping one loss.
// Where the page leaves a choice: the governor starts with remeasure_steps plain calibration
// steps; the baseline is the mean ms per token of the last baseline_samples (64) plain samples;
// a win needs speculative ms per token strictly below the baseline; parks count committed tokens.
#include <algorithm>
#include <deque>
#include <new>
#include <utility>

#include "sdv.h"

struct sdv_governor {
    enum State { CALIBRATE = 0, PROBE = 1, HOLD = 2, REMEASURE = 3, PARKED = 4 };
    sdv_governor_cfg cfg{};
    State state = CALIBRATE;
    std::deque<std::pair<double, double>> plain;  // (ms, tokens) of the recent plain samples
    std::deque<std::pair<double, double>> window; // the last hold steps
    double probe_ms = 0, probe_tok = 0;
    int left = 0, zero_streak = 0, next_probe = 0, park_len = 0, park_left = 0, hold_steps = 0;
    bool first_parked = false;
    int wins = 0, losses = 0, parked_steps = 0;
    double spec_ms = 0, spec_tok = 0;

    double baseline() const {
        double m = 0, t = 0;
        for (const auto &s : plain) m += s.first, t += s.second;
        return t > 0 ? m / t : -1.0;
    }
    void add_plain(double ms, double tok) {
        plain.emplace_back(ms, tok);
        while (static_cast<int>(plain.size()) > cfg.baseline_samples) plain.pop_front();
    }
    void start_probe() {
        state = PROBE;
        left = next_probe;
        probe_ms = probe_tok = 0;
        zero_streak = 0;
    }
    void loss() {
        ++losses;
        state = PARKED;
        park_left = park_len;
        park_len = std::min(2 * park_len, cfg.max_park);
        first_parked = true;
        next_probe = cfg.reprobe_steps;
    }
    void win() {
        ++wins;
        state = HOLD;
        window.clear();
        hold_steps = 0;
        park_len = cfg.first_park;
        next_probe = cfg.probe_steps;
    }
    void record(bool spec, double ms, int committed, int drafted, int accepted) {
        if (spec) {
            const double tok = drafted == 0 ? 1.0 : static_cast<double>(committed);
            spec_ms += ms;
            spec_tok += tok;
            if (state == PROBE) {
                probe_ms += ms;
                probe_tok += tok;
                zero_streak = accepted == 0 ? zero_streak + 1 : 0;
                --left;
                if (zero_streak >= cfg.zero_accept_end) {
                    loss();
                } else if (left == 0) {
                    const double base = baseline();
                    if (base >= 0 && probe_ms / probe_tok < base) win();
                    else loss();
                }
            } else if (state == HOLD) {
                window.emplace_back(ms, tok);
                while (static_cast<int>(window.size()) > cfg.hold_window) window.pop_front();
                ++hold_steps;
                double m = 0, t = 0;
                for (const auto &s : window) m += s.first, t += s.second;
                const double base = baseline();
                if (static_cast<int>(window.size()) == cfg.hold_window && base >= 0 && m / t >= base) {
                    loss();
                } else if (hold_steps >= cfg.remeasure_every) {
                    state = REMEASURE;
                    left = cfg.remeasure_steps;
                }
            }
            return;
        }
        if (state == CALIBRATE || state == REMEASURE) {
            add_plain(ms, committed);
            if (--left == 0) {
                if (state == CALIBRATE) {
                    start_probe();
                } else {
                    state = HOLD;
                    hold_steps = 0;
                }
            }
        } else if (state == PARKED) {
            if (first_parked) first_parked = false;
            else add_plain(ms, committed);
            ++parked_steps;
            park_left -= committed;
            if (park_left <= 0) start_probe();
        }
    }
};

extern "C" {

int sdv_governor_create(const sdv_governor_cfg *cfg, sdv_governor **out) {
    if (!out) return SDV_ERR_ARG;
    sdv_governor_cfg c{8, 3, 32, 256, 8, 64, 3, 4, 64};
    if (cfg) c = *cfg;
    if (c.probe_steps < 1 || c.reprobe_steps < 1 || c.first_park < 1 || c.max_park < c.first_park ||
        c.hold_window < 1 || c.remeasure_every < 1 || c.remeasure_steps < 1 || c.zero_accept_end < 1 ||
        c.baseline_samples < 1)
        return SDV_ERR_ARG;
    sdv_governor *g = new (std::nothrow) sdv_governor();
    if (!g) return SDV_ERR_ARG;
    g->cfg = c;
    g->left = c.remeasure_steps;
    g->next_probe = c.probe_steps;
    g->park_len = c.first_park;
    *out = g;
    return SDV_OK;
}

int sdv_governor_destroy(sdv_governor *g) {
    delete g;
    return SDV_OK;
}

int sdv_governor_decide(sdv_governor *g, int32_t *h_speculate) {
    if (!g || !h_speculate) return SDV_ERR_ARG;
    *h_speculate = (g->state == sdv_governor::PROBE || g->state == sdv_governor::HOLD) ? 1 : 0;
    return SDV_OK;
}

int sdv_governor_record(sdv_governor *g, int speculative, float ms, int committed, int drafted, int accepted) {
    if (!g || !(ms >= 0.f) || committed < 0 || drafted < 0 || accepted < 0 || accepted > drafted) return SDV_ERR_ARG;
    g->record(speculative != 0, ms, committed, drafted, accepted);
    return SDV_OK;
}

int sdv_governor_new_request(sdv_governor *g) {
    if (!g) return SDV_ERR_ARG;
    if (g->state == sdv_governor::PARKED) g->park_left = std::min(g->park_left, g->cfg.first_park);
    g->park_len = g->cfg.first_park;
    return SDV_OK;
}

int sdv_governor_stats(sdv_governor *g, sdv_governor_report *out) {
    if (!g || !out) return SDV_ERR_ARG;
    out->plain_ms_per_tok = static_cast<float>(g->baseline());
    out->spec_ms_per_tok = g->spec_tok > 0 ? static_cast<float>(g->spec_ms / g->spec_tok) : -1.f;
    out->wins = g->wins;
    out->losses = g->losses;
    out->parked_steps = g->parked_steps;
    out->state = static_cast<int>(g->state);
    return SDV_OK;
}

}  // extern "C"
