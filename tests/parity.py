"""Comparison helpers for the GPU parity tests (CUDA path vs oracle on the same bytes).

Decision rule: a discrete output (token id, accepted length, eval mask, L_j) must equal the
oracle's unless the oracle's decision margin is below MARGIN; such decisions are counted as
excluded.  Continuous outputs must agree within RTOL relative (ATOL absolute floor for values
near zero)."""
import numpy as np

MARGIN = 1e-5
RTOL = 1e-5


class Tally:
    def __init__(self):
        self.total = 0
        self.excluded = 0

    def check_fraction(self):
        # under 0.01% of decisions, or at most one when fewer than 10^4 were made
        if self.total >= 10_000:
            assert self.excluded <= 1e-4 * self.total, (self.excluded, self.total)
        else:
            assert self.excluded <= 1, (self.excluded, self.total)


def close(got, ref, rtol=RTOL, atol=1e-6, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bad = ~(np.abs(got - ref) <= rtol * np.abs(ref) + atol)
    bad &= ~(np.isnan(got) & np.isnan(ref))
    assert not bad.any(), f"{what}: {int(bad.sum())} values off; first {got[bad][:5]} vs {ref[bad][:5]}"


def compare_block(tally, got_tok, got_lse, got_zat, ref, T, j=None):
    """One request's sampled block vs the oracle's (tokens, lse, zat, margins).  Returns the
    number of leading positions that agree (comparison stops after an excluded decision)."""
    rtok, rlse, rzat, rmg = ref
    for i in range(len(rtok)):
        tally.total += 1
        if got_tok[i] != rtok[i]:
            assert rmg[i] < MARGIN, f"request {j} position {i + 1}: token {got_tok[i]} vs {rtok[i]} (margin {rmg[i]})"
            tally.excluded += 1
            return i
        if T > 0:
            close([got_lse[i]], [rlse[i]], what=f"draft_lse j={j} i={i + 1}")
        else:
            assert np.isnan(got_lse[i])
        close([got_zat[i]], [rzat[i]], what=f"z_at_tok j={j} i={i + 1}")
    return len(rtok)
