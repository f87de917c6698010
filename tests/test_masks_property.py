"""Property tests (CPU): the library's host mask builders against the oracle's
token-level definitions on random schedules and parameters."""
import numpy as np
import pytest
from hypothesis import HealthCheck, given, settings, strategies as st

import oracle
import visual_autoregressive_next_var_b300 as V
from tests.test_abi import _csr_to_token_mask


@st.composite
def schedules(draw):
    """Increasing sides: a sink prefix (side <= sink), then multiples of 8 up to 48."""
    sink = draw(st.sampled_from([2, 4, 8]))
    head = [s for s in (1, 2, 3, 4, 6, 8) if s <= sink]
    n_head = draw(st.integers(1, len(head)))
    tail_pool = [s for s in (8, 12, 16, 20, 24, 32, 40, 48) if s > sink]
    tail = sorted(draw(st.lists(st.sampled_from(tail_pool), min_size=1, max_size=4, unique=True)))
    return tuple(head[:n_head] + tail), sink


@settings(max_examples=25, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(schedules(), st.integers(0, 3))
def test_static_mask_matches_oracle(sched, radius):
    sides, sink = sched
    step = len(sides) - 1
    if sides[step] % 8:
        return
    p = V.problem(1, 1, 64, sides)
    rp, en, sink_len = V.var_block_mask_build(p, step, 8, radius, sink)
    got = _csr_to_token_mask(sides, step, 8, rp, en, sink_len)
    ref = oracle.block_mask_rows(oracle.mask_spec(sides, step, 8, radius, sink), 0, sides[step] ** 2)
    assert np.array_equal(got, ref.astype(bool))


@settings(max_examples=25, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(schedules(), st.floats(0.0, 1.0), st.integers(0, 2 ** 31 - 1), st.data())
def test_dynamic_mask_matches_oracle(sched, tau, seed, data):
    sides, sink = sched
    cand = [i for i, s in enumerate(sides) if s > sink and s % 8 == 0]
    if not cand:
        return
    d = data.draw(st.sampled_from(cand))
    targets = [i for i in range(d, len(sides)) if sides[i] % 8 == 0]
    k_step = data.draw(st.sampled_from(targets))
    p = V.problem(1, 1, 64, sides)
    U, n_sink = V.var_sparvar_units(p, d, sink)
    _, units, ns = oracle.sparvar_units(sides, d, sink)
    assert (U, n_sink) == (len(units), ns)
    rng = np.random.default_rng(seed)
    A = rng.random(((sides[d] // 8) ** 2, U))
    A[:, rng.integers(0, U, size=U // 3)] = 0.25       # equal scores
    rp, en, sink_len = V.var_sparvar_mask_build(p, d, k_step, sink, A, tau)
    got = _csr_to_token_mask(sides, k_step, 8, rp, en, sink_len)
    ref = oracle.sparvar_keep_mask(sides, d, k_step, units, oracle.sparvar_select(A, ns, tau), sink)
    assert np.array_equal(got, ref.astype(bool))
