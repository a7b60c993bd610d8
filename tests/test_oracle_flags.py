"""Pins of the oracle's flagged draws (R8: a draw within 1e-6 of a decision
boundary is flagged, and the parity tests stop comparing tokens bit for bit
from its output slot on). The boundary cases are built from the uniforms the
oracle itself draws, so a flag that never fires, fires at the wrong slot or
uses an absolute instead of a mass-relative margin fails here."""
import numpy as np
import pytest

from oracle import spec_oracle as O

SEED = 0x5EED1234


def test_coin_margin():
    assert O.coin_flagged(0.5, 0.5)
    assert O.coin_flagged(0.5, 0.5 + 9e-7) and O.coin_flagged(0.5, 0.5 - 9e-7)
    assert not O.coin_flagged(0.5, 0.5 + 2e-6) and not O.coin_flagged(0.5, 0.5 - 2e-6)


@pytest.mark.parametrize("scale", [1.0, 1000.0, 1e-3])
def test_inverse_cdf_margin_is_relative_to_the_mass(scale):
    w = np.array([0.25, 0.25, 0.5]) * scale   # cumulative 0.25, 0.5, 1.0 of the mass
    x, fl = O.inverse_cdf(w, 0.25)            # exactly on the first step
    assert x == 1 and fl
    x, fl = O.inverse_cdf(w, 0.25 + 5e-7)     # inside the margin, above it
    assert x == 1 and fl
    x, fl = O.inverse_cdf(w, 0.5 - 5e-7)      # inside the margin, below the next step
    assert x == 1 and fl
    x, fl = O.inverse_cdf(w, 0.25 + 1e-5)     # clear of both steps
    assert x == 1 and not fl
    x, fl = O.inverse_cdf(w, 0.75)
    assert x == 2 and not fl


def _two_token_request(p0, q0, d):
    """One request, one draft: V = 2 logits whose softmax at T = 1 is
    (p0, 1 - p0) for the target and (q0, 1 - q0) for the draft."""
    target = np.log(np.array([[p0, 1 - p0], [0.5, 0.5]]))
    draft = np.log(np.array([[q0, 1 - q0]]))
    return O.verify_linear(target, draft, np.array([d]), np.array([0, 1]), np.array([1.0]),
                           SEED, max_k=1)


def test_coin_on_the_acceptance_ratio_flags_slot_zero():
    u = O.uniform(SEED, 0, 1, O.STREAM_COIN)
    q0 = 0.9
    r = _two_token_request(u * q0, q0, 0)      # a = p(d)/q(d) = u up to rounding
    assert abs(r["pq"][0, 0] / r["pq"][0, 1] - u) < 1e-12
    assert r["flag_slot"][0] == 0
    # the same coin against a ratio 0.01 away is not flagged at slot 0
    a = u + 0.01 if u < 0.5 else u - 0.01
    r = _two_token_request(a * q0, q0, 0)
    assert r["flag_slot"][0] != 0


def test_bonus_draw_on_a_cdf_step_flags_its_slot():
    """A request without drafts: the bonus draw from p_1 at u(seed, 0, 1, 2)
    with p = (u, 1 - u) puts u*Z on the first cumulative."""
    u = O.uniform(SEED, 0, 1, O.STREAM_BONUS)
    target = np.log(np.array([[u, 1 - u]]))
    draft = np.zeros((0, 2))
    r = O.verify_linear(target, draft, np.zeros(0, dtype=np.int64), np.array([0, 0]),
                        np.array([1.0]), SEED, max_k=0)
    assert r["accepted"][0] == 0 and r["flag_slot"][0] == 0
    # moved off the step: not flagged
    v = u + 0.01 if u < 0.5 else u - 0.01
    target = np.log(np.array([[v, 1 - v]]))
    r = O.verify_linear(target, draft, np.zeros(0, dtype=np.int64), np.array([0, 0]),
                        np.array([1.0]), SEED, max_k=0)
    assert r["flag_slot"][0] == -1


def test_greedy_requests_are_never_flagged():
    """Greedy decisions compare integers (argmax) and draw nothing."""
    u = O.uniform(SEED, 0, 1, O.STREAM_COIN)
    target = np.log(np.array([[u, 1 - u], [0.5 + 1e-9, 0.5 - 1e-9]]))
    draft = np.log(np.array([[u, 1 - u]]))
    r = O.verify_linear(target, draft, np.array([0]), np.array([0, 1]), np.array([0.0]),
                        SEED, max_k=1)
    assert r["flag_slot"][0] == -1


def _one_child_tree(p0, q0):
    """A root with one child (token 0): target rows of the root and the
    child, the root's draft row; V = 2, T = 1."""
    target = np.log(np.array([[p0, 1 - p0], [0.5, 0.5]]))
    draft = np.log(np.array([[q0, 1 - q0], [0.5, 0.5]]))
    return O.verify_tree(target, draft, np.array([-1, 0]), np.array([-1, 0]),
                         np.array([0, 2]), np.array([1.0]), SEED, 1)


def test_tree_coin_on_the_acceptance_ratio_flags_depth_zero():
    """The child's coin is keyed by its node index (1); with a = p(x)/q(x)
    equal to it, the root's decision is flagged."""
    u = O.uniform(SEED, 0, 1, O.STREAM_COIN)
    q0 = 0.9
    assert _one_child_tree(u * q0, q0)["flag_slot"][0] == 0
    a = u + 0.01 if u < 0.5 else u - 0.01
    assert _one_child_tree(a * q0, q0)["flag_slot"][0] != 0
