"""Plant plausible mistakes in a copy of the oracle and check that every one
of them fails at least one pin.

Each mutation is a textual edit of the oracle's source (a dropped term, a
wrong sign or index, a transposed operand, a swapped clip or boundary
value); the edited source is loaded as a throwaway module on the CPU and
run against the pins of ``tests/pins.py``.  A mutation that survives every
pin would be a hole in the pins.
"""
import types

import pytest

from oracle import rlca_ref
from tests import pins

SOURCE = open(rlca_ref.__file__).read()

MUTATIONS = [
    ("affine: transposed operands", "A = a[:, t] + b[:, t] * A", "A = b[:, t] + a[:, t] * A"),
    ("successor: truncation takes the bootstrap",
     "nxt = np.where(trunc[:, t], tv[:, t], nxt)", "nxt = np.where(trunc[:, t], boot, nxt)"),
    ("successor: termination ignored",
     "np.where(term[:, t], 0.0, nxt)", "np.where(term[:, t], nxt, nxt)"),
    ("continues: truncation does not cut",
     "~(term[:, t] | trunc[:, t])", "~term[:, t]"),
    ("GAE: dropped lambda", "adv[:, t] = delta + gamma * lam *", "adv[:, t] = delta + gamma *"),
    ("GAE: sign of the value", "boot) - v[:, t]\n        adv", "boot) + v[:, t]\n        adv"),
    ("GAE: returns subtract the value", "return adv, adv + v", "return adv, adv - v"),
    ("GAE: value of the same step", "v_next = v[:, t + 1] if t + 1 < T else None\n        delta = r[:, t] + gamma",
     "v_next = v[:, t] if t + 1 < T else None\n        delta = r[:, t] + gamma"),
    ("discounted: dropped gamma",
     "ret[:, t] = r[:, t] + gamma * _successor(t, T, later,",
     "ret[:, t] = r[:, t] + _successor(t, T, later,"),
    ("TD(lambda): value index", "(1.0 - lam) * v[:, t + 1] + lam * later",
     "(1.0 - lam) * v[:, t] + lam * later"),
    ("TD(lambda): swapped weights", "(1.0 - lam) * v[:, t + 1] + lam * later",
     "lam * v[:, t + 1] + (1.0 - lam) * later"),
    ("V-Trace: rho clipped at c_bar", "rho = np.minimum(rho_bar, ratio)", "rho = np.minimum(c_bar, ratio)"),
    ("V-Trace: c clipped at rho_bar", "c = lam * np.minimum(c_bar, ratio)", "c = lam * np.minimum(rho_bar, ratio)"),
    ("V-Trace: c without lambda", "c = lam * np.minimum(c_bar, ratio)", "c = np.minimum(c_bar, ratio)"),
    ("V-Trace: trace uses rho", "gap = delta + gamma * c[:, t]", "gap = delta + gamma * rho[:, t]"),
    ("V-Trace: pg bootstraps from V", "_successor(t, T, later_vs,", "_successor(t, T, v_next,"),
    ("V-Trace: ratio inverted", "np.exp(_f64(logp_target) - _f64(logp_behaviour))",
     "np.exp(_f64(logp_behaviour) - _f64(logp_target))"),
    ("Retrace: trace of the same step", "c[:, t + 1] * (later - q_taken[:, t + 1])",
     "c[:, t] * (later - q_taken[:, t + 1])"),
    ("Retrace: Q of the taken action instead of E_pi Q", "ev[:, t + 1] + c[:, t + 1]",
     "q_taken[:, t + 1] + c[:, t + 1]"),
    ("Retrace: inverted ratio", "np.minimum(1.0, p_taken / _f64(mu_a))",
     "np.minimum(1.0, _f64(mu_a) / p_taken)"),
    ("Retrace: E_pi Q without pi", "ev = np.sum(P * Q, axis=-1)", "ev = np.sum(Q, axis=-1) / A"),
    ("Retrace: no lambda", "c = lam * np.minimum(1.0", "c = np.minimum(1.0"),
    ("eligibility: reset keyed on the same step", "else done[:, t - 1]\n        prev",
     "else done[:, t]\n        prev"),
    ("eligibility: dropped lambda", "prev = xs[:, t] + gamma * lam *", "prev = xs[:, t] + gamma *"),
    ("prefix sum: exclusive ignored", "out[:, t] = before if exclusive else running",
     "out[:, t] = running if exclusive else running"),
    ("prefix sum: start flag read one step late",
     "starts = np.ones(E, bool) if t == 0 else flag[:, t]\n",
     "starts = np.ones(E, bool) if t == 0 else flag[:, t - 1]\n"),
    ("prefix sum: end flag read on the same step",
     "starts = np.ones(E, bool) if t == 0 else flag[:, t - 1]\n",
     "starts = np.ones(E, bool) if t == 0 else flag[:, t]\n"),
]


def _mutant(old, new):
    assert SOURCE.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(SOURCE.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, old, new):
    mod = _mutant(old, new)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mod)
        except (AssertionError, FloatingPointError, ValueError, IndexError, TypeError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches: {name}"
