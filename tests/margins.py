"""Worst observed parity errors, collected across a test session.

Each parity check records (quantity, worst value, bound) under the test that
ran it; conftest.py prints the table at the end of the session, so a passing
run still shows how much room each kernel leaves under its bound.
"""
import contextlib
import os

_ROWS = {}
_OFF = [0]


def _test_id() -> str:
    cur = os.environ.get("PYTEST_CURRENT_TEST", "")
    return cur.split(" (")[0] if cur else "-"


def record(quantity: str, value: float, bound):
    if _OFF[0]:
        return
    key = (_test_id(), quantity)
    old = _ROWS.get(key)
    if old is None or value > old[0]:
        _ROWS[key] = (float(value), bound)


def rows():
    return [(t, q, v, b) for (t, q), (v, b) in sorted(_ROWS.items())]


def worst_by_quantity():
    out = {}
    for (t, q), (v, b) in _ROWS.items():
        if q not in out or v > out[q][0]:
            out[q] = (v, b, t)
    return out


@contextlib.contextmanager
def suspended():
    """Checks run inside this block record nothing (tests of the checks)."""
    _OFF[0] += 1
    try:
        yield
    finally:
        _OFF[0] -= 1
