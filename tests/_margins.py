"""Achieved errors of the parity tests, printed at the end of the run.

Tests call ``record(name, err, tol)``; tests/conftest.py prints every
recorded error beside its tolerance in pytest's terminal summary, so the
margins to each bar are visible in the log of a passing run.
"""
RECORDS = []


def record(name: str, err: float, tol: float) -> float:
    RECORDS.append((name, float(err), float(tol)))
    return float(err)
