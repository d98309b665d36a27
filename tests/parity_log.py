"""Per-test parity figures, printed in pytest's terminal summary.

The checks in moe_check.py add one entry per call: the near-tie counts of the
routing check (boundary near-ties, where the oracle's k-th and (k+1)-th
probabilities differ by less than 1e-6; slot-order near-ties inside the
top-k; and how many tokens the GPU actually chose or ordered differently) and
the output check's max|err| / RMS(oracle).  conftest.py prints the table at
the end of the run, so a test log shows every figure the bounds were
checked against.
"""
from __future__ import annotations

import os

ENTRIES: list[tuple[str, str, dict]] = []


def current_test() -> str:
    name = os.environ.get("PYTEST_CURRENT_TEST", "?")
    return name.rsplit(" ", 1)[0]


def record(kind: str, **fields) -> None:
    ENTRIES.append((current_test(), kind, fields))


def lines() -> list[str]:
    out = []
    for test, kind, f in ENTRIES:
        body = " ".join(f"{k}={v:.3e}" if isinstance(v, float) else f"{k}={v}" for k, v in f.items())
        out.append(f"{kind:7s} {body}  [{test}]")
    return out
