"""Per-case parity figures collected by the GPU parity tests and printed at the end of
the pytest session (tests/conftest.py): the gated output metric
max |y - r| / (|r| + rms(r)), the plain ratio max |y - r| / max |r|, and the near-tie
counts the parity criteria exempt (tokens whose k-th and (k+1)-th logits, or two
selected logits, or two rerouting candidates, lie within 1e-4)."""

RECORDS = []


def record(case: str, **fields):
    RECORDS.append((case, fields))


def lines():
    out = []
    for case, f in RECORDS:
        parts = [f"{k}={v:.2e}" if isinstance(v, float) else f"{k}={v}" for k, v in f.items()]
        out.append(f"{case}: " + ", ".join(parts))
    return out
