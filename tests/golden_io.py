"""Parser for the small text fixtures under tests/golden/ (key: values lines)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_pairs(name):
    """Return the fixture's (key, value-string) pairs in file order, comments dropped."""
    pairs = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = line.split(":", 1)
            pairs.append((key.strip(), val.strip()))
    return pairs


def floats(s):
    return [float(t) for t in s.split()]
