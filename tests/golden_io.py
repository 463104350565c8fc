"""Reader for the small text fixtures under tests/golden/ (key: values lines,
'#' comments carry the citation of the page the values come from)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            vals = val.split()
            try:
                parsed = [int(v) for v in vals]
            except ValueError:
                parsed = [float(v) for v in vals]
            out[key.strip()] = parsed if len(parsed) != 1 else parsed[0]
    return out
