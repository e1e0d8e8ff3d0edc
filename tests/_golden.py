"""Reader for the text fixtures under tests/golden (``name: v1 v2 ...`` lines, ``#`` comments)."""
import os

GOLDEN_DIR = os.path.join(os.path.dirname(__file__), "golden")


def read_kv(name):
    out = {}
    with open(os.path.join(GOLDEN_DIR, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = line.split(":", 1)
            out[key.strip()] = [float(x) for x in val.split()]
    return out


def read_columns(name):
    rows = []
    with open(os.path.join(GOLDEN_DIR, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([float(x) for x in line.split()])
    return rows
