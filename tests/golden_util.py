"""Reader for the text fixtures under tests/golden/ ("key: v1 v2 ..." lines,
'#' comments carry the citation of each value)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    out = {}
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if ":" in line:
                k, v = line.split(":", 1)
                out[k.strip()] = v.split()
            else:
                rows.append(line.split())
    if rows:
        out["_rows"] = rows
    return out
