"""Reader for the small ``key = value`` text fixtures in this folder."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def load(name):
    out = {}
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            if ";" in val:
                out[key] = [[float(x) for x in row.split()] for row in val.split(";")]
            else:
                out[key] = float(val)
    return out
