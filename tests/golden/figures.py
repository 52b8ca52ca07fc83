"""Loader for ``pages_figures.txt`` (figures quoted from the lecture pages)."""
import os

_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "pages_figures.txt")


def load():
    out = {}
    with open(_PATH) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val, _src = [p.strip() for p in line.split("|", 2)]
            out[key] = float(val)
    return out
