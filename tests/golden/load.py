"""Reader for the small text fixtures in this folder.

Lines starting with '#' are comments (they carry the citation and the
derivation).  Every other line is `name = rows`, rows separated by ';' and
values by whitespace; a single row comes back as a 1-D array.
"""
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))


def load(name):
    out = {}
    with open(os.path.join(_HERE, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            rows = [[float(t) for t in r.split()] for r in val.split(";")]
            arr = np.array(rows, dtype=np.float64)
            if arr.shape[1] == 1:
                arr = arr[:, 0]
            if arr.ndim == 1 and arr.shape[0] == 1:
                arr = arr[0]
            out[key] = arr
    return out
