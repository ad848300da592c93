"""Loader for the hand-worked fixtures in this folder (plain text, see each file's header)."""
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent


def load(name: str) -> dict:
    out = {}
    toks = []
    for line in (HERE / name).read_text().splitlines():
        line = line.split("#", 1)[0].strip()
        if line:
            toks.extend(line.split())
    i = 0
    while i < len(toks):
        kind = toks[i]
        if kind == "scalar":
            val = toks[i + 2]
            out[toks[i + 1]] = float(val) if "." in val else int(val)
            i += 3
        elif kind == "array":
            name_, typ = toks[i + 1], toks[i + 2]
            j = i + 3
            dims = []
            while j < len(toks) and toks[j] not in ("scalar", "array") and len(dims) < 8:
                # dims end where the value list starts: values count = prod(dims)
                dims.append(int(toks[j]))
                j += 1
                n = int(np.prod(dims))
                rest = toks[j:]
                # stop reading dims once the remaining tokens up to the next
                # keyword are exactly prod(dims) values
                nxt = next((q for q, t in enumerate(rest) if t in ("scalar", "array")), len(rest))
                if nxt == n:
                    break
            n = int(np.prod(dims))
            vals = toks[j:j + n]
            dtype = np.int32 if typ == "int" else np.float64
            out[name_] = np.array([float(v) for v in vals], dtype=np.float64).astype(dtype).reshape(dims)
            i = j + n
        else:
            raise ValueError(f"bad token {kind!r} in {name}")
    return out
