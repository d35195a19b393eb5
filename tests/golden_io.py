"""Reader for the hand-worked fixtures under tests/golden/."""
import math
import os
from fractions import Fraction

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

_SYMS = {"ln3": math.log(3.0), "ln2": math.log(2.0)}


def num(tok: str) -> float:
    """Parses '3/4', '-31/20', 'ln3/2', 'ln3-1', '-ln3', 'ln3-2*ln2' into a float."""
    t = tok.strip()
    if any(name in t for name in _SYMS):
        for name, val in _SYMS.items():
            t = t.replace(name, repr(val))
        return float(eval(t, {"__builtins__": {}}))  # fixture-only arithmetic
    return float(Fraction(t))


def read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([num(x) for x in line.split()])
    return rows


def read_recurrence(name):
    """Returns dict with dk, dv, S0 [dk][dv], per-token lists, o rows, ST."""
    d = {"alpha": [], "beta": [], "k": [], "v": [], "q": [], "o": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            xs = [num(x) for x in vals]
            if key in ("dk", "dv"):
                d[key] = int(xs[0])
            elif key in ("S0", "ST"):
                d[key] = xs
            elif key == "beta":
                d[key].append(xs[0])
            else:
                d[key].append(xs)
    return d
