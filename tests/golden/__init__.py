"""Hand-derived fixtures; ``load`` turns their symbolic entries into floats."""

import json
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))

_SYMBOLS = {
    "ln2": math.log(2.0),
    "ln3": math.log(3.0),
    "ln4": math.log(4.0),
    "-ln2": -math.log(2.0),
    "sqrt2*ln2": math.sqrt(2.0) * math.log(2.0),
}


def _value(x):
    if isinstance(x, str):
        return _SYMBOLS[x]
    if isinstance(x, list):
        if len(x) == 2 and all(isinstance(e, int) for e in x):
            return x[0] / x[1]  # [numerator, denominator]
        return [_value(e) for e in x]
    return float(x)


def load(name: str) -> dict:
    with open(os.path.join(_HERE, name)) as fh:
        raw = json.load(fh)
    skip = ("what", "source", "derivation", "note")
    return {k: (v if k in skip else _value(v)) for k, v in raw.items()}
