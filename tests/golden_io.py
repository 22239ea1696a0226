"""Readers for the hand-worked fixtures under tests/golden/ (text, one record per line)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                key, _, rest = ln.partition(":")
                yield key.strip(), rest.strip()


def matrix(text, dtype=float):
    return np.array([[dtype(v) for v in row.split()] for row in text.split(";")])


def vector(text, dtype=float):
    return np.array([dtype(v) for v in text.split()])
