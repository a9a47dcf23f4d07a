"""Small text fixtures of values the pages print, each with its citation.

Format: ``key = value`` lines; ``#`` starts a comment.
"""
import os

_HERE = os.path.dirname(os.path.abspath(__file__))


def read_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(_HERE, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("=", 1))
                out[k] = v
    return out
