"""Readers for the small text fixtures in this folder (each cites its page)."""

import os

HERE = os.path.dirname(os.path.abspath(__file__))


def rows(name):
    out = []
    with open(os.path.join(HERE, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def constants(name):
    return {k: float(v) for k, v in rows(name)}
