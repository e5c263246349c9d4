"""Readers for the hand-worked fixtures under tests/golden/."""

import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            raw = raw.strip()
            if raw and not raw.startswith("#"):
                yield raw.split()


def table(name):
    """Fixture lines 'key v1 v2 ...' as a dict key -> list of tokens."""
    return {t[0]: t[1:] for t in lines(name)}
