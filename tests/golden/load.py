"""Parse the hand-worked golden fixtures (hex bytes in named sections)."""
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def load(name: str) -> dict:
    sections, cur = {}, None
    with open(os.path.join(HERE, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = line.strip("[]")
                sections[cur] = bytearray()
                continue
            for tok in line.split():
                sections[cur] += bytes.fromhex(tok)
    return {k: np.frombuffer(bytes(v), np.uint8) for k, v in sections.items()}
