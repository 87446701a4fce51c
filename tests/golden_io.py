"""Reader for the text fixtures under tests/golden/ (test helper, no arithmetic)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _float(tok: str) -> float:
    if tok in ("0", "-0"):
        return -0.0 if tok.startswith("-") else 0.0
    return float.fromhex(tok)


def load_blocks(name: str = "blocks.txt"):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest}
            elif key == "format":
                cur["format"] = rest
            elif key == "why":
                cur["why"] = rest
            elif key == "bytes":
                cur["bytes"] = np.array([int(t, 16) for t in rest.split()], np.uint8)
            elif key == "expect_f32":
                cur["f32"] = np.array([_float(t) for t in rest.split()], np.float32)
            elif key == "expect_f16":
                cur["f16"] = np.array([int(t, 16) for t in rest.split()], np.uint16)
            elif key == "end":
                cases.append(cur)
                cur = None
    return cases
