"""Parser for tests/golden/kquant_blocks.txt (hand-built blocks with hand-derived decodes)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kquant_blocks.txt")


def _hex_tokens(tokens):
    out = []
    i = 0
    while i < len(tokens):
        t = tokens[i]
        if "x[" in t:                      # Nx[HH HH ... HH]
            n, first = t.split("x[")
            group = [first]
            while not group[-1].endswith("]"):
                i += 1
                group.append(tokens[i])
            group[-1] = group[-1][:-1]
            out += [int(h, 16) for h in group if h] * int(n)
        elif "x" in t:                     # NxHH
            n, h = t.split("x")
            out += [int(h, 16)] * int(n)
        else:
            out.append(int(t, 16))
        i += 1
    return out


def load():
    blocks = []
    cur = None
    with open(GOLDEN) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            key = tok[0]
            if key == "block":
                cur = {"name": tok[1], "fmt": tok[2], "bytes": [], "q": {}, "value": {}}
            elif key == "hex":
                cur["bytes"] += _hex_tokens(tok[1:])
            elif key in ("d", "dmin"):
                cur[key] = float(tok[1])
            elif key in ("sc", "m"):
                cur[key] = [int(v) for v in tok[1:]]
            elif key == "q":
                cur["q"][int(tok[1])] = int(tok[2])
            elif key == "value":
                cur["value"][int(tok[1])] = float(tok[2])
            elif key == "end":
                cur["bytes"] = np.array(cur["bytes"], dtype=np.uint8)
                blocks.append(cur)
                cur = None
            else:
                raise ValueError(f"bad golden line: {raw!r}")
    return blocks
