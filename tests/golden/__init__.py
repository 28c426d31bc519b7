"""Readers for the hand-derived fixtures in this folder."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def read_kv(name):
    """Parse 'key v1 v2 ...' lines and 'items'/'leaves' ... 'end' blocks."""
    out, block, rows = {}, None, []
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if block is not None:
                if line == "end":
                    out[block] = rows
                    block, rows = None, []
                else:
                    rows.append([int(x) for x in line.split()])
                continue
            parts = line.split()
            if len(parts) == 1:
                block = parts[0]
                continue
            out[parts[0]] = [float(x) for x in parts[1:]]
    return out
