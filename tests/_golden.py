"""Reader for the text fixtures under tests/golden/.

Format: '#' comment lines (the citation), 'key = value' lines, and table rows
whose first token is a row tag (anything without '=').
"""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(tok):
    try:
        return int(tok)
    except ValueError:
        try:
            return float(tok)
        except ValueError:
            return tok


def load(name):
    kv, rows = {}, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if " = " in line:
                k, v = line.split("=", 1)
                toks = v.split()
                kv[k.strip()] = _num(toks[0]) if len(toks) == 1 else [_num(t) for t in toks]
            else:
                rows.append(line.split())
    return kv, rows
