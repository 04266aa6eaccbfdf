"""Parsers for the small text fixtures in this folder (each file cites its source)."""
import os

_HERE = os.path.dirname(os.path.abspath(__file__))


def _num(tok: str):
    tok = tok.strip()
    if tok.lower().startswith("0x"):
        return int(tok, 16)
    try:
        return int(tok)
    except ValueError:
        return float(tok)


def load_kv(name: str) -> dict:
    """`key v1 v2 ...` lines -> {key: [values]} (scalars unwrapped); '#' lines skipped."""
    out = {}
    with open(os.path.join(_HERE, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            v = [_num(t) for t in vals]
            out[key] = v[0] if len(v) == 1 else v
    return out


def load_table(name: str) -> list:
    """Whitespace-separated rows of numbers; '#' lines skipped."""
    rows = []
    with open(os.path.join(_HERE, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([_num(t) for t in line.split()])
    return rows
