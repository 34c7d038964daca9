"""Reader for the hand-derived fixtures under tests/golden/.

Values are small arithmetic expressions (numbers, ln, exp, + - * / and
parentheses); they are evaluated with no builtins available."""
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_NS = {"__builtins__": {}, "ln": math.log, "exp": math.exp}


def _val(tok: str) -> float:
    return float(eval(tok, _NS))  # fixture expressions only


def _matrix(text: str) -> np.ndarray:
    rows = [r.split() for r in text.split(";")]
    return np.array([[_val(t) for t in r] for r in rows], dtype=np.float64)


def _split_values(rest: str):
    """Tokens are separated by spaces except inside parentheses."""
    toks, depth, cur = [], 0, ""
    for ch in rest:
        if ch == "(":
            depth += 1
        elif ch == ")":
            depth -= 1
        if ch.isspace() and depth == 0:
            if cur:
                toks.append(cur)
            cur = ""
        else:
            cur += ch
    if cur:
        toks.append(cur)
    return toks


def _parse_line(line: str):
    key, _, rest = line.partition(" ")
    rows = [_split_values(r) for r in rest.split(";")]
    return key, np.array([[_val(t) for t in r] for r in rows], dtype=np.float64)


def load_cases(name: str) -> dict:
    cases, cur, cname = {}, None, None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                cname, cur = line.split()[1], {}
            elif line == "end":
                cases[cname] = cur
                cur = None
            else:
                key, arr = _parse_line(line)
                cur[key] = arr
    return cases


def load_single(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if " " in line and line.split()[0] in ("LSE", "O"):
                key, _, rest = line.partition(" ")
                out[key] = _val(rest)
            else:
                key, arr = _parse_line(line)
                out[key] = arr
    return out


def load_philox_kat(name: str = "philox4x32_10_kat.txt"):
    """(counter[4], key[2], expected[4]) triples of 32-bit words."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            toks = line.split()
            assert toks[0] == "kat" and toks[7] == "->" and len(toks) == 12, line
            words = [int(t, 16) for t in toks[1:7] + toks[8:12]]
            out.append((words[0:4], words[4:6], words[6:10]))
    return out
