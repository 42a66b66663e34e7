"""Reader for the hand-worked example fixtures under tests/golden/."""
from __future__ import annotations

import os
import re

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _expand_groups(text: str) -> str:
    """"(a b)*n" -> the group written n times."""
    pat = re.compile(r"\(([^()]*)\)\*(\d+)")
    while True:
        new = pat.sub(lambda m: " ".join([m.group(1)] * int(m.group(2))), text)
        if new == text:
            return text
        text = new


def _hex_list(text: str):
    text = _expand_groups(text)
    out = []
    for tok in text.split():
        if "*" in tok:
            v, n = tok.split("*")
            out.extend([int(v, 16)] * int(n))
        else:
            out.append(int(tok, 16))
    return out


def load_quant_examples(name: str = "quant_examples.txt"):
    cases, cur = [], None
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = (s.strip() for s in line.partition("="))
            if key == "case":
                cur = {"case": val}
                cases.append(cur)
            elif key in ("x",):
                cur[key] = np.array(_hex_list(val), np.uint16)
            elif key in ("q", "q_in", "s_in", "q_out", "s_out"):
                cur[key] = np.array(_hex_list(val), np.uint8)
            elif key in ("scale", "scale_f32"):
                cur[key] = int(val, 16)
            elif key in ("clamped", "rows", "saturated", "top_code", "blocks_saturated",
                         "blocks_collapsed"):
                cur[key] = int(val)
            elif key == "row_sat":
                cur[key] = [int(t) for t in val.split()]
            else:
                cur[key] = val
    return cases
