"""Assemble the hand-built fixtures of ``tests/golden/kq_closed_forms.json``.

Only byte placement lives here: each field of a fixture is written at its
GGUF offset inside the superblock.  No decode and no fold.
"""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kq_closed_forms.json")
FMT = {"Q4_K": 1, "Q5_K": 2, "Q6_K": 3}

# (offset, length) of each field inside the disk superblock
FIELDS = {
    "Q4_K": {"d": (0, 2), "dmin": (2, 2), "scales12": (4, 12), "qs": (16, 128)},
    "Q5_K": {"d": (0, 2), "dmin": (2, 2), "scales12": (4, 12), "qh": (16, 32), "qs": (48, 128)},
    "Q6_K": {"ql": (0, 128), "qh": (128, 64), "scales16": (192, 16), "d": (208, 2)},
}
SIZE = {"Q4_K": 144, "Q5_K": 176, "Q6_K": 210}


def load():
    with open(GOLDEN) as f:
        return json.load(f)


def fill_array(spec, n, dtype):
    """A {'fill': v, 'set': {i: v}, 'set_range': [a, b, v]} description -> array."""
    if isinstance(spec, list):
        return np.array(spec, dtype=dtype)
    a = np.full(n, spec.get("fill", 0), dtype=dtype)
    if "set_range" in spec:
        lo, hi, v = spec["set_range"]
        a[lo:hi] = v
    for k, v in spec.get("set", {}).items():
        a[int(k)] = v
    return a


def block_bytes(fmt_name, block):
    raw = np.zeros(SIZE[fmt_name], np.uint8)
    for name, (off, ln) in FIELDS[fmt_name].items():
        if name not in block:
            continue
        val = block[name]
        if name in ("d", "dmin"):
            bits = int(val, 16)
            raw[off] = bits & 0xFF
            raw[off + 1] = bits >> 8
        elif name == "scales16":
            raw[off:off + ln] = fill_array(val, ln, np.int8).view(np.uint8)
        else:
            raw[off:off + ln] = fill_array(val, ln, np.int64).astype(np.uint8)
    return raw


def act_planes(act):
    d8 = np.array([[act["d8"]]], np.float32)
    q8 = fill_array(act["q8"], 256, np.int8)[None, :]
    bs = fill_array(act["bsums"], 16, np.int16)[None, :]
    return d8, q8, bs
