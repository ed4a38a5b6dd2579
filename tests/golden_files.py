"""Readers of the hand-written fixtures under tests/golden/ (shared by the oracle pins
and the GPU tests; no arithmetic of the method here)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def q8_1_blocks():
    """tests/golden/q8_1_handmade.txt: name -> {"x" float32[32], "q" int64[32], and,
    when given, "d"/"s" (float values) or "dbits"/"sbits" (float32 bit patterns)}."""
    out, cur = {}, None
    for line in open(os.path.join(GOLDEN, "q8_1_handmade.txt")):
        t = line.split("#")[0].split()
        if not t:
            continue
        if t[0] == "block":
            cur = {"x": np.zeros(32, np.float32), "q": np.zeros(32, np.int64)}
            out[t[1]] = cur
        elif t[0] == "end":
            cur = None
        elif t[0] in ("d", "s"):
            cur[t[0]] = float(t[1])
        elif t[0] in ("dbits", "sbits"):
            cur[t[0]] = int(t[1], 16)
        else:
            p = int(t[0])
            cur["x"][p] = np.float32(float(t[1]))
            cur["q"][p] = int(t[2])
    return out


def q8_1_byte_vector():
    """tests/golden/q8_1_bytes_2x256.txt: (x float32 [2, 256], expected bytes uint8[640])."""
    x, buf = None, None
    for line in open(os.path.join(GOLDEN, "q8_1_bytes_2x256.txt")):
        t = line.split("#")[0].split()
        if not t:
            continue
        if t[0] == "size":
            buf = np.zeros(int(t[1]), np.uint8)
            x = np.zeros((int(t[2]), int(t[3])), np.float32)
        elif t[0] == "x":
            x[int(t[1]), int(t[2])] = np.float32(float(t[3]))
        elif t[0] == "byte":
            buf[int(t[1])] = int(t[2], 16)
    return x, buf
