"""Parser for the hand-worked fixtures under tests/golden/ (plain text)."""
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
CONTAINER_FIXTURES = ["bf16_five_elements.txt", "bf16_two_chunks_ragged.txt", "e5m2_nine_elements.txt",
                      "fp16_nine_elements.txt"]
DTYPES = {"bf16": 0, "e5m2": 1, "fp16": 2}


def _lines(name):
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                yield line.split()


def load_container(name):
    """Return dict(dtype, chunk_elems, input bits, codebook, expected bytes)."""
    fx = {"bytes": []}
    inputs = []
    for tok in _lines(name):
        key = tok[0]
        if key == "dtype":
            fx["dtype"] = DTYPES[tok[1]]
        elif key in ("chunk_elems", "n", "size"):
            fx[key] = int(tok[1])
        elif key == "input_default":
            fx["default"] = int(tok[1], 16)
        elif key == "input":
            inputs.append((int(tok[1]), int(tok[2], 16)))
        elif key == "codebook":
            fx["codebook"] = np.array([int(t, 16) for t in tok[1:]], dtype=np.uint8)
        elif key == "bytes":
            fx["bytes"].append((int(tok[1]), [int(t, 16) for t in tok[2:]]))
        else:
            raise ValueError("unknown fixture key %r in %s" % (key, name))
    bits = np.uint8 if fx["dtype"] == 1 else np.uint16
    x = np.full(fx["n"], fx["default"], dtype=bits)
    for i, v in inputs:
        x[i] = v
    blob = np.zeros(fx["size"], dtype=np.uint8)
    for off, vals in fx["bytes"]:
        blob[off : off + len(vals)] = vals
    fx["input"] = x
    fx["expected"] = blob
    return fx


def load_calibration_cases(name="calibration_ties.txt"):
    cases = []
    for tok in _lines(name):
        if tok[0] == "case":
            cases.append({"dtype": DTYPES[tok[1]], "hist": np.zeros(256, np.uint64)})
        elif tok[0] == "hist":
            cases[-1]["hist"][int(tok[1])] = int(tok[2])
        elif tok[0] == "expect":
            cases[-1]["expect"] = np.array([int(t) for t in tok[1:]], dtype=np.uint8)
    return cases
