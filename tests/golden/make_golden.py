"""Writes the small regression fixtures of tests/golden/ from the oracle only.

    python tests/golden/make_golden.py

Each fixture is a text file: a header line of JSON (the call), then the input
blocks and the expected gathered outputs as rows of hexadecimal 16-bit words.
They freeze the oracle's answers on tiny, hand-checkable cases of the
all-gather (iris #594 "Multi-GPU CI": block i of every member's output is
member i's input) and the all-to-all (member d's block i = member i's block d).
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

CASES = {
    "gather_w3_strided.txt": dict(kind="all_gather", H=6, group=[1, 2, 3], M=2, N=3),
    "all_to_all_w3.txt": dict(kind="all_to_all", H=3, group=[0, 1, 3], M=2, N=3),
}


def inputs(case):
    """Input of member h: element (m, n) = 0x1000*h + 0x100*m + n (readable in hex)."""
    start, stride, W = case["group"]
    rows = W * case["M"] if case["kind"] == "all_to_all" else case["M"]
    out = {}
    for i in range(W):
        h = start + i * stride
        m = np.arange(rows).reshape(rows, 1)
        n = np.arange(case["N"]).reshape(1, case["N"])
        out[h] = (0x1000 * h + 0x100 * m + n).astype(np.uint16)
    return out


def run(case):
    start, stride, W = case["group"]
    M, N = case["M"], case["N"]
    ins = inputs(case)
    rows = ins[start].shape[0]
    in_off, out_off = 0, rows * N * 2
    part = out_off + W * M * N * 2
    heap = np.zeros(case["H"] * part, dtype=np.uint8)
    for h, blk in ins.items():
        heap[h * part: h * part + blk.nbytes] = blk.view(np.uint8).ravel()
    orc = oracle.Oracle()
    fn = orc.all_to_all if case["kind"] == "all_to_all" else orc.all_gather
    fn(heap, part, in_off, N, out_off, N, M, N, 2, tuple(case["group"]))
    outs = {h: heap[h * part + out_off: (h + 1) * part].view(np.uint16).reshape(W * M, N)
            for h in ins}
    return ins, outs


def render(case, ins, outs):
    lines = [json.dumps(case)]
    for h in sorted(ins):
        lines.append(f"input {h}")
        lines += [" ".join(f"{v:04x}" for v in row) for row in ins[h]]
    for h in sorted(outs):
        lines.append(f"output {h}")
        lines += [" ".join(f"{v:04x}" for v in row) for row in outs[h]]
    return "\n".join(lines) + "\n"


def main():
    for name, case in CASES.items():
        ins, outs = run(case)
        with open(os.path.join(HERE, name), "w") as f:
            f.write(render(case, ins, outs))


if __name__ == "__main__":
    main()
