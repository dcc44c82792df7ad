"""Write tests/golden/tiny_seed1.txt from the oracle alone.

The pages print no worked numeric example, so this fixture is a regression pin
of the oracle on the tiny workload (1 layer, 2 heads, d 64, 64 slots, seed 1):
after every operation it records the stored position of each slot, the K and
V scales of each (head, slot), a checksum of the codes, and the first output
row of every attention call.  Run: python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth_inputs as si  # noqa: E402


def run(seed: int = 1):
    s = si.TINY
    oc = oracle.OracleCache(s.layers, s.heads, s.head_dim, s.slots, s.rope_base)
    lines = []
    step = 0
    q = None
    for op in si.tiny_schedule():
        if op[0] == "write":
            _, layer, p0, n = op
            k, v, q = si.tiny_tensors(seed, step, "cpu")
            oc.write(layer, k, v, np.arange(p0, p0 + n))
            step += 1
            tag = f"write {p0} {n}"
        elif op[0] == "delta":
            oc.delta_rotate(op[1])
            tag = f"delta {op[1]}"
        else:
            out = oc.attend(op[1], q)
            lines.append("attend row0 " + " ".join(f"{x:.17g}" for x in out[0].reshape(-1)))
            continue
        st = oc.export(0)
        lines.append(tag)
        lines.append("pos " + " ".join(str(int(p)) if p != oracle.EMPTY else "E" for p in st["pos"]))
        for h in range(s.heads):
            lines.append(f"kscale{h} " + " ".join(f"{x:.9g}" for x in st["kscale"][h]))
            lines.append(f"vscale{h} " + " ".join(f"{x:.9g}" for x in st["vscale"][h]))
        lines.append("kcodesum %d vcodesum %d" % (int(st["kcodes"].astype(np.int64).sum()),
                                                  int(st["vcodes"].astype(np.int64).sum())))
    return lines


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_seed1.txt")
    with open(path, "w") as f:
        f.write("# oracle regression fixture, tiny workload, seed 1; written by make_golden.py\n")
        f.write("\n".join(run(1)) + "\n")
    print("wrote", path)
