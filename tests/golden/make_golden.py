"""Write the oracle's worked-example fixtures under tests/golden/.

Calls only ``oracle/``.  The pages print no worked example of the delayed
eviction rule, so these fixtures are regression records of the oracle on small
hand-checkable cases (each row can be verified by hand from the rule in
"Inference-Time Hyper-Scaling with KV Cache Compression", AI research-map
summary, "Approach": a marked token leaves the cache w steps after it entered,
and the slot it frees is taken by the token appended in that step).

Run:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle.dms_oracle import SlotSimulator, retained_length, visibility_mask  # noqa: E402

CASES = [
    # (name, window, decisions as a 0/1 string, capacity)
    ("w3_mixed", 3, "1011001110", 8),
    ("w1_eager", 1, "1101011", 4),
    ("w4_all_evict", 4, "111111111", 4),
]


def main():
    out = os.path.join(HERE, "delayed_eviction_examples.txt")
    with open(out, "w") as f:
        f.write("# Delayed-eviction worked examples (one sequence, one KV head).\n")
        f.write("# Written by tests/golden/make_golden.py from oracle/ only.\n")
        f.write("# Rule: 'Inference-Time Hyper-Scaling with KV Cache Compression', AI research-map\n")
        f.write("# summary, 'Approach' (decision executed after a delay window).\n")
        f.write("# Columns: case window t decision visible_positions retained slot_map(len slots)\n")
        for name, w, bits, cap in CASES:
            e = np.array([c == "1" for c in bits])
            sim = SlotSimulator(1, 1, cap, w)
            for t in range(len(bits)):
                sim.append(e[t:t + 1].reshape(1, 1))
                vis = np.nonzero(visibility_mask(e, t, w))[0].tolist()
                ret = retained_length(e, t + 1, w)
                slots = sim.occupied_positions(0, 0).tolist()
                f.write(f"{name} {w} {t} {int(e[t])} {','.join(map(str, vis))} {ret} "
                        f"{','.join(map(str, slots))}\n")
    print("wrote", out)


if __name__ == "__main__":
    main()
