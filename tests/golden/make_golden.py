"""Write oracle_regression.txt: the fp64 oracle's results on small seeded cases.

Calls only oracle/ (and the numpy input generator), never the CUDA library.  The file
guards the oracle against unintended change: tests/test_golden.py re-runs these cases and
compares bit for bit.  Regenerate only together with a reasoned change to the oracle.

    python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from adaptive_gradient_summation_gb300.workloads import numpy_case  # noqa: E402

#: (seed, K, segment lengths, bf16)
CASES = [
    (1, 2, [13], False),
    (2, 4, [5, 0, 9, 1], False),
    (3, 8, [17, 3], False),
    (4, 16, [7, 8], True),
    (5, 4, [1, 2, 3, 4, 5], True),
]


def render() -> str:
    lines = ["# fp64 oracle results (hex floats) for the seeded cases of make_golden.py",
             "# case <seed> <K> <lengths> <dtype>  then one line per output element"]
    for seed, K, lengths, bf16 in CASES:
        grads, offs = numpy_case(seed, K, lengths, bf16)
        r = oracle.adasum_reduce(grads, offs, want_ortho=True)
        dt = "bf16" if bf16 else "f32"
        lines.append(f"case {seed} {K} {','.join(map(str, lengths))} {dt}")
        lines += [float(x).hex() for x in r["out64"]]
        lines.append("ortho " + " ".join(float(x).hex() for x in r["ortho"]))
    return "\n".join(lines) + "\n"


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_regression.txt"), "w") as fh:
        fh.write(render())
