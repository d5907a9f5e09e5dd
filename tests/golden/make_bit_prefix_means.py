"""Writes bit_prefix_means.txt: exact prefix means of V[j, c] = (j >> c) & 1.

With Q = 0 every visible score is equal, so Eq. (1) of the VPP technical
review (§2.2, "VPP: Virtual Pipeline Parallelism for Efficient Chunked
Prefill in Long-Context LLM Inference") gives, for the query at absolute
position p under the causal rule (keys 0..p), the plain mean of V[0..p].
For V[j, c] = bit c of j that mean is (number of j <= p with bit c set) /
(p + 1).  This script counts those bits directly (no oracle, no GPU) and
stores numerator and denominator as integers.
"""

import os

POSITIONS = [0, 1, 2, 3, 63, 64, 65, 127, 128, 129, 191, 255, 256, 300, 511]
BITS = 10


def main():
    here = os.path.dirname(os.path.abspath(__file__))
    with open(os.path.join(here, "bit_prefix_means.txt"), "w") as f:
        f.write("# p c count denominator   (mean = count / denominator)\n")
        f.write("# V[j, c] = (j >> c) & 1, Q = 0, keys 0..p visible; VPP review §2.2 Eq. (1)\n")
        for p in POSITIONS:
            for c in range(BITS):
                count = sum((j >> c) & 1 for j in range(p + 1))
                f.write(f"{p} {c} {count} {p + 1}\n")


if __name__ == "__main__":
    main()
