"""Writes the stored oracle outputs under tests/golden/.  Calls only the
oracle and the seeded input generator; never the CUDA path."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from draft_token_markov_gb300 import workloads as W  # noqa: E402


def main():
    w = W.TINY
    head, embed = W.make_weights(w)
    c = W.make_call(w)
    toks, _ = oracle.chain(oracle.bf16_bits(c["base"]), oracle.bf16_bits(head),
                           oracle.bf16_bits(embed), c["anchor"].numpy(),
                           c["temperature"].numpy(), c["seeds"].numpy(),
                           c["row_state_idx"].numpy(), w.mode)
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny_chain.txt")
    with open(out, "w") as f:
        f.write("# Oracle tokens of the tiny chain workload (V=4096, r=64, 1 row, N=4,\n"
                "# Gumbel, T=1, seed 1), written by tests/golden/make_golden.py from\n"
                "# oracle/ alone.  A regression pin: it changes only with the oracle's\n"
                "# arithmetic or the input generator.\n")
        f.write("tokens: " + " ".join(str(int(t)) for t in toks.ravel()) + "\n")
    print(open(out).read())


if __name__ == "__main__":
    main()
