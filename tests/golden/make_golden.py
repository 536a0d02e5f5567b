"""Writes the fixtures of this folder from the fp64 oracle alone (no CUDA
code is involved).  The pages print no worked example of the method, so no
fixture here comes from them; these pin the oracle against accidental change:

  e4m3_codes.txt, e5m2_codes.txt : the value of every 8-bit code (also fixed
      by the OCP FP8 format definitions, which test_oracle_pins checks);
  f16_specials.txt               : binary16 fixed points;
  workload1_decode.txt           : the oracle's decode of the tiny paged
      decode workload (4 sequences, lens {1, 7, 16, 33}, 4 q / 2 kv heads,
      head_dim 64, bf16, seed 1001): per (sequence, head) its lse and out.

Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from paged_kv_attention_14_gb300 import workloads as W  # noqa: E402


def codes(fn, path):
    with open(path, "w") as f:
        for c in range(256):
            f.write(f"{c:#04x} {fn(c)!r}\n")


def main():
    codes(oracle.e4m3_decode, os.path.join(HERE, "e4m3_codes.txt"))
    codes(oracle.e5m2_decode, os.path.join(HERE, "e5m2_codes.txt"))
    with open(os.path.join(HERE, "f16_specials.txt"), "w") as f:
        for c in (0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x3C01, 0x7BFF, 0x7C00, 0xFC00, 0xC000):
            f.write(f"{c:#06x} {oracle.f16_decode(c)!r}\n")
    b = W.workload(1, poison=True)
    out, lse = oracle.decode(oracle.KV_BF16, 16, b.num_kv_heads, b.num_q_heads, b.head_dim, b.q_decode,
                             b.k_pool, b.v_pool, b.block_tables_decode, b.context_lens_decode, b.scale)
    with open(os.path.join(HERE, "workload1_decode.txt"), "w") as f:
        f.write("# seq head lse out[0..63]  (fp64 oracle, repr)\n")
        for i in range(out.shape[0]):
            s, h = divmod(i, b.num_q_heads)
            f.write(f"{s} {h} {float(lse[i])!r} " + " ".join(repr(float(x)) for x in out[i]) + "\n")


if __name__ == "__main__":
    main()
