"""Writes the stored expected values under tests/golden/ from the fp64 oracle only.

Run from the repository root: ``python tests/golden/make_golden.py``. It calls
nothing but ``oracle`` and the seeded generator; no value comes from the CUDA path.
"""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
from relu_linear_attention_gb300 import synthetic as syn  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def main():
    w = syn.tiny_fp32(0)
    out, _, _ = O.rla2_prefill(w.q, w.k, w.v, w.gamma_q, w.gamma_k, w.eps_norm, w.rope_base,
                               w.eps_den)
    np.savetxt(os.path.join(HERE, "tiny_fp32_out.txt"), out.reshape(-1, out.shape[-1]),
               fmt="%.17e",
               header="RLA-2 causal output, tiny fp32 workload B=1 L=64 H=2 d=16 seed 0, "
                      "rows = (b, t, h) row-major, fp64 oracle")


if __name__ == "__main__":
    main()
