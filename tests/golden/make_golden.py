"""Writes tests/golden/tiny_oracle.txt: digests of the oracle's results on the
small end-to-end case (256x256 fp32 weights with 328 outliers, seed 0; one bf16
activation row, seed 1).  Calls only the oracle and the seeded input module, so
the stored values never come from the CUDA path.  The test that reads the file
checks that the oracle stays deterministic across machines and edits.

Run:  python tests/golden/make_golden.py
"""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from ternary_weight_fwht128_gb300 import synth  # noqa: E402


def digests():
    orc = oracle.load()
    W, xb = synth.tiny_config()
    T, S = orc.quantize(W)
    c2 = orc.pack2(T)
    c3 = orc.pack3(T)
    y = orc.gemv(T, S, synth.bf16_bits_to_f32(xb))
    return {
        "codes2_sha256": hashlib.sha256(c2.tobytes()).hexdigest(),
        "codes3_sha256": hashlib.sha256(c3.tobytes()).hexdigest(),
        "scales_sha256": hashlib.sha256(S.tobytes()).hexdigest(),
        "y_sha256": hashlib.sha256(y.tobytes()).hexdigest(),
        "zero_trits": int((T == 0).sum()),
        "y0": float(y[0, 0]).hex(),
    }


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.txt")
    with open(out, "w") as f:
        f.write("# written by tests/golden/make_golden.py from the oracle only\n")
        for k, v in digests().items():
            f.write(f"{k} {v}\n")
    print(open(out).read())
