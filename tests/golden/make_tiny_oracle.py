"""Writes tiny_oracle.json: fp64 oracle outputs for one tiny seeded case.

Calls only the oracle package and the seeded input generators; run it from the
repository root with ``python tests/golden/make_tiny_oracle.py``.  The fixture is
a regression guard: a later change to the oracle's arithmetic that moves these
numbers must say which passage of the pages justifies it.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from attention_forward_07_gb300 import inputs as inp  # noqa: E402

B, Hq, Hkv, S, d, SEED, CAUSAL, SCALE = 1, 2, 1, 12, 4, 20240, True, 0.5


def main():
    q, k, v = inp.qkv(B, Hq, Hkv, S, d, inp.F16, SEED)
    bits = inp.pack_bits(inp.bernoulli_mask(B, S, SEED))
    o, lse = oracle.attn_fwd(inp.as_u16(q), inp.as_u16(k), inp.as_u16(v), inp.F16, bits, CAUSAL, SCALE)
    out = {"shape": [B, Hq, Hkv, S, d], "seed": SEED, "causal": CAUSAL, "scale": SCALE,
           "o": [x.hex() for x in o.reshape(-1).tolist()],
           "lse": [x.hex() for x in lse.reshape(-1).tolist()]}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json"), "w") as f:
        json.dump(out, f, indent=0)
        f.write("\n")


if __name__ == "__main__":
    main()
