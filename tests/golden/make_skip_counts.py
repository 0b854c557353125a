"""Writes skip_counts.json: for each custom-mask workload of the benchmark, the number of
(query tile, key tile) blocks the kernel must compute and the number it must skip, from
the oracle's block map.

A block is computed iff it holds a kept entry (the tile-skip rule of the page "Opus 4.6 +
AutoResearch驱动25轮迭代...", first code excerpt); with a custom mask the query tiles are
the compacted ones (the 16-row blocks that keep anything, in ascending order, eight per
tile), as include/attn.h states for attn_fwd_visited.  Calls only the oracle package, the
seeded input generators and the test helper that applies that tile layout to the oracle's
(16-row, 128-key) map; run it from the repository root with
``python tests/golden/make_skip_counts.py``.  Each entry carries the sha1 of the mask words
it was computed on, so a reader can tell whether its inputs are the same.
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(HERE))

from attention_forward_07_gb300 import inputs as inp  # noqa: E402
from gpu_util import expected_visited  # noqa: E402


def main():
    out = {}
    names = list(inp.WORKLOADS)
    for name, w in inp.WORKLOADS.items():
        if w.mask == "none":
            continue
        seed = w.seed(names.index(name))
        _, _, _, bits = w.make(seed)
        vis = expected_visited(bits, False, w.B, w.Hq, w.S, w.S, w.causal)
        out[name] = {"seed": seed, "mask_sha1": hashlib.sha1(bits.tobytes()).hexdigest(),
                     "blocks": int(vis.size), "computed": int(vis.sum()), "skipped": int(vis.size - vis.sum())}
    with open(os.path.join(HERE, "skip_counts.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
