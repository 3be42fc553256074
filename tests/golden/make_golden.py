"""Writes tests/golden/shard_tiles.json.  Calls only the oracle (no CUDA path).

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

CASES = [
    # the benchmark workloads' (L, n, layout), causal, tile 128
    ("causal_contig_8k", 8192, 8, "contiguous"),
    ("causal_contig_8k_as_zigzag", 8192, 8, "zigzag"),
    ("zigzag_gqa_32k", 32768, 8, "zigzag"),
    ("zigzag_gqa_32k_as_contiguous", 32768, 8, "contiguous"),
    ("zigzag_gqa_128k", 131072, 8, "zigzag"),
    ("zigzag_gqa_64k_train", 65536, 16, "zigzag"),
]


def main():
    out = {
        "source": "oracle.shard_tiles (brute force over tile pairs); sizes from the pages",
        "page_sizes": {
            "citation": "agentalpha 'Ring Attention vs tensor parallelism', standard answer and "
                        "follow-up 1: 128K tokens over 8 devices, 16K per device, block size 128",
            "L": 131072, "n": 8, "tokens_per_device": 16384, "block": 128,
        },
        "cases": [],
    }
    for name, L, n, layout in CASES:
        tiles = oracle.shard_tiles(L, n, True, layout, 128).tolist()
        out["cases"].append({"name": name, "L": L, "n": n, "causal": True, "layout": layout,
                             "tile": 128, "tiles_per_shard": tiles})
    with open(os.path.join(HERE, "shard_tiles.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
