"""Write tests/golden/tiny_layout.txt from the CPU oracle (calls only oracle/).

The tiny workload (4 ranks x 128 tokens, 16 experts, top-4, seed 0) is the
functional configuration of the MSCCL++ EP multi-rank tests (num_ranks*4
experts, top-4).  The summary pins the input generator and the oracle's
layout against drift.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from workloads import CONFIGS, make_case  # noqa: E402


def main():
    cfg = CONFIGS["tiny"]
    c = make_case(cfg, with_hidden=False)
    L = oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks)
    lines = [
        "# written by tests/golden/make_golden.py from the CPU oracle; tiny workload",
        "recv_base: " + " ".join(map(str, L.recv_base.tolist())),
        "num_tokens_per_rank: " + " ".join(map(str, L.num_tokens_per_rank.ravel().tolist())),
        "num_tokens_per_expert: " + " ".join(map(str, L.num_tokens_per_expert.ravel().tolist())),
        "slot_first_8_tokens: " + " ".join(map(str, L.slot[:8].ravel().tolist())),
    ]
    with open(os.path.join(HERE, "tiny_layout.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
