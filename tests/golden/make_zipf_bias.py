"""Write the fitted router bias of the Zipf-skewed 2048-token workload.

Calls only the oracle (for routing counts) and the input generator. The bias is
fitted on a calibration token draw that is independent of the workload's own
tokens, so expert popularity is a property of the layer, not of one batch.

    python tests/golden/make_zipf_bias.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import moe_synth as ms  # noqa: E402
from oracle import moe_oracle as mo  # noqa: E402


def main():
    shape = ms.CONFIGS["zipf2048"]
    cal = ms.calibration_tokens(shape, shape.tokens)
    logits = mo.router_logits(cal, ms.router_weights(shape))

    def count_fn(bias):
        ids, _, _ = mo.select_topk(logits, bias, shape.top_k)
        return mo.expert_counts(ids, shape.experts)[0]

    b = ms.fit_zipf_bias(shape, count_fn, shape.tokens)
    counts = count_fn(b)
    target = ms.zipf_targets(shape, shape.tokens)
    path = ms.zipf_bias_path(shape)
    with open(path, "w") as f:
        f.write("# fp32 router bias (hex bits, value) fitted so that routed row counts of\n")
        f.write(f"# {shape.tokens} calibration tokens follow Zipf(s={shape.zipf_s}) over a seeded\n")
        f.write("# expert ranking; written by tests/golden/make_zipf_bias.py (oracle routing).\n")
        f.write(f"# max count {counts.max()}, experts under 10 rows {(counts < 10).sum()}\n")
        for v in b:
            f.write(f"{np.float32(v).view(np.uint32):08x} {float(v):.9g}\n")
    order = np.argsort(-target)
    print("top targets", np.round(target[order[:6]]), "counts", counts[order[:6]])
    print("tail targets", np.round(target[order[-6:]], 1), "counts", counts[order[-6:]])
    print("max", counts.max(), "under10", (counts < 10).sum(), "wrote", path)


if __name__ == "__main__":
    main()
