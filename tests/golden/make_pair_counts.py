"""Writes pair_counts.json: the number of (query, key) pairs the float64
oracle's mask admits for one head of each benchmark workload, at full size.

It calls only the oracle: with K = 0 every allowed score is 0, so a row's LSE
is ln(number of keys it may attend) and exp(LSE) summed over the rows counts
the admitted pairs. The shapes are those of the workloads in workloads.py
(TransformerEngine PR #3705: compact-THD causal D128 with Hq32/Hkv8 and
lengths up to 4096; PR #3527 "Problem": sliding-window layers, left window
1024; PR #3527 "Performance": b2 hq8 hkv4 d512 causal, here with Sq 2048 and
Sk 8192 bottom-right and non-causal; a 32K-token causal context).

    python tests/golden/make_pair_counts.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402
from oracle import oracle  # noqa: E402


def oracle_pairs(sq, sk, mask, window):
    q = np.ones((1, sq, 1, 1))
    k = np.zeros((1, sk, 1, 1))
    v = np.zeros((1, sk, 1, 1))
    _, lse = oracle.fwd(q, k, v, layout="bshd", mask=mask, scale=1.0, window=window)
    finite = np.isfinite(lse)
    return int(round(float(np.sum(np.exp(lse[finite])))))


def main():
    out = {"_about": "pairs per head admitted by the oracle's mask; written by make_pair_counts.py", "workloads": {}}
    for w in workloads.ALL:
        if w.layout == "thd":
            lens = [int(x) for x in workloads.thd_lengths(w)]
            per_seq = [oracle_pairs(n, n, w.mask, w.window) for n in lens]
            out["workloads"][w.name] = {"lengths": lens, "mask": w.mask, "window": list(w.window),
                                        "pairs_per_sequence": per_seq}
        else:
            out["workloads"][w.name] = {"seqlen_q": w.seqlen_q, "seqlen_kv": w.seqlen_kv, "mask": w.mask,
                                        "window": list(w.window),
                                        "pairs": oracle_pairs(w.seqlen_q, w.seqlen_kv, w.mask, w.window)}
        print(w.name, out["workloads"][w.name], flush=True)
    with open(os.path.join(HERE, "pair_counts.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
