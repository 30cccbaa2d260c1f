#!/usr/bin/env python
"""Axis ablation on the GPU: the key/value axis errors and the kernels' speed, as JSON lines.

Draws seeded keys, values and queries of a workload (the harness's input generator lives beside
this script, outside the library package), then runs the library's axis-ablation harness
(bit_asymmetric_kv_kvq_gb300.ablation): score and output error of the four key/value axis choices
at 2, 3 and 4 bits, and the time of each ablation kernel at 2 bits.
"""
import argparse
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    import torch

    import synth
    from bit_asymmetric_kv_kvq_gb300 import ablation

    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", type=int, default=1, help="index into synth.WORKLOADS")
    ap.add_argument("--units", type=int, default=32, help="(sequence, kv head) units")
    ap.add_argument("--tokens", type=int, default=4096, help="tokens per unit")
    ap.add_argument("--group", type=int, default=32, help="group size G")
    args = ap.parse_args(argv)
    w = synth.WORKLOADS[args.workload]
    w = w.scaled(batch=1, kv_heads=args.units, q_heads=args.units * w.group_q, prefill_tokens=args.tokens,
                 decode_steps=1)
    dev = torch.device("cuda:0")
    K = torch.from_numpy(np.ascontiguousarray(synth.keys(w)[0, :, :args.tokens])).to(dev)
    V = torch.from_numpy(np.ascontiguousarray(synth.values(w)[0, :, :args.tokens])).to(dev)
    Q = torch.from_numpy(np.ascontiguousarray(synth.queries(w, 0)[0].reshape(args.units, w.group_q, -1))).to(dev)
    for bits in (2, 3, 4):
        for (ka, va), e in ablation.axis_errors(K, V, Q, bits, args.group, w.softmax_scale).items():
            print(json.dumps({"bits": bits, "group": args.group, "key_axis": ka, "value_axis": va,
                              **{k: round(v, 6) for k, v in e.items()}}))
    for name, r in ablation.time_kernels(K, V, Q, 2, args.group, w.softmax_scale).items():
        print(json.dumps({"kernel": name, "us": round(r["s"] * 1e6, 2), "bytes": r["bytes"],
                          "GBps": round(r["GBps"], 1)}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
