"""Write tests/golden/<workload>_inputs.json for every workload.

Two facts about the synthetic inputs cannot be drawn blindly and are computed
here with the CPU oracle (and nothing else):

* ``bias`` (skew workload only): a per-expert router bias fitted so that the
  oracle's per-expert counts follow the Zipf(1.2) targets of
  ``gen.zipf_target_counts`` -- 200 rounds of b_e += 0.5 (ln c_e - ln(n_e + 0.5))
  on the fp64 base logits, top-k by the oracle.
* ``retry``: per-token redraw counters.  Every token whose k-th and (k+1)-th
  oracle logits are within 1e-3 of each other has its x row redrawn (its
  stream shifted by one) until no such token is left, so the selected expert
  set cannot depend on the summation order of an fp32 versus an fp64 router.

Also recorded, for reference only: the oracle's per-expert counts and the
smallest routing margin.  Usage: python tests/golden/make_inputs_meta.py [names]
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import gen  # noqa: E402
import oracle  # noqa: E402

MARGIN = 1e-3


def fit_zipf_bias(w, x, wr, rounds=200):
    target = gen.zipf_target_counts(w)
    L0 = oracle.router_logits(x, wr, None)
    b = np.zeros(w.E, dtype=np.float32)
    for _ in range(rounds):
        idx = oracle.topk(L0 + b.astype(np.float64), w.k)[0]
        n = np.bincount(idx.ravel(), minlength=w.E).astype(np.float64)
        b = (b.astype(np.float64) + 0.5 * (np.log(target) - np.log(n + 0.5))).astype(np.float32)
    return b


def enforce_margin(w, wr, bias):
    retry = np.zeros(w.T, dtype=np.int32)
    x = gen.x_rows(w.T, w.d, retry)
    gap = oracle.route(x, wr, bias, w.k)["gap"]
    rounds = 0
    while True:
        bad = np.nonzero(gap <= MARGIN)[0]
        if bad.size == 0:
            break
        rounds += 1
        assert rounds < 64, "margin enforcement does not converge"
        retry[bad] += 1
        x = gen.x_rows(w.T, w.d, retry)
        gap[bad] = oracle.route(x[bad], wr, bias, w.k)["gap"]
    return retry, x, gap


def make(name):
    w = gen.WORKLOADS[name]
    wr = gen.router_w(w)
    meta = {"workload": name, "shape": w.describe()}
    if w.bias and w.bias[0] == "zipf":
        x0 = gen.x_rows(w.T, w.d)
        bias = fit_zipf_bias(w, x0, wr)
        meta["bias"] = [float(v) for v in bias]
        meta["zipf_target"] = [round(float(c), 3) for c in gen.zipf_target_counts(w)]
    bias = gen.router_bias(w, meta=meta)
    retry, x, gap = enforce_margin(w, wr, bias)
    meta["retry"] = {str(int(t)): int(retry[t]) for t in np.nonzero(retry)[0]}
    r = oracle.route(x, wr, bias, w.k)
    counts = np.bincount(r["idx"].ravel(), minlength=w.E)
    meta["oracle_counts"] = [int(c) for c in counts]
    meta["min_margin"] = float(r["gap"].min()) if w.k < w.E else None
    with open(os.path.join(HERE, f"{name}_inputs.json"), "w") as fh:
        json.dump(meta, fh, indent=1)
        fh.write("\n")
    print(name, "redrawn rows:", len(meta["retry"]), "min margin:", meta["min_margin"],
          "max count:", counts.max(), "min count:", counts.min())


if __name__ == "__main__":
    names = sys.argv[1:] or list(gen.WORKLOADS)
    for n in names:
        make(n)
