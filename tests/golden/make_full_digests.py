"""Write tests/golden/full_digests.json: the oracle's results on the full-size
workloads, as digests the GPU tests compare against.

Calls only ``oracle/`` and the seeded generators of
``exl3_trellis_weight_gb300.inputs``; nothing here touches the CUDA path.
For each matrix it stores the digests of the input bytes (W, su, sv), of the
rotated matrix R and of the reconstruction W-hat, sigma_R, the scale, the MSE
(the evaluation chain of the page "EXL3 Intel Arc Quantizer", Core items 7, 1,
5 and 10), and per 128-row band the digests of the packed codes and of the
fp32 tile costs.  For the golden-section workload (page "alpha2beta/JEV-9B-EXL3-K2",
section 2) it runs the oracle's 12-evaluation search over g in [0.5, 2] and
stores every evaluation the same way, plus the search's choice.

Workloads: 4096x4096 bf16 K=2 with 0.1 % outliers (g = 1); the golden-section
search on 4096x4096 bf16 K=2; 12288x4096 bf16 Student-t K=4 (g = 1); the seven
projections of the 4096/12288 decoder layer at K=3 (g = 1).  About 1.8 M tile
encodes in all: hours of CPU time.  The file is rewritten after each matrix,
and a rerun skips what is already stored (--force recomputes).

    python tests/golden/make_full_digests.py [--only NAME ...] [--threads N] [--force]
"""
from __future__ import annotations

import argparse
import os
import platform
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import oracle  # noqa: E402
from exl3_trellis_weight_gb300 import inputs  # noqa: E402
import digests as D  # noqa: E402

ORDER = ["linear4096_k2", "gss4096_k2", "mlp12288_t5_k4",
         "layer4096_k3/q", "layer4096_k3/k", "layer4096_k3/v", "layer4096_k3/o",
         "layer4096_k3/gate", "layer4096_k3/up", "layer4096_k3/down"]


def _matrix(key):
    name, _, proj = key.partition("/")
    for lab, W, su, sv, K in inputs.workload(name):
        if not proj or lab == proj:
            return W, su, sv, K
    raise KeyError(key)


def _evaluate(W, su, sv, K, g, threads):
    Wf = W.float().numpy()
    r = oracle.evaluate_matrix(Wf, su.numpy(), sv.numpy(), K, g, threads=threads)
    rows, cols = Wf.shape
    return {
        "g": D.fhex(g), "sigma": D.fhex(r["sigma"]), "scale": D.fhex(r["scale"]),
        "mse": D.fhex(r["mse"]), "R": D.sha(r["R"]), "What": D.sha(r["What"]),
        "bands": D.band_digests(r["codes"], r["costs"], rows, cols, K),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--only", nargs="*", default=None)
    ap.add_argument("--threads", type=int, default=None)
    ap.add_argument("--force", action="store_true")
    a = ap.parse_args()
    store = D.load()
    store.setdefault("_about", {})
    store["_about"].update({
        "generated_by": "python tests/golden/make_full_digests.py",
        "host": f"{platform.machine()} {platform.python_version()} numpy {np.__version__}",
        "band_rows": D.BAND_ROWS,
    })
    for key in ORDER:
        if a.only and key not in a.only and key.split("/")[0] not in a.only:
            continue
        if key in store and not a.force:
            print(f"{key}: stored, skipped", flush=True)
            continue
        t0 = time.time()
        W, su, sv, K = _matrix(key)
        rows, cols = W.shape
        entry = {"rows": rows, "cols": cols, "K": K, "inputs": D.input_digests(W, su, sv)}
        if key == "gss4096_k2":
            evals = []

            def f(g):
                e = _evaluate(W, su, sv, K, g, a.threads)
                evals.append(e)
                print(f"  {key} eval {len(evals)}: g={g:.9f} mse={D.unhex(e['mse']):.9e} "
                      f"({time.time() - t0:.0f} s)", flush=True)
                return D.unhex(e["mse"])

            best_g, best_f, hist = oracle.golden_section_search(f, 0.5, 2.0, 12)
            entry.update({"lo": D.fhex(0.5), "hi": D.fhex(2.0), "n_eval": 12,
                          "best_g": D.fhex(best_g), "best_mse": D.fhex(best_f), "evals": evals})
        else:
            entry.update(_evaluate(W, su, sv, K, 1.0, a.threads))
        entry["oracle_seconds"] = round(time.time() - t0, 1)
        store[key] = entry
        D.save(store)
        print(f"{key}: done in {time.time() - t0:.0f} s", flush=True)


if __name__ == "__main__":
    main()
