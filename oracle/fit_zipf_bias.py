"""Fit the per-expert popularity offsets of the Zipf(1.1) workloads.

Writes ``synth/data/zipf_bias_<workload>.txt`` (one FP32 value per expert, added
to the selection bias).  Uses only the oracle's router (test infrastructure)
and the seeded generators; run once, output committed:

    python -m oracle.fit_zipf_bias

Procedure: a calibration batch of 16,384 hidden rows (own seed) is routed with
bias b + o; each of 80 iterations moves o_e by eta_i times the log-ratio between
the target pick rate f_e = min(1, c * rank_e^-s) (sum f = K) and the observed
rate, eta_i = 0.08 * 0.96^i (the sigmoid scores spread over about 0.2, so a
bias step much larger than that overshoots).
The router matrix and base bias are the workload's own, so the offsets carry
over to every token count of that workload.
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

if __package__ in (None, ""):
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from oracle import moe_oracle as O  # noqa: E402
from synth import WORKLOADS, make_calibration_x, router_params, zipf_targets  # noqa: E402


def fit(name: str, n_cal: int = 16384, iters: int = 80) -> np.ndarray:
    shape = WORKLOADS[name]
    rp = router_params(shape, with_popularity=False)
    x = make_calibration_x(shape, n_cal).float().numpy().astype(np.float64)
    z, _ = O.router_logits(x, rp["w_router"].numpy())
    s = O.sigmoid_scores(z.astype(np.float32))
    b = rp["bias"].numpy().astype(np.float32)
    E, K = shape.n_experts, shape.top_k
    target = zipf_targets(E, K, shape.zipf_s, shape.weight_seed)
    o = np.zeros(E, dtype=np.float32)
    for it in range(iters):
        bias = (b + o).astype(np.float32)
        ids = O.select_batch(s, bias, shape.n_group, shape.topk_group, K)
        counts = np.bincount(ids.reshape(-1), minlength=E).astype(np.float64)
        f_obs = np.clip(counts / n_cal, 0.5 / n_cal, 1.0)
        eta = 0.08 * 0.96 ** it
        o = (o + eta * (np.log(target) - np.log(f_obs))).astype(np.float32)
        err = np.abs(f_obs - target).max()
        rel = np.abs(np.log(f_obs / target)).max()
        print(f"{name} iter {it:2d}: max |f_obs - f_target| = {err:.4f}  max |log ratio| = {rel:.3f}", flush=True)
    return o


def main():
    out_dir = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "synth", "data")
    os.makedirs(out_dir, exist_ok=True)
    for name in ("nano_prefill", "super_nvfp4"):
        t0 = time.time()
        o = fit(name)
        np.savetxt(os.path.join(out_dir, f"zipf_bias_{name}.txt"), o.astype(np.float64), fmt="%.9g")
        print(f"{name}: written in {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main()
